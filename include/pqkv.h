/*
 * pqkv.h -- C-ABI of libpqkv: quantize-and-append into a paged KV cache and
 * paged decode / speculative-verify attention over it, on one GB300 (sm_103a).
 *
 * The operations follow the KV design on the ReVolta README (pages
 * "ReVolta" README and "v0.1.3" release note):
 *   - "Weight and KV formats": the KV cache is stored compressed as FP8 E4M3
 *     (calibrated per-layer K and V scales, "E4M3 KV"), INT8 ("INT8 KV") or
 *     FP16, and widened to FP16 for the arithmetic;
 *   - "Quick start", launch: MTP verify with 4 speculative tokens, i.e. one
 *     committed and four draft query positions per sequence, causally masked
 *     among themselves; GQA through the model's query / KV head counts;
 *   - "Hardware" and "Quick start": decode context parallelism splits a
 *     sequence's keys across GPUs and combines the partial results; here the
 *     split is across thread blocks of one GPU and the partials are merged by
 *     log-sum-exp;
 *   - release note "Known issues": 16-token kernel pages.
 *
 * Pool layout (this library's choice):
 *   pages[num_pages][num_kv_heads][2][page_size][head_dim]
 * where index 0 of the third axis is K and 1 is V; elements are 1-byte codes
 * (E4M3, INT8) or fp16.  Slot s of the pool is token s % page_size of page
 * s / page_size.  For one (page, kv-head) the K tile and the V tile are
 * contiguous (4 KB for 8-bit codes), which is what the attention kernel
 * streams.
 * PQKV_KV_INT8_ROW pools carry a scale area right after the codes, in the same
 * allocation (num_pages*num_kv_heads*4096 bytes from the start of `pages`):
 *   fp16 row_scale[num_pages][num_kv_heads][8][4]
 * (IEEE binary16), where [p][h][i] holds the scales of K row i, K row i+8,
 * V row i and V row i+8 of page p, kv-head h -- the order in which the
 * attention kernel's matrix fragments consume them.  That is 64 bytes per
 * (page, kv-head); the allocation is num_pages*num_kv_heads*4160 bytes.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers owned by the caller.  Nothing
 *     is allocated, freed or retained.  Between calls the library keeps only
 *     a per-device cache of device properties, and -- the one exception --
 *     the scratch area of pqkv_paged_attention_noalloc (a file-scope device
 *     array present on every GPU that loads the library, its per-device
 *     address cache and the last call's contents; see that entry point).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream), in stream order.  Most kernels are launched with
 *     programmatic dependent launch allowed: their blocks may become resident
 *     while the previous kernel on the stream finishes, but they wait for it
 *     to complete (and its writes to be visible) before touching memory, so
 *     the ordering is that of a plain launch.  The return value reports
 *     argument validation and launch errors only.
 *   - Errors that only the device can see are OR-ed as PQKV_DEV_* bits into
 *     `*status` (a device int32, may be NULL).  The offending work is skipped;
 *     no kernel traps, asserts or waits without a bound.
 */
#ifndef PQKV_H
#define PQKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* KV element formats. */
typedef enum {
  PQKV_KV_FP16 = 0,     /* fp16 values, scales ignored                          */
  PQKV_KV_FP8_E4M3 = 1, /* OCP E4M3 ("FN": max 448, no Inf), value = dec(c)*scale */
  PQKV_KV_INT8 = 2,     /* symmetric int8 in [-127, 127], value = c*scale         */
  PQKV_KV_INT8_ROW = 3  /* int8 with its own scale per (token, kv-head) row of K
                           and of V, computed when the row is written (ReVolta
                           README, "Weight and KV formats", "INT8 KV": scales
                           derived from the data at run time, no calibration);
                           value = c * row_scale.  Scale area: see the layout. */
} pqkv_kv_dtype;

/* Host-side return codes. */
enum {
  PQKV_OK = 0,
  PQKV_EINVAL = -1,       /* null pointer, bad size, misaligned pointer         */
  PQKV_EUNSUPPORTED = -2, /* valid but not implemented (head_dim != 128, ...)   */
  PQKV_ERANGE = -3,       /* a size is outside the supported range              */
  PQKV_EWORKSPACE = -4,   /* workspace missing or smaller than required         */
  PQKV_ECUDA = -5         /* a CUDA runtime call or a launch failed             */
};

/* Device-side status bits (OR-ed into *status). */
enum {
  PQKV_DEV_SLOT_RANGE = 1,    /* append: slot >= num_pages*page_size; token skipped */
  PQKV_DEV_SEQ_RANGE = 2,     /* attention: seq_len < q_len or beyond its block-table row */
  PQKV_DEV_BAD_SCALE = 4,     /* a scale is not finite and > 0; work skipped        */
  PQKV_DEV_TIMEOUT = 8,       /* a pipeline wait ran out (about 1 s); outputs invalid */
  PQKV_DEV_PAGE_RANGE = 16    /* attention: block-table entry outside [0, num_pages); read as zeros */
};

/* Largest supported sizes. */
#define PQKV_HEAD_DIM 128
#define PQKV_PAGE_SIZE 16
#define PQKV_MAX_Q_LEN 8
#define PQKV_MAX_ROWS 32          /* (num_q_heads / num_kv_heads) * q_len        */
#define PQKV_MAX_SEQS 2048
#define PQKV_MAX_SPLITS 128
#define PQKV_MAX_SEQ_LEN 524288   /* ReVolta README, "Performance": 512K boundary */

/*
 * pqkv_kv_append_quant -- quantize new K and V tokens and write them into
 * their pool slots.  (ReVolta README, "Weight and KV formats": KV is stored
 * compressed; E4M3 uses calibrated per-layer scales, INT8 a scale per head.)
 *
 * For every token t with slot_mapping[t] >= 0, kv-head h and dim d:
 *     pages[slot/ps][h][0][slot%ps][d] = Q(fp32(k[t,h,d]) / fp32(k_scale[h']))
 *     pages[slot/ps][h][1][slot%ps][d] = Q(fp32(v[t,h,d]) / fp32(v_scale[h']))
 * where the quotient is the correctly rounded IEEE binary32 division, h' = h
 * if scale_per_head else 0, and Q is
 *     E4M3: round to nearest, ties to even, saturate to +-448 (Inf -> +-448,
 *           NaN -> 0x7F), zero keeps its sign;
 *     INT8: round half to even, clamp to [-127, 127] (NaN -> 0);
 *     FP16: the fp16 bits unchanged (scales ignored, may be NULL).
 * INT8_ROW: for each written (token, kv-head) row x of K (and of V) the row's
 * scale r = fp16(amax / 127), the binary16 value nearest the exact quotient
 * (ties to even), amax = the largest |x_d| of the row (NaNs ignored; 0 for a
 * row of zeros), is stored in the scale area at the row's slot and the codes
 * are the INT8 codes of fp32(x_d) / fp32(r).  A zero r (amax <= 127 * 2^-25)
 * gives 0/0 = NaN -> code 0 and +-x/0 -> +-127, all worth 0.  k_scale /
 * v_scale are ignored (may be NULL).  V rows with amax above 32512 exceed what the attention kernel's
 * fp16 products hold (probability <= 256 times the row scale).
 *
 *   k, v            fp16 [num_tokens][num_kv_heads][head_dim]; heads and dims
 *                   contiguous, tokens `k_token_stride` / `v_token_stride`
 *                   ELEMENTS apart (>= num_kv_heads*head_dim), so K and V may
 *                   be column slices of a fused QKV buffer.
 *   slot_mapping    int64 [num_tokens]; negative = skip the token (padding).
 *                   Two tokens with the same slot: the result is unspecified.
 *   k_scale/v_scale fp32 [1] or [num_kv_heads] (device).
 *   pages           the pool (layout above); num_pages pages.
 * Requires head_dim == 128, page_size == 16, all pointers 16-byte aligned and
 * token strides multiples of 8 elements.  num_tokens == 0 is a no-op.
 */
int pqkv_kv_append_quant(const void* k, int64_t k_token_stride, const void* v,
                         int64_t v_token_stride, const int64_t* slot_mapping,
                         int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                         int32_t kv_dtype, const float* k_scale, const float* v_scale,
                         int32_t scale_per_head, void* pages, int64_t num_pages,
                         int32_t page_size, int32_t* status, void* stream);

/*
 * pqkv_paged_attention_workspace_size -- bytes of device workspace that
 * pqkv_paged_attention needs for these sizes and split mode (0 if none).
 * num_splits as in pqkv_paged_attention.  Pure host function; it queries the
 * current device's SM count.  The first PQKV_COUNTER_BYTES(num_seqs,
 * num_kv_heads) bytes of the workspace are merge counters: they must be zero
 * before the first call, and every call that returns with *status clean
 * leaves them zero again.  Zero the whole workspace once after allocating it
 * (and again after a call that reported PQKV_DEV_TIMEOUT).
 */
size_t pqkv_paged_attention_workspace_size(int32_t num_seqs, int32_t q_len,
                                           int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t num_splits);

/*
 * pqkv_paged_attention -- decode (q_len == 1) or verify (q_len > 1)
 * attention of each sequence's new query positions over its paged,
 * quantized K/V, with GQA and split-KV partitions merged by log-sum-exp.
 * (ReVolta README, "Quick start": MTP4 verify and the FLASH_ATTN_V100
 * backend; "Weight and KV formats": K/V dequantized for compute; "Hardware":
 * decode context parallel split of the keys.)
 *
 * For sequence s with L = seq_lens[s] cached tokens (its q_len new tokens
 * already appended), query i < q_len sits at position p = L - q_len + i and
 * attends to tokens j <= p.  Query head hq reads kv-head
 * hq / (num_q_heads / num_kv_heads).  With K_j = dec(kcode_j) * k_scale and
 * V_j = dec(vcode_j) * v_scale:
 *     out[s*q_len + i][hq][:] = sum_j softmax_j(q . K_j / sqrt(head_dim)) V_j
 * computed in fp32 with fp16 tensor-core products, and rounded to fp16.
 *
 *   q, out            fp16 [num_seqs*q_len][num_q_heads][head_dim], contiguous.
 *   pages             the pool (layout above), num_pages pages, 16-byte aligned.
 *   block_table       int32 [num_seqs][max_pages_per_seq]: the pool page of
 *                     each logical 16-token page of the sequence.
 *   seq_lens          int32 [num_seqs] (device), q_len <= L <= max_pages_per_seq*16.
 *   k_scale, v_scale  fp32 [1] or [num_kv_heads] (device); ignored for FP16
 *                     and INT8_ROW (whose K_j, V_j use the row scales stored
 *                     at token j's slot).
 *   num_splits        0: balanced split -- the key pages of all sequences and
 *                     kv-heads are cut into one equal contiguous share per
 *                     resident thread block, and a sequence's shares are
 *                     merged by log-sum-exp;  k >= 1: every (sequence, kv-head)
 *                     is cut into k near-equal partitions (k == 1: no merge).
 *   max_seq_len       an upper bound of seq_lens used to size the balanced
 *                     grid (0: max_pages_per_seq*16).
 *   workspace         device scratch of pqkv_paged_attention_workspace_size()
 *                     bytes (may be NULL when that size is 0), 256-byte
 *                     aligned; see the counter rule above.  Calls that share a
 *                     workspace must not overlap on the device.
 * Requires head_dim == 128, page_size == 16, 1 <= q_len <= 8,
 * (num_q_heads/num_kv_heads)*q_len <= 32, num_seqs <= 2048.
 * The result does not depend on the order of pages in the pool; for a fixed
 * split mode and device it is bitwise reproducible run to run.
 */
int pqkv_paged_attention(const void* q, void* out, const void* pages, int64_t num_pages,
                         const int32_t* block_table, int32_t max_pages_per_seq,
                         const int32_t* seq_lens, int32_t num_seqs, int32_t q_len,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t page_size, int32_t kv_dtype, const float* k_scale,
                         const float* v_scale, int32_t scale_per_head, int32_t num_splits,
                         int32_t max_seq_len, void* workspace, size_t workspace_bytes,
                         int32_t* status, void* stream);

/*
 * pqkv_paged_attention_window -- pqkv_paged_attention with a sliding window:
 * query position p attends to the `window` most recent keys, itself included,
 * i.e. keys j with p - window < j <= p.  (ReVolta README, "DFlash2
 * speculative decoding": the drafter's sliding-window layers use a 2048-token
 * window.)  Pages that lie wholly before every query's window are not read, so
 * the cost follows the window, not the cache length.
 *
 * Same arguments as pqkv_paged_attention, plus:
 *   window   >= 1: the window in tokens; 0: no window (exactly
 *            pqkv_paged_attention); negative: PQKV_EINVAL.
 * The workspace rules are those of pqkv_paged_attention (its size query
 * covers this call).
 */
int pqkv_paged_attention_window(const void* q, void* out, const void* pages, int64_t num_pages,
                                const int32_t* block_table, int32_t max_pages_per_seq,
                                const int32_t* seq_lens, int32_t num_seqs, int32_t q_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t page_size, int32_t kv_dtype, const float* k_scale,
                                const float* v_scale, int32_t scale_per_head, int32_t num_splits,
                                int32_t max_seq_len, int32_t window, void* workspace,
                                size_t workspace_bytes, int32_t* status, void* stream);

/*
 * pqkv_paged_attention_partial -- one rank's part of a decode context
 * parallel split (ReVolta README, "Hardware": TP4 + DCP2; "Quick start",
 * launch: --decode-context-parallel-size 2): each rank holds a contiguous,
 * page-aligned share of every sequence's keys, attends over it, and the ranks'
 * results are combined by pqkv_lse_merge (after an all-gather across ranks).
 *
 * Same arguments as pqkv_paged_attention, except:
 *   seq_lens   int32 [num_seqs]: keys of each sequence held here (0 allowed);
 *   q_pos      int32 [num_seqs] (device): local index of query 0's position,
 *              i.e. its global position minus the global index of this
 *              share's first key; query i sees local keys j <= q_pos + i
 *              (any value: negative hides every key from the row);
 *   out_o      fp32 [num_seqs*q_len][num_q_heads][head_dim]: O / l of the
 *              share (0 for a row that sees no key);
 *   out_lse    fp32 [num_seqs*q_len][num_q_heads]: m + ln(l), the natural-log
 *              log-sum-exp of the row's scores over the share (-inf when the
 *              row sees no key).
 * Scores are q . K_j / sqrt(head_dim) as in pqkv_paged_attention.  out_o must
 * be 16-byte aligned.
 */
int pqkv_paged_attention_partial(const void* q, const void* pages, int64_t num_pages,
                                 const int32_t* block_table, int32_t max_pages_per_seq,
                                 const int32_t* seq_lens, const int32_t* q_pos, int32_t num_seqs,
                                 int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t page_size, int32_t kv_dtype,
                                 const float* k_scale, const float* v_scale,
                                 int32_t scale_per_head, int32_t num_splits, int32_t max_seq_len,
                                 float* out_o, float* out_lse, void* workspace,
                                 size_t workspace_bytes, int32_t* status, void* stream);

/*
 * pqkv_lse_merge -- combine partial results of the same rows (the merge step
 * of the split above): with parts p = 0 .. num_parts-1,
 *     LSE = ln sum_p e^{lse_p},   out = sum_p e^{lse_p - LSE} o_p   (fp16)
 * Parts with lse_p = -inf contribute nothing; a row with no finite lse_p
 * gets out = 0 and LSE = -inf.
 *   part_o    fp32 [num_parts][num_rows][head_dim], 16-byte aligned;
 *   part_lse  fp32 [num_parts][num_rows];
 *   out       fp16 [num_rows][head_dim], 16-byte aligned;
 *   out_lse   fp32 [num_rows] or NULL (for a further merge level).
 * num_rows = num_seqs*q_len*num_q_heads for pqkv_paged_attention_partial's
 * outputs.  Requires head_dim == 128.
 */
int pqkv_lse_merge(const float* part_o, const float* part_lse, int32_t num_parts,
                   int64_t num_rows, int32_t head_dim, void* out, float* out_lse, void* stream);

/* Size of the library-owned scratch area used by pqkv_paged_attention_noalloc
 * (16 MiB, held on every GPU that loads the library until the process exits). */
#define PQKV_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * pqkv_paged_attention_noalloc -- pqkv_paged_attention for callers that cannot
 * allocate device memory.  (No counterpart on the ReVolta pages: an addition of
 * this library for callers such as runtimes that budget all device memory up
 * front and forbid cudaMalloc at call time, hooks running inside another
 * framework's step that must not bypass its allocator, or C callers with no
 * allocator at all.)
 *
 * Same arguments and result as pqkv_paged_attention without the workspace:
 * the library uses its own fixed scratch area of PQKV_NOALLOC_SCRATCH_BYTES, a
 * file-scope device array.  Nothing is allocated or freed, by the library or by
 * any routine it calls.
 *   - Returns PQKV_ERANGE when the workspace of the launch this call makes
 *     exceeds PQKV_NOALLOC_SCRATCH_BYTES.  That is the grid the call actually
 *     uses, not the largest one pqkv_paged_attention_workspace_size() assumes:
 *     with RP = (num_q_heads/num_kv_heads)*q_len rounded up to a multiple of
 *     8, it needs PQKV_COUNTER_BYTES(num_seqs, num_kv_heads) plus about
 *     n*RP*520 bytes, where n = num_seqs*num_kv_heads*num_splits for
 *     num_splits >= 2, and n = num_seqs*num_kv_heads + G for num_splits == 0,
 *     G the balanced grid (at most the blocks resident on the device at once:
 *     one per SM in this build); num_splits == 1 needs none.
 *   - All arguments are checked before anything is queued: a rejected call
 *     leaves the scratch area untouched.
 *   - The first call on a device that needs scratch looks up the array's
 *     device address (cudaGetSymbolAddress) with that device current; make
 *     that first call before any stream capture begins.
 *   - Every call on a device shares the one scratch area and it keeps the last
 *     call's contents; each call clears the part that must start at zero
 *     (cudaMemsetAsync on `stream`, queued just before the kernel).  Calls that
 *     overlap on the GPU (different streams, or concurrent host threads) race
 *     on it and must be serialised by the caller.
 */
int pqkv_paged_attention_noalloc(const void* q, void* out, const void* pages, int64_t num_pages,
                                 const int32_t* block_table, int32_t max_pages_per_seq,
                                 const int32_t* seq_lens, int32_t num_seqs, int32_t q_len,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t page_size, int32_t kv_dtype, const float* k_scale,
                                 const float* v_scale, int32_t scale_per_head, int32_t num_splits,
                                 int32_t max_seq_len, int32_t* status, void* stream);

/* Bytes at the start of the workspace that hold merge counters. */
#define PQKV_COUNTER_BYTES(num_seqs, num_kv_heads) \
  ((((size_t)(num_seqs) * (size_t)(num_kv_heads) * 4u) + 255u) & ~(size_t)255u)

/* Static description of a return code, or of a device status word holding any
 * combination of OR-ed PQKV_DEV_* bits ("device: a; b"); "unknown status" for
 * anything else.  The returned string lives until the process exits. */
const char* pqkv_status_string(int code);

/* Library version as "major.minor.patch". */
const char* pqkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PQKV_H */
