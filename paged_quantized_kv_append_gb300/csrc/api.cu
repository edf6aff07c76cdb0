// C-ABI entry points of libpqkv (declared in include/pqkv.h): argument
// validation, TMA tensor-map encoding, grid sizing and workspace carve-up.
// Everything the device computes happens in append.cu / attention_*.cu.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "pqkv_internal.h"

namespace pqkv {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGrid = 1024;           // upper bound of the balanced grid
constexpr int kMinPagesPerBlock = 8;     // smallest balanced share worth a block
// 8-row decodes of 8-bit pools with at most this many (page, kv-head) units
// per SM run as two 8-warp blocks per SM (one 16-warp block otherwise):
// short contexts gain from the two blocks' unsynchronised start-up and
// fragment ends, long ones stream faster with one block.
constexpr int64_t kPairMaxUnitsPerSm = 1024;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PQKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev[dev].ready) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return PQKV_ECUDA;
    g_dev[dev].sms = n;
    g_dev[dev].ready = true;
  }
  *sms = g_dev[dev].sms;
  return PQKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int kv_dtype) { return kv_dtype == PQKV_KV_FP16 ? 2 : 1; }

// formats whose k_scale / v_scale arguments are read
bool uses_scale_args(int kv_dtype) {
  return kv_dtype == PQKV_KV_FP8_E4M3 || kv_dtype == PQKV_KV_INT8;
}

// INT8_ROW: the row scales follow the codes in the pool allocation
uint16_t* row_scale_area(void* pages, int64_t num_pages, int32_t num_kv_heads) {
  return reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(pages) +
                                  num_pages * num_kv_heads * 2 * kPageSize * kHeadDim);
}

int blocks_per_sm(int kv_dtype, int nt, bool pair, int num_seqs) {
  switch (kv_dtype) {
    case PQKV_KV_FP16: return attention_blocks_per_sm_fp16(nt, pair, num_seqs);
    case PQKV_KV_FP8_E4M3: return attention_blocks_per_sm_e4m3(nt, pair, num_seqs);
    case PQKV_KV_INT8: return attention_blocks_per_sm_int8(nt, pair, num_seqs);
    case PQKV_KV_INT8_ROW: return attention_blocks_per_sm_int8_row(nt, pair, num_seqs);
  }
  return 0;
}

int plan_attention(int32_t num_seqs, int32_t q_len, int32_t hq, int32_t hkv, int32_t num_splits,
                   int grid, AttnPlan* pl) {
  pl->rows = (hq / hkv) * q_len;
  pl->rp = rows_padded(pl->rows);
  pl->nt = pl->rp / 8;
  const int64_t segs = (int64_t)num_seqs * hkv;
  if (num_splits == 1) {
    pl->slots = 0;
  } else if (num_splits > 1) {
    pl->slots = segs * num_splits;             // slot = block index
  } else {
    pl->slots = segs + grid;                   // slot = segment + block index
  }
  if (pl->slots == 0) {
    pl->total = 0;
    return PQKV_OK;
  }
  pl->counter_bytes = PQKV_COUNTER_BYTES(num_seqs, hkv);
  pl->o_bytes = (size_t)pl->slots * pl->rp * kHeadDim * 4;
  pl->ml_bytes = (size_t)pl->slots * 2 * pl->rp * 4;
  pl->total = pl->counter_bytes + ((pl->o_bytes + 255) & ~size_t(255)) + pl->ml_bytes;
  return PQKV_OK;
}

int validate_common(int32_t head_dim, int32_t page_size, int32_t kv_dtype) {
  if (kv_dtype < PQKV_KV_FP16 || kv_dtype > PQKV_KV_INT8_ROW) return PQKV_EINVAL;
  if (head_dim != kHeadDim || page_size != kPageSize) return PQKV_EUNSUPPORTED;
  return PQKV_OK;
}

int validate_heads(int32_t num_seqs, int32_t q_len, int32_t hq, int32_t hkv) {
  if (num_seqs < 0 || q_len < 1 || hq < 1 || hkv < 1) return PQKV_EINVAL;
  if (hq % hkv != 0) return PQKV_EINVAL;
  if (num_seqs > PQKV_MAX_SEQS || q_len > PQKV_MAX_Q_LEN) return PQKV_ERANGE;
  if ((hq / hkv) * q_len > PQKV_MAX_ROWS) return PQKV_EUNSUPPORTED;
  return PQKV_OK;
}

}  // namespace
}  // namespace pqkv

using namespace pqkv;

extern "C" int pqkv_kv_append_quant(const void* k, int64_t k_token_stride, const void* v,
                                    int64_t v_token_stride, const int64_t* slot_mapping,
                                    int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t kv_dtype, const float* k_scale, const float* v_scale,
                                    int32_t scale_per_head, void* pages, int64_t num_pages,
                                    int32_t page_size, int32_t* status, void* stream) {
  int rc = validate_common(head_dim, page_size, kv_dtype);
  if (rc) return rc;
  if (num_tokens < 0 || num_kv_heads < 1 || num_pages < 0) return PQKV_EINVAL;
  if (num_tokens == 0) return PQKV_OK;
  if (!k || !v || !slot_mapping || !pages) return PQKV_EINVAL;
  if (uses_scale_args(kv_dtype) && (!k_scale || !v_scale)) return PQKV_EINVAL;
  if (k_token_stride < (int64_t)num_kv_heads * head_dim ||
      v_token_stride < (int64_t)num_kv_heads * head_dim)
    return PQKV_EINVAL;
  if (k_token_stride % 8 || v_token_stride % 8) return PQKV_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(pages, 16) || !aligned(slot_mapping, 8))
    return PQKV_EINVAL;
  int sms = 0;
  rc = current_device_sms(&sms);
  if (rc) return rc;
  AppendParams p;
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.k_stride = k_token_stride;
  p.v_stride = v_token_stride;
  p.slots = slot_mapping;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.scale_per_head = scale_per_head ? 1 : 0;
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.pages = static_cast<uint8_t*>(pages);
  p.num_pages = num_pages;
  p.row_scales = kv_dtype == PQKV_KV_INT8_ROW ? row_scale_area(pages, num_pages, num_kv_heads)
                                              : nullptr;
  p.status = status;
  // one pass when the chunk fits the resident blocks, grid-stride beyond
  // that: at most one wave of the blocks that fit on every SM at once
  const int per_sm = append_blocks_per_sm(kv_dtype);
  if (per_sm < 1) return PQKV_ECUDA;
  const int64_t work = (int64_t)num_tokens * num_kv_heads * (kHeadDim / 16);
  const int64_t per_block = (int64_t)kAppendThreads * kAppendUnroll;
  const int64_t blocks = (work + per_block - 1) / per_block;
  const int grid = (int)std::min<int64_t>(blocks, (int64_t)sms * per_sm);
  if (launch_append(p, kv_dtype, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PQKV_ECUDA;
  return PQKV_OK;
}

extern "C" size_t pqkv_paged_attention_workspace_size(int32_t num_seqs, int32_t q_len,
                                                      int32_t num_q_heads, int32_t num_kv_heads,
                                                      int32_t head_dim, int32_t num_splits) {
  if (head_dim != kHeadDim) return 0;
  if (validate_heads(num_seqs, q_len, num_q_heads, num_kv_heads)) return 0;
  if (num_splits < 0 || num_splits > PQKV_MAX_SPLITS) return 0;
  AttnPlan pl;
  plan_attention(num_seqs, q_len, num_q_heads, num_kv_heads, num_splits, kMaxGrid, &pl);
  return pl.total;
}

namespace pqkv {

int plan_attention_launch(const AttnArgs& a, AttnLaunch* L) {
  int rc = validate_common(a.head_dim, a.page_size, a.kv_dtype);
  if (rc) return rc;
  rc = validate_heads(a.num_seqs, a.q_len, a.num_q_heads, a.num_kv_heads);
  if (rc) return rc;
  if (a.num_splits < 0 || a.num_splits > PQKV_MAX_SPLITS) return PQKV_ERANGE;
  if (a.num_seqs == 0) return PQKV_OK;
  if (!a.q || !a.pages || !a.block_table || !a.seq_lens) return PQKV_EINVAL;
  if (uses_scale_args(a.kv_dtype) && (!a.k_scale || !a.v_scale)) return PQKV_EINVAL;
  if (a.num_pages < 1 || a.num_pages > INT32_MAX || a.max_pages_per_seq < 1) return PQKV_EINVAL;
  if ((int64_t)a.max_pages_per_seq * a.page_size > PQKV_MAX_SEQ_LEN + a.page_size)
    return PQKV_ERANGE;
  if (a.max_seq_len < 0) return PQKV_EINVAL;
  if (!aligned(a.q, 16) || !aligned(a.pages, 16) || !aligned(a.block_table, 4) ||
      !aligned(a.seq_lens, 4))
    return PQKV_EINVAL;
  int sms = 0;
  rc = current_device_sms(&sms);
  if (rc) return rc;
  const int rows = (a.num_q_heads / a.num_kv_heads) * a.q_len;
  const int nt = rows_padded(rows) / 8;

  // grid
  int grid;
  bool pair = false;
  if (a.num_splits == 0) {
    const int64_t cap_len = (int64_t)a.max_pages_per_seq * a.page_size;
    int64_t lmax = a.max_seq_len > 0 ? std::min<int64_t>(a.max_seq_len, cap_len) : cap_len;
    // a sliding window reads at most window + q_len - 1 keys per sequence,
    // over one page more than they fill
    if (a.window > 0)
      lmax = std::min<int64_t>(lmax, (int64_t)a.window + a.q_len - 1 + a.page_size);
    const int64_t units =
        (int64_t)a.num_seqs * a.num_kv_heads * ((lmax + a.page_size - 1) / a.page_size);
    pair = nt == 1 && a.kv_dtype != PQKV_KV_FP16 && a.window == 0 &&
           units <= kPairMaxUnitsPerSm * sms;
    const int per_sm = blocks_per_sm(a.kv_dtype, nt, pair, a.num_seqs);
    if (per_sm <= 0) return PQKV_ECUDA;
    const int64_t want = (units + kMinPagesPerBlock - 1) / kMinPagesPerBlock;
    const int64_t cap = std::min<int64_t>((int64_t)sms * per_sm, (int64_t)kMaxGrid);
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, cap));
  } else {
    const int64_t g = (int64_t)a.num_seqs * a.num_kv_heads * a.num_splits;
    if (g > INT32_MAX) return PQKV_ERANGE;
    grid = (int)g;
  }
  plan_attention(a.num_seqs, a.q_len, a.num_q_heads, a.num_kv_heads, a.num_splits, grid, &L->pl);
  L->grid = grid;
  L->nt = nt;
  L->pair = pair;
  L->rows = rows;
  return PQKV_OK;
}

int bind_attention(const AttnArgs& a, const AttnLaunch& L, void* workspace,
                   size_t workspace_bytes, int32_t* status, AttnParams* pp, CUtensorMap* mapp) {
  const AttnPlan& pl = L.pl;
  if (pl.total > 0) {
    if (!workspace) return PQKV_EWORKSPACE;
    if (!aligned(workspace, 256) || workspace_bytes < pl.total) return PQKV_EWORKSPACE;
  }

  // TMA map over the pool: [num_pages][Hkv][lines][128 bytes]
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return PQKV_ECUDA;
  const int eb = elem_bytes(a.kv_dtype);
  const cuuint32_t lines = (cuuint32_t)(2 * a.page_size * a.head_dim * eb / 128);
  CUtensorMap& map = *mapp;
  std::memset(&map, 0, sizeof(map));
  const cuuint64_t dims[4] = {(cuuint64_t)(128 / eb), lines, (cuuint64_t)a.num_kv_heads,
                              (cuuint64_t)a.num_pages};
  const cuuint64_t strides[3] = {128, (cuuint64_t)lines * 128,
                                 (cuuint64_t)lines * 128 * a.num_kv_heads};
  const cuuint32_t box[4] = {(cuuint32_t)(128 / eb), lines, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult cr = enc(&map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                          4, const_cast<void*>(a.pages), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return PQKV_ECUDA;

  AttnParams& p = *pp;
  p.q = static_cast<const uint16_t*>(a.q);
  p.out = nullptr;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  // INT8_ROW reads no scale arguments: its k_scale slot carries the row-scale area
  p.k_scale = a.kv_dtype == PQKV_KV_INT8_ROW
                  ? reinterpret_cast<const float*>(
                        row_scale_area(const_cast<void*>(a.pages), a.num_pages, a.num_kv_heads))
                  : a.k_scale;
  p.v_scale = a.v_scale;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = pl.total ? reinterpret_cast<int32_t*>(ws) : nullptr;
  p.part_o = pl.total ? reinterpret_cast<float*>(ws + pl.counter_bytes) : nullptr;
  p.part_ml = pl.total ? reinterpret_cast<float*>(ws + pl.counter_bytes +
                                                  ((pl.o_bytes + 255) & ~size_t(255)))
                       : nullptr;
  p.status = status;
  p.num_pages = a.num_pages;
  p.bt_stride = a.max_pages_per_seq;
  p.num_seqs = a.num_seqs;
  p.q_len = a.q_len;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.rows = L.rows;
  p.scale_per_head = a.scale_per_head ? 1 : 0;
  p.num_splits = a.num_splits;
  p.sm_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a.head_dim));
  return PQKV_OK;
}

cudaError_t launch_attention(int kv_dtype, const AttnParams& p, const CUtensorMap& map, int grid,
                             int nt, bool pair, cudaStream_t st) {
  switch (kv_dtype) {
    case PQKV_KV_FP16: return launch_attention_fp16(p, map, grid, nt, pair, st);
    case PQKV_KV_FP8_E4M3: return launch_attention_e4m3(p, map, grid, nt, pair, st);
    case PQKV_KV_INT8_ROW: return launch_attention_int8_row(p, map, grid, nt, pair, st);
    default: return launch_attention_int8(p, map, grid, nt, pair, st);
  }
}

int check_output_args(const AttnArgs& a, bool bad_outputs) {
  if (a.num_seqs > 0 && bad_outputs) {
    const int rc0 = validate_common(a.head_dim, a.page_size, a.kv_dtype);
    if (rc0) return rc0;
    const int rc1 = validate_heads(a.num_seqs, a.q_len, a.num_q_heads, a.num_kv_heads);
    return rc1 ? rc1 : PQKV_EINVAL;
  }
  return PQKV_OK;
}

}  // namespace pqkv

extern "C" int pqkv_paged_attention(const void* q, void* out, const void* pages,
                                    int64_t num_pages, const int32_t* block_table,
                                    int32_t max_pages_per_seq, const int32_t* seq_lens,
                                    int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                    int32_t kv_dtype, const float* k_scale, const float* v_scale,
                                    int32_t scale_per_head, int32_t num_splits,
                                    int32_t max_seq_len, void* workspace, size_t workspace_bytes,
                                    int32_t* status, void* stream) {
  const AttnArgs a{q, pages, num_pages, block_table, max_pages_per_seq, seq_lens, num_seqs, q_len,
                   num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, k_scale, v_scale,
                   scale_per_head, num_splits, max_seq_len};
  int rc = check_output_args(a, !out || !aligned(out, 16));
  if (rc) return rc;
  AttnLaunch L;
  rc = plan_attention_launch(a, &L);
  if (rc || num_seqs == 0) return rc;
  AttnParams p;
  CUtensorMap map;
  rc = bind_attention(a, L, workspace, workspace_bytes, status, &p, &map);
  if (rc) return rc;
  p.out = static_cast<uint16_t*>(out);
  const cudaError_t e =
      launch_attention(kv_dtype, p, map, L.grid, L.nt, L.pair, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PQKV_OK : PQKV_ECUDA;
}

extern "C" int pqkv_paged_attention_window(const void* q, void* out, const void* pages,
                                           int64_t num_pages, const int32_t* block_table,
                                           int32_t max_pages_per_seq, const int32_t* seq_lens,
                                           int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t page_size, int32_t kv_dtype,
                                           const float* k_scale, const float* v_scale,
                                           int32_t scale_per_head, int32_t num_splits,
                                           int32_t max_seq_len, int32_t window, void* workspace,
                                           size_t workspace_bytes, int32_t* status, void* stream) {
  AttnArgs a{q, pages, num_pages, block_table, max_pages_per_seq, seq_lens, num_seqs, q_len,
             num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, k_scale, v_scale,
             scale_per_head, num_splits, max_seq_len};
  int rc = check_output_args(a, !out || !aligned(out, 16));
  if (rc) return rc;
  if (window < 0) return PQKV_EINVAL;
  if (window == 0)      // no window: the plain kernel
    return pqkv_paged_attention(q, out, pages, num_pages, block_table, max_pages_per_seq,
                                seq_lens, num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                                page_size, kv_dtype, k_scale, v_scale, scale_per_head,
                                num_splits, max_seq_len, workspace, workspace_bytes, status,
                                stream);
  a.window = window;
  AttnLaunch L;
  rc = plan_attention_launch(a, &L);
  if (rc || num_seqs == 0) return rc;
  AttnWindowParams p;
  CUtensorMap map;
  rc = bind_attention(a, L, workspace, workspace_bytes, status, &p, &map);
  if (rc) return rc;
  p.out = static_cast<uint16_t*>(out);
  p.window = window;
  cudaError_t e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (kv_dtype) {
    case PQKV_KV_FP16: e = launch_attention_window_fp16(p, map, L.grid, L.nt, st); break;
    case PQKV_KV_FP8_E4M3: e = launch_attention_window_e4m3(p, map, L.grid, L.nt, st); break;
    case PQKV_KV_INT8_ROW: e = launch_attention_window_int8_row(p, map, L.grid, L.nt, st); break;
    default: e = launch_attention_window_int8(p, map, L.grid, L.nt, st); break;
  }
  return e == cudaSuccess ? PQKV_OK : PQKV_ECUDA;
}

extern "C" int pqkv_paged_attention_partial(
    const void* q, const void* pages, int64_t num_pages, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* q_pos, int32_t num_seqs,
    int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int32_t kv_dtype, const float* k_scale, const float* v_scale, int32_t scale_per_head,
    int32_t num_splits, int32_t max_seq_len, float* out_o, float* out_lse, void* workspace,
    size_t workspace_bytes, int32_t* status, void* stream) {
  const AttnArgs a{q, pages, num_pages, block_table, max_pages_per_seq, seq_lens, num_seqs, q_len,
                   num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, k_scale, v_scale,
                   scale_per_head, num_splits, max_seq_len};
  int rc = check_output_args(a, !q_pos || !out_o || !out_lse || !aligned(q_pos, 4) ||
                                    !aligned(out_o, 16) || !aligned(out_lse, 4));
  if (rc) return rc;
  AttnLaunch L;
  rc = plan_attention_launch(a, &L);
  if (rc || num_seqs == 0) return rc;
  AttnPartialParams p;
  CUtensorMap map;
  rc = bind_attention(a, L, workspace, workspace_bytes, status, &p, &map);
  if (rc) return rc;
  p.q_pos = q_pos;
  p.out_o = out_o;
  p.out_lse = out_lse;
  cudaError_t e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (kv_dtype) {
    case PQKV_KV_FP16: e = launch_attention_partial_fp16(p, map, L.grid, L.nt, L.pair, st); break;
    case PQKV_KV_FP8_E4M3: e = launch_attention_partial_e4m3(p, map, L.grid, L.nt, L.pair, st); break;
    case PQKV_KV_INT8_ROW: e = launch_attention_partial_int8_row(p, map, L.grid, L.nt, L.pair, st); break;
    default: e = launch_attention_partial_int8(p, map, L.grid, L.nt, L.pair, st); break;
  }
  return e == cudaSuccess ? PQKV_OK : PQKV_ECUDA;
}

extern "C" int pqkv_lse_merge(const float* part_o, const float* part_lse, int32_t num_parts,
                              int64_t num_rows, int32_t head_dim, void* out, float* out_lse,
                              void* stream) {
  if (head_dim != kHeadDim) return PQKV_EUNSUPPORTED;
  if (num_parts < 1 || num_rows < 0) return PQKV_EINVAL;
  if (num_rows == 0) return PQKV_OK;
  if (num_rows > ((int64_t)1 << 34)) return PQKV_ERANGE;
  if (!part_o || !part_lse || !out || !aligned(part_o, 16) || !aligned(part_lse, 4) ||
      !aligned(out, 16) || (out_lse && !aligned(out_lse, 4)))
    return PQKV_EINVAL;
  const cudaError_t e = launch_lse_merge(part_o, part_lse, num_parts, num_rows,
                                         static_cast<uint16_t*>(out), out_lse,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PQKV_OK : PQKV_ECUDA;
}

namespace pqkv {
namespace {

constexpr int kDevBits = 5;   // PQKV_DEV_SLOT_RANGE .. PQKV_DEV_PAGE_RANGE

const char* device_bit_text(int bit) {
  switch (bit) {
    case PQKV_DEV_SLOT_RANGE: return "slot beyond the pool (token skipped)";
    case PQKV_DEV_SEQ_RANGE: return "seq_len out of range (clamped)";
    case PQKV_DEV_BAD_SCALE: return "scale not finite and positive";
    case PQKV_DEV_TIMEOUT: return "pipeline wait timed out";
    case PQKV_DEV_PAGE_RANGE: return "block-table page id out of range (read as zeros)";
  }
  return "";
}

// "device: a; b; ..." for every combination of the device status bits, built
// once (a status word may hold several OR-ed bits).
const std::string& device_bits_text(int bits) {
  static const std::vector<std::string> table = [] {
    std::vector<std::string> t(1u << kDevBits);
    for (int c = 1; c < (1 << kDevBits); ++c) {
      std::string s = "device: ";
      bool first = true;
      for (int b = 0; b < kDevBits; ++b) {
        if (!(c & (1 << b))) continue;
        if (!first) s += "; ";
        s += device_bit_text(1 << b);
        first = false;
      }
      t[c] = s;
    }
    return t;
  }();
  return table[bits];
}

}  // namespace
}  // namespace pqkv

extern "C" const char* pqkv_status_string(int code) {
  switch (code) {
    case PQKV_OK: return "ok";
    case PQKV_EINVAL: return "invalid argument (null/misaligned pointer or bad size)";
    case PQKV_EUNSUPPORTED: return "unsupported configuration";
    case PQKV_ERANGE: return "size outside the supported range";
    case PQKV_EWORKSPACE: return "workspace missing, misaligned or too small";
    case PQKV_ECUDA: return "CUDA runtime call or kernel launch failed";
  }
  if (code > 0 && code < (1 << pqkv::kDevBits)) return pqkv::device_bits_text(code).c_str();
  return "unknown status";
}

extern "C" const char* pqkv_version(void) { return "0.1.0"; }
