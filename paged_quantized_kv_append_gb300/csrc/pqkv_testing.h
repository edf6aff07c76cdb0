// Testing entry points of libpqkv.  Not part of the public interface
// (include/pqkv.h is); the test suite reaches them through ctypes.
#pragma once

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pqkv_testing_attention_wait_timeout -- pqkv_paged_attention (same
 * arguments, E4M3 pools with 17..24 query rows per kv-head only) in a test
 * mode of its bounded waits: block `skip_block` never issues the tile copy of
 * page `skip_page` of its share, so the warp that owns that page waits for a
 * tile that never arrives.  Waits give up after 1 ms (instead of 1 s); the
 * kernel then sets PQKV_DEV_TIMEOUT in *status, waits for every copy it did
 * issue, and returns.  The outputs are invalid and the workspace must be
 * zeroed again, as after any timeout.  No copy is left in flight and nothing
 * traps, so the context stays usable.
 */
int pqkv_testing_attention_wait_timeout(
    const void* q, void* out, const void* pages, int64_t num_pages, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t q_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int32_t kv_dtype, const float* k_scale, const float* v_scale, int32_t scale_per_head,
    int32_t num_splits, int32_t max_seq_len, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream, int32_t skip_block, int32_t skip_page);

#ifdef __cplusplus
}
#endif
