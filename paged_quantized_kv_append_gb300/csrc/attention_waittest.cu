// Test instantiation of the paged attention kernel for its bounded waits (see
// pqkv_testing.h): the E4M3 24-row kernel with one page's copy never issued
// and a 1 ms wait limit.  Kept in a translation unit of its own, so the
// production kernels are compiled exactly as without it.
#include "attention_launch.cuh"
#include "pqkv_testing.h"

namespace pqkv {

cudaError_t launch_attention_wait_test_e4m3(const AttnWaitTestParams& p, const CUtensorMap& map,
                                            int grid, int nt, cudaStream_t stream) {
  constexpr int KVT = PQKV_KV_FP8_E4M3, NT = 3;
  if (nt != NT) return cudaErrorInvalidValue;
  using Cfg = AttnCfg<KVT, NT>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = opt_in_smem(paged_attention_kernel<KVT, NT, AttnWaitTestParams>,
                                    Cfg::smem_bytes(PQKV_MAX_SEQS), attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_attention_kernel<KVT, NT, AttnWaitTestParams>, grid, Cfg::kThreads,
                    Cfg::smem_bytes(p.num_seqs), stream, map, p);
}

}  // namespace pqkv

using namespace pqkv;

extern "C" int pqkv_testing_attention_wait_timeout(
    const void* q, void* out, const void* pages, int64_t num_pages, const int32_t* block_table,
    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t q_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
    int32_t kv_dtype, const float* k_scale, const float* v_scale, int32_t scale_per_head,
    int32_t num_splits, int32_t max_seq_len, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream, int32_t skip_block, int32_t skip_page) {
  const AttnArgs a{q, pages, num_pages, block_table, max_pages_per_seq, seq_lens, num_seqs, q_len,
                   num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, k_scale, v_scale,
                   scale_per_head, num_splits, max_seq_len};
  int rc = check_output_args(a, !out || (reinterpret_cast<uintptr_t>(out) % 16) != 0);
  if (rc) return rc;
  AttnLaunch L;
  rc = plan_attention_launch(a, &L);
  if (rc || num_seqs == 0) return rc;
  if (kv_dtype != PQKV_KV_FP8_E4M3 || L.nt != 3) return PQKV_EUNSUPPORTED;
  if (skip_block < 0 || skip_block >= L.grid || skip_page < 0) return PQKV_EINVAL;
  AttnWaitTestParams p;
  CUtensorMap map;
  rc = bind_attention(a, L, workspace, workspace_bytes, status, &p, &map);
  if (rc) return rc;
  p.out = static_cast<uint16_t*>(out);
  p.skip_block = skip_block;
  p.skip_page = skip_page;
  return launch_attention_wait_test_e4m3(p, map, L.grid, L.nt,
                                         static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PQKV_OK
             : PQKV_ECUDA;
}
