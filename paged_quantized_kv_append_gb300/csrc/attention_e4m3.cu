// Paged attention instantiations for one KV format (kept in its own
// translation unit so the formats compile in parallel).
#include "attention_launch.cuh"

namespace pqkv {

cudaError_t launch_attention_e4m3(const AttnParams& p, const CUtensorMap& map, int grid,
                                  int nt, bool pair, cudaStream_t stream) {
  return launch_attention_dtype<PQKV_KV_FP8_E4M3>(p, map, grid, nt, pair, stream);
}

int attention_blocks_per_sm_e4m3(int nt, bool pair, int num_seqs) {
  return blocks_per_sm_dtype<PQKV_KV_FP8_E4M3>(nt, pair, num_seqs);
}

cudaError_t launch_attention_partial_e4m3(const AttnPartialParams& p, const CUtensorMap& map,
                                          int grid, int nt, bool pair, cudaStream_t stream) {
  return launch_attention_partial_dtype<PQKV_KV_FP8_E4M3>(p, map, grid, nt, pair, stream);
}

cudaError_t launch_attention_window_e4m3(const AttnWindowParams& p, const CUtensorMap& map,
                                         int grid, int nt, cudaStream_t stream) {
  return launch_attention_window_dtype<PQKV_KV_FP8_E4M3>(p, map, grid, nt, stream);
}

}  // namespace pqkv
