// Paged attention instantiations for INT8 with a scale per (token, kv-head)
// row (kept in its own translation unit so the formats compile in parallel).
#include "attention_launch.cuh"

namespace pqkv {

cudaError_t launch_attention_int8_row(const AttnParams& p, const CUtensorMap& map, int grid,
                                      int nt, bool pair, cudaStream_t stream) {
  return launch_attention_dtype<PQKV_KV_INT8_ROW>(p, map, grid, nt, pair, stream);
}

int attention_blocks_per_sm_int8_row(int nt, bool pair, int num_seqs) {
  return blocks_per_sm_dtype<PQKV_KV_INT8_ROW>(nt, pair, num_seqs);
}

cudaError_t launch_attention_partial_int8_row(const AttnPartialParams& p, const CUtensorMap& map,
                                              int grid, int nt, bool pair, cudaStream_t stream) {
  return launch_attention_partial_dtype<PQKV_KV_INT8_ROW>(p, map, grid, nt, pair, stream);
}

cudaError_t launch_attention_window_int8_row(const AttnWindowParams& p, const CUtensorMap& map,
                                             int grid, int nt, cudaStream_t stream) {
  return launch_attention_window_dtype<PQKV_KV_INT8_ROW>(p, map, grid, nt, stream);
}

}  // namespace pqkv
