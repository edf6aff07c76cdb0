// Log-sum-exp merge of partial attention results, the combine step of a decode
// context parallel split of the keys across ranks (ReVolta README, "Hardware"
// and "Quick start": DCP2).  Each rank attends over its share of the keys and
// gives, per (query, q-head) row, O_p = (sum_j e^{s_j - m_p} V_j) / l_p and
// lse_p = m_p + ln l_p; the full result is
//     O = sum_p e^{lse_p - LSE} O_p,   LSE = ln sum_p e^{lse_p}.
// One warp per row; lane d4 owns dims 4*d4 .. 4*d4 + 3.
#include "pqkv_common.cuh"

namespace pqkv {

__global__ void __launch_bounds__(256) lse_merge_kernel(const float* part_o, const float* part_lse,
                                                        int num_parts, int64_t rows,
                                                        uint16_t* out, float* out_lse) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float M = -INFINITY;
  for (int q = 0; q < num_parts; ++q) M = fmaxf(M, __ldg(part_lse + (int64_t)q * rows + row));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float sum = 0.f;
  if (M > -INFINITY) {
    for (int q = 0; q < num_parts; ++q) {
      const float lq = __ldg(part_lse + (int64_t)q * rows + row);
      if (!(lq > -INFINITY)) continue;                 // a share with no visible key
      const float w = expf(lq - M);
      const float4 v = __ldg(reinterpret_cast<const float4*>(part_o + ((int64_t)q * rows + row) *
                                                                          kHeadDim) + lane);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
      sum += w;
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  __half2 h01 = __floats2half2_rn(acc.x * inv, acc.y * inv);
  __half2 h23 = __floats2half2_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&h01);
  pk.y = *reinterpret_cast<uint32_t*>(&h23);
  *reinterpret_cast<uint2*>(out + row * kHeadDim + 4 * lane) = pk;
  if (out_lse && lane == 0) out_lse[row] = sum > 0.f ? M + logf(sum) : -INFINITY;
}

cudaError_t launch_lse_merge(const float* part_o, const float* part_lse, int num_parts,
                             int64_t rows, uint16_t* out, float* out_lse, cudaStream_t stream) {
  const int64_t blocks = (rows + 7) / 8;
  return launch_pdl(lse_merge_kernel, (unsigned)blocks, 256, 0, stream, part_o, part_lse,
                    num_parts, rows, out, out_lse);
}

}  // namespace pqkv
