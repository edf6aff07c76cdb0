// Host-side launchers of the paged attention kernel (one set per KV format,
// instantiated by attention_<format>.cu).
#pragma once

#include <atomic>

#include "attention_impl.cuh"

namespace pqkv {

// The dynamic shared-memory opt-in of a kernel is a per-device setting: set
// it once on each device the kernel is launched on (devices 0..63 tracked in
// `done`; higher ordinals set it on every launch).
template <class Kernel>
cudaError_t opt_in_smem(Kernel* kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

template <int KVT, int NT, bool kPair = false>
cudaError_t launch_attention_t(const AttnParams& p, const CUtensorMap& map, int grid,
                               cudaStream_t stream) {
  using Cfg = AttnCfg<KVT, NT, kPair>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = opt_in_smem(paged_attention_kernel<KVT, NT, AttnParams, kPair>,
                                    Cfg::smem_bytes(PQKV_MAX_SEQS), attr_done);
  if (e != cudaSuccess) return e;
  if constexpr (Cfg::kFlat && !kPair && KVT == PQKV_KV_FP16) {
    // one segment over at most 8 blocks: a cluster, merged in shared memory
    if (p.num_splits == 0 && p.num_seqs * p.num_kv_heads == 1 && grid > 1 && grid <= 8)
      return launch_cluster(paged_attention_kernel<KVT, NT, AttnParams, kPair>, grid,
                            Cfg::kThreads, Cfg::smem_bytes(p.num_seqs), stream, (unsigned)grid,
                            attention_uses_pdl<KVT, NT, AttnParams, kPair>(), map, p);
  }
  if constexpr (attention_uses_pdl<KVT, NT, AttnParams, kPair>()) {
    return launch_pdl(paged_attention_kernel<KVT, NT, AttnParams, kPair>, grid, Cfg::kThreads,
                      Cfg::smem_bytes(p.num_seqs), stream, map, p);
  } else {
    paged_attention_kernel<KVT, NT, AttnParams, kPair>
        <<<grid, Cfg::kThreads, Cfg::smem_bytes(p.num_seqs), stream>>>(map, p);
    return cudaGetLastError();
  }
}

template <int KVT, int NT, bool kPair = false>
int blocks_per_sm_t(int num_seqs) {
  using Cfg = AttnCfg<KVT, NT, kPair>;
  static std::atomic<uint64_t> attr_done{0};
  if (opt_in_smem(paged_attention_kernel<KVT, NT, AttnParams, kPair>,
                  Cfg::smem_bytes(PQKV_MAX_SEQS), attr_done) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, paged_attention_kernel<KVT, NT, AttnParams, kPair>, Cfg::kThreads,
          Cfg::smem_bytes(num_seqs)) != cudaSuccess)
    return 0;
  return n;
}

template <int KVT, int NT, bool kPair = false>
cudaError_t launch_attention_partial_t(const AttnPartialParams& p, const CUtensorMap& map,
                                       int grid, cudaStream_t stream) {
  using Cfg = AttnCfg<KVT, NT, kPair>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = opt_in_smem(paged_attention_kernel<KVT, NT, AttnPartialParams, kPair>,
                                    Cfg::smem_bytes(PQKV_MAX_SEQS), attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_attention_kernel<KVT, NT, AttnPartialParams, kPair>, grid,
                    Cfg::kThreads, Cfg::smem_bytes(p.num_seqs), stream, map, p);
}

// Sliding-window mode: the kernel also keeps each sequence's first page read
// (num_seqs ints after the sequence lengths).
template <int KVT, int NT>
cudaError_t launch_attention_window_t(const AttnWindowParams& p, const CUtensorMap& map, int grid,
                                      cudaStream_t stream) {
  using Cfg = AttnCfg<KVT, NT, false, true>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = opt_in_smem(paged_attention_kernel<KVT, NT, AttnWindowParams>,
                                    Cfg::smem_bytes(PQKV_MAX_SEQS) + 4 * PQKV_MAX_SEQS, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(paged_attention_kernel<KVT, NT, AttnWindowParams>, grid, Cfg::kThreads,
                    Cfg::smem_bytes(p.num_seqs) + 4 * p.num_seqs, stream, map, p);
}

template <int KVT>
cudaError_t launch_attention_window_dtype(const AttnWindowParams& p, const CUtensorMap& map,
                                          int grid, int nt, cudaStream_t stream) {
  switch (nt) {
    case 1: return launch_attention_window_t<KVT, 1>(p, map, grid, stream);
    case 2: return launch_attention_window_t<KVT, 2>(p, map, grid, stream);
    case 3: return launch_attention_window_t<KVT, 3>(p, map, grid, stream);
    case 4: return launch_attention_window_t<KVT, 4>(p, map, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// pair: the 8-row decode as two 8-warp blocks per SM (8-bit formats only)
template <int KVT>
cudaError_t launch_attention_partial_dtype(const AttnPartialParams& p, const CUtensorMap& map,
                                           int grid, int nt, bool pair, cudaStream_t stream) {
  switch (nt) {
    case 1:
      if constexpr (KVT != PQKV_KV_FP16)
        if (pair) return launch_attention_partial_t<KVT, 1, true>(p, map, grid, stream);
      return launch_attention_partial_t<KVT, 1>(p, map, grid, stream);
    case 2: return launch_attention_partial_t<KVT, 2>(p, map, grid, stream);
    case 3: return launch_attention_partial_t<KVT, 3>(p, map, grid, stream);
    case 4: return launch_attention_partial_t<KVT, 4>(p, map, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int KVT>
cudaError_t launch_attention_dtype(const AttnParams& p, const CUtensorMap& map, int grid, int nt,
                                   bool pair, cudaStream_t stream) {
  switch (nt) {
    case 1:
      if constexpr (KVT != PQKV_KV_FP16)
        if (pair) return launch_attention_t<KVT, 1, true>(p, map, grid, stream);
      return launch_attention_t<KVT, 1>(p, map, grid, stream);
    case 2: return launch_attention_t<KVT, 2>(p, map, grid, stream);
    case 3: return launch_attention_t<KVT, 3>(p, map, grid, stream);
    case 4: return launch_attention_t<KVT, 4>(p, map, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int KVT>
int blocks_per_sm_dtype(int nt, bool pair, int num_seqs) {
  switch (nt) {
    case 1:
      if constexpr (KVT != PQKV_KV_FP16)
        if (pair) return blocks_per_sm_t<KVT, 1, true>(num_seqs);
      return blocks_per_sm_t<KVT, 1>(num_seqs);
    case 2: return blocks_per_sm_t<KVT, 2>(num_seqs);
    case 3: return blocks_per_sm_t<KVT, 3>(num_seqs);
    case 4: return blocks_per_sm_t<KVT, 4>(num_seqs);
    default: return 0;
  }
}

}  // namespace pqkv
