// pqkv_paged_attention_noalloc: paged attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: code that runs under a
// runtime which forbids cudaMalloc at call time (its memory is budgeted up
// front), hooks that execute inside another framework's step and must not
// bypass its allocator, or plain C callers with no allocator at all.  This
// entry point serves them by using a scratch area that the library itself
// owns: a fixed-size file-scope device array that every GPU that loads the
// library holds until the process exits.  It allocates nothing and calls no
// allocating routine; it is otherwise the same computation as
// pqkv_paged_attention, planned and launched by the same internal steps with
// the scratch area as workspace.
#include <cstring>
#include <mutex>

#include "pqkv_internal.h"

namespace {

// The library's own scratch area (PQKV_NOALLOC_SCRATCH_BYTES, 16 MiB).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PQKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's
// name in host code is only a host-side stand-in, so its device address is
// looked up once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PQKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PQKV_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PQKV_OK;
}

}  // namespace

extern "C" int pqkv_paged_attention_noalloc(const void* q, void* out, const void* pages,
                                            int64_t num_pages, const int32_t* block_table,
                                            int32_t max_pages_per_seq, const int32_t* seq_lens,
                                            int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t page_size, int32_t kv_dtype,
                                            const float* k_scale, const float* v_scale,
                                            int32_t scale_per_head, int32_t num_splits,
                                            int32_t max_seq_len, int32_t* status, void* stream) {
  using namespace pqkv;
  const AttnArgs a{q, pages, num_pages, block_table, max_pages_per_seq, seq_lens, num_seqs, q_len,
                   num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, k_scale, v_scale,
                   scale_per_head, num_splits, max_seq_len};
  int rc = check_output_args(a, !out || (reinterpret_cast<uintptr_t>(out) % 16) != 0);
  if (rc) return rc;
  // Every check runs before anything is queued on the stream: a call that is
  // rejected leaves the shared scratch area alone.
  AttnLaunch L;
  rc = plan_attention_launch(a, &L);
  if (rc || num_seqs == 0) return rc;
  // the workspace of the grid this call launches (not the largest grid)
  if (L.pl.total > PQKV_NOALLOC_SCRATCH_BYTES) return PQKV_ERANGE;
  void* scratch = nullptr;
  if (L.pl.total > 0) {
    rc = scratch_address(&scratch);
    if (rc) return rc;
  }
  AttnParams p;
  CUtensorMap map;
  rc = bind_attention(a, L, scratch, L.pl.total > 0 ? (size_t)PQKV_NOALLOC_SCRATCH_BYTES : 0,
                      status, &p, &map);
  if (rc) return rc;
  p.out = static_cast<uint16_t*>(out);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (L.pl.total > 0) {
    // The array keeps the previous call's contents; the merge counters at its
    // start must be zero when the kernel begins.
    if (cudaMemsetAsync(scratch, 0, L.pl.counter_bytes, st) != cudaSuccess) return PQKV_ECUDA;
  }
  return launch_attention(kv_dtype, p, map, L.grid, L.nt, L.pair, st) == cudaSuccess ? PQKV_OK
                                                                              : PQKV_ECUDA;
}
