// kv_append_quant: quantize new K/V rows and scatter them into their pool
// slots.  ReVolta README, "Weight and KV formats" ("E4M3 KV", "INT8 KV"): the
// cache holds E4M3 codes under calibrated per-layer scales, INT8 codes under a
// per-head scale, or plain fp16.
//
// One thread owns 16-element vectors of (token, kv-head) rows for both K and
// V -- two per pass, whose loads are all issued before any arithmetic: per
// vector it reads 32 B of fp16 per tensor (two 16-byte streaming loads), forms
// the correctly rounded fp32 quotient x / scale for each element, converts
// with round-to-nearest-even and saturation, and stores 16 codes (one 16-byte
// store; 32 B for fp16).  Consecutive threads cover consecutive vectors of a
// row, so loads are fully coalesced and each (token, head) row lands as one
// 128-byte line of its page tile.
//
// INT8 with a scale per row (the README's INT8 KV with run-time scales): the
// eight threads of a row -- eight consecutive lanes of one warp -- exchange
// their partial |x| maxima with shuffles, divide the row maximum by 127, encode
// under that scale and the row's first thread stores the scale at the row's
// slot of the scale area that follows the codes.
#include "pqkv_common.cuh"

namespace pqkv {

__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  // cvt packs its first source into the upper byte
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t int8_from_f32(float x) {
  int i;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(i) : "f"(x));  // NaN -> 0, saturating
  i = max(-127, min(127, i));
  return static_cast<uint32_t>(i) & 0xFFu;
}

__device__ __forceinline__ bool scale_ok(float s) { return s > 0.0f && s <= 3.4e38f; }

// largest |x| of 16 fp16 values (NaNs drop out of fmaxf), starting from 0
__device__ __forceinline__ float amax16(const uint4& a, const uint4& b) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    m = fmaxf(m, fmaxf(fabsf(__low2float(h)), fabsf(__high2float(h))));
  }
  return m;
}

// maximum over the 8 consecutive lanes that hold one row
__device__ __forceinline__ float row_max8(float m) {
  const unsigned mask = 0xFFu << (threadIdx.x & 24);
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(mask, m, o));
  return m;
}

// 16 fp16 values (as 8 words) -> 16 codes (4 words)
template <int KVT>
__device__ __forceinline__ uint4 quantize16(const uint4& a, const uint4& b, float scale) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[2 * i + j]);
      f[2 * j] = __fdiv_rn(__low2float(h), scale);
      f[2 * j + 1] = __fdiv_rn(__high2float(h), scale);
    }
    if (KVT == PQKV_KV_FP8_E4M3) {
      out[i] = e4m3x2_from_f32(f[0], f[1]) | (e4m3x2_from_f32(f[2], f[3]) << 16);
    } else {
      out[i] = int8_from_f32(f[0]) | (int8_from_f32(f[1]) << 8) | (int8_from_f32(f[2]) << 16) |
               (int8_from_f32(f[3]) << 24);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int KVT>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
  constexpr int kVecPerRow = kHeadDim / 16;
  constexpr int kElem = (KVT == PQKV_KV_FP16) ? 2 : 1;
  constexpr int64_t kTile = (int64_t)kPageSize * kHeadDim * kElem;  // one K (or V) tile
  constexpr int U = kAppendUnroll;
  const int64_t total = (int64_t)p.num_tokens * p.num_kv_heads * kVecPerRow;
  const int64_t pool_slots = p.num_pages * kPageSize;
  const int64_t stride = (int64_t)gridDim.x * kAppendThreads * U;
  for (int64_t i0 = (int64_t)blockIdx.x * kAppendThreads * U + threadIdx.x; i0 < total;
       i0 += stride) {
    // ---- all loads of this pass first.  Vector u is i0 + u * blockDim; the
    //      eight vectors of one (token, kv-head) row sit in eight consecutive
    //      lanes, so a row is either wholly in range or wholly out.
    int64_t slot[U], t[U];
    int h[U], c[U];
    uint4 k0[U], k1[U], v0[U], v1[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + (int64_t)u * kAppendThreads;
      slot[u] = -1;
      if (i < total) {
        c[u] = (int)(i % kVecPerRow);
        const int64_t th = i / kVecPerRow;
        h[u] = (int)(th % p.num_kv_heads);
        t[u] = th / p.num_kv_heads;
        slot[u] = __ldg(p.slots + t[u]);
        const uint4* ks = reinterpret_cast<const uint4*>(p.k + t[u] * p.k_stride +
                                                         h[u] * kHeadDim + c[u] * 16);
        const uint4* vs = reinterpret_cast<const uint4*>(p.v + t[u] * p.v_stride +
                                                         h[u] * kHeadDim + c[u] * 16);
        k0[u] = __ldcs(ks);
        k1[u] = __ldcs(ks + 1);
        v0[u] = __ldcs(vs);
        v1[u] = __ldcs(vs + 1);
      }
    }
    // ---- then convert and store
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + (int64_t)u * kAppendThreads;
      if (i >= total || slot[u] < 0) continue;
      if (slot[u] >= pool_slots) {
        if (c[u] == 0 && h[u] == 0) report(p.status, PQKV_DEV_SLOT_RANGE);
        continue;
      }
      const int64_t page = slot[u] / kPageSize;
      const int off = (int)(slot[u] % kPageSize);
      uint8_t* tile = p.pages + (page * p.num_kv_heads + h[u]) * 2 * kTile;
      uint8_t* kd = tile + (int64_t)off * kHeadDim * kElem + c[u] * 16 * kElem;
      uint8_t* vd = kd + kTile;
      if (KVT == PQKV_KV_FP16) {
        reinterpret_cast<uint4*>(kd)[0] = k0[u];
        reinterpret_cast<uint4*>(kd)[1] = k1[u];
        reinterpret_cast<uint4*>(vd)[0] = v0[u];
        reinterpret_cast<uint4*>(vd)[1] = v1[u];
      } else if (KVT == PQKV_KV_INT8_ROW) {
        // all eight threads of the row reach this point together
        const float kscale = __fdiv_rn(row_max8(amax16(k0[u], k1[u])), 127.f);
        const float vscale = __fdiv_rn(row_max8(amax16(v0[u], v1[u])), 127.f);
        *reinterpret_cast<uint4*>(kd) = quantize16<PQKV_KV_INT8>(k0[u], k1[u], kscale);
        *reinterpret_cast<uint4*>(vd) = quantize16<PQKV_KV_INT8>(v0[u], v1[u], vscale);
        if (c[u] == 0) {
          float* rs = p.row_scales + (page * p.num_kv_heads + h[u]) * 2 * kPageSize + off;
          rs[0] = kscale;
          rs[kPageSize] = vscale;
        }
      } else {
        const int sh = p.scale_per_head ? h[u] : 0;
        const float kscale = __ldg(p.k_scale + sh);
        const float vscale = __ldg(p.v_scale + sh);
        if (!scale_ok(kscale) || !scale_ok(vscale)) {
          if (c[u] == 0) report(p.status, PQKV_DEV_BAD_SCALE);
          continue;
        }
        *reinterpret_cast<uint4*>(kd) = quantize16<KVT>(k0[u], k1[u], kscale);
        *reinterpret_cast<uint4*>(vd) = quantize16<KVT>(v0[u], v1[u], vscale);
      }
    }
  }
}

cudaError_t launch_append(const AppendParams& p, int kv_dtype, int grid, cudaStream_t stream) {
  switch (kv_dtype) {
    case PQKV_KV_FP16:
      append_kernel<PQKV_KV_FP16><<<grid, kAppendThreads, 0, stream>>>(p);
      break;
    case PQKV_KV_FP8_E4M3:
      append_kernel<PQKV_KV_FP8_E4M3><<<grid, kAppendThreads, 0, stream>>>(p);
      break;
    case PQKV_KV_INT8:
      append_kernel<PQKV_KV_INT8><<<grid, kAppendThreads, 0, stream>>>(p);
      break;
    case PQKV_KV_INT8_ROW:
      append_kernel<PQKV_KV_INT8_ROW><<<grid, kAppendThreads, 0, stream>>>(p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pqkv
