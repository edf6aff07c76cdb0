// kv_append_quant: quantize new K/V rows and scatter them into their pool
// slots.  ReVolta README, "Weight and KV formats" ("E4M3 KV", "INT8 KV"): the
// cache holds E4M3 codes under calibrated per-layer scales, INT8 codes under a
// per-head scale, or plain fp16.
//
// One thread owns 16-element vectors of (token, kv-head) rows for both K and
// V, whose loads are all issued before any arithmetic: per vector it reads
// 32 B of fp16 per tensor (two 16-byte streaming loads), encodes the correctly
// rounded fp32 quotient x / scale of each element with round-to-nearest-even
// and saturation, and stores 16 codes (one 16-byte store; 32 B for fp16).
// Consecutive threads cover consecutive vectors of a row, so loads are fully
// coalesced and each (token, head) row lands as one 128-byte line of its page
// tile.
//
// The code of RN(x / s) is found without a division (the encode is
// otherwise bound by the issue of IEEE divisions).  With r = RN(1/s), the
// product RN(x r) equals the quotient t = x / s up to a factor
// (1 + e1)(1 + e2), |e1|, |e2| <= 2^-24, and RN(t) is within a factor 2^-24 of
// t.  That holds while r and the products are normal numbers: s in
// [2^-125, 2^125] (other scales take the division); a product below the normal
// range belongs to a quotient below 2^-125, and every value there encodes as
// a zero of x's sign.
//  * E4M3: the products with RN(r (1 - 2^-20)) and RN(r (1 + 2^-20)) lie on
//    either side of RN(t) (the margin 2^-20 exceeds the three roundings'
//    3.01 * 2^-24), and the encode is monotone: where both give the same
//    code, RN(t) gives it too.
//  * INT8: z = RN(x r) rounds to the integer c (added to 1.5 * 2^23, which
//    leaves c in the low bits); RN(t), within 2^-15.4 of z while
//    |z| <= 127.25, rounds to c too when |z - c| <= 0.5 - 2^-14.  Beyond
//    127.25 the code is +-127.
// Where the check fails, RN(t) lies within about 2^-19 of the boundary m
// between two adjacent codes (an E4M3 midpoint, or a half-integer).  Then
// x - s m is a multiple of the last bit of the product s m and smaller than
// 2^20 of them, so one fused multiply-add gives it exactly, and comparing it
// with s h (h half an ulp of m, an exact product) decides: RN(t) is above m,
// below m, or m itself -- a tie of the encode, which goes to the even code.
//
// INT8 with a scale per row (the README's INT8 KV with run-time scales): the
// eight threads of a row -- eight consecutive lanes of one warp -- exchange
// their partial |x| maxima with shuffles, round the row maximum over 127 to
// the nearest fp16 value, encode under that scale and the row's first thread
// stores the fp16 scale at the row's place in the scale area that follows the
// codes.
#include <atomic>

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

// 16 fp16 values (as 8 words) -> 16 codes (4 words), through the correctly
// rounded division x / scale
template <int KVT>
__device__ __forceinline__ uint4 quantize16_div(const uint4& a, const uint4& b, float scale) {
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

// The reciprocal brackets of a scale for the division-free encode
struct Recip {
  float r, lo, hi;    // RN(1/s), RN(r (1 - 2^-20)), RN(r (1 + 2^-20))
  bool fast;          // s in [2^-125, 2^125]
};

__device__ __forceinline__ Recip recip_of(float s) {
  Recip q;
  q.fast = s >= 0x1p-125f && s <= 0x1p125f;
  q.r = __frcp_rn(s);
  q.lo = __fmul_rn(q.r, 1.0f - 0x1p-20f);
  q.hi = __fmul_rn(q.r, 1.0f + 0x1p-20f);
  return q;
}

// Magnitude code of RN(a / s), a >= 0, when RN(a / s) lies next to the
// boundary m between the adjacent magnitude codes c_lo < c_hi (see the head
// of this file); m_pow2: m is a power of two, so the ulp below it is half.
__device__ __forceinline__ uint32_t resolve_boundary(float a, float s, float m, uint32_t c_lo,
                                                     uint32_t c_hi, bool m_pow2) {
  const float rho = fmaf(-s, m, a);                                   // a - s m, exact
  const float h = __uint_as_float((__float_as_uint(m) & 0x7F800000u) - (24u << 23));
  const float hs = __fmul_rn(s, h);                                   // exact
  if (rho > hs) return c_hi;
  if (rho < (m_pow2 ? -0.5f * hs : -hs)) return c_lo;
  return (c_lo & 1u) ? c_hi : c_lo;                                   // RN(a / s) == m
}

// E4M3: the code of x whose bracket codes cl != ch
__device__ __forceinline__ uint32_t e4m3_boundary(float x, float s, uint32_t cl, uint32_t ch) {
  const uint32_t ml = cl & 0x7Fu, mh = ch & 0x7Fu;
  const uint32_t c_lo = min(ml, mh), c_hi = max(ml, mh);
  uint32_t v;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(v)
      : "r"(c_lo | (c_hi << 8)));
  const __half2 hv = *reinterpret_cast<const __half2*>(&v);
  const float m = 0.5f * (__low2float(hv) + __high2float(hv));        // exact
  // the only power-of-two midpoint lies between 0 and the smallest subnormal
  return resolve_boundary(fabsf(x), s, m, c_lo, c_hi, c_lo == 0) | (cl & 0x80u);
}

// INT8: the code byte of x whose fast check failed
__device__ __forceinline__ uint32_t int8_boundary(float x, float s, float z) {
  if (z != z) return 0;                                               // NaN
  if (fabsf(z) > 127.25f) return z > 0.f ? 127u : 0x81u;
  constexpr float kMagic = 12582912.0f;
  const float za = fabsf(z);
  const float ca = __fsub_rn(__fadd_rn(za, kMagic), kMagic);          // rint(za)
  const float m = za > ca ? ca + 0.5f : ca - 0.5f;                    // the half-integer near za
  const uint32_t c_lo = (uint32_t)(m - 0.5f);
  const uint32_t mag = resolve_boundary(fabsf(x), s, m, c_lo, c_lo + 1, m == 0.5f);
  return (x < 0.f ? 0u - mag : mag) & 0xFFu;
}

__device__ __forceinline__ float half_of(const uint32_t (&w)[8], int k) {
  const __half2 h = *reinterpret_cast<const __half2*>(&w[k >> 1]);
  return (k & 1) ? __high2float(h) : __low2float(h);
}

// 16 fp16 values -> 16 codes of RN(x / scale); see the head of this file.
// Each group of four codes comes from the fast path first; the rare group
// with an element next to a rounding boundary then decides that element.
template <int KVT>
__device__ __forceinline__ uint4 quantize16(const uint4& a, const uint4& b, float scale,
                                            const Recip& rc) {
  if (!rc.fast) return quantize16_div<KVT>(a, b, scale);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = half_of(w, 4 * i + e);
    uint32_t fix = 0;
    if (KVT == PQKV_KV_FP8_E4M3) {
      out[i] = e4m3x2_from_f32(__fmul_rn(f[0], rc.lo), __fmul_rn(f[1], rc.lo)) |
               (e4m3x2_from_f32(__fmul_rn(f[2], rc.lo), __fmul_rn(f[3], rc.lo)) << 16);
      fix = out[i] ^ (e4m3x2_from_f32(__fmul_rn(f[0], rc.hi), __fmul_rn(f[1], rc.hi)) |
                      (e4m3x2_from_f32(__fmul_rn(f[2], rc.hi), __fmul_rn(f[3], rc.hi)) << 16));
    } else {
      constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
      uint32_t y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float z = __fmul_rn(f[e], rc.r);
        const float yf = __fadd_rn(z, kMagic);
        const float d = __fsub_rn(z, __fsub_rn(yf, kMagic));
        y[e] = __float_as_uint(yf);
        fix |= (fabsf(z) <= 127.25f && fabsf(d) <= 0.5f - 0x1p-14f) ? 0u : 0xFFu << (8 * e);
      }
      out[i] = __byte_perm(__byte_perm(y[0], y[1], 0x0040), __byte_perm(y[2], y[3], 0x0040),
                           0x5410);
    }
    if (fix) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (!((fix >> (8 * e)) & 0xFFu)) continue;
        uint32_t c;
        if (KVT == PQKV_KV_FP8_E4M3) {
          const uint32_t cl = (out[i] >> (8 * e)) & 0xFFu;
          const uint32_t ch = e4m3x2_from_f32(__fmul_rn(f[e], rc.hi), 0.f) & 0xFFu;
          c = e4m3_boundary(f[e], scale, cl, ch);
        } else {
          c = int8_boundary(f[e], scale, __fmul_rn(f[e], rc.r));
        }
        out[i] = (out[i] & ~(0xFFu << (8 * e))) | (c << (8 * e));
      }
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Six resident blocks per SM (40 registers) for the formats with one scale;
// the row-scale format keeps its registers (it would spill under that cap).
template <int KVT>
__global__ void __launch_bounds__(kAppendThreads, KVT == PQKV_KV_INT8_ROW ? 1 : 6)
    append_kernel(const AppendParams p) {
  constexpr int kVecPerRow = kHeadDim / 16;
  constexpr int kElem = (KVT == PQKV_KV_FP16) ? 2 : 1;
  constexpr int64_t kTile = (int64_t)kPageSize * kHeadDim * kElem;  // one K (or V) tile
  constexpr int U = kAppendUnroll;
  grid_dependency_wait();
  grid_dependents_launch();
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
        // the row scale is the binary16 nearest to amax / 127 (rounding the
        // binary32 quotient once more is exact: 24 >= 2 * 11 + 2)
        const __half kh = __float2half_rn(__fdiv_rn(row_max8(amax16(k0[u], k1[u])), 127.f));
        const __half vh = __float2half_rn(__fdiv_rn(row_max8(amax16(v0[u], v1[u])), 127.f));
        const float kscale = __half2float(kh);
        const float vscale = __half2float(vh);
        *reinterpret_cast<uint4*>(kd) =
            quantize16<PQKV_KV_INT8>(k0[u], k1[u], kscale, recip_of(kscale));
        *reinterpret_cast<uint4*>(vd) =
            quantize16<PQKV_KV_INT8>(v0[u], v1[u], vscale, recip_of(vscale));
        if (c[u] == 0) {
          // the (page, kv-head)'s 32 scales are ordered for the attention
          // kernel's fragments: [i][K row i, K row i+8, V row i, V row i+8]
          uint16_t* rs = p.row_scales + (page * p.num_kv_heads + h[u]) * 2 * kPageSize +
                         (off & 7) * 4 + (off >> 3);
          rs[0] = __half_as_ushort(kh);
          rs[2] = __half_as_ushort(vh);
        }
      } else {
        const int sh = p.scale_per_head ? h[u] : 0;
        const float kscale = __ldg(p.k_scale + sh);
        const float vscale = __ldg(p.v_scale + sh);
        if (!scale_ok(kscale) || !scale_ok(vscale)) {
          if (c[u] == 0) report(p.status, PQKV_DEV_BAD_SCALE);
          continue;
        }
        *reinterpret_cast<uint4*>(kd) = quantize16<KVT>(k0[u], k1[u], kscale, recip_of(kscale));
        *reinterpret_cast<uint4*>(vd) = quantize16<KVT>(v0[u], v1[u], vscale, recip_of(vscale));
      }
    }
  }
}

// Resident blocks per SM of the append kernel for `kv_dtype` on the current
// device (register-limited), cached per device ordinal 0..63; 0 on error.
int append_blocks_per_sm(int kv_dtype) {
  static std::atomic<int> cache[4][64];
  int dev = 0;
  if (kv_dtype < 0 || kv_dtype > 3 || cudaGetDevice(&dev) != cudaSuccess) return 0;
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    const int n = cache[kv_dtype][dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (kv_dtype) {
    case PQKV_KV_FP16:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, append_kernel<PQKV_KV_FP16>,
                                                        kAppendThreads, 0);
      break;
    case PQKV_KV_FP8_E4M3:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, append_kernel<PQKV_KV_FP8_E4M3>,
                                                        kAppendThreads, 0);
      break;
    case PQKV_KV_INT8:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, append_kernel<PQKV_KV_INT8>,
                                                        kAppendThreads, 0);
      break;
    default:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, append_kernel<PQKV_KV_INT8_ROW>,
                                                        kAppendThreads, 0);
      break;
  }
  if (e != cudaSuccess || n < 1) return 0;
  if (cached) cache[kv_dtype][dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_append(const AppendParams& p, int kv_dtype, int grid, cudaStream_t stream) {
  switch (kv_dtype) {
    case PQKV_KV_FP16:
      return launch_pdl(append_kernel<PQKV_KV_FP16>, grid, kAppendThreads, 0, stream, p);
    case PQKV_KV_FP8_E4M3:
      return launch_pdl(append_kernel<PQKV_KV_FP8_E4M3>, grid, kAppendThreads, 0, stream, p);
    case PQKV_KV_INT8:
      return launch_pdl(append_kernel<PQKV_KV_INT8>, grid, kAppendThreads, 0, stream, p);
    case PQKV_KV_INT8_ROW:
      return launch_pdl(append_kernel<PQKV_KV_INT8_ROW>, grid, kAppendThreads, 0, stream, p);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pqkv
