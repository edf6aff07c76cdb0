// Paged decode / speculative-verify attention over an FP16, E4M3, INT8 or
// INT8-with-row-scales KV pool, with split-KV partitions merged by
// log-sum-exp; a partial mode gives one rank's share of a decode context
// parallel split as O / l and LSE per row.
//
// What it computes: ReVolta README, "Quick start" (MTP verify of 1 committed +
// 4 draft positions with a causal mask among them, GQA) and "Weight and KV
// formats" (KV stored compressed, widened to fp16 for the products); the split
// of a sequence's keys with partial results combined afterwards is the
// one-GPU counterpart of the decode-context-parallel split on the same page
// ("Hardware", "Quick start").
//
// Design (GB300, sm_103a):
//  * Work.  The key pages of every (sequence, kv-head) segment are laid end to
//    end; in the balanced mode each of the C resident thread blocks takes one
//    equal contiguous share of that list (so a block may finish one segment
//    and start the next, and a long segment is shared by several blocks).  In
//    the fixed mode block c takes partition c % k of segment c / k.  A block
//    that holds a whole segment writes the output directly; otherwise it
//    writes an unnormalised partial (O, m, l) and the last block to finish a
//    segment (an atomic ticket; no block ever waits on another) merges the
//    partials in a fixed order.
//  * Data movement.  Every warp feeds itself: the block's pages are dealt
//    round-robin to its warps, and each warp streams its own (page, kv-head)
//    tiles -- 16 K rows followed by 16 V rows, 4 KB for 8-bit codes -- with
//    4-D TMA loads (cp.async.bulk.tensor, 128-byte swizzle) into ring stages
//    that only it uses, each guarded by an mbarrier; a stage is refilled as
//    soon as its warp has read it.  A warp's lanes look up the pool pages of
//    its next 32 tiles at once, one batch ahead.  Out-of-range page ids read
//    as zeros (TMA bounds) and are reported.
//  * Math.  Per page a warp dequantises the codes in registers (exact fp16),
//    computes S^T = K Q^T with mma.sync m16n8k16 (tokens as M, the G*q_len
//    query rows padded to 8, 16, 24 or 32 as N), keeps an fp32 online softmax
//    in the log2 domain whose reference maximum is only raised when a score
//    exceeds it by more than 2^8 (so probabilities stay <= 256 in fp16),
//    transposes P with movmatrix and accumulates O^T = V^T P^T with a second
//    mma.  Warps merge their states through shared memory at the end of each
//    segment share.
#pragma once

#include <type_traits>

#include "pqkv_common.cuh"

namespace pqkv {

template <int KVT, int NT, bool kPair = false, bool kWideTree = false>
struct AttnCfg {
  // One block per SM.  Every warp is a consumer and feeds its own slice of the
  // TMA ring: page i of the block goes to warp i % kW and stage i % kStages,
  // and kStages is a multiple of kW, so each stage always belongs to one warp
  // (an mbarrier phase is tracked by one parity bit; a stage shared by warps
  // could be waited on for a later round while an earlier load is still in
  // flight).  Warp counts follow the register need of the row width and are
  // multiples of 4, because registers are allotted per scheduler (a quarter
  // of the SM): 8 warps get 255 registers each, 12 get 168, 16 get 128.
  // 8 query rows (NT 1) run 16 warps, 16 rows 12, and 24 or 32 rows 8.
  static constexpr int kW =
      (KVT == PQKV_KV_FP16 || kPair) ? 8 : (NT == 1 ? 16 : (NT == 2 ? 12 : 8));
  // kPair (8 query rows, 8-bit codes, short contexts): two 8-warp blocks per
  // SM at 128 registers, each with half the ring, instead of one 16-warp
  // block; the two blocks' start-up and fragment ends do not wait on each
  // other.
  static constexpr int kMinBlocks = kPair ? 2 : 1;
  // Balanced shares that charge each segment boundary this many units (a
  // fragment end, a query reload and, usually, the segment's merge): the
  // paired short decodes (60, measured best among 1..220 on the 8-sequence
  // E4M3 decode), the sliding-window kernels (60: the 131K verify with a
  // 2048-token window 34.3 -> 30.9 us; from 130 on, the shares get too small
  // for the constant-time partial count) and the 24-row INT8_ROW verify (120:
  // 567 -> 556 us on the 131K verify).  The other kernels balance units: the
  // same charge made the 24-row E4M3 verify's page loop compile 8 % slower,
  // and the 32-row one gained nothing.
  static constexpr int kFragUnits =
      kPair ? 60 : ((KVT == PQKV_KV_INT8_ROW && NT == 3) ? 120 : (kWideTree ? 60 : 0));
  static_assert(!kPair || (NT == 1 && KVT != PQKV_KV_FP16), "paired blocks: 8-row 8-bit decode only");
  static constexpr int kThreads = kW * 32;
  static constexpr int kLines = (KVT == PQKV_KV_FP16) ? 64 : 32;   // 128-B lines per tile
  static constexpr int kTileBytes = kLines * 128;
  static constexpr int kStagesPerWarp =
      (KVT == PQKV_KV_FP16 || kPair || (kWideTree && (NT == 2 || NT == 3 || NT == 4)))
          ? 2
          : (kW <= 8 ? 4 : (kW == 12 ? 3 : 2));
  static constexpr int kStages = kW * kStagesPerWarp;
  static constexpr int kRP = 8 * NT;                               // padded query rows
  static constexpr int kQfBytes = 8 * NT * 32 * 8;
  // shared-memory carve-up (offsets from a 1024-aligned base)
  static constexpr int kRingOff = 0;
  static constexpr int kOOff = kRingOff + kStages * kTileBytes;
  // Fragment-end combine of the warps' O.  8 and 16 query rows (kTree): a
  // tree (in each round the upper half of the remaining warps hands its O to
  // the lower half, kW / 2 buffers in the first round; warp 0 writes the
  // result from registers), or for 8 rows the flat combine below; these
  // kernels also share the one-pass merge and the early fragment set-up.
  // 24 and 32 rows: groups of four warps take turns on a group
  // buffer (8 warps: one group), then the group buffers are added in fixed
  // order -- the 24-row page loop compiled slower with the tree epilogue,
  // and the 32-row kernel has no shared memory left for its buffers.
  // kWideTree: the sliding-window kernel, a separate instantiation: the tree
  // (the flat combine for 24 rows) for 24 and 32 rows too (8-bit formats),
  // and two ring stages per warp for 16, 24 and 32 rows so its buffers and
  // per-sequence array fit
  static constexpr bool kTree = NT <= 2 || (kWideTree && KVT != PQKV_KV_FP16);
  // 8 query rows (not the sliding-window kernels) and the 24-row 8-bit
  // sliding-window kernel: instead of the tree every warp writes its O to a
  // buffer of its own, and after one barrier every thread adds one float4 of
  // the output over the warps (the window kernel takes two ring stages per
  // warp to make room: 29.7 -> 27.3 us on the 131K verify with a 2048-token
  // window)
  static constexpr bool kFlat =
      (NT == 1 && !kWideTree) || (kWideTree && NT == 3 && KVT != PQKV_KV_FP16);
  static constexpr int kCombGroups = kW >= 12 ? kW / 4 : 1;
  static constexpr int kCombSize = kW / kCombGroups;
  static constexpr int kOBytes = kRP * kHeadDim * 4;     // one buffer
  static constexpr int kOBuffers = kFlat ? kW : (kTree ? kW / 2 : kCombGroups);
  static constexpr int kMLOff = kOOff + kOBuffers * kOBytes;
  static constexpr int kQOff = kMLOff + kW * 2 * kRP * 4;
  static constexpr int kQfOff = kQOff + kRP * kHeadDim * 2;
  // INT8_ROW: the 32 fp16 row scales (16 K, 16 V) of each stage's (page, kv-head)
  static constexpr bool kRowScaled = (KVT == PQKV_KV_INT8_ROW);
  static constexpr int kScOff = kQfOff + kQfBytes;
  static constexpr int kScBytes = kRowScaled ? kStages * 64 : 0;
  static constexpr int kBarOff = kScOff + kScBytes;
  static constexpr int kMiscOff = kBarOff + kStages * 8;
  // 32 query rows (NT 4) are short of registers: there the per-row causal
  // limits live in shared memory and the rescale test recomputes its
  // threshold from the reference maximum instead of keeping it per row
  // (fewer spills; with fewer rows the registers are faster)
  static constexpr bool kRowsInSmem = (NT == 4);
  static constexpr int kMiscBytes = 64 + kW * 4 + 2 * kRP * 4 + 128 + (kRowsInSmem ? kRP * 4 : 0);
  static constexpr int kPreOff = kMiscOff + kMiscBytes;
  static __host__ __device__ constexpr int smem_bytes(int num_seqs) {
    return kPreOff + (2 * num_seqs + 1) * 4 + 1024;
  }
  static_assert(kStages % kW == 0, "each ring stage must belong to one warp");
  // the largest launch (PQKV_MAX_SEQS sequences; the sliding-window kernel
  // also keeps one int per sequence) fits the 227 KB a block may opt into
  static_assert(smem_bytes(PQKV_MAX_SEQS) + (kWideTree ? 4 * PQKV_MAX_SEQS : 0) <= 232448,
                "shared memory of the largest launch");
  static_assert(kW % kCombGroups == 0, "whole combine groups");
  static_assert(kOBytes / 4 >= 1024, "the merge's slot list (<= 1024 blocks) must fit the O buffer");
};

// Initial reference maximum of a row: finite, so exp2(score - ref) needs no
// special case, and far below any score (the first page always raises it).
constexpr float kNoScore = -1.0e30f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Work split: fragments of the concatenated (sequence, kv-head) page list
// ---------------------------------------------------------------------------
struct Frag {
  int s, h, pg0, pg1;   // sequence, kv-head, page range [pg0, pg1)
  int seg;              // s * H + h
  int64_t a, b;         // the segment's span in the concatenated list
};

// kCost: the balanced shares equalise cost rather than units, where every
// segment after the first adds F units of cost at its start.  A block whose
// share crosses into the next segment pays a fragment end and a query reload;
// charging them keeps such blocks from finishing last.  Deterministic: the
// shares depend only on the sequence lengths and the grid.
template <bool kCost> struct SplitCost {};
template <> struct SplitCost<true> {
  int F;                // cost units charged per segment boundary
  int64_t Ctot;         // P + F * (B * H - 1)
};

template <bool kCost>
struct SplitT : SplitCost<kCost> {
  const int* pre;       // [B + 1] page prefix per sequence
  int B, H;
  int64_t P;            // total (page, kv-head) units
  int C;                // blocks
  int k;                // 0 = balanced

  // cost of unit x: x plus F for every segment starting at or before x but
  // the first (segments are never empty here: every sequence holds a key)
  __device__ int64_t cost(int64_t x) const {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)pre[mid] * H <= x) lo = mid; else hi = mid - 1;
    }
    const int64_t h = (x - (int64_t)pre[lo] * H) / pages(lo);
    return x + (int64_t)this->F * ((int64_t)lo * H + h);
  }
  // first unit of block c's share
  __device__ int64_t start(int c) const {
    if constexpr (!kCost) {
      return (int64_t)c * P / C;
    } else {
      const int F = this->F;
      if (c <= 0) return 0;
      if (c >= C) return P;
      const int64_t T = ((int64_t)c * this->Ctot + C - 1) / C;   // smallest cost in the share
      int lo = 0, hi = B - 1;                                  // sequence of cost T
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)pre[mid] * H + (int64_t)F * mid * H <= T) lo = mid; else hi = mid - 1;
      }
      const int64_t base = (int64_t)pre[lo] * H, np = pages(lo);
      const int64_t rel = T - base - (int64_t)F * lo * H;
      const int64_t h = rel / (np + F), off = rel - h * (np + F);
      if (h >= H) return (int64_t)pre[lo + 1] * H;           // cost between sequences
      return base + h * np + (off < np ? off : np);           // in a segment, or just after it
    }
  }
  // the block whose (non-empty) share holds unit x
  __device__ __forceinline__ int cta_of(int64_t x) const {
    if constexpr (!kCost) return (int)(((x + 1) * C - 1) / P);
    else return (int)(cost(x) * C / this->Ctot);
  }
  __device__ __forceinline__ int pages(int s) const { return pre[s + 1] - pre[s]; }

  // number of partial results of segment seg
  __device__ int count(int seg, int64_t a, int64_t b) const {
    if (k > 0) return min(k, pages(seg / H));
    int n = 0;
    for (int64_t x = a; x < b; x = start(cta_of(x) + 1)) ++n;
    return n;
  }

  // n / d for n >= 0, d > 0, in 32-bit arithmetic when both fit (a 64-bit
  // division is a long dependent chain, and one thread computes these while
  // the block waits at the fragment end)
  static __device__ __forceinline__ int64_t udiv(int64_t n, int64_t d) {
    if (((uint64_t)n | (uint64_t)d) <= 0xFFFFFFFFull) return (uint32_t)n / (uint32_t)d;
    return n / d;
  }
  // cta_of with those divisions (the same values)
  __device__ __forceinline__ int cta_of_q(int64_t x) const {
    if constexpr (!kCost) {
      return (int)udiv((x + 1) * C - 1, P);
    } else {
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)pre[mid] * H <= x) lo = mid; else hi = mid - 1;
      }
      const int64_t h = udiv(x - (int64_t)pre[lo] * H, pages(lo));
      const int64_t cx = x + (int64_t)this->F * ((int64_t)lo * H + h);
      return (int)udiv(cx * C, this->Ctot);
    }
  }

  // The same in constant time when every block's share is non-empty (P >= C):
  // the blocks holding units of [a, b) are then exactly first .. first + n - 1.
  __device__ __forceinline__ int count_fast(int seg, int64_t a, int64_t b, int& first) const {
    if (k > 0) {
      first = 0;
      return min(k, pages(seg / H));
    }
    // with equal shares every share is non-empty when P >= C; with cost
    // shares when every share spans at least F + 1 cost values (a share can
    // then not fall inside the F-value gap a segment boundary adds);
    // otherwise walk the blocks
    bool walk;
    if constexpr (kCost) walk = this->Ctot < (int64_t)(this->F + 1) * C;
    else walk = P < C;
    if (walk) {
      first = -1;
      return count(seg, a, b);
    }
    first = cta_of_q(a);
    return cta_of_q(b - 1) - first + 1;
  }
};

template <bool kCost>
struct FragIterT {
  SplitT<kCost> sp;
  int c;
  int64_t x, e;
  int s;
  bool fixed_done;

  __device__ void init(const SplitT<kCost>& split, int cta) {
    sp = split;
    c = cta;
    s = 0;
    fixed_done = false;
    if (sp.k == 0) {
      x = sp.start(c);
      e = sp.start(c + 1);
    }
  }
  // the same with the block's share [x0, x1) already known
  __device__ void init_range(const SplitT<kCost>& split, int cta, int64_t x0, int64_t x1) {
    sp = split;
    c = cta;
    s = 0;
    fixed_done = false;
    x = x0;
    e = x1;
  }

  __device__ bool next(Frag& f) {
    if (sp.k > 0) {
      if (fixed_done) return false;
      fixed_done = true;
      const int seg = c / sp.k, p = c % sp.k;
      if (seg >= sp.B * sp.H) return false;
      f.s = seg / sp.H;
      f.h = seg % sp.H;
      const int np = sp.pages(f.s);
      f.pg0 = (int)((int64_t)p * np / sp.k);
      f.pg1 = (int)((int64_t)(p + 1) * np / sp.k);
      f.seg = seg;
      f.a = (int64_t)sp.pre[f.s] * sp.H + (int64_t)f.h * np;
      f.b = f.a + np;
      return f.pg1 > f.pg0;
    }
    if (x >= e) return false;
    while ((int64_t)sp.pre[s + 1] * sp.H <= x) ++s;
    const int np = sp.pages(s);
    const int64_t base = (int64_t)sp.pre[s] * sp.H;
    const int64_t off = x - base;
    f.s = s;
    f.h = (int)(off / np);
    f.pg0 = (int)(off % np);
    f.seg = s * sp.H + f.h;
    f.a = base + (int64_t)f.h * np;
    f.b = f.a + np;
    const int64_t fe = min(e, f.b);
    f.pg1 = f.pg0 + (int)(fe - x);
    x = fe;
    return true;
  }
};

using Split = SplitT<false>;
using FragIter = FragIterT<false>;

static_assert(sizeof(FragIterT<true>) + sizeof(Frag) <= 128, "iterator state must fit its smem slot");

// ---------------------------------------------------------------------------
// Per-page work of one consumer warp
// ---------------------------------------------------------------------------
// Physical head dims of the 4 K elements a lane feeds to k-step kk of QK^T
// (order: b0.lo, b0.hi, b1.lo, b1.hi); they are 4 consecutive dims.
template <int KVT>
__device__ __forceinline__ int k_dim_base(int t, int kk) {
  if (KVT == PQKV_KV_FP16) {
    const int c1 = (t & 1) | ((t & 2) << 1);     // chunks {0,1,4,5} of a 64-dim line
    const int q = kk >> 1;                        // which of the lane's 4 chunks
    const int lh = q >> 1;                        // line half (dims 0-63 / 64-127)
    const int ch = c1 + ((q & 1) << 1);
    return 64 * lh + 8 * ch + 4 * (kk & 1);
  } else {
    return 32 * t + 4 * kk;
  }
}

__device__ __forceinline__ uint4 lds128(const uint8_t* base, int line, int chunk) {
  return *reinterpret_cast<const uint4*>(base + line * 128 + ((chunk ^ (line & 7)) << 4));
}

// The Q^T B-fragments live in a shared table [4][NT][32] of 16-byte entries:
// a lane's fragments of k-steps 2*k2 and 2*k2 + 1 of one row tile side by
// side, so one 16-byte load serves two k-steps.
template <int NT>
struct QFrags {
  const uint4* tab;
  __device__ __forceinline__ uint4 get2(int k2, int nt, int lane) const {
    return tab[(k2 * NT + nt) * 32 + lane];
  }
};

template <int KVT>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if (KVT == PQKV_KV_FP8_E4M3) e4m3_word(w, lo, hi);
  else int8_word(w, lo, hi);
}

// S^T[16 tokens][8*NT rows] = K Q^T for one page tile.  Lane (g, t) feeds the
// K rows of tokens g and g+8 and gets back S^T for tokens (g, g+8) and query
// rows (8nt + 2t, 8nt + 2t + 1).  Codes are widened just before each k-step.
template <int KVT, int NT>
__device__ __forceinline__ void page_qk(const uint8_t* T, int g, int t, int lane,
                                        const QFrags<NT>& qf, float (&sc)[NT][4]) {
  if (KVT == PQKV_KV_FP16) {
    const int c1 = (t & 1) | ((t & 2) << 1);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int lh = q >> 1, ch = c1 + ((q & 1) << 1);
      const uint4 x = lds128(T, 2 * g + lh, ch);
      const uint4 y = lds128(T, 2 * (g + 8) + lh, ch);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 b = qf.get2(q, nt, lane);
        mma_16816(sc[nt], x.x, y.x, x.y, y.y, b.x, b.y);
        mma_16816(sc[nt], x.z, y.z, x.w, y.w, b.z, b.w);
      }
    }
  } else {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint4 x = lds128(T, g, 2 * t + half), y = lds128(T, g + 8, 2 * t + half);
      const uint32_t wx[4] = {x.x, x.y, x.z, x.w}, wy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        uint4 b[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) b[nt] = qf.get2(2 * half + j2, nt, lane);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * j2 + jj;
          uint32_t a0, a1, a2, a3;
          dequant_word<KVT>(wx[j], a0, a2);
          dequant_word<KVT>(wy[j], a1, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816(sc[nt], a0, a1, a2, a3, jj ? b[nt].z : b[nt].x, jj ? b[nt].w : b[nt].y);
        }
      }
    }
  }
}

// Zero the halves of tokens at or beyond `valid` (tokens 2t, 2t+1 in a0/a1 and
// 2t+8, 2t+9 in a2/a3 of a V^T fragment).
struct VMask {
  uint32_t m01, m89;
  __device__ __forceinline__ void init(int t, int valid) {
    m01 = (2 * t < valid ? 0x0000FFFFu : 0u) | (2 * t + 1 < valid ? 0xFFFF0000u : 0u);
    m89 = (2 * t + 8 < valid ? 0x0000FFFFu : 0u) | (2 * t + 9 < valid ? 0xFFFF0000u : 0u);
  }
};

// O^T[128 dims][8*NT rows] += V^T P^T for one page tile.  V^T m-tile mt holds
// dims 16g + 2mt (A rows g) and 16g + 2mt + 1 (A rows g + 8) of tokens
// (2t, 2t+1) and (2t+8, 2t+9).  When `masked`, tokens past the sequence end
// are zeroed: their probability is 0, but a stale NaN code times 0 is NaN.
template <int KVT, int NT, class AfterLoads>
__device__ __forceinline__ void page_pv(const uint8_t* T, int g, int t,
                                        const uint32_t (&pb)[NT][2], bool masked, const VMask& vm,
                                        float (&o)[8][NT][4], AfterLoads after_loads) {
  auto mma_mt = [&](int mt, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
    if (masked) {
      a0 &= vm.m01;
      a1 &= vm.m01;
      a2 &= vm.m89;
      a3 &= vm.m89;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
  };
  if (KVT == PQKV_KV_FP16) {
    const int lh = g >> 2, ch = 2 * (g & 3);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint4 A = lds128(T, 32 + 2 * (2 * t) + lh, ch + hh);
      const uint4 B = lds128(T, 32 + 2 * (2 * t + 1) + lh, ch + hh);
      const uint4 C = lds128(T, 32 + 2 * (2 * t + 8) + lh, ch + hh);
      const uint4 D = lds128(T, 32 + 2 * (2 * t + 9) + lh, ch + hh);
      const uint32_t a[4] = {A.x, A.y, A.z, A.w}, b[4] = {B.x, B.y, B.z, B.w};
      const uint32_t c[4] = {C.x, C.y, C.z, C.w}, d[4] = {D.x, D.y, D.z, D.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        mma_mt(4 * hh + j, __byte_perm(a[j], b[j], 0x5410), __byte_perm(a[j], b[j], 0x7632),
               __byte_perm(c[j], d[j], 0x5410), __byte_perm(c[j], d[j], 0x7632));
    }
  } else {
    const uint4 A = lds128(T, 16 + 2 * t, g), B = lds128(T, 17 + 2 * t, g);
    const uint4 C = lds128(T, 24 + 2 * t, g), D = lds128(T, 25 + 2 * t, g);
    const uint32_t a[4] = {A.x, A.y, A.z, A.w}, b[4] = {B.x, B.y, B.z, B.w};
    const uint32_t c[4] = {C.x, C.y, C.z, C.w}, d[4] = {D.x, D.y, D.z, D.w};
    after_loads();
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      if (KVT == PQKV_KV_FP8_E4M3) {
        // the two halves of each interleaved word feed the conversions directly
        uint32_t x0, x1, x2, x3;
        e4m3_word(__byte_perm(a[wi], b[wi], 0x5140), x0, x1);
        e4m3_word(__byte_perm(c[wi], d[wi], 0x5140), x2, x3);
        mma_mt(2 * wi, x0, x1, x2, x3);
        e4m3_word(__byte_perm(a[wi], b[wi], 0x7362), x0, x1);
        e4m3_word(__byte_perm(c[wi], d[wi], 0x7362), x2, x3);
        mma_mt(2 * wi + 1, x0, x1, x2, x3);
      } else {
        mma_mt(2 * wi, i8pair(__byte_perm(a[wi], b[wi], 0x0400)),
               i8pair(__byte_perm(a[wi], b[wi], 0x0501)), i8pair(__byte_perm(c[wi], d[wi], 0x0400)),
               i8pair(__byte_perm(c[wi], d[wi], 0x0501)));
        mma_mt(2 * wi + 1, i8pair(__byte_perm(a[wi], b[wi], 0x0602)),
               i8pair(__byte_perm(a[wi], b[wi], 0x0703)), i8pair(__byte_perm(c[wi], d[wi], 0x0602)),
               i8pair(__byte_perm(c[wi], d[wi], 0x0703)));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Programmatic dependent launch (see pqkv_common.cuh) for every instantiation
// but two, which are launched without it: the plain 24-row E4M3 kernel (with
// the grid-dependency wait in it, its page loop compiled about 1 us slower,
// and its launches gained nothing from an early start) and the paired
// short-decode kernel (back-to-back decodes ran 0.3-0.5 us faster without).
template <int KVT, int NT, class PP, bool kPair>
constexpr bool attention_uses_pdl() {
  constexpr bool kPlain = std::is_same<PP, AttnParams>::value;
  return !(kPlain && ((KVT == PQKV_KV_FP8_E4M3 && NT == 3 && !kPair) || kPair));
}

template <class PP> struct IsPartial { static constexpr bool value = false; };
template <> struct IsPartial<AttnPartialParams> { static constexpr bool value = true; };
template <class PP> struct IsWaitTest { static constexpr bool value = false; };
template <> struct IsWaitTest<AttnWaitTestParams> { static constexpr bool value = true; };
template <class PP> struct IsWindow { static constexpr bool value = false; };
template <> struct IsWindow<AttnWindowParams> { static constexpr bool value = true; };
constexpr uint64_t kTestWaitLimitNs = 1000000ull;   // 1 ms in the wait test

template <int KVT, int NT, class PP = AttnParams, bool kPair = false>
__global__ void __launch_bounds__(AttnCfg<KVT, NT, kPair>::kThreads,
                                  AttnCfg<KVT, NT, kPair>::kMinBlocks)
    paged_attention_kernel(const __grid_constant__ CUtensorMap map, const PP p) {
  using Cfg = AttnCfg<KVT, NT, kPair, IsWindow<PP>::value>;
  constexpr bool kPartial = IsPartial<PP>::value;
  constexpr bool kWaitTest = IsWaitTest<PP>::value;
  constexpr bool kWin = IsWindow<PP>::value;
  constexpr uint64_t kLimitNs = kWaitTest ? kTestWaitLimitNs : kWaitLimitNs;
  constexpr int W = Cfg::kW, S = Cfg::kStages, SPW = Cfg::kStagesPerWarp, RP = Cfg::kRP;
  constexpr int nthr = W * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem + Cfg::kRingOff;
  float* sO = reinterpret_cast<float*>(smem + Cfg::kOOff);
  float* sML = reinterpret_cast<float*>(smem + Cfg::kMLOff);
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem + Cfg::kQOff);
  uint4* sQf = reinterpret_cast<uint4*>(smem + Cfg::kQfOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  int* misc = reinterpret_cast<int*>(smem + Cfg::kMiscOff);
  volatile int* abort_flag = misc + 0;
  volatile int* merge_flag = misc + 1;
  volatile int* has_frag = misc + 2;
  volatile int* frag_cnt = misc + 3;
  volatile int* frag_first = misc + 4;    // first block of the fragment's segment (or -1)
  float* sWarp = reinterpret_cast<float*>(misc + 16);          // [W] per-warp scratch
  float* sMrow = sWarp + W;                                    // [RP]
  float* sLrow = sMrow + RP;                                   // [RP]
  // cost shares (not in the partial mode, where a sequence may hold no key
  // and a segment may be empty; in the sliding-window mode every sequence
  // reads at least one page)
  constexpr bool kCostSplit = Cfg::kFragUnits > 0 && !kPartial;
  FragIterT<kCostSplit>* sit = reinterpret_cast<FragIterT<kCostSplit>*>(sLrow + RP);
  Frag* sf = reinterpret_cast<Frag*>(sit + 1);
  int* pre = reinterpret_cast<int*>(smem + Cfg::kPreOff);
  int* sLim = reinterpret_cast<int*>(smem + Cfg::kPreOff - RP * 4);   // [RP] if kRowsInSmem
  int* slen = pre + p.num_seqs + 1;
  int* sfp = slen + p.num_seqs;     // sliding window: each sequence's first page read

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int B = p.num_seqs, H = p.num_kv_heads;
  if constexpr (attention_uses_pdl<KVT, NT, PP, kPair>()) {
    grid_dependency_wait();
    grid_dependents_launch();
  }

  // -- per-sequence lengths (clamped into the valid range) and page prefix
  for (int s = tid; s < B; s += nthr) {
    int L = p.seq_lens[s];
    const int Lmax = p.bt_stride * kPageSize;
    const int Lmin = kPartial ? 0 : p.q_len;    // a rank's share of keys may be empty
    if (L < Lmin || L > Lmax) {
      if (blockIdx.x == 0) report(p.status, PQKV_DEV_SEQ_RANGE);
      L = max(Lmin, min(L, Lmax));
    }
    slen[s] = L;
    pre[s + 1] = (L + kPageSize - 1) / kPageSize;
    if constexpr (kWin) {
      // the first key any query of the sequence sees, and its page
      const int fp = max(0, L - p.q_len - p.window + 1) / kPageSize;
      sfp[s] = fp;
      pre[s + 1] -= fp;
    }
  }
  if (tid == 0) {
    pre[0] = 0;
    misc[0] = 0;
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < B; base += 32) {
      int v = (base + lane < B) ? pre[base + lane + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (base + lane < B) pre[base + lane + 1] = run + v;
      run += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();

  if constexpr (kPartial) {
    // rows of sequences with no local keys: O = 0, LSE = -inf
    for (int s = blockIdx.x; s < B; s += gridDim.x) {
      if (slen[s] != 0) continue;
      const int64_t r0 = (int64_t)s * p.q_len * p.num_q_heads;
      const int nr = p.q_len * p.num_q_heads;
      for (int idx = tid; idx < nr * kHeadDim; idx += nthr) p.out_o[r0 * kHeadDim + idx] = 0.f;
      for (int idx = tid; idx < nr; idx += nthr) p.out_lse[r0 + idx] = -INFINITY;
    }
  }

  SplitT<kCostSplit> sp;
  sp.pre = pre;
  sp.B = B;
  sp.H = H;
  sp.P = (int64_t)pre[B] * H;
  sp.C = gridDim.x;
  sp.k = p.num_splits;
  if constexpr (kCostSplit) {
    sp.F = Cfg::kFragUnits;
    sp.Ctot = sp.P + (int64_t)sp.F * ((int64_t)B * H - 1);
  }

  // -- this block's contiguous range [x0, x1) of the (page, kv-head) unit list
  int64_t x0 = 0, x1 = 0;
  if (sp.k == 0) {
    x0 = sp.start(blockIdx.x);
    x1 = sp.start(blockIdx.x + 1);
  } else {
    const int seg = blockIdx.x / sp.k, q = blockIdx.x % sp.k;
    if (seg < B * H) {
      const int s0 = seg / H, np = sp.pages(s0);
      const int64_t a = (int64_t)pre[s0] * H + (int64_t)(seg % H) * np;
      x0 = a + (int64_t)q * np / sp.k;
      x1 = a + (int64_t)(q + 1) * np / sp.k;
    }
  }
  const int ntot = (int)(x1 - x0);

  // Tree-combine kernels whose query rows take one vector per thread (8 and
  // 16 rows): the query rows and scales of the block's first segment are read
  // now, beside the first block-table lookups.
  constexpr bool kEarlyQ = Cfg::kTree && RP * 16 <= nthr;
  uint4 q_early = make_uint4(0, 0, 0, 0);
  int early_seg = -1;
  float ks0 = 1.f, vs0 = 1.f;
  int qpos0 = 0;
  if constexpr (kEarlyQ) {
    if (ntot > 0) {
      int s0 = 0, h0 = 0;
      if (sp.k == 0) {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if ((int64_t)pre[mid] * H <= x0) lo = mid; else hi = mid - 1;
        }
        s0 = lo;
        h0 = (int)((x0 - (int64_t)pre[lo] * H) / sp.pages(lo));
      } else {
        const int seg = blockIdx.x / sp.k;
        s0 = seg / H;
        h0 = seg % H;
      }
      early_seg = s0 * H + h0;
      if constexpr (KVT != PQKV_KV_FP16 && KVT != PQKV_KV_INT8_ROW) {
        const int sh = p.scale_per_head ? h0 : 0;
        ks0 = __ldg(p.k_scale + sh);
        vs0 = __ldg(p.v_scale + sh);
      }
      if constexpr (kPartial) qpos0 = p.q_pos[s0];
      if (tid < RP * 16) {
        const int r = tid >> 4, c8 = tid & 15;
        if (r < p.rows) {
          const int i = r / p.group, gh = r % p.group;
          const int64_t row = ((int64_t)s0 * p.q_len + i) * p.num_q_heads + h0 * p.group + gh;
          q_early = __ldg(reinterpret_cast<const uint4*>(p.q + row * kHeadDim) + c8);
        }
      }
    }
  }

  // -- tile feed: warp w streams the block's pages w, w+W, w+2W, ... into its
  //    own stages.  Its u-th page is i = w + u*W; lane l caches the kv-head
  //    and pool page of the warp's pages u in [ubase, ubase+32) (cur) and the
  //    next 32 (nxt).
  const uint64_t policy = l2_evict_first_policy();
  // INT8_ROW: two kv-heads' row scales share a 128-byte line and are read by
  // different blocks at about the same time; they stay in L2 for the second
  uint64_t scale_policy = policy;
  if constexpr (Cfg::kRowScaled) scale_policy = l2_evict_last_policy();
  if (tid == 0) prefetch_tensormap(&map);
  auto lookup = [&](int u, int& id, int& h) {
    const int i = warp + u * W;
    id = 0;
    h = 0;
    if (i >= ntot) return;
    const int64_t x = x0 + i;
    int lo = 0, hi = B - 1;                       // sequence holding unit x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)pre[mid] * H <= x) lo = mid; else hi = mid - 1;
    }
    const int np = pre[lo + 1] - pre[lo];
    const int64_t off = x - (int64_t)pre[lo] * H;
    h = (int)(off / np);
    const int pg = (int)(off % np);
    if constexpr (kWin)
      id = __ldg(p.block_table + (int64_t)lo * p.bt_stride + sfp[lo] + pg);
    else
      id = __ldg(p.block_table + (int64_t)lo * p.bt_stride + pg);
    if (id < 0 || (int64_t)id >= p.num_pages) report(p.status, PQKV_DEV_PAGE_RANGE);
  };
  int cur_id, cur_h, nxt_id, nxt_h, ubase = 0;
  lookup(lane, cur_id, cur_h);
  lookup(32 + lane, nxt_id, nxt_h);
  int issued_u = 0;                      // pages of this warp issued so far
  int skipped_u = -1;                    // wait test: the page whose copy was never issued
  auto issue_next = [&]() {
    const int u = issued_u;
    const int i = warp + u * W;
    if (i >= ntot) return;
    if (u - ubase >= 32) {
      cur_id = nxt_id;
      cur_h = nxt_h;
      ubase += 32;
      lookup(ubase + 32 + lane, nxt_id, nxt_h);
    }
    const int id = __shfl_sync(0xffffffffu, cur_id, u - ubase);
    const int h = __shfl_sync(0xffffffffu, cur_h, u - ubase);
    if constexpr (kWaitTest) {
      if ((int)blockIdx.x == p.skip_block && i == p.skip_page) {
        skipped_u = u;
        issued_u = u + 1;
        return;
      }
    }
    if (lane == 0) {
      const int stage = i % S;
      if constexpr (Cfg::kRowScaled) {
        // the page's 32 fp16 row scales travel with its tile (one bulk copy on
        // the same barrier); a page id outside the pool (reported, its codes
        // read as zeros) gets zero scales, written before the barrier is armed
        uint16_t* dst = reinterpret_cast<uint16_t*>(smem + Cfg::kScOff) + stage * 32;
        const bool id_ok = id >= 0 && (int64_t)id < p.num_pages;
        if (!id_ok) {
#pragma unroll
          for (int k = 0; k < 4; ++k) reinterpret_cast<uint4*>(dst)[k] = make_uint4(0, 0, 0, 0);
        }
        mbar_arrive_expect_tx(&full[stage], Cfg::kTileBytes + (id_ok ? 64 : 0));
        tma_load_4d(ring + stage * Cfg::kTileBytes, &map, &full[stage], 0, 0, h, id, policy);
        if (id_ok)
          bulk_load(dst,
                    reinterpret_cast<const uint16_t*>(p.k_scale) +
                        ((int64_t)id * p.num_kv_heads + h) * 32,
                    64, &full[stage], scale_policy);
      } else {
        mbar_arrive_expect_tx(&full[stage], Cfg::kTileBytes);
        tma_load_4d(ring + stage * Cfg::kTileBytes, &map, &full[stage], 0, 0, h, id, policy);
      }
    }
    issued_u = u + 1;
  };
#pragma unroll 1
  for (int k = 0; k < SPW; ++k) issue_next();
  if constexpr (kEarlyQ) {
    if (early_seg >= 0 && tid < RP * 16) reinterpret_cast<uint4*>(sQ)[tid] = q_early;
  }

  // -- walk the fragments of the block's range in lock step
  if (tid == 0) {
    if constexpr (Cfg::kTree) sit->init_range(sp, blockIdx.x, x0, x1);
    else sit->init(sp, blockIdx.x);
  }
  uint32_t n0 = 0;
  int consumed_u = 0;
  int cur_seg = -1, cur_L = 0;
  QFrags<NT> qf;
  qf.tab = sQf;
  float qk_scale = 0.f, inv_qk_scale = 0.f, v_mult = 1.f;
  int lim[NT][2];
  int lim_min = 0;
  bool dead = false;

  // Launched as a cluster (one segment split over at most 8 blocks; the FP16
  // 8-row kernel only, the others have no registers to spare for it): each
  // block leaves its combined O, m and l in its idle ring, and
  // block 0 of the cluster merges them through distributed shared memory at
  // the end, instead of global partials and a ticket.
  constexpr bool kClusterMerge = Cfg::kFlat && !kPair && !kWin && KVT == PQKV_KV_FP16;
  uint32_t ncl = 1;
  if constexpr (kClusterMerge) ncl = cluster_nctarank();
  const bool clu = kClusterMerge && ncl > 1;
  bool clu_written = false;
  for (;;) {
    if (tid == 0) *has_frag = sit->next(*sf) ? 1 : 0;
    __syncthreads();
    if (!*has_frag) break;
    const int f_s = sf->s, f_h = sf->h, f_pg0 = sf->pg0, f_pg1 = sf->pg1, f_seg = sf->seg;
    // ---- (re)load the query rows of this (sequence, kv-head)
    if (f_seg != cur_seg) {
      const int L = slen[f_s];
      // tree-combine kernels: the scales (and the partial mode's query
      // position) are read beside the query rows, not after the barrier
      float ks_e = 1.f, vs_e = 1.f;
      int qpos_e = 0;
      const bool q_read = kEarlyQ && f_seg == early_seg;
      if constexpr (Cfg::kTree) {
        if (q_read) {
          ks_e = ks0;
          vs_e = vs0;
          qpos_e = qpos0;
        } else {
          if constexpr (KVT != PQKV_KV_FP16 && KVT != PQKV_KV_INT8_ROW) {
            const int sh = p.scale_per_head ? f_h : 0;
            ks_e = __ldg(p.k_scale + sh);
            vs_e = __ldg(p.v_scale + sh);
          }
          if constexpr (kPartial) qpos_e = p.q_pos[f_s];
        }
      }
      for (int v = tid; v < RP * 16 && !q_read; v += nthr) {
        const int r = v >> 4, c8 = v & 15;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < p.rows) {
          const int i = r / p.group, gh = r % p.group;
          const int64_t row = ((int64_t)f_s * p.q_len + i) * p.num_q_heads + f_h * p.group + gh;
          val = __ldg(reinterpret_cast<const uint4*>(p.q + row * kHeadDim) + c8);
        }
        reinterpret_cast<uint4*>(sQ)[v] = val;
      }
      __syncthreads();
      if (warp == 0) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int db = k_dim_base<KVT>(t, kk);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            reinterpret_cast<uint2*>(sQf)[(((kk >> 1) * NT + nt) * 32 + lane) * 2 + (kk & 1)] =
                *reinterpret_cast<const uint2*>(sQ + (8 * nt + g) * kHeadDim + db);
        }
      }
      const int sh = p.scale_per_head ? f_h : 0;
      if constexpr (KVT == PQKV_KV_FP16 || KVT == PQKV_KV_INT8_ROW) {
        // FP16 has no scale; INT8_ROW applies its row scales per token
        qk_scale = p.sm_scale_log2;
        v_mult = 1.f;
      } else {
        const float ks = Cfg::kTree ? ks_e : __ldg(p.k_scale + sh);
        const float vs = Cfg::kTree ? vs_e : __ldg(p.v_scale + sh);
        if (!(ks > 0.f && ks <= 3.4e38f && vs > 0.f && vs <= 3.4e38f))
          report(p.status, PQKV_DEV_BAD_SCALE);
        qk_scale = ks * p.sm_scale_log2;
        v_mult = vs;
      }
      inv_qk_scale = 1.f / qk_scale;
      if constexpr (kPartial) lim_min = Cfg::kTree ? qpos_e : p.q_pos[f_s];
      else lim_min = L - p.q_len;
      // causal limit per row: the last key position row r may see
      if constexpr (Cfg::kRowsInSmem) {
        for (int r = tid; r < RP; r += nthr)
          sLim[r] = r < p.rows ? lim_min + r / p.group : 0x7fffffff;
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int r = 8 * nt + 2 * t + c;
            lim[nt][c] = r < p.rows ? lim_min + r / p.group : 0x7fffffff;
          }
      }
      cur_seg = f_seg;
      cur_L = L;
      __syncthreads();
    }

    // ---- stream this warp's pages of the fragment
    float o[8][NT][4];
    float mref[NT][2], lsum[NT][2], thr[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        mref[nt][c] = kNoScore;
        if constexpr (!Cfg::kRowsInSmem) thr[nt][c] = (kNoScore + 8.f) * inv_qk_scale;
        lsum[nt][c] = 0.f;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    }
    const int npg = f_pg1 - f_pg0;
    const int first = (int)((warp - (int)(n0 % W) + W) % W);
    for (int j = first; j < npg; j += W) {
      const uint32_t gi = n0 + j;
      const int stage = gi % S;
      if (!dead) {
        // one try first: the tile is usually there, and the abort flag (a
        // shared-memory read) only matters once some wait has run out
        bool ok = mbar_try_wait(&full[stage], (gi / S) & 1) ||
                  (!*abort_flag && mbar_wait<kLimitNs>(&full[stage], (gi / S) & 1));
        ok = __all_sync(0xffffffffu, ok);       // keep the warp's control flow uniform
        if (!ok) {
          dead = true;
          if (lane == 0) {
            *abort_flag = 1;
            report(p.status, PQKV_DEV_TIMEOUT);
          }
        }
      }
      if (dead) continue;
      const uint8_t* T = ring + stage * Cfg::kTileBytes;
      const int pos0 = (kWin ? sfp[f_s] + f_pg0 + j : f_pg0 + j) * kPageSize;

      // S^T = K Q^T
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
      page_qk<KVT, NT>(T, g, t, lane, qf, sc);
      if constexpr (Cfg::kRowScaled) {
        // INT8_ROW: scores of token g and token g+8 times their K row scales
        // (the stage's scales are [i][K row i, K row i+8, V row i, V row i+8])
        const float2 ks = __half22float2(
            *reinterpret_cast<const __half2*>(smem + Cfg::kScOff + stage * 64 + g * 8));
        const float ks_g = ks.x, ks_g8 = ks.y;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          sc[nt][0] *= ks_g;
          sc[nt][1] *= ks_g;
          sc[nt][2] *= ks_g8;
          sc[nt][3] *= ks_g8;
        }
      }

      // Raw scores; masked -> -inf.  The log2-domain score is sc * qk_scale.
      if (pos0 + kPageSize - 1 > lim_min) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = pos0 + g + ((e & 2) ? 8 : 0);
            const int lm = Cfg::kRowsInSmem ? sLim[8 * nt + 2 * t + (e & 1)] : lim[nt][e & 1];
            if (tok > lm) sc[nt][e] = -INFINITY;
          }
      }
      if constexpr (kWin) {
        // keys before a row's window: row r (limit lm) sees keys > lm - window
        if (pos0 <= lim_min + p.q_len - 1 - p.window) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = pos0 + g + ((e & 2) ? 8 : 0);
              const int lm = Cfg::kRowsInSmem ? sLim[8 * nt + 2 * t + (e & 1)] : lim[nt][e & 1];
              if (tok <= lm - p.window) sc[nt][e] = -INFINITY;
            }
        }
      }
      // The reference maximum of a row only moves when one of its scores
      // exceeds it by more than 8 (probabilities then stay <= 2^8).  Each lane
      // tests its own raw scores against thr = (mref + 8) / qk_scale (with 32
      // rows: raw * qk_scale - mref against 8); only then does the warp form
      // the exact page maximum across the 8 lanes that share a row and
      // rescale.
      bool raise = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float mx = fmaxf(sc[nt][c], sc[nt][c + 2]);
          if constexpr (Cfg::kRowsInSmem) raise |= fmaf(mx, qk_scale, -mref[nt][c]) > 8.f;
          else raise |= mx > thr[nt][c];
        }
      if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float m = fmaxf(sc[nt][c], sc[nt][c + 2]);
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            m *= qk_scale;
            if (m > mref[nt][c] + 8.f) {
              const float fct = ex2(mref[nt][c] - m);
              mref[nt][c] = m;
              if constexpr (!Cfg::kRowsInSmem) thr[nt][c] = (m + 8.f) * inv_qk_scale;
              lsum[nt][c] *= fct;
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) {
                o[mt][nt][c] *= fct;
                o[mt][nt][c + 2] *= fct;
              }
            }
          }
      }
      // probabilities (<= 2^8), row sums, and P^T -> B fragments
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[e] = ex2(fmaf(sc[nt][e], qk_scale, -mref[nt][e & 1]));
        lsum[nt][0] += pr[0] + pr[2];
        lsum[nt][1] += pr[1] + pr[3];
        if constexpr (Cfg::kRowScaled) {
          // O accumulates p_j * vscale_j * vcode_j; the row sums keep p_j
          // alone.  Tokens past the sequence end may hold stale scales, and
          // their probability 0 must not meet a NaN.
          const float2 vs = __half22float2(
              *reinterpret_cast<const __half2*>(smem + Cfg::kScOff + stage * 64 + g * 8 + 4));
          const float vs_g = pos0 + g < cur_L ? vs.x : 0.f;
          const float vs_g8 = pos0 + g + 8 < cur_L ? vs.y : 0.f;
          pb[nt][0] = movmatrix_trans(pack_half2(pr[0] * vs_g, pr[1] * vs_g));
          pb[nt][1] = movmatrix_trans(pack_half2(pr[2] * vs_g8, pr[3] * vs_g8));
        } else {
          pb[nt][0] = movmatrix_trans(pack_half2(pr[0], pr[1]));
          pb[nt][1] = movmatrix_trans(pack_half2(pr[2], pr[3]));
        }
      }
      // O^T += V^T P^T
      {
        const bool tail = pos0 + kPageSize > cur_L;
        VMask vm;
        vm.init(t, cur_L - pos0);
        if constexpr (Cfg::kRowScaled) {
          // the stage is free once its V codes are in registers: refill it
          // with this warp's page S ahead before the PV products
          page_pv<KVT, NT>(T, g, t, pb, tail, vm, o, [&]() {
            __syncwarp();
            fence_proxy_async_smem();
            consumed_u += 1;
            issue_next();
          });
        } else {
          page_pv<KVT, NT>(T, g, t, pb, tail, vm, o, []() {});
        }
      }
      if constexpr (!Cfg::kRowScaled) {
        // the stage is free again: refill it with this warp's page S ahead
        __syncwarp();
        fence_proxy_async_smem();
        consumed_u += 1;
        issue_next();
      }
    }
    n0 += npg;

    if constexpr (!Cfg::kTree) {
    // ---- combine the warps' states of this fragment: every warp publishes
    // its (m, l) per row, then the warps add their rescaled O into their
    // group's shared buffer, the members of a group in turn (all groups at
    // once); the output step adds the group buffers in order.  Fixed order
    // throughout, so the result is deterministic.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float l = lsum[nt][c];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (g == 0) {
          const int r = 8 * nt + 2 * t + c;
          sML[(warp * 2 + 0) * RP + r] = mref[nt][c];
          sML[(warp * 2 + 1) * RP + r] = l;
        }
      }
    __syncthreads();
    float fw[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int r = 8 * nt + 2 * t + c;
        float M = sML[r];
#pragma unroll
        for (int w = 1; w < W; ++w) M = fmaxf(M, sML[(w * 2) * RP + r]);
        fw[nt][c] = ex2(mref[nt][c] - M);
      }
    const int comb_group = Cfg::kCombGroups > 1 ? warp / Cfg::kCombSize : 0;
    const int comb_member = Cfg::kCombGroups > 1 ? warp % Cfg::kCombSize : warp;
#pragma unroll 1
    for (int w = 0; w < Cfg::kCombSize; ++w) {
      if (comb_member == w) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int r = 8 * nt + 2 * t + c;
            float4* dst = reinterpret_cast<float4*>(sO + ((size_t)comb_group * RP + r) * kHeadDim +
                                                    16 * g);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              float4 v = make_float4(o[2 * k4][nt][c] * fw[nt][c], o[2 * k4][nt][c + 2] * fw[nt][c],
                                     o[2 * k4 + 1][nt][c] * fw[nt][c],
                                     o[2 * k4 + 1][nt][c + 2] * fw[nt][c]);
              if (w > 0) {
                const float4 u4 = dst[k4];
                v.x += u4.x;
                v.y += u4.y;
                v.z += u4.z;
                v.w += u4.w;
              }
              dst[k4] = v;
            }
          }
      }
      __syncthreads();
    }

    const int cnt = sp.count(f_seg, sf->a, sf->b);
    const int slot = sp.k > 0 ? (int)blockIdx.x : f_seg + (int)blockIdx.x;
    const int64_t out_row0 = (int64_t)f_s * p.q_len;
    for (int idx = tid; idx < p.rows * kHeadDim; idx += nthr) {
      const int r = idx / kHeadDim, d = idx % kHeadDim;
      float M = sML[r];
#pragma unroll
      for (int w = 1; w < W; ++w) M = fmaxf(M, sML[(w * 2) * RP + r]);
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) l += ex2(sML[(w * 2) * RP + r] - M) * sML[(w * 2 + 1) * RP + r];
      float acc = sO[(size_t)r * kHeadDim + d];
#pragma unroll
      for (int gi = 1; gi < Cfg::kCombGroups; ++gi) acc += sO[((size_t)gi * RP + r) * kHeadDim + d];
      if (cnt == 1) {
        const int i = r / p.group, gh = r % p.group;
        const int64_t orow = (out_row0 + i) * p.num_q_heads + f_h * p.group + gh;
        const float val = l > 0.f ? acc / l * v_mult : 0.f;
        if constexpr (kPartial) {
          p.out_o[orow * kHeadDim + d] = val;
          if (d == 0) p.out_lse[orow] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
        } else {
          p.out[orow * kHeadDim + d] = __half_as_ushort(__float2half_rn(val));
        }
      } else {
        p.part_o[((size_t)slot * RP + r) * kHeadDim + d] = acc;
        if (d == 0) {
          p.part_ml[(size_t)slot * 2 * RP + r] = M;
          p.part_ml[(size_t)slot * 2 * RP + RP + r] = l;
        }
      }
    }
    if (cnt > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int ticket = atomicAdd(p.counters + f_seg, 1);
        *merge_flag = (ticket == cnt - 1);
      }
      __syncthreads();
      if (*merge_flag) {
        __threadfence();
        // gather the segment's partial slots (fixed order) into shared memory
        int* slots = reinterpret_cast<int*>(sO);
        if (tid == 0) {
          int nsl = 0;
          if (sp.k > 0) {
            const int np = sp.pages(f_s);
            for (int q = 0; q < sp.k; ++q)
              if ((int64_t)(q + 1) * np / sp.k > (int64_t)q * np / sp.k)
                slots[nsl++] = f_seg * sp.k + q;
          } else {
            for (int64_t x = sf->a; x < sf->b;) {
              const int cc = sp.cta_of(x);
              slots[nsl++] = f_seg + cc;
              x = sp.start(cc + 1);
            }
          }
        }
        __syncthreads();
        // per-row maximum and normaliser
        if (tid < p.rows) {
          const int r = tid;
          float M = kNoScore;
          for (int q = 0; q < cnt; ++q)
            M = fmaxf(M, __ldcg(p.part_ml + (size_t)slots[q] * 2 * RP + r));
          float l = 0.f;
          for (int q = 0; q < cnt; ++q) {
            const float mq = __ldcg(p.part_ml + (size_t)slots[q] * 2 * RP + r);
            l += ex2(mq - M) * __ldcg(p.part_ml + (size_t)slots[q] * 2 * RP + RP + r);
          }
          sMrow[r] = M;
          sLrow[r] = l;
        }
        __syncthreads();
        const int dq = lane, rg = warp;
        for (int r = rg; r < p.rows; r += W) {
          const float M = sMrow[r];
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int q = 0; q < cnt; ++q) {
            const size_t sl = slots[q];
            const float wq = ex2(__ldcg(p.part_ml + sl * 2 * RP + r) - M);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                                        p.part_o + (sl * RP + r) * kHeadDim) +
                                    dq);
            acc.x += wq * v.x;
            acc.y += wq * v.y;
            acc.z += wq * v.z;
            acc.w += wq * v.w;
          }
          const float inv = sLrow[r] > 0.f ? v_mult / sLrow[r] : 0.f;
          const int i = r / p.group, gh = r % p.group;
          const int64_t orow = (out_row0 + i) * p.num_q_heads + f_h * p.group + gh;
          if constexpr (kPartial) {
            *reinterpret_cast<float4*>(p.out_o + orow * kHeadDim + 4 * dq) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (dq == 0)
              p.out_lse[orow] = sLrow[r] > 0.f ? (M + __log2f(sLrow[r])) * kLn2 : -INFINITY;
          } else {
            __half2 h01 = __floats2half2_rn(acc.x * inv, acc.y * inv);
            __half2 h23 = __floats2half2_rn(acc.z * inv, acc.w * inv);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&h01);
            pk.y = *reinterpret_cast<uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + 4 * dq) = pk;
          }
        }
        if (tid == 0) p.counters[f_seg] = 0;
      }
    }
    } else {
    // ---- fragment end.  Every warp publishes its (m, l) per row; each warp
    // rescales its O to the block's row maximum; then either the flat
    // combine (kFlat: every warp's O to its own buffer, every thread adds one
    // float4 over the warps and writes it) or a tree adds the warps' O (in
    // each round the upper half of the remaining warps hands its O to the
    // lower half through shared memory, so warp 0 ends with the fragment's O
    // in registers and writes the output or the partial from there).  Fixed
    // order throughout, so the result is deterministic.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float l = lsum[nt][c];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (g == 0) {
          const int r = 8 * nt + 2 * t + c;
          sML[(warp * 2 + 0) * RP + r] = mref[nt][c];
          sML[(warp * 2 + 1) * RP + r] = l;
        }
      }
    if (tid == 0) {
      int first;
      *frag_cnt = sp.count_fast(f_seg, sf->a, sf->b, first);
      *frag_first = first;
    }
    __syncthreads();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int r = 8 * nt + 2 * t + c;
        float M = sML[r];
#pragma unroll
        for (int w = 1; w < W; ++w) M = fmaxf(M, sML[(w * 2) * RP + r]);
        const float fw = ex2(mref[nt][c] - M);
        mref[nt][c] = M;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][nt][c] *= fw;
          o[mt][nt][c + 2] *= fw;
        }
      }
    if constexpr (Cfg::kFlat) {
      // every warp's rescaled O to its own buffer (the lane's four float4
      // slots of a row permuted by g / 2: conflict-free stores) ...
      {
        float4* dst = reinterpret_cast<float4*>(sO + (size_t)warp * RP * kHeadDim);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              dst[((8 * nt + 2 * t + c) * kHeadDim + 16 * g) / 4 + (k4 ^ (g >> 1))] =
                  make_float4(o[2 * k4][nt][c], o[2 * k4][nt][c + 2], o[2 * k4 + 1][nt][c],
                              o[2 * k4 + 1][nt][c + 2]);
      }
      __syncthreads();
    }
    if constexpr (!Cfg::kFlat) {
#pragma unroll 1
    for (int n = W; n > 1;) {
      const int half = (n + 1) >> 1;
      if (warp >= half && warp < n) {
        float4* dst = reinterpret_cast<float4*>(sO + (size_t)(warp - half) * RP * kHeadDim);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              dst[((8 * nt + 2 * t + c) * kHeadDim + 16 * g) / 4 + k4] =
                  make_float4(o[2 * k4][nt][c], o[2 * k4][nt][c + 2], o[2 * k4 + 1][nt][c],
                              o[2 * k4 + 1][nt][c + 2]);
      }
      __syncthreads();
      if (warp < n - half) {
        const float4* src = reinterpret_cast<const float4*>(sO + (size_t)warp * RP * kHeadDim);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const float4 v = src[((8 * nt + 2 * t + c) * kHeadDim + 16 * g) / 4 + k4];
              o[2 * k4][nt][c] += v.x;
              o[2 * k4][nt][c + 2] += v.y;
              o[2 * k4 + 1][nt][c] += v.z;
              o[2 * k4 + 1][nt][c + 2] += v.w;
            }
      }
      __syncthreads();
      n = half;
    }

    }
    const int cnt = *frag_cnt;
    const int slot = sp.k > 0 ? (int)blockIdx.x : f_seg + (int)blockIdx.x;
    const int64_t out_row0 = (int64_t)f_s * p.q_len;
    if constexpr (Cfg::kFlat) {
      // ... then thread (r, dq) adds float4 dq of row r over the warps and
      // writes the output or the partial.  Launched as a cluster (one
      // segment split over the cluster's blocks), each block keeps its result
      // in its (now idle) ring and block 0 merges them through distributed
      // shared memory, instead of global partials and a ticket.
      float4* cP = reinterpret_cast<float4*>(ring);
      float* cML = reinterpret_cast<float*>(ring + RP * kHeadDim * 4);
      for (int it = tid; it < p.rows * 32; it += nthr) {
        const int r = it >> 5, dq = it & 31;
        const int sidx = r * 32 + (dq & ~3) + ((dq & 3) ^ (dq >> 3));
        float M = sML[r];
#pragma unroll
        for (int w = 1; w < W; ++w) M = fmaxf(M, sML[(w * 2) * RP + r]);
        float l = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < W; ++w) {
          l += ex2(sML[(w * 2) * RP + r] - M) * sML[(w * 2 + 1) * RP + r];
          const float4 v = reinterpret_cast<const float4*>(sO + (size_t)w * RP * kHeadDim)[sidx];
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        if (clu) {
          cP[r * 32 + dq] = acc;
          if (dq == 0) {
            cML[r] = M;
            cML[RP + r] = l;
          }
          clu_written = true;
          continue;
        }
        const int i = r / p.group, gh = r % p.group;
        const int64_t orow = (out_row0 + i) * p.num_q_heads + f_h * p.group + gh;
        if (cnt == 1) {
          const float f = l > 0.f ? v_mult / l : 0.f;
          if constexpr (kPartial) {
            *reinterpret_cast<float4*>(p.out_o + orow * kHeadDim + 4 * dq) =
                make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
            if (dq == 0) p.out_lse[orow] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
          } else {
            __half2 h01 = __floats2half2_rn(acc.x * f, acc.y * f);
            __half2 h23 = __floats2half2_rn(acc.z * f, acc.w * f);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&h01);
            pk.y = *reinterpret_cast<uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + 4 * dq) = pk;
          }
        } else {
          *reinterpret_cast<float4*>(p.part_o + ((size_t)slot * RP + r) * kHeadDim + 4 * dq) = acc;
          if (dq == 0) {
            p.part_ml[(size_t)slot * 2 * RP + r] = M;
            p.part_ml[(size_t)slot * 2 * RP + RP + r] = l;
          }
        }
      }
      // the buffers are read; the next fragment's warps may write them
      __syncthreads();
    } else {
    if (warp == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int r = 8 * nt + 2 * t + c;
          if (r >= p.rows) continue;
          const float M = mref[nt][c];
          float l = 0.f;
#pragma unroll
          for (int w = 0; w < W; ++w) l += ex2(sML[(w * 2) * RP + r] - M) * sML[(w * 2 + 1) * RP + r];
          const int i = r / p.group, gh = r % p.group;
          const int64_t orow = (out_row0 + i) * p.num_q_heads + f_h * p.group + gh;
          if (cnt == 1) {
            const float f = l > 0.f ? v_mult / l : 0.f;
            if constexpr (kPartial) {
              float4* dst = reinterpret_cast<float4*>(p.out_o + orow * kHeadDim + 16 * g);
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
                dst[k4] = make_float4(o[2 * k4][nt][c] * f, o[2 * k4][nt][c + 2] * f,
                                      o[2 * k4 + 1][nt][c] * f, o[2 * k4 + 1][nt][c + 2] * f);
              if (g == 0) p.out_lse[orow] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
            } else {
              uint32_t hv[8];
#pragma unroll
              for (int mt = 0; mt < 8; ++mt)
                hv[mt] = pack_half2(o[mt][nt][c] * f, o[mt][nt][c + 2] * f);
              uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kHeadDim + 16 * g);
              dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
              dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + ((size_t)slot * RP + r) * kHeadDim +
                                                    16 * g);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              dst[k4] = make_float4(o[2 * k4][nt][c], o[2 * k4][nt][c + 2], o[2 * k4 + 1][nt][c],
                                    o[2 * k4 + 1][nt][c + 2]);
            if (g == 0) {
              p.part_ml[(size_t)slot * 2 * RP + r] = M;
              p.part_ml[(size_t)slot * 2 * RP + RP + r] = l;
            }
          }
        }
    }
    }
        if (cnt > 1 && !clu) {
      // warp 0's partial writes, ordered by the barrier before thread 0's
      // release; the last block's acquire, then the barrier, orders its
      // partial loads after every other block's release
      __syncthreads();
      if (tid == 0) {
        int ticket;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(ticket)
                     : "l"(p.counters + f_seg)
                     : "memory");
        *merge_flag = (ticket == cnt - 1);
      }
      __syncthreads();
      if (*merge_flag) {
        // gather the segment's partial slots (fixed order) into shared memory
        int* slots = reinterpret_cast<int*>(sO);
        if (tid == 0) {
          int nsl = 0;
          if (sp.k > 0) {
            const int np = sp.pages(f_s);
            for (int q = 0; q < sp.k; ++q)
              if ((int64_t)(q + 1) * np / sp.k > (int64_t)q * np / sp.k)
                slots[nsl++] = f_seg * sp.k + q;
          } else if (*frag_first >= 0) {
            for (int q = 0; q < cnt; ++q) slots[nsl++] = f_seg + *frag_first + q;
          } else {
            for (int64_t x = sf->a; x < sf->b;) {
              const int cc = sp.cta_of(x);
              slots[nsl++] = f_seg + cc;
              x = sp.start(cc + 1);
            }
          }
        }
        __syncthreads();
        // One pass: thread (r, dq) loads the (m, l) and the float4 dq of row r
        // of eight partials at once and folds them in with a running rescale
        // (fixed order, so the result is deterministic).
        for (int it = tid; it < p.rows * 32; it += nthr) {
          const int r = it >> 5, dq = it & 31;
          float M = kNoScore, l = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int q0 = 0; q0 < cnt; q0 += 8) {
            float mq[8], lq[8];
            float4 vq[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const bool in = q0 + k < cnt;
              const size_t sl = slots[in ? q0 + k : 0];
              mq[k] = in ? __ldcg(p.part_ml + sl * 2 * RP + r) : kNoScore;
              lq[k] = in ? __ldcg(p.part_ml + sl * 2 * RP + RP + r) : 0.f;
              vq[k] = in ? __ldcg(reinterpret_cast<const float4*>(p.part_o + (sl * RP + r) *
                                                                             kHeadDim) + dq)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float Mn = M;
#pragma unroll
            for (int k = 0; k < 8; ++k) Mn = fmaxf(Mn, mq[k]);
            const float f = ex2(M - Mn);
            l *= f;
            acc.x *= f;
            acc.y *= f;
            acc.z *= f;
            acc.w *= f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float wq = ex2(mq[k] - Mn);
              l += wq * lq[k];
              acc.x += wq * vq[k].x;
              acc.y += wq * vq[k].y;
              acc.z += wq * vq[k].z;
              acc.w += wq * vq[k].w;
            }
            M = Mn;
          }
          const float inv = l > 0.f ? v_mult / l : 0.f;
          const int i = r / p.group, gh = r % p.group;
          const int64_t orow = (out_row0 + i) * p.num_q_heads + f_h * p.group + gh;
          if constexpr (kPartial) {
            *reinterpret_cast<float4*>(p.out_o + orow * kHeadDim + 4 * dq) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (dq == 0) p.out_lse[orow] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
          } else {
            __half2 h01 = __floats2half2_rn(acc.x * inv, acc.y * inv);
            __half2 h23 = __floats2half2_rn(acc.z * inv, acc.w * inv);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&h01);
            pk.y = *reinterpret_cast<uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + 4 * dq) = pk;
          }
        }
        if (tid == 0) p.counters[f_seg] = 0;
      }
    }
    }
    __syncthreads();
  }

  if constexpr (kClusterMerge) {
    if (clu) {
      // a block whose share was empty leaves a neutral partial; every block
      // arrives at both cluster barriers exactly once
      float4* cP = reinterpret_cast<float4*>(ring);
      float* cML = reinterpret_cast<float*>(ring + RP * kHeadDim * 4);
      if (!__syncthreads_or(clu_written)) {
        for (int it = tid; it < p.rows * 32; it += nthr) {
          const int r = it >> 5, dq = it & 31;
          cP[r * 32 + dq] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (dq == 0) {
            cML[r] = kNoScore;
            cML[RP + r] = 0.f;
          }
        }
      }
      __syncthreads();
      cluster_sync_all();
      if (cluster_ctarank() == 0) {
        // the cluster's one segment: sequence 0, kv-head 0; 8-warp flat
        // kernels are FP16, so no V scale
        for (int it = tid; it < p.rows * 32; it += nthr) {
          const int r = it >> 5, dq = it & 31;
          float M = kNoScore;
          for (uint32_t c = 0; c < ncl; ++c)
            M = fmaxf(M, ld_cluster_f32(cluster_map(smem_u32(cML + r), c)));
          float l = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (uint32_t c = 0; c < ncl; ++c) {
            const float w = ex2(ld_cluster_f32(cluster_map(smem_u32(cML + r), c)) - M);
            l += w * ld_cluster_f32(cluster_map(smem_u32(cML + RP + r), c));
            const float4 v = ld_cluster_f4(cluster_map(smem_u32(cP + r * 32 + dq), c));
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
          }
          const float f = l > 0.f ? 1.f / l : 0.f;
          const int i = r / p.group, gh = r % p.group;
          const int64_t orow = (int64_t)i * p.num_q_heads + gh;
          if constexpr (kPartial) {
            *reinterpret_cast<float4*>(p.out_o + orow * kHeadDim + 4 * dq) =
                make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
            if (dq == 0) p.out_lse[orow] = l > 0.f ? (M + __log2f(l)) * kLn2 : -INFINITY;
          } else {
            __half2 h01 = __floats2half2_rn(acc.x * f, acc.y * f);
            __half2 h23 = __floats2half2_rn(acc.z * f, acc.w * f);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&h01);
            pk.y = *reinterpret_cast<uint32_t*>(&h23);
            *reinterpret_cast<uint2*>(p.out + orow * kHeadDim + 4 * dq) = pk;
          }
        }
      }
      // every block's shared memory stays until block 0 has read it
      cluster_sync_all();
    }
  }

  // ---- drain: never leave with a tile copy in flight (only after a timeout
  //      can this warp have issued pages it did not consume)
  if (lane == 0 && *abort_flag) {
    for (int u = consumed_u; u < issued_u; ++u) {
      if (kWaitTest && u == skipped_u) continue;     // nothing in flight there
      const int i = warp + u * W;
      (void)mbar_wait<kLimitNs>(&full[i % S], (i / S) & 1);
    }
  }
}

}  // namespace pqkv
