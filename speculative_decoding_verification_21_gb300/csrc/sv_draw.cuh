// sv_draw.cuh -- the draw of the target's own token by the inverse transform.
//
// After a rejection at n the token comes from norm(max(0, p_n - q_n)), after a
// clean sweep from p_gamma ("Fast Inference from Transformers via Speculative
// Decoding", section "The loop", step 3).  The draw takes one uniform U in
// [0, 1) with 53 random bits and returns the smallest v, in vocabulary order,
// whose cumulative weight exceeds U times the total weight.  The weights are
// formed in fp32 up to a common factor and summed per run of consecutive
// entries (8 per lane here, 16 per chunk in the fused LM head) in order, in
// fp32.  Each run sum is then taken as the fixed-point integer nearest
// sum * 2^f (f chosen from V so that no total can overflow 64 bits), and
// everything above the runs is added in 64-bit integers: exact, so the totals
// do not depend on the order of the additions and every level of the search
// agrees with the level above it.  t = floor(U W) in the same fixed point; a
// warp walks down the levels (per-CTA totals, segments, lanes) to the run
// whose cumulative end first exceeds t, and within it to the entry whose fp32
// prefix (in fixed point) does.  A GB300 SM runs fp64 at a small fraction of
// its integer rate, so no double arithmetic (nor a conversion to a 64-bit
// integer) is used.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"

namespace sv {

constexpr int kDrawLaneEntries = 8;
constexpr int kDrawSegEntries = 32 * kDrawLaneEntries;  // one warp

struct DrawArgs {
  const void* zt;
  const void* zd;
  int B, gamma;
  int64_t V;
  uint64_t seed, round;
  uint32_t* alpha_cnt;  // [B] counters of the optional overlap kernel, zeroed here
  uint32_t* done;       // [B] CTAs of the batch row that finished their segments (zeroed
                        // by the sweep that precedes the draw)
  uint64_t* segsum;     // [B][nseg] segment sums (fixed point)
  uint64_t* ctot;       // [B][nsplit] per-CTA totals of those
  int fsh;              // fixed-point scale, fix_shift(V)
  int nseg;             // segments per row, ceil(V / 256)
  int nsplit;           // CTAs per batch row
  int spc;              // segments per CTA
  bool vec;             // 16-byte loads of 8 entries are aligned in every row
  int32_t* out_tokens;
  uint8_t* out_flags;
};

// The uniform of the draw at position pos as its 53-bit integer k (U = k 2^-53):
// Philox4x32-10 at counter (0, 1<<24 | pos, b, round); the top 21 bits of word
// 0 and word 1.
__device__ __forceinline__ uint64_t draw_uniform53(uint64_t seed, uint32_t pos, uint32_t b,
                                                   uint64_t round) {
  const uint4 r = philox4x32_10(sv_counter(0u, 1u, pos, b, round), (uint32_t)seed,
                                (uint32_t)(seed >> 32));
  return ((uint64_t)(r.x >> 11) << 32) | (uint64_t)r.y;
}

// Fixed-point scale f for a row of V entries: every weight is at most 1, so
// totals stay below V 2^f <= 2^62.
inline int fix_shift(int64_t V) {
  int lg = 0;
  while (((int64_t)1 << lg) < V) ++lg;
  const int f = 62 - lg;
  return f > 48 ? 48 : (f < 20 ? 20 : f);
}

// A run sum (fp32, >= 0, finite, at most 16) as the nearest integer to
// sum * 2^f, ties to even, from its bits (integer operations only: the
// conversion instruction to 64-bit integers runs on the slow fp64 pipe).
__device__ __forceinline__ uint64_t to_fix(float x, int f) {
  const uint32_t u = __float_as_uint(x);
  const int ex = (int)(u >> 23);  // the sign bit is 0
  if (ex == 0) return 0ull;       // zero or below 2^-126
  const uint64_t m = (uint64_t)((u & 0x7FFFFFu) | 0x800000u);
  const int sh = ex - 150 + f;    // x 2^f = m 2^(ex - 150 + f)
  if (sh >= 0) return m << sh;    // x <= 16: below 2^(f + 5)
  if (sh < -24) return 0ull;      // below 1/2
  const int r = -sh;
  const uint64_t q = m >> r, rem = m & ((1ull << r) - 1ull), half = 1ull << (r - 1);
  return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

// floor(U W) for U = k 2^-53: the high 64 bits of (k 2^11) W.
__device__ __forceinline__ uint64_t scale_fix(uint64_t k53, uint64_t W) {
  return __umul64hi(k53 << 11, W);
}

// Weight of one entry up to the common factor 2^-mct / St: p_n is
// 2^(zt c - mct); the residual is that minus 2^(zd c + K - mct) where positive
// (K = log2 of the normaliser ratio).  Below a row's top-k threshold the entry
// has probability 0 in that row.  Explicit intrinsics only, so that the
// summing pass and the select get the same bits.
template <bool RESID, bool TOPK>
__device__ __forceinline__ float draw_weight(float zt, float zd, const DrawState& st, float kd) {
  if (TOPK && zt < st.tt) zt = -kInf;
  const float et = ex2(__fmaf_rn(zt, st.c, -st.mct));
  if (!RESID) return et;
  if (TOPK && zd < st.td) zd = -kInf;
  const float ed = ex2(__fmaf_rn(zd, st.c, kd));
  return (et > ed) ? __fsub_rn(et, ed) : 0.0f;
}

// Eight consecutive entries of a row as raw bits: one 16-byte vector of bf16
// or two of fp32.
template <int DT>
struct Raw8 {
  uint4 v[DT == SV_F32 ? 2 : 1];
};

template <int DT>
__device__ __forceinline__ Raw8<DT> load_raw8(const char* row, int64_t v0, int64_t V, bool vec,
                                              float pad) {
  Raw8<DT> r;
  if (vec && v0 + kDrawLaneEntries <= V) {
    const uint4* p = reinterpret_cast<const uint4*>(row + v0 * (DT == SV_F32 ? 4 : 2));
#pragma unroll
    for (int i = 0; i < (DT == SV_F32 ? 2 : 1); ++i) r.v[i] = __ldg(p + i);
  } else {
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = (v0 + e < V) ? load_logit<DT>(row, v0 + e) : pad;
    if constexpr (DT == SV_F32) {
      r.v[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
      r.v[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                          __float_as_uint(f[7]));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)  // the values are bf16-exact: re-pack their bits
        w[i] = (__float_as_uint(f[2 * i]) >> 16) | (__float_as_uint(f[2 * i + 1]) & 0xFFFF0000u);
      r.v[0] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  return r;
}

template <int DT>
__device__ __forceinline__ void unpack8(const Raw8<DT>& r, float (&f)[8]) {
  if constexpr (DT == SV_F32) {
    unpack<SV_F32>(r.v[0], f);
    unpack<SV_F32>(r.v[1], f + 4);
  } else {
    unpack<SV_BF16>(r.v[0], f);
  }
}

// The eight weights of a lane and their sum, added in order.
template <int DT, bool RESID, bool TOPK>
__device__ __forceinline__ float lane_weights(const Raw8<DT>& rt, const Raw8<DT>& rd,
                                              const DrawState& st, float kd, float (&w)[8]) {
  float zt[8], zd[8];
  unpack8<DT>(rt, zt);
  if (RESID) unpack8<DT>(rd, zd);
  float s = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    w[e] = draw_weight<RESID, TOPK>(zt[e], RESID ? zd[e] : 0.0f, st, kd);
    s = __fadd_rn(s, w[e]);
  }
  return s;
}

// Sum over the warp's lanes (the same value in every lane).
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Segment sums of segments [s0, s1) of one row, warps round-robin, U segments
// of a warp in flight together; returns the warp's total.
template <int DT, bool RESID, bool TOPK>
__device__ __forceinline__ uint64_t segment_sums(const char* rt, const char* rd, int64_t V,
                                                 bool vec, const DrawState& st, int s0, int s1,
                                                 int warp, int nwarps, int fsh, uint64_t* seg) {
  uint64_t total = 0;  // this warp's segments
  constexpr int U = (DT == SV_F32) ? 2 : 4;  // the same bytes in flight for both types
  const int lane = threadIdx.x & 31;
  const float kd = RESID ? __fsub_rn(st.K, st.mct) : 0.0f;
  for (int s = s0 + warp; s < s1; s += U * nwarps) {
    Raw8<DT> xt[U], xd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int su = s + u * nwarps;
      if (su < s1) {
        const int64_t v0 = (int64_t)su * kDrawSegEntries + lane * kDrawLaneEntries;
        xt[u] = load_raw8<DT>(rt, v0, V, vec, -kInf);
        if (RESID) xd[u] = load_raw8<DT>(rd, v0, V, vec, -kInf);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int su = s + u * nwarps;
      if (su < s1) {
        float w[8];
        const uint64_t S =
            warp_sum_u64(to_fix(lane_weights<DT, RESID, TOPK>(xt[u], xd[u], st, kd, w), fsh));
        if (lane == 0) seg[su] = S;
        total += S;
      }
    }
  }
  return total;  // the same in every lane
}

// Sum of n fixed-point words by one warp (the same in every lane).
__device__ __forceinline__ uint64_t warp_total(const uint64_t* v, int n) {
  uint64_t x = 0;
  for (int j = (int)(threadIdx.x & 31); j < n; j += 32) x += __ldcg(v + j);
  return warp_sum_u64(x);
}

// One warp: the first j in [0, n) whose cumulative end base + v[0] + .. + v[j]
// exceeds t, with *before = base + v[0] + .. + v[j-1]; R consecutive words per
// lane, 32 R per round of loads.  -1 if there is none (base + total <= t).
// The same result in every lane.
template <int R>
__device__ __forceinline__ int warp_find(const uint64_t* v, int n, uint64_t t, uint64_t base,
                                         uint64_t* before) {
  const int lane = threadIdx.x & 31;
  for (int j0 = 0; j0 < n; j0 += 32 * R) {
    uint64_t x[R], ls = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j = j0 + lane * R + r;
      x[r] = (j < n) ? __ldcg(v + j) : 0ull;
      ls += x[r];
    }
    uint64_t P = ls;  // inclusive prefix over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, P, o);
      if (lane >= o) P += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, base + P > t);
    if (hit) {
      const int l = __ffs((int)hit) - 1;
      int idx = 0;
      uint64_t acc = base + P - ls;
      if (lane == l) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (acc + x[r] > t) {
            idx = j0 + lane * R + r;
            break;
          }
          acc += x[r];
        }
      }
      *before = __shfl_sync(0xffffffffu, acc, l);
      return __shfl_sync(0xffffffffu, idx, l);
    }
    base += __shfl_sync(0xffffffffu, P, 31);
  }
  *before = base;
  return -1;
}

// warp_find over all n <= 32 kPickAll words in one round of loads, with W (the
// total) and t = floor(U W) taken from the same registers.  -1 when W = 0.
constexpr int kPickAll = 16;
__device__ __forceinline__ int warp_pick_all(const uint64_t* v, int n, uint64_t k53,
                                             uint64_t* W, uint64_t* t, uint64_t* before) {
  const int lane = threadIdx.x & 31;
  uint64_t x[kPickAll], ls = 0;
#pragma unroll
  for (int r = 0; r < kPickAll; ++r) {
    const int j = lane * kPickAll + r;
    x[r] = (j < n) ? __ldcg(v + j) : 0ull;
    ls += x[r];
  }
  uint64_t P = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, P, o);
    if (lane >= o) P += y;
  }
  *W = __shfl_sync(0xffffffffu, P, 31);
  *t = scale_fix(k53, *W);
  *before = 0;
  if (*W == 0) return -1;
  const unsigned hit = __ballot_sync(0xffffffffu, P > *t);
  const int l = __ffs((int)hit) - 1;
  int idx = 0;
  uint64_t acc = P - ls;
  if (lane == l) {
#pragma unroll
    for (int r = 0; r < kPickAll; ++r) {
      if (acc + x[r] > *t) {
        idx = lane * kPickAll + r;
        break;
      }
      acc += x[r];
    }
  }
  *before = __shfl_sync(0xffffffffu, acc, l);
  return __shfl_sync(0xffffffffu, idx, l);
}

// The entry of a run of weights w[0..M) holding trel (fixed point, measured
// from `lo`, the run's start): the first e whose fp32 prefix, added in order,
// ends past it.  The run's own sum is the prefix at M - 1, so an entry is
// found whenever trel lies below lo + to_fix(sum); -1 otherwise.
template <int M>
__device__ __forceinline__ int pick_in_run(const float (&w)[M], uint64_t lo, uint64_t trel,
                                           int fsh) {
  float a32 = 0.0f;
  int pick = -1;
#pragma unroll
  for (int e = 0; e < M; ++e) {
    a32 = __fadd_rn(a32, w[e]);
    if (pick < 0 && w[e] > 0.0f && lo + to_fix(a32, fsh) > trel) pick = e;
  }
  return pick;
}

// The select, by one warp of the CTA of the batch row that arrives last, after
// every segment sum of the row is in `seg`: W, t = floor(U W), the CTA range
// holding t (from the per-CTA totals `ctot`, ngrp of them with spc segments
// each; or, ctot null, the segments directly), the segment, then the lane
// (the same lane sums recomputed, their prefix) and the entry.  Returns the
// token in every lane; -1 when no weight is positive.
template <int DT, bool RESID, bool TOPK>
__device__ int draw_select_warp(const char* rt, const char* rd, int64_t V, bool vec,
                                const DrawState& st, const uint64_t* seg, int nseg,
                                const uint64_t* ctot, int ngrp, int spc, int fsh, uint64_t k53) {
  const int lane = threadIdx.x & 31;
  uint64_t W, t, base = 0;
  int s = 0;
  if (nseg <= 32 * kPickAll) {
    // one round of loads: all segment sums at once give W, t and the segment
    s = warp_pick_all(seg, nseg, k53, &W, &t, &base);
    if (W == 0) return -1;
  } else {
    W = ctot ? warp_total(ctot, ngrp) : warp_total(seg, nseg);
    if (W == 0) return -1;
    t = scale_fix(k53, W);  // < W
    int s0 = 0, cnt = nseg;
    if (ctot) {
      const int c = warp_find<2>(ctot, ngrp, t, 0ull, &base);
      s0 = c * spc;
      cnt = min(nseg - s0, spc);
    }
    s = s0 + warp_find<4>(seg + s0, cnt, t, base, &base);
  }
  const float kd = RESID ? __fsub_rn(st.K, st.mct) : 0.0f;
  const int64_t v0 = (int64_t)s * kDrawSegEntries + lane * kDrawLaneEntries;
  const Raw8<DT> xt = load_raw8<DT>(rt, v0, V, vec, -kInf);
  Raw8<DT> xd = xt;
  if (RESID) xd = load_raw8<DT>(rd, v0, V, vec, -kInf);
  float w[8];
  const uint64_t L = to_fix(lane_weights<DT, RESID, TOPK>(xt, xd, st, kd, w), fsh);
  uint64_t P = L;  // inclusive prefix over the lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, P, o);
    if (lane >= o) P += y;
  }
  const uint64_t trel = t - base;  // below the segment's sum, P at lane 31
  const unsigned cross = __ballot_sync(0xffffffffu, P > trel);
  const int ln = __ffs((int)cross) - 1;
  int tok = -1;
  if (lane == ln) {
    const int e = pick_in_run<8>(w, P - L, trel, fsh);
    if (e >= 0) tok = (int)(v0 + e);
  }
  return __shfl_sync(0xffffffffu, tok, ln < 0 ? 0 : ln);
}

}  // namespace sv
