// sv_gumbel.cuh -- the draw of the target's own token by Gumbel-max.
//
// After a rejection at n the token comes from norm(max(0, p_n - q_n)), after a
// clean sweep from p_gamma ("Fast Inference from Transformers via Speculative
// Decoding", section "The loop", step 3).  The token is the argmax over the
// entries of positive weight w_v of log w_v + g_v, g_v = -ln(-ln u_v) Gumbel
// noise, ties to the lowest index; u_v comes from Philox4x32-10 with tag 1 at
// the draw position n (counter (v>>2, 1<<24 | n, b, lo32(round)), lane v&3).
//
// On the GPU the race is run in ratio form: with E_v = -log2 u_v (an
// exponential variate in log2 units), argmax log w_v + g_v = argmax w_v / E_v,
// and the weights need only be known up to a factor common to the row.  Each
// lane keeps its two largest keys w_v / E_v (a reciprocal and a product per
// entry, the update by selects); the warp, then the merge, keep the best two of
// those.  Most entries never reach the key: once a warp holds two candidates,
// an entry whose Philox word shows an E_v too large for any weight of its block
// of four (one Philox block) to beat the second-best key is dropped by one
// integer compare.  When the two best keys lie within 2^-10 of each other, they
// are re-decided in double precision from the logits (the key's definition,
// log w + g), so that the winner differs from an exact evaluation only where
// the exact keys themselves are within the rounding of the row sums.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_decide.cuh"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_plan.h"

namespace sv {

// A candidate: its key w/E as a float and its index (-1: none, key -inf).
struct KeyIdx {
  float k;
  int i;
};
__device__ __forceinline__ bool key_beats(const KeyIdx& a, const KeyIdx& b) {
  if (a.i < 0) return false;
  if (b.i < 0) return true;
  return a.k > b.k || (a.k == b.k && a.i < b.i);
}
struct KeyTop2 {
  KeyIdx a, b;
};
__device__ __forceinline__ KeyTop2 key_top2_empty() {
  return KeyTop2{KeyIdx{-kInf, -1}, KeyIdx{-kInf, -1}};
}
// An entry in its lane's increasing index order (strictly larger keys win, so
// an equal key keeps the earlier, lower index): selects only.
__device__ __forceinline__ void top2_push(KeyTop2& t, float k, int i) {
  const bool g1 = k > t.a.k, g2 = k > t.b.k;
  t.b.k = g1 ? t.a.k : (g2 ? k : t.b.k);
  t.b.i = g1 ? t.a.i : (g2 ? i : t.b.i);
  t.a.k = g1 ? k : t.a.k;
  t.a.i = g1 ? i : t.a.i;
}
__device__ __forceinline__ void key_insert(KeyTop2& t, const KeyIdx& c) {
  if (key_beats(c, t.a)) {
    t.b = t.a;
    t.a = c;
  } else if (key_beats(c, t.b)) {
    t.b = c;
  }
}
__device__ __forceinline__ KeyTop2 key_warp(KeyTop2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const KeyIdx a{__shfl_xor_sync(0xffffffffu, t.a.k, o), __shfl_xor_sync(0xffffffffu, t.a.i, o)};
    const KeyIdx b{__shfl_xor_sync(0xffffffffu, t.b.k, o), __shfl_xor_sync(0xffffffffu, t.b.i, o)};
    key_insert(t, a);
    key_insert(t, b);
  }
  return t;
}

// A candidate as one 64-bit word that is never zero (a zeroed slot means "not
// written yet"): the key's bits low, index + 1 high; an empty candidate has
// key -1.
__device__ __forceinline__ uint64_t key_word(const KeyIdx& c) {
  return ((uint64_t)(uint32_t)(c.i + 1) << 32) | (uint64_t)__float_as_uint(c.i < 0 ? -1.0f : c.k);
}
__device__ __forceinline__ KeyIdx key_unword(uint64_t w) {
  const int i = (int)(uint32_t)(w >> 32) - 1;
  return KeyIdx{i < 0 ? -kInf : __uint_as_float((uint32_t)w), i};
}

// The Gumbel noise -ln(-ln u) of entry v in double (the re-decision of a near tie).
__device__ __forceinline__ double gumbel_f64(int64_t v, int pos, int b, uint64_t seed,
                                             uint64_t round, uint32_t tag) {
  const uint4 rnd = philox4x32_10(sv_counter((uint32_t)(v >> 2), tag, (uint32_t)pos, (uint32_t)b, round),
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t lanes[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  return -log(sv_neglog_u_f64(lanes[v & 3]));
}

// Entries of one draw, for the re-decision in double: p_n(v) = exp(zt_v / T -
// mt) / St and q_n(v) likewise (mt, md: the rows' largest scaled logits), with
// entries below a top-k threshold at weight 0.
struct DrawRowsF64 {
  double invT, mt, md, St, Sd;
  float tt, td;  // top-k thresholds (-inf: none)
  bool resid;
};
__device__ __forceinline__ double draw_key_f64(const DrawRowsF64& r, float zt, float zd,
                                               double g) {
  if (!(zt >= r.tt) || zt == -kInf) return -HUGE_VAL;
  if (!r.resid) return (double)zt * r.invT + g;  // log p_n(v) + g up to the row's constant
  const double p = exp((double)zt * r.invT - r.mt) / r.St;
  const double q = (zd >= r.td && zd > -kInf) ? exp((double)zd * r.invT - r.md) / r.Sd : 0.0;
  const double w = p - q;
  return (w > 0.0) ? log(w) + g : -HUGE_VAL;
}

// The winner of a top-2 whose keys lie within 2^-10 of each other, by their
// double keys (ties to the lower index); otherwise the fp32 winner.
template <class F>
__device__ __forceinline__ int race_pick(const KeyTop2& t, F key_f64) {
  if (t.a.i < 0) return -1;
  if (t.b.i < 0 || t.b.k < t.a.k * (1.0f - 0x1p-10f)) return t.a.i;
  const double ka = key_f64(t.a.i), kb = key_f64(t.b.i);
  if (kb > ka || (kb == ka && t.b.i < t.a.i)) return t.b.i;
  return t.a.i;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The weight of one entry of the race up to the common factor 2^-mct / St:
// p_n's, or the residual max(0, p_n - q_n) (RESID); 0 below a row's top-k
// threshold (TOPK).
template <bool RESID, bool TOPK>
__device__ __forceinline__ float race_weight(float a, float d, const DrawState& st, float kd) {
  if (TOPK && a < st.tt) a = -kInf;
  float w = ex2(__fmaf_rn(a, st.c, -st.mct));
  if (RESID) {
    if (TOPK && d < st.td) d = -kInf;
    const float ed = ex2(__fmaf_rn(d, st.c, kd));
    w = (w > ed) ? __fsub_rn(w, ed) : 0.0f;
  }
  return w;
}
// Its key w / E from its Philox word; -inf for a weight of 0 (no candidate).
__device__ __forceinline__ float race_key(float w, uint32_t r) {
  return (w > 0.0f) ? w * rcp_approx(neglog2_u(r)) : -kInf;
}

// The largest logit of a run of eight (NaN ignored).
template <int DT>
__device__ __forceinline__ float run_max(const Raw8<DT>& x) {
  if constexpr (DT == SV_F32)
    return fmaxf(vmax<SV_F32>(x.v[0]), vmax<SV_F32>(x.v[1]));
  else
    return vmax<SV_BF16>(x.v[0]);
}

// Entry e (0..7, not known at compile time) of a run, by selects (no local
// array).
template <int DT>
__device__ __forceinline__ float run_at(const Raw8<DT>& x, int e) {
  if constexpr (DT == SV_F32) {
    const uint4 q = (e & 4) ? x.v[1] : x.v[0];
    const uint32_t lo = (e & 1) ? q.y : q.x, hi = (e & 1) ? q.w : q.z;
    return __uint_as_float((e & 2) ? hi : lo);
  } else {
    const uint4 q = x.v[0];
    const uint32_t lo = (e & 2) ? q.y : q.x, hi = (e & 2) ? q.w : q.z;
    const uint32_t w = (e & 4) ? hi : lo;
    return (e & 1) ? bf16hi(w) : bf16lo(w);
  }
}
__device__ __forceinline__ uint32_t word_at(const uint32_t (&r)[8], int e) {
  const uint32_t m0 = (e & 1) ? r[1] : r[0], m1 = (e & 1) ? r[3] : r[2];
  const uint32_t m2 = (e & 1) ? r[5] : r[4], m3 = (e & 1) ? r[7] : r[6];
  const uint32_t n0 = (e & 2) ? m1 : m0, n1 = (e & 2) ? m3 : m2;
  return (e & 4) ? n1 : n0;
}

// The two Philox blocks of the run at v0 (a multiple of 8): word e is entry v0 + e's.
__device__ __forceinline__ void run_words(int64_t v0, uint32_t c1, uint32_t c2, uint32_t c3,
                                          const PhiloxKeys& pk, uint32_t (&r)[8]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 x = philox_rk(make_uint4((uint32_t)(v0 >> 2) + (uint32_t)h, c1, c2, c3), pk);
    r[4 * h] = x.x;
    r[4 * h + 1] = x.y;
    r[4 * h + 2] = x.z;
    r[4 * h + 3] = x.w;
  }
}

// The key of a run's largest-logit entry (the first of equal ones), from the
// run's Philox words rw: a seed for the pruning bound.  -inf when that entry
// has no weight.
template <int DT, bool RESID, bool TOPK>
__device__ __forceinline__ float run_seed_key(const Raw8<DT>& xt, const Raw8<DT>& xd, float zmax,
                                              const uint32_t (&rw)[8], const DrawState& st,
                                              float kd) {
  int es = 0;
  for (int e = 7; e >= 0; --e)
    if (run_at<DT>(xt, e) == zmax) es = e;
  return race_key(race_weight<RESID, TOPK>(run_at<DT>(xt, es), RESID ? run_at<DT>(xd, es) : 0.0f,
                                           st, kd),
                  word_at(rw, es));
}

// Pruning of a block of four entries (one Philox block): their weights are at
// most Wb = 2^(max z c - mct) (the residual's lie below p_n's), so an entry's
// key w_v / E_v stays below th whenever E_v > Wb / th; with u_v = (m_v + 1/2)
// 2^-23 that holds when m_v < 2^(23 - Wb / th) (1 - 2^-10).  The slack of
// 2^-10 covers the approximate ex2 / lg2 / reciprocal many times over, so a
// pruned entry's computed key is below th as well.  tau = (1 + 2^-10) / th, or
// 0 when th is no positive key.  Returns R: an entry whose Philox word is below
// R is pruned (0: none).
__device__ __forceinline__ float prune_tau(float th) {
  return (th > 0.0f) ? (1.0f + 0x1p-10f) * rcp_approx(th) : 0.0f;
}
__device__ __forceinline__ uint32_t prune_word(float zmax, const DrawState& st, float tau) {
  const float Wb = ex2(__fmaf_rn(zmax, st.c, -st.mct));
  const float y = ex2(23.0f - Wb * tau) * (1.0f - 0x1p-10f);
  if (!(tau > 0.0f) || !(y >= 1.0f)) return 0u;  // no bound yet; also NaN
  return __float2uint_rz(fminf(y, 8388607.0f)) << 9;
}

// The largest logit of entries 4h..4h+3 of a run (NaN ignored).
template <int DT>
__device__ __forceinline__ float half_max(const Raw8<DT>& x, int h) {
  if constexpr (DT == SV_F32) {
    return vmax<SV_F32>(x.v[h]);
  } else {
    const uint32_t a = h ? x.v[0].z : x.v[0].x, b = h ? x.v[0].w : x.v[0].y;
    uint32_t m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    return fmaxf(bf16lo(m), bf16hi(m));
  }
}

// A lower bound of the second-best key over a warp's candidates: the larger
// of every lane's second key and the second largest first key.  At least two
// distinct entries hold keys >= the bound, so an entry whose key lies below it
// is in no final best two.  The same value in every lane; -inf while there is
// no such pair.
__device__ __forceinline__ float warp_second_bound(const KeyTop2& t) {
  const float m1 = warp_max(t.a.k);
  return warp_max(t.a.k == m1 ? t.b.k : t.a.k);
}

// Runs of eight per lane and round of loads (the same bytes for both types),
// 16-byte vectors per run and row, and the shared memory a racing warp stages
// its rounds in: two rounds of both rows.
template <int DT>
struct RaceStage {
  static constexpr int kRuns = (DT == SV_F32) ? 2 : 4;
  static constexpr int kVecs = (DT == SV_F32) ? 2 : 1;
  static constexpr int kRound = kRuns * 2 * kVecs * 32;  // uint4 per round, both rows
};
constexpr int kRaceStages = 3;  // rounds staged per warp: one raced, the others in flight
constexpr size_t kRaceWarpSmem = kRaceStages * 4 * 2 * 32 * sizeof(uint4);  // 4 KB a round

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A round of the race: entries [lo, hi) of the draw row (hi <= lo: none; V <
// 2^31, so entry indices fit in 32 bits).
struct RaceRound {
  int32_t lo, hi;
};

// The race over the rounds `next()` hands out (warp-uniform; once it returns an
// empty round it returns no other) of row n (and of draft row n for a
// residual): a round holds at most kRuns runs of eight per lane, lane l taking
// the runs at lo + 8 (l + 32 u).  Whole 16-byte runs go through the warp's
// shared memory `sb` (kRaceWarpSmem bytes) by cp.async, the next
// kRaceStages - 1 rounds' copies in flight while one round is raced; a run cut
// by the row's end (or any run of rows that do not start on 16-byte
// boundaries, !vec) is loaded directly.  Each lane reads back only its own
// copies.  Round starts are multiples of 8.  A round computes its Philox words
// first, then waits for its copies and for the shared bound (the words cover
// both latencies).  `th` (the same in every lane) is the warp's bound on the
// second-best key, carried from one call to the next; while it is unset, the
// largest-logit entry of each lane's first run is keyed first to set it, and
// in that first round residual entries of certainly zero weight are dropped
// too.  `thw` (or null) is a bound shared by every warp racing the same draw:
// each round reads it and raises it to th afterwards when th rose above what
// it is known to hold (any warp's bound holds for the union of their
// candidates).
template <int DT, bool RESID, bool TOPK, class Next>
__device__ __forceinline__ void race_rounds(const char* rt, const char* rd, int64_t V, bool vec,
                                            const DrawState& st, float kd, uint64_t seed,
                                            uint64_t round, int b, KeyTop2& t, float& th,
                                            uint32_t* thw, uint4* sb, Next&& next) {
  using RS = RaceStage<DT>;
  constexpr int kRuns = RS::kRuns, kVecs = RS::kVecs;
  constexpr int kElem = (DT == SV_F32) ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const PhiloxKeys pk = philox_keys(seed);
  // th into the shared bound when it is above what the word is known to hold
  // (no reply waited for; keys are positive, so their bits order as integers)
  float known = 0.0f;
  auto share = [&]() {
    if (thw != nullptr && th > known) {
      if (lane == 0)
        asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(thw), "r"(__float_as_uint(th))
                     : "memory");
      known = th;
    }
  };
  const uint32_t c1 = (1u << 24) | (uint32_t)st.pos, c2 = (uint32_t)b, c3 = (uint32_t)round;
  auto nruns = [](const RaceRound& q) { return q.hi > q.lo ? (int)((q.hi - q.lo + 7) >> 3) : 0; };
  // slot of (round buffer s, run u, row w, vector q) for this lane
  auto slot = [&](int s, int u, int w, int q) {
    return sb + s * RS::kRound + ((u * 2 + w) * kVecs + q) * 32 + lane;
  };
  auto whole = [&](int64_t v0) { return vec && v0 + 8 <= V; };
  auto issue = [&](const RaceRound& q, int s) {
    const int n = nruns(q);
#pragma unroll
    for (int u = 0; u < kRuns; ++u) {
      const int r = lane + 32 * u;
      const int64_t v0 = q.lo + 8 * (int64_t)r;
      if (r < n && whole(v0)) {
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
          cp_async16(slot(s, u, 0, k), rt + v0 * kElem + 16 * k);
          if (RESID) cp_async16(slot(s, u, 1, k), rd + v0 * kElem + 16 * k);
        }
      }
    }
    cp_async_commit_group();  // (possibly empty: the count of groups stays the same)
  };
  // q[0] is raced from buffer s, q[k] is in flight in buffer (s + k) mod kRaceStages
  RaceRound q[kRaceStages];
#pragma unroll
  for (int k = 0; k < kRaceStages - 1; ++k) {
    q[k] = next();
    issue(q[k], k);
  }
  for (int s = 0; q[0].hi > q[0].lo; s = (s + 1 == kRaceStages) ? 0 : s + 1) {
    uint32_t g = 0u;
    if (thw != nullptr && lane == 0)
      asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(g) : "l"(thw) : "memory");
    q[kRaceStages - 1] = next();
    issue(q[kRaceStages - 1], (s + kRaceStages - 1) % kRaceStages);  // the buffer raced last
    const int64_t lo = q[0].lo;
    const int nrun = nruns(q[0]);
    // the Philox words of all runs first (independent chains, interleaved): they
    // need neither this round's copies nor the shared bound, whose latencies
    // they cover
    uint32_t rw[kRuns][8];
#pragma unroll
    for (int u = 0; u < kRuns; ++u) run_words(lo + 8 * (int64_t)(lane + 32 * u), c1, c2, c3, pk, rw[u]);
    cp_async_wait_group<kRaceStages - 1>();  // this round's copies have landed
    // run u of this lane (from its own copies; a ragged tail from global memory),
    // read when it is pruned so that only one run's logits are held at a time
    auto load_run = [&](int u, Raw8<DT>& a, Raw8<DT>& d) {
      const int64_t v0 = lo + 8 * (int64_t)(lane + 32 * u);
      if (whole(v0)) {
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
          a.v[k] = *slot(s, u, 0, k);
          if (RESID) d.v[k] = *slot(s, u, 1, k);
        }
      } else {
        a = load_raw8<DT>(rt, v0, V, vec, -kInf);
        if (RESID) d = load_raw8<DT>(rd, v0, V, vec, -kInf);
      }
    };
    g = __shfl_sync(0xffffffffu, g, 0);
    if (g != 0u) {
      th = fmaxf(th, __uint_as_float(g));
      known = fmaxf(known, __uint_as_float(g));
    }
    const bool seeded = !(th > 0.0f);  // this warp's first round: its bound is still loose
    if (seeded) {  // the same in every lane: seeds from each lane's first run
      float k = -kInf;
      if (lane < nrun) {
        Raw8<DT> a, d;
        load_run(0, a, d);
        k = run_seed_key<DT, RESID, TOPK>(a, d, run_max<DT>(a), rw[0], st, kd);
      }
      // the second largest seed over the lanes (distinct entries)
      const float m1 = warp_max(k);
      const unsigned top = __ballot_sync(0xffffffffu, k == m1);
      th = fmaxf(th, (__popc(top) > 1) ? m1 : warp_max(k == m1 ? -kInf : k));
      share();
    }
    // the pruning of each block of four against one bound, then the rare
    // entries left, in increasing order
    const float tau = prune_tau(fmaxf(th, t.b.k));
#pragma unroll
    for (int u = 0; u < kRuns; ++u) {
      const int r = lane + 32 * u;
      if (r >= nrun) continue;
      Raw8<DT> xt, xd;
      load_run(u, xt, xd);
      uint32_t live = 0u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t R = prune_word(half_max<DT>(xt, h), st, tau);
#pragma unroll
        for (int e = 4 * h; e < 4 * h + 4; ++e) live |= (rw[u][e] >= R ? 1u : 0u) << e;
      }
      if (RESID && !TOPK && seeded) {
        // under the loose first bound, also drop the entries whose residual weight
        // is certainly 0: 2^a below 2^d by far more than the error of ex2 (their
        // key would be -inf, which never enters the best two)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float a = __fmaf_rn(run_at<DT>(xt, e), st.c, -st.mct);
          const float d = __fmaf_rn(run_at<DT>(xd, e), st.c, kd);
          if (a < d - 0x1p-6f) live &= ~(1u << e);
        }
      }
      const int64_t v0 = lo + 8 * (int64_t)r;
      while (live != 0u) {
        const int e = __ffs((int)live) - 1;
        live &= live - 1u;
        const float w = race_weight<RESID, TOPK>(run_at<DT>(xt, e),
                                                 RESID ? run_at<DT>(xd, e) : 0.0f, st, kd);
        top2_push(t, race_key(w, word_at(rw[u], e)), (int)(v0 + e));
      }
    }
    th = fmaxf(th, warp_second_bound(t));
    share();
#pragma unroll
    for (int k = 0; k < kRaceStages - 1; ++k) q[k] = q[k + 1];
  }
  cp_async_wait_group<0>();  // nothing left in flight
}

// Entries per round of the race (kRuns runs of eight per lane).
template <int DT>
constexpr int64_t race_round_entries() {
  return (int64_t)32 * 8 * RaceStage<DT>::kRuns;
}

// The race of a draw in the mode the decision set (residual, or p_n), into t,
// over the rounds `next()` hands out.  thw: the bound shared by the warps
// racing this draw, or null; sb: the warp's kRaceWarpSmem bytes of shared
// memory.
template <int DT, bool TOPK, class Next>
__device__ __forceinline__ void race_draw_rounds(const SweepCtx& x, int b, const DrawState& st,
                                                 bool resid, bool vec, KeyTop2& t, float& th,
                                                 uint32_t* thw, uint4* sb, Next&& next) {
  const int gamma = x.gamma;
  const int64_t V = x.V;
  const char* rt = row_ptr<DT>(x.zt, x.zd, b, st.pos, gamma, V);
  if (resid) {
    const char* rd = row_ptr<DT>(x.zt, x.zd, b, gamma + 1 + st.pos, gamma, V);
    race_rounds<DT, true, TOPK>(rt, rd, V, vec, st, __fsub_rn(st.K, st.mct), x.seed, x.round, b,
                                t, th, thw, sb, next);
  } else {
    race_rounds<DT, false, TOPK>(rt, rt, V, vec, st, 0.0f, x.seed, x.round, b, t, th, thw, sb,
                                 next);
  }
}

// The same over the contiguous entries [lo, hi) (lo a multiple of 8).
template <int DT, bool TOPK>
__device__ __forceinline__ void race_draw(const SweepCtx& x, int b, const DrawState& st, bool resid,
                                          int64_t lo, int64_t hi, bool vec, KeyTop2& t,
                                          float& th, uint32_t* thw, uint4* sb) {
  int64_t at = lo;
  race_draw_rounds<DT, TOPK>(x, b, st, resid, vec, t, th, thw, sb, [&]() {
    const int64_t e = at + race_round_entries<DT>() < hi ? at + race_round_entries<DT>() : hi;
    const RaceRound q{(int32_t)at, (int32_t)e};
    if (e > at) at = e;
    return q;
  });
}

// The token from the best two keys T over the whole row of the race that drew
// it (the residual's when use_resid, else p_n's), re-decided in double near a
// tie; token 0 and ZERO_MASS when there is none.  fl: the flags so far.  One
// warp; lane 0 writes the token and the flags.
template <int DT>
__device__ __noinline__ void race_emit(const SweepCtx& x, int b, const DrawState& st,
                                       const KeyTop2& T, bool use_resid, int fl) {
  const int lane = threadIdx.x & 31;
  const int gamma = x.gamma;
  const int64_t V = x.V;
  const char* rt = row_ptr<DT>(x.zt, x.zd, b, st.pos, gamma, V);
  const char* rd = use_resid ? row_ptr<DT>(x.zt, x.zd, b, gamma + 1 + st.pos, gamma, V) : rt;
  DrawRowsF64 rr;
  rr.invT = (double)st.invT;
  rr.mt = (double)st.zmt * rr.invT;
  rr.md = (double)st.zmd * rr.invT;
  rr.St = (double)st.st;
  rr.Sd = (double)st.sd;
  rr.tt = st.tt;
  rr.td = st.td;
  rr.resid = use_resid;
  int tok = race_pick(T, [&](int v) {
    const float zt = load_logit<DT>(rt, v);
    const float zd = use_resid ? load_logit<DT>(rd, v) : 0.0f;
    return draw_key_f64(rr, zt, zd, gumbel_f64(v, st.pos, b, x.seed, x.round, 1u));
  });
  if (lane == 0) {
    if (tok < 0 || (int64_t)tok >= V) {
      tok = 0;
      fl |= SV_FLAG_ZERO_MASS;
    }
    x.out_tokens[(int64_t)b * (gamma + 1) + st.pos] = tok;
    if (x.out_flags) x.out_flags[b] = (uint8_t)fl;
  }
}

// The empty-residual fallback: p_n raced over the whole row by one warp (rare:
// max(0, p_n - q_n) has no positive entry in floating point), then emitted;
// sb: the warp's kRaceWarpSmem bytes of shared memory.
template <int DT, bool TOPK>
__device__ __noinline__ void race_fallback_emit(const SweepCtx& x, int b, const DrawState& st,
                                                bool vec, int fl, uint4* sb) {
  KeyTop2 t = key_top2_empty();
  float th = -kInf;
  race_draw<DT, TOPK>(x, b, st, false, 0, x.V, vec, t, th, nullptr, sb);  // p_n: keys of its own
  t = key_warp(t);
  race_emit<DT>(x, b, st, t, false, fl | SV_FLAG_RESIDUAL_FALLBACK);
}

}  // namespace sv
