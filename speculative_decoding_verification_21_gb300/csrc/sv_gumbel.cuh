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
// and the weights need only be known up to a factor common to the row.  Lanes
// keep their two best entries, compared by cross products (no division); the
// warp, then the merge, keep the best two of those.  When the two best keys lie
// within 2^-10 of each other, they are re-decided in double precision from the
// logits (the key's definition, log w + g), so that the winner differs from an
// exact evaluation only where the exact keys themselves are within the
// rounding of the row sums.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_decide.cuh"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_plan.h"

namespace sv {

// One entry of the race: weight w (>= 0), exponential variate E (> 0), index.
struct RaceCand {
  float w, E;
  int idx;
};
struct RaceTop2 {
  RaceCand a, b;  // best, second best
};

__device__ __forceinline__ RaceCand race_empty() { return RaceCand{0.0f, 1.0f, -1}; }
__device__ __forceinline__ RaceTop2 race_top2_empty() { return RaceTop2{race_empty(), race_empty()}; }

// w/E beats c (w_c/E_c): larger ratio, ties to the lower index (-1 loses).
__device__ __forceinline__ bool race_beats(float w, float E, int i, const RaceCand& c) {
  const float l = w * c.E, r = c.w * E;
  return l > r || (l == r && (unsigned)i < (unsigned)c.idx);
}

__device__ __forceinline__ void race_insert(RaceTop2& t, float w, float E, int i) {
  if (!(w > 0.0f)) return;
  if (race_beats(w, E, i, t.b)) {
    if (race_beats(w, E, i, t.a)) {
      t.b = t.a;
      t.a = RaceCand{w, E, i};
    } else {
      t.b = RaceCand{w, E, i};
    }
  }
}

__device__ __forceinline__ void race_insert(RaceTop2& t, const RaceCand& c) {
  if (c.idx >= 0) race_insert(t, c.w, c.E, c.idx);
}

__device__ __forceinline__ RaceCand race_shfl(const RaceCand& c, int o) {
  return RaceCand{__shfl_xor_sync(0xffffffffu, c.w, o), __shfl_xor_sync(0xffffffffu, c.E, o),
                  __shfl_xor_sync(0xffffffffu, c.idx, o)};
}

// The best two of the warp's lanes (the same in every lane).
__device__ __forceinline__ RaceTop2 race_warp(RaceTop2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const RaceCand a = race_shfl(t.a, o), b = race_shfl(t.b, o);
    race_insert(t, a);
    race_insert(t, b);
  }
  return t;
}

// A finished candidate: its key w/E as a float and its index (-1: none).
struct KeyIdx {
  float k;
  int i;
};
__device__ __forceinline__ KeyIdx race_key(const RaceCand& c) {
  return (c.idx < 0) ? KeyIdx{-1.0f, -1} : KeyIdx{__fdiv_rn(c.w, c.E), c.idx};
}
__device__ __forceinline__ bool key_beats(const KeyIdx& a, const KeyIdx& b) {
  if (a.i < 0) return false;
  if (b.i < 0) return true;
  return a.k > b.k || (a.k == b.k && a.i < b.i);
}
struct KeyTop2 {
  KeyIdx a, b;
};
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
  return KeyIdx{__uint_as_float((uint32_t)w), (int)(uint32_t)(w >> 32) - 1};
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

// One run of eight consecutive entries v0..v0+7 of the race: weights of the
// residual max(0, p_n - q_n) (RESID) and of p_n, up to the common factor
// 2^-mct / St, and their exponential variates from the Philox blocks of the
// run.  Entries past V carry -inf logits (weight 0); below a row's top-k
// threshold the weight is 0 (TOPK).
template <bool RESID, bool TOPK>
__device__ __forceinline__ void race_run8(const float (&zt)[8], const float (&zd)[8], int64_t v0,
                                          const DrawState& st, float kd, uint32_t k0, uint32_t k1,
                                          uint32_t c1, uint32_t c2, uint32_t c3, RaceTop2& tr,
                                          RaceTop2& tp) {
  uint32_t r[8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 x = philox4x32_10(make_uint4((uint32_t)(v0 >> 2) + (uint32_t)h, c1, c2, c3), k0, k1);
    r[4 * h] = x.x;
    r[4 * h + 1] = x.y;
    r[4 * h + 2] = x.z;
    r[4 * h + 3] = x.w;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float a = zt[e];
    if (TOPK && a < st.tt) a = -kInf;
    const float et = ex2(__fmaf_rn(a, st.c, -st.mct));
    const float E = neglog2_u(r[e]);
    const int v = (int)(v0 + e);
    if (RESID) {
      float d = zd[e];
      if (TOPK && d < st.td) d = -kInf;
      const float ed = ex2(__fmaf_rn(d, st.c, kd));
      race_insert(tr, (et > ed) ? __fsub_rn(et, ed) : 0.0f, E, v);
    }
    race_insert(tp, et, E, v);
  }
}

// The race over entries [lo, hi) of row n (and of draft row n for a residual):
// lane l takes the runs of eight at lo + 8 (l + 32 i), kRunsInFlight of them
// with their loads in flight together.  lo is a multiple of 8; `vec`: rows start
// on 16-byte boundaries (16-byte loads).
constexpr int kRaceRunsInFlight = 2;
template <int DT, bool RESID, bool TOPK>
__device__ __forceinline__ void race_range(const char* rt, const char* rd, int64_t lo, int64_t hi,
                                           int64_t V, bool vec, const DrawState& st, float kd,
                                           uint64_t seed, uint64_t round, int b, RaceTop2& tr,
                                           RaceTop2& tp) {
  const int lane = threadIdx.x & 31;
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  const uint32_t c1 = (1u << 24) | (uint32_t)st.pos, c2 = (uint32_t)b, c3 = (uint32_t)round;
  const int nrun = (int)((hi - lo + 7) >> 3);
  for (int r0 = 0; r0 < nrun; r0 += 32 * kRaceRunsInFlight) {
    Raw8<DT> xt[kRaceRunsInFlight], xd[kRaceRunsInFlight];
#pragma unroll
    for (int u = 0; u < kRaceRunsInFlight; ++u) {
      const int r = r0 + lane + 32 * u;
      if (r < nrun) {
        const int64_t v0 = lo + 8 * (int64_t)r;
        xt[u] = load_raw8<DT>(rt, v0, V, vec, -kInf);
        if (RESID) xd[u] = load_raw8<DT>(rd, v0, V, vec, -kInf);
      }
    }
#pragma unroll
    for (int u = 0; u < kRaceRunsInFlight; ++u) {
      const int r = r0 + lane + 32 * u;
      if (r < nrun) {
        float zt[8], zd[8];
        unpack8<DT>(xt[u], zt);
        if (RESID) unpack8<DT>(xd[u], zd);
        race_run8<RESID, TOPK>(zt, zd, lo + 8 * (int64_t)r, st, kd, k0, k1, c1, c2, c3, tr, tp);
      }
    }
  }
}

// The token from the best two of the residual race (R) and of p_n (P) over the
// whole row: the residual's when it has a positive entry, else p_n's with the
// fallback flag; re-decided in double near a tie; token 0 and ZERO_MASS when
// there is none.  One warp; lane 0 writes the token and the flags.
template <int DT>
__device__ void race_emit(const SweepCtx& x, int b, const DrawState& st, const KeyTop2& R,
                          const KeyTop2& P, bool lost) {
  const int lane = threadIdx.x & 31;
  const int gamma = x.gamma;
  const int64_t V = x.V;
  const bool resid = st.mode == kDrawResidual;
  int fl = st.flags;
  bool use_resid = false;
  KeyTop2 T = P;
  if (resid) {
    if (R.a.i >= 0) {
      T = R;
      use_resid = true;
    } else {
      fl |= SV_FLAG_RESIDUAL_FALLBACK;  // no positive residual entry: p_n, the same noise
    }
  }
  const char* rt = row_ptr<DT>(x.zt, x.zd, b, st.pos, gamma, V);
  const char* rd = resid ? row_ptr<DT>(x.zt, x.zd, b, gamma + 1 + st.pos, gamma, V) : rt;
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
    if (lost) fl |= SV_FLAG_TIMEOUT | SV_FLAG_NONFINITE;
    if (tok < 0 || (int64_t)tok >= V) {
      tok = 0;
      fl |= SV_FLAG_ZERO_MASS;
    }
    x.out_tokens[(int64_t)b * (gamma + 1) + st.pos] = tok;
    if (x.out_flags) x.out_flags[b] = (uint8_t)fl;
  }
}

}  // namespace sv
