// sv_decide.cuh -- the decision of one round for one batch row (accept test,
// prefix, set-up of the draw), shared by the logits path and the fused LM-head
// path, plus the row-combine of chunk partials.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"

namespace sv {

__device__ __forceinline__ float inv_temperature(float T) { return 1.0f / T; }
__device__ __forceinline__ float log2_scale(float invT) { return invT * kLog2e; }
__device__ __forceinline__ bool temperature_ok(float T) { return T > 0.0f && T < kInf; }

// Row k of batch row b: target rows k = 0..gamma, draft rows k = gamma+1..2gamma.
template <int DT>
__device__ __forceinline__ const char* row_ptr(const void* zt, const void* zd, int b, int k,
                                               int gamma, int64_t V) {
  constexpr int kBytes = (DT == SV_F32) ? 4 : 2;
  if (k <= gamma)
    return reinterpret_cast<const char*>(zt) + (((int64_t)b * (gamma + 1) + k) * V) * kBytes;
  return reinterpret_cast<const char*>(zd) + (((int64_t)b * gamma + (k - gamma - 1)) * V) * kBytes;
}

// --------------------------------------------------------------------------
// Row combine and decision (the start of k_race and k_draw; k_lm_finish on the fused path).
// --------------------------------------------------------------------------
struct SweepCtx {
  const void* zt;
  const void* zd;
  const int32_t* xt;
  int B, gamma;
  int64_t V;
  float temperature;
  const float* row_T;
  uint64_t seed, round;
  int np;                // partials per logit row: 4 KB chunks (vector sweep) or splits
  float2* part;          // [B][R1][np] (largest logit as given, sum of 2^(y - max y))
  RowStat* rowstat;      // [B][R1]
  DrawState* state;      // [B]
  int32_t* out_tokens;
  int32_t* out_counts;
  float* out_p;
  float* out_q;
  uint8_t* out_flags;
  float inv_lenience;    // 1/l of the lenient comparison u <= p/(l q); 1: the exact round
  const float* thr;      // [B][R1] top-k thresholds (logits below have weight 0) or null
  uint32_t* done;        // [B] arrival counters of the inverse-transform draw, zeroed by
                         // every sweep
  uint32_t* thw;         // [B][kThwStride] the race's shared lower bound on its second-best
                         // key (float bits, 0: none yet; word 0 of each row's line), zeroed
                         // by every sweep
};

// The partials of one logit row, in row order: [np] consecutive entries.  Each
// covers a piece of the row counted from the row's start (a 4 KB chunk, or a
// kChunkSweep-logit split), so they do not depend on where the row sits in
// memory.
struct RowParts {
  float2* p;
  int n;
  __device__ __forceinline__ float2* at(int j) const { return p + j; }
};
template <int DT>
__device__ __forceinline__ RowParts row_parts(const SweepCtx& x, int64_t rid) {
  return RowParts{x.part + rid * x.np, x.np};
}

// Online (max, sum) of a lane's share of one row's chunk partials.
// A partial is (largest logit z, sum of 2^(y - z c)) with c the row's scale; the
// fused LM head's partials carry the scaled max itself (c = 1).
struct RowAcc {
  float m, s;
  int bits;
  float z;
};
__device__ __forceinline__ RowAcc row_acc_init() { return RowAcc{-kInf, 0.0f, 0, -kInf}; }
__device__ __forceinline__ void row_acc_add(RowAcc& a, float2 p, float c) {
  if (p.x != p.x) a.bits |= kRowNaN;
  if (p.y < 0.0f) a.bits |= kRowTimeout;
  a.z = fmaxf(a.z, p.x);
  const float m = p.x * c;  // the partial's own scaled max, bit for bit
  if (m > a.m) {
    a.s = (a.m == -kInf) ? 0.0f : a.s * exp2f(a.m - m);
    a.m = m;
  }
  if (m > -kInf) a.s += p.y * exp2f(m - a.m);
}
// The warp's combined statistics, kept by lane 0 and written to *out.
__device__ __forceinline__ RowStat row_acc_finish(const RowAcc& a, RowStat* out) {
  const int lane = threadIdx.x & 31;
  const float M = warp_max(a.m);
  float sl = (a.m > -kInf) ? a.s * exp2f(a.m - M) : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sl += __shfl_xor_sync(0xffffffffu, sl, o);
  const int bits = __reduce_or_sync(0xffffffffu, a.bits);
  RowStat rs;
  rs.mc = M;
  rs.bits = bits;
  rs.s = (bits & kRowNaN) ? CUDART_NAN_F : sl;
  rs.z = warp_max(a.z);
  if (lane == 0 && out) *out = rs;
  return rs;
}

// Row statistics of row r from its chunk partials (one warp, all loads of a
// lane in flight together), kept by lane 0 and written to rowstat[r].
__device__ __forceinline__ RowStat combine_row(const float2* pr, int nch, RowStat* out,
                                               float c) {
  const int lane = threadIdx.x & 31;
  RowAcc a = row_acc_init();
#pragma unroll 4
  for (int j = lane; j < nch; j += 32) row_acc_add(a, __ldcg(pr + j), c);
  return row_acc_finish(a, out);
}

// The same over a row's partials in any layout.
__device__ __forceinline__ RowStat combine_parts(const RowParts& p, RowStat* out, float c) {
  const int lane = threadIdx.x & 31;
  RowAcc a = row_acc_init();
#pragma unroll 4
  for (int j = lane; j < p.n; j += 32) row_acc_add(a, __ldcg(p.at(j)), c);
  return row_acc_finish(a, out);
}

// Two rows by one warp with the loads of both in flight together (p1.n may be
// 0: no second row); each row's arithmetic is that of combine_row.
__device__ __forceinline__ void combine_parts2(const RowParts& p0, const RowParts& p1,
                                               RowStat* out0, RowStat* out1, RowStat& r0,
                                               RowStat& r1, float c) {
  const int lane = threadIdx.x & 31;
  RowAcc a0 = row_acc_init(), a1 = row_acc_init();
  const int n = max(p0.n, p1.n);
#pragma unroll 4
  for (int j = lane; j < n; j += 32) {
    const float2 x0 = (j < p0.n) ? __ldcg(p0.at(j)) : make_float2(-kInf, 0.0f);
    const float2 x1 = (j < p1.n) ? __ldcg(p1.at(j)) : make_float2(-kInf, 0.0f);
    row_acc_add(a0, x0, c);
    row_acc_add(a1, x1, c);
  }
  r0 = row_acc_finish(a0, out0);
  r1 = row_acc_finish(a1, p1.n ? out1 : nullptr);
}

// log2 of the unnormalised probability, e = z c - mc, carried in two floats:
// z c = ph + pl exactly (FMA residual) and ph - mc by TwoSum, so e = hi + lo
// to about 2^-48 relative.
struct Exp2 {
  float hi, lo;
};
__device__ __forceinline__ Exp2 exponent_at(float z, float c, float mc) {
  const float ph = z * c;
  const float pl = fmaf(z, c, -ph);
  const float a = ph - mc;
  const float bv = a - ph;
  const float err = (ph - (a - bv)) + (-mc - bv);
  return Exp2{a, err + pl};
}
// p(x) from its exponent and the row sum (0 for a -inf logit or an empty row).
__device__ __forceinline__ float prob_from(float z, const Exp2& e, float s) {
  if (!(s > 0.0f)) return (s == 0.0f) ? 0.0f : s;  // NaN stays NaN
  if (z == -kInf) return 0.0f;
  return exp2f(e.hi) * fmaf(e.lo, kLn2, 1.0f) / s;
}

// The decision for batch row b (one warp): accept test, prefix, draw set-up.
// srs[k] holds the statistics of row k of the batch row.  With `emit` the
// warp writes the outputs (prefix, counts, p, q, the draw state, the flags of a
// finished row); the draw state also goes to *st_out (shared memory) if given.
// Draft token i of a batch row and the two logits at it.
struct DraftAt {
  int32_t x;
  float zt, zd;
};

template <int DT>
__device__ void decide_batch_row(const SweepCtx& x, int b, const RowStat* srs,
                                 const DraftAt* sda, bool emit = true,
                                 DrawState* st_out = nullptr) {
  const int lane = threadIdx.x & 31;
  const int gamma = x.gamma;
  const int64_t V = x.V;
  const int R1 = 2 * gamma + 1;
  const float T = x.row_T ? __ldg(x.row_T + b) : x.temperature;
  const float invT = inv_temperature(T);
  const float c = log2_scale(invT);

  int fl = 0;
  for (int k = lane; k < R1; k += 32) {
    const RowStat v = srs[k];
    if (v.mc == -kInf) fl |= SV_FLAG_ZERO_MASS;
    if (!(v.s < kInf) || v.mc == kInf || !temperature_ok(T)) fl |= SV_FLAG_NONFINITE;
    if (v.bits & kRowTimeout) fl |= SV_FLAG_TIMEOUT | SV_FLAG_NONFINITE;
  }
  bool accept = false, bad = false, qzero = false;
  float P = 0.0f, Q = 0.0f;
  int32_t xi = 0;
  if (lane < gamma) {
    const DraftAt da = sda[lane];
    xi = da.x;
    bad = (xi < 0 || (int64_t)xi >= V);
    float ratio = CUDART_NAN_F;  // a bad token: p = q = 0, rejected
    if (!bad) {
      const float zx = da.zt;
      const float zy = da.zd;
      const RowStat rt = srs[lane], rd = srs[gamma + 1 + lane];
      const float st_ = rt.s, sd_ = rd.s;
      const Exp2 ep = exponent_at(zx, c, rt.mc), eq = exponent_at(zy, c, rd.mc);
      P = prob_from(zx, ep, st_);
      Q = prob_from(zy, eq, sd_);
      // p/q from the exponent difference (no underflow of p and q themselves);
      // q = 0 with p > 0 gives inf (accept), p = q = 0 gives NaN (reject)
      const bool p0 = !(st_ > 0.0f) || zx == -kInf, q0 = !(sd_ > 0.0f) || zy == -kInf;
      if (st_ != st_ || sd_ != sd_) {
        ratio = CUDART_NAN_F;
      } else if (p0 || q0) {
        ratio = p0 ? (q0 ? CUDART_NAN_F : 0.0f) : kInf;
      } else {
        const float d = (ep.hi - eq.hi) + (ep.lo - eq.lo);
        ratio = exp2f(d) * __fdiv_rn(sd_, st_) * x.inv_lenience;
      }
      qzero = q0 || !(sd_ == sd_);
    } else {
      qzero = true;
    }
    const uint4 rnd = philox4x32_10(sv_counter(0u, 0u, (uint32_t)lane, (uint32_t)b, x.round),
                                    (uint32_t)x.seed, (uint32_t)(x.seed >> 32));
    accept = (sv_u01(rnd.x) <= ratio);
    if (emit && x.out_p) x.out_p[(int64_t)b * gamma + lane] = P;
    if (emit && x.out_q) x.out_q[(int64_t)b * gamma + lane] = Q;
  }
  const unsigned rej = ~__ballot_sync(0xffffffffu, accept);
  const int n = (rej == 0u) ? 32 : min(__ffs((int)rej) - 1, gamma);
  // flags: bad tokens anywhere, q(x) = 0 at a tested position (i <= n, i < gamma)
  if (__ballot_sync(0xffffffffu, bad)) fl |= SV_FLAG_BAD_TOKEN;
  if (__ballot_sync(0xffffffffu, lane < gamma && lane <= n && qzero)) fl |= SV_FLAG_NONFINITE;
  fl = __reduce_or_sync(0xffffffffu, fl);
  int32_t* tok = x.out_tokens + (int64_t)b * (gamma + 1);
  if (emit) {
    if (lane < n) tok[lane] = xi;  // n <= gamma <= 32
    for (int i = lane; i <= gamma; i += 32)
      if (i > n) tok[i] = -1;
  }
  if (lane == 0) {
    // set up the draw of the target's own token
    const float mct = srs[n].mc;
    const float St = srs[n].s;
    DrawState st{};
    st.pos = n;
    st.zmt = srs[n].z;
    st.zmd = (n < gamma) ? srs[gamma + 1 + n].z : -kInf;
    st.c = c;
    st.invT = invT;
    st.tt = x.thr ? x.thr[(int64_t)b * R1 + n] : -kInf;
    st.td = (x.thr && n < gamma) ? x.thr[(int64_t)b * R1 + gamma + 1 + n] : -kInf;
    const bool t_ok = (St > 0.0f) && (St < kInf) && (mct < kInf);
    if (n == gamma) {
      if (t_ok) {
        st.mode = kDrawSampleRow;
        st.mct = mct;
        st.st = St;
      } else {
        st.mode = kDrawDone;
      }
    } else {
      const float mcd = srs[gamma + 1 + n].mc;
      const float Sd = srs[gamma + 1 + n].s;
      const bool d_nonfinite = !(Sd < kInf) || mcd == kInf;
      if (!t_ok || d_nonfinite) {
        // p_n has no mass (or a row is not finite): the residual and its fallback
        // are empty; token 0
        st.mode = kDrawDone;
        if (St == 0.0f) fl |= SV_FLAG_RESIDUAL_FALLBACK;
      } else if (Sd == 0.0f) {
        st.mode = kDrawSampleRow;  // q_n has no mass: max(0, p_n - q_n) = p_n
        st.mct = mct;
        st.st = St;
      } else {
        st.mode = kDrawResidual;
        st.mct = mct;
        st.st = St;
        st.mcd = mcd;
        st.sd = Sd;
        st.K = (mct - mcd) + (log2f(St) - log2f(Sd));
      }
    }
    st.flags = fl;
    if (st_out) *st_out = st;
    if (emit) {
      x.state[b] = st;
      x.out_counts[b] = n;
      if (st.mode == kDrawDone) {
        tok[n] = 0;
        if (x.out_flags) x.out_flags[b] = (uint8_t)fl;
      }
    }
  }
}

}  // namespace sv
