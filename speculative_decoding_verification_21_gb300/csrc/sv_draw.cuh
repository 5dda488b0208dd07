// sv_draw.cuh -- the draw of the target's own token: Gumbel-max in the
// exponential-race form over 4-entry Philox groups, top-2 merges and the
// double-precision re-decision of near ties.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"

namespace sv {

struct DrawArgs {
  const void* zt;
  const void* zd;
  int B, gamma;
  int64_t V;
  uint64_t seed, round;
  DrawState* state;        // [B] (written by the first draw CTA of each batch row)
  uint32_t* alpha_cnt;     // [B] counters of the optional overlap kernel, zeroed here
  Top2* part3;             // [B][nsplit3]
  int nsplit3;             // CTAs per batch row
  int gpc;                 // 4-entry groups per CTA
  int32_t* out_tokens;
  uint8_t* out_flags;
};

// Keys of one 4-entry Philox group v = v0 .. v0+3 from already loaded logits;
// the running best is kept as a fraction num/den and compared by cross-products.
// With TOPK, logits below the rows' top-k thresholds (st.tt, st.td) have weight 0.
template <bool RESID, bool TOPK>
__device__ __forceinline__ void draw_keys(const float* ztv, const float* zdv, int v0,
                                          const DrawState& st, uint4 rnd, float& bn, float& bd,
                                          int& bi) {
  const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float zt = (TOPK && ztv[e] < st.tt) ? -kInf : ztv[e];
    const float et = ex2(fmaf(zt, st.c, -st.mct));
    float wgt;
    bool cand;
    if (RESID) {
      // weight p - q up to the common factor 2^-mct / St: 2^(zt c - mct) minus
      // 2^(zd c + K - mct) (K = log2 of the normaliser ratio); p > q iff the
      // first is larger.  Where p and q nearly agree the difference loses
      // relative precision, but only for weights far below the top keys, and any
      // misordering of the top two is re-decided in double (refine)
      const float zd = (TOPK && zdv[e] < st.td) ? -kInf : zdv[e];
      const float ed = ex2(fmaf(zd, st.c, st.K - st.mct));
      cand = et > ed;
      wgt = et - ed;
    } else {
      cand = zt > -kInf;
      wgt = et;
    }
    const float E = neglog2_u(rr[e]);
    if (cand && wgt * bd > bn * E) {
      bn = wgt;
      bd = E;
      bi = v0 + e;
    }
  }
}

// Raw 4-entry group of a row (bf16: 8 bytes, fp32: 16 bytes) and its widening.
template <int DT>
struct Group;
template <>
struct Group<SV_BF16> {
  uint2 v;
};
template <>
struct Group<SV_F32> {
  float4 v;
};

template <int DT>
__device__ __forceinline__ Group<DT> load_group(const char* row, int g, int V, bool vec_ok,
                                                float pad) {
  Group<DT> out;
  const int v0 = 4 * g;
  if (vec_ok && v0 + 3 < V) {
    if constexpr (DT == SV_F32)
      out.v = __ldg(reinterpret_cast<const float4*>(row) + g);
    else
      out.v = __ldg(reinterpret_cast<const uint2*>(row) + g);
  } else {
    float f[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = (v0 + e < V) ? load_logit<DT>(row, v0 + e) : pad;
    if constexpr (DT == SV_F32) {
      out.v = make_float4(f[0], f[1], f[2], f[3]);
    } else {
      // re-pack as bf16 bits (the values are bf16-exact)
      out.v.x = (__float_as_uint(f[0]) >> 16) | (__float_as_uint(f[1]) & 0xFFFF0000u);
      out.v.y = (__float_as_uint(f[2]) >> 16) | (__float_as_uint(f[3]) & 0xFFFF0000u);
    }
  }
  return out;
}

template <int DT>
__device__ __forceinline__ void widen(const Group<DT>& g, float* f) {
  if constexpr (DT == SV_F32) {
    f[0] = g.v.x; f[1] = g.v.y; f[2] = g.v.z; f[3] = g.v.w;
  } else {
    f[0] = bf16lo(g.v.x); f[1] = bf16hi(g.v.x); f[2] = bf16lo(g.v.y); f[3] = bf16hi(g.v.y);
  }
}

// This thread's best key over groups [g0, g1); all loads of a step in flight together.
template <int DT, bool RESID, bool TOPK>
__device__ __forceinline__ KI draw_range(const char* rt, const char* rd, int g0, int g1, int V,
                                         bool vec_ok, const DrawState& st, uint32_t b,
                                         const PhiloxKeys& pk, uint64_t round) {
  float bn = -1.0f, bd = 1.0f;
  int bi = -1;
  constexpr int U = 4;  // 4 groups in flight per row keeps 64 registers: 4 CTAs per SM
  const int stride = (int)blockDim.x;
  for (int g = g0 + (int)threadIdx.x; g < g1; g += U * stride) {
    Group<DT> gt[U], gd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gg = g + u * stride;
      if (gg < g1) {
        gt[u] = load_group<DT>(rt, gg, V, vec_ok, -kInf);
        if (RESID) gd[u] = load_group<DT>(rd, gg, V, vec_ok, 0.0f);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gg = g + u * stride;
      if (gg < g1) {
        float zt4[4], zd4[4];
        widen<DT>(gt[u], zt4);
        if (RESID) widen<DT>(gd[u], zd4);
        const uint4 rnd = philox_rk(sv_counter((uint32_t)gg, 1u, (uint32_t)st.pos, b, round), pk);
        draw_keys<RESID, TOPK>(zt4, zd4, 4 * gg, st, rnd, bn, bd, bi);
      }
    }
  }
  KI r;
  r.i = bi;
  r.k = (bi >= 0) ? bn / bd : -kInf;
  return r;
}

// Double-precision key with the oracle-level definition, for the refinement.
template <int DT>
__device__ double draw_key_f64(const char* rt, const char* rd, int64_t v, const DrawState& st,
                               bool resid, uint32_t b, uint64_t seed, uint64_t round) {
  const uint4 rnd = philox4x32_10(sv_counter((uint32_t)(v >> 2), 1u, (uint32_t)st.pos, b, round),
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t lanes[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  const double lnE = log(sv_neglog_u_f64(lanes[v & 3]));
  const float zt32 = load_logit<DT>(rt, v);
  const double zt = (zt32 < st.tt) ? -CUDART_INF : (double)zt32;  // top-k: below the threshold
  if (!resid) return zt * (double)st.invT - lnE;
  const float zd32 = load_logit<DT>(rd, v);
  const double zd = (zd32 < st.td) ? -CUDART_INF : (double)zd32;
  const double P = exp2(zt * (double)st.c - (double)st.mct) / st.st;
  const double Q = exp2(zd * (double)st.c - (double)st.mcd) / st.sd;
  const double r = P - Q;
  return (r > 0.0) ? log(r) - lnE : -CUDART_INF;
}

__device__ __forceinline__ Top2 block_top2(KI mine) {
  __shared__ Top2 sm[kThreads / 32];
  Top2 t{mine, KI{-kInf, -1}};
  t = warp_reduce_top2(t);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sm[warp] = t;
  __syncthreads();
  Top2 r{KI{-kInf, -1}, KI{-kInf, -1}};
  if (warp == 0) {
    if (lane < (int)(blockDim.x >> 5)) r = sm[lane];
    r = warp_reduce_top2(r);
  }
  return r;  // valid in warp 0
}

template <int DT>
__device__ int refine(const Top2& t, const char* rt, const char* rd, const DrawState& st,
                      bool resid, uint32_t b, uint64_t seed, uint64_t round) {
  if (t.a.i < 0) return -1;
  if (t.b.i < 0 || !(t.a.k - t.b.k <= t.a.k * 0x1p-10f)) return t.a.i;
  const double ka = draw_key_f64<DT>(rt, rd, t.a.i, st, resid, b, seed, round);
  const double kb = draw_key_f64<DT>(rt, rd, t.b.i, st, resid, b, seed, round);
  if (kb > ka || (kb == ka && t.b.i < t.a.i)) return t.b.i;
  return t.a.i;
}

}  // namespace sv
