// sv_sampling.cu -- sampling verify on sm_103a.
//
// One round for B independent batch rows, after Algorithm 1 of "Fast Inference
// from Transformers via Speculative Decoding" (section "The loop: draft, verify
// in one pass, keep a prefix") and the course notes "Speculative Decoding"
// ("The algorithm"):
//
//   k_sweep   every CTA streams one chunk of one of the 2*gamma+1 logit rows of
//             a batch row with 16-byte loads and keeps an online (max, sum of
//             2^(y - max)) with y = z * T^-1 * log2 e; one partial per CTA.
//   k_decide  one CTA per batch row: combines the partials (double), gathers
//             p(x_i), q(x_i), draws u_i, accepts iff u_i <= p/q, finds the first
//             rejection with a warp ballot, writes the accepted prefix, and sets
//             up the draw of the target's own token.
//   k_draw    Gumbel-max over the bonus row p_gamma or the residual
//             max(0, p_n - q_n), in the exponential-race form argmax w_v / E_v
//             (E_v = -ln u_v), which has the same argmax as log w_v + g_v; the
//             last CTA of a batch row merges the per-CTA top-2 and, when the two
//             best fp32 keys are within 2^-10 of each other, re-decides between
//             them in double with the oracle-level definition.
//   k_alpha   optional overlap sum_v min(p_i, q_i), "The acceptance rate is the
//             overlap of p and q".
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

// Visit elements [lo, hi) of a row: an unaligned head as scalars, then 16-byte
// vectors, then the tail.  Every thread sees its own elements in increasing
// index order.  `row` must be a row start; `f_vec(v0, vec)` / `f_one(v, z)`.
template <int DT, int UNROLL, class FV, class FS>
__device__ __forceinline__ void for_each_in_chunk(const char* row, int64_t lo, int64_t hi,
                                                  FV&& f_vec, FS&& f_one) {
  constexpr int VE = VecInfo<DT>::kElems;
  constexpr int kBytes = (DT == SV_F32) ? 4 : 2;
  const int tid = threadIdx.x;
  // first element at or after lo whose address is 16-byte aligned
  const uintptr_t addr_lo = reinterpret_cast<uintptr_t>(row) + lo * kBytes;
  const int64_t head = (int64_t)(((16 - (addr_lo & 15)) & 15) / kBytes);
  int64_t a0 = lo + head;
  if (a0 > hi) a0 = hi;
  const int64_t nvec = (hi - a0) / VE;
  const int64_t a1 = a0 + nvec * VE;
  for (int64_t v = lo + tid; v < a0; v += blockDim.x) f_one(v, load_logit<DT>(row, v));
  const uint4* vp = reinterpret_cast<const uint4*>(row + a0 * kBytes);
  for (int64_t j = tid; j < nvec; j += (int64_t)UNROLL * blockDim.x) {
    uint4 buf[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t jj = j + (int64_t)u * blockDim.x;
      if (jj < nvec) buf[u] = ld_stream16(vp + jj);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t jj = j + (int64_t)u * blockDim.x;
      if (jj < nvec) f_vec(a0 + jj * VE, buf[u]);
    }
  }
  for (int64_t v = a1 + tid; v < hi; v += blockDim.x) f_one(v, load_logit<DT>(row, v));
}

// --------------------------------------------------------------------------
// k_sweep: online softmax statistics per (row, chunk).
// --------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads, 4)
k_sweep(const void* __restrict__ zt, const void* __restrict__ zd, int gamma, int64_t V,
        float temperature, const float* __restrict__ row_T, int nsplit,
        float2* __restrict__ part) {
  const int R1 = 2 * gamma + 1;
  const int64_t item = blockIdx.x;  // (row, split) flattened: rows are B*R1
  const int64_t r = item / nsplit;
  const int split = (int)(item - r * nsplit);
  const int b = (int)(r / R1), k = (int)(r - (int64_t)b * R1);
  const float T = row_T ? __ldg(row_T + b) : temperature;
  const float c = log2_scale(inv_temperature(T));
  const char* row = row_ptr<DT>(zt, zd, b, k, gamma, V);
  const int64_t lo = (int64_t)split * kChunkSweep;
  const int64_t hi = min(V, lo + kChunkSweep);

  float zmax = -kInf, mc = -kInf, s = 0.0f;
  auto raise_max = [&](float m) {
    if (m > zmax) {
      const float mcn = m * c;
      s = (zmax == -kInf) ? 0.0f : s * ex2(mc - mcn);
      mc = mcn;
      zmax = m;
    }
  };
  for_each_in_chunk<DT, 4>(
      row, lo, hi,
      [&](int64_t, const uint4& vec) {
        raise_max(vmax<DT>(vec));
        if (zmax > -kInf) {
          float f[VecInfo<DT>::kElems];
          unpack<DT>(vec, f);
          float acc = 0.0f;
#pragma unroll
          for (int e = 0; e < VecInfo<DT>::kElems; ++e) acc += ex2(fmaf(f[e], c, -mc));
          s += acc;
        }
      },
      [&](int64_t, float z) {
        raise_max(z);
        if (zmax > -kInf) s += ex2(fmaf(z, c, -mc));
      });

  MS v = warp_reduce_ms(MS{mc, s});
  __shared__ MS sm[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = (lane < (int)(blockDim.x >> 5)) ? sm[lane] : MS{-kInf, 0.0f};
    v = warp_reduce_ms(v);
    if (lane == 0) part[item] = make_float2(v.m, v.s);
  }
}

// --------------------------------------------------------------------------
// k_decide: one CTA (128 threads) per batch row.
// --------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(128)
k_decide(const void* __restrict__ zt, const void* __restrict__ zd,
         const int32_t* __restrict__ xt, int gamma, int64_t V, float temperature,
         const float* __restrict__ row_T, uint64_t seed, uint64_t round, int nsplit,
         const float2* __restrict__ part, RowStat* __restrict__ rowstat,
         DrawState* __restrict__ state, uint32_t* __restrict__ counters, int B,
         int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_counts,
         float* __restrict__ out_p, float* __restrict__ out_q, uint8_t* __restrict__ out_flags) {
  const int b = blockIdx.x;
  const int R1 = 2 * gamma + 1;
  const int tid = threadIdx.x;
  // the draw and overlap kernels that follow count their CTAs here: start at zero
  // whatever an earlier call (of any shape) left in this part of the workspace
  if (tid == 0) {
    counters[b] = 0u;
    counters[B + b] = 0u;
  }
  __shared__ float s_mc[65];
  __shared__ double s_s[65];
  __shared__ int s_flag;
  if (tid == 0) s_flag = 0;
  const float T = row_T ? __ldg(row_T + b) : temperature;
  const float invT = inv_temperature(T);
  const float c = log2_scale(invT);
  __syncthreads();

  // 1. combine the split partials of every row (double sum)
  for (int k = tid; k < R1; k += blockDim.x) {
    const float2* pr = part + ((int64_t)b * R1 + k) * nsplit;
    float m = -kInf;
    bool nan_m = false;
    for (int j = 0; j < nsplit; ++j) {
      const float mj = pr[j].x;
      nan_m |= (mj != mj);
      m = fmaxf(m, mj);
    }
    double s = 0.0;
    if (m > -kInf) {
      for (int j = 0; j < nsplit; ++j) {
        const float2 pj = pr[j];
        if (pj.x > -kInf) s += (double)pj.y * exp2((double)pj.x - (double)m);
        else if (pj.y != 0.0f) s += (double)pj.y;  // NaN/inf propagate
      }
    }
    if (nan_m) s = CUDART_NAN;
    s_mc[k] = m;
    s_s[k] = s;
    rowstat[(int64_t)b * R1 + k] = RowStat{m, 0.0f, s};
    int f = 0;
    if (m == -kInf) f |= SV_FLAG_ZERO_MASS;
    if (!(s < CUDART_INF) || m == kInf || !temperature_ok(T)) f |= SV_FLAG_NONFINITE;
    if (f) atomicOr(&s_flag, f);
  }
  __syncthreads();

  // 2. accept test on warp 0, one lane per draft position
  if (tid < 32) {
    const int lane = tid;
    bool accept = false;
    double P = 0.0, Q = 0.0;
    int bad = 0;
    if (lane < gamma) {
      const int32_t x = __ldg(xt + (int64_t)b * gamma + lane);
      if (x < 0 || (int64_t)x >= V) {
        bad = 1;
      } else {
        const double cd = (double)c;
        const double zx = (double)load_logit<DT>(row_ptr<DT>(zt, zd, b, lane, gamma, V), x);
        const double zy =
            (double)load_logit<DT>(row_ptr<DT>(zt, zd, b, gamma + 1 + lane, gamma, V), x);
        const double St = s_s[lane], Sd = s_s[gamma + 1 + lane];
        P = (St > 0.0) ? exp2(zx * cd - (double)s_mc[lane]) / St : (St == 0.0 ? 0.0 : St);
        Q = (Sd > 0.0) ? exp2(zy * cd - (double)s_mc[gamma + 1 + lane]) / Sd
                       : (Sd == 0.0 ? 0.0 : Sd);
      }
      const double ratio = P / Q;  // IEEE: p/0 = inf (accept), 0/0 = NaN (reject)
      const uint4 rnd = philox4x32_10(sv_counter(0u, 0u, (uint32_t)lane, (uint32_t)b, round),
                                      (uint32_t)seed, (uint32_t)(seed >> 32));
      const double u = (double)sv_u01(rnd.x);
      accept = (u <= ratio);
      if (out_p) out_p[(int64_t)b * gamma + lane] = (float)P;
      if (out_q) out_q[(int64_t)b * gamma + lane] = (float)Q;
    }
    const unsigned mask = __ballot_sync(0xffffffffu, accept);
    const unsigned rej = ~mask;
    const int n = (rej == 0u) ? 32 : min(__ffs((int)rej) - 1, gamma);
    // flags: bad tokens anywhere, q(x)=0 at a tested position (i <= n, i < gamma)
    const unsigned badm = __ballot_sync(0xffffffffu, bad);
    const unsigned qz = __ballot_sync(0xffffffffu, lane < gamma && lane <= n && !(Q > 0.0));
    if (lane == 0) {
      int f = s_flag;
      if (badm) f |= SV_FLAG_BAD_TOKEN;
      if (qz) f |= SV_FLAG_NONFINITE;
      s_flag = f;
    }
    __syncwarp();
    int32_t* tok = out_tokens + (int64_t)b * (gamma + 1);
    for (int i = lane; i <= gamma; i += 32) {
      if (i < n) tok[i] = __ldg(xt + (int64_t)b * gamma + i);
      else if (i > n) tok[i] = -1;
    }
    if (lane == 0) {
      out_counts[b] = n;
      // 3. set up the draw of the target's own token
      DrawState st{};
      st.pos = n;
      st.c = c;
      st.invT = invT;
      int f = s_flag;
      const float mct = s_mc[n];
      const double St = s_s[n];
      const bool t_ok = (St > 0.0) && (St < 1e308) && (mct < kInf);
      if (n == gamma) {
        if (!t_ok) {
          st.mode = kDrawDone;
          tok[n] = 0;
        } else {
          st.mode = kDrawSampleRow;
          st.mct = mct;
          st.st = St;
        }
      } else {
        const float mcd = s_mc[gamma + 1 + n];
        const double Sd = s_s[gamma + 1 + n];
        const bool d_nonfinite = !(Sd < 1e308) || mcd == kInf;
        if (!t_ok || d_nonfinite) {
          // p_n has no mass (or the row is not finite): the residual is empty and
          // so is its fallback; emit token 0
          st.mode = kDrawDone;
          tok[n] = 0;
          if (St == 0.0) f |= SV_FLAG_RESIDUAL_FALLBACK;
        } else if (Sd == 0.0) {
          // q_n has no mass: max(0, p_n - q_n) = p_n
          st.mode = kDrawSampleRow;
          st.mct = mct;
          st.st = St;
        } else {
          st.mode = kDrawResidual;
          st.mct = mct;
          st.st = St;
          st.mcd = mcd;
          st.sd = Sd;
          st.K = (float)(((double)mct + log2(St)) - ((double)mcd + log2(Sd)));
        }
      }
      state[b] = st;
      if (out_flags) out_flags[b] = (uint8_t)f;
    }
  }
}

// --------------------------------------------------------------------------
// k_draw: Gumbel-max of the target's own token.
// --------------------------------------------------------------------------
struct DrawArgs {
  const void* zt;
  const void* zd;
  int gamma;
  int64_t V;
  uint64_t seed, round;
  int nsplit;
  const DrawState* state;
  Top2* part;
  uint32_t* counter;
  int32_t* out_tokens;
  uint8_t* out_flags;
};

// Keys of one 4-entry Philox group v = 4g .. 4g+3 (entries >= V skipped).
template <int DT, bool RESID>
__device__ __forceinline__ void draw_group(const char* rt, const char* rd, int64_t g, int64_t V,
                                           bool vec_ok, const DrawState& st, uint32_t b,
                                           uint64_t seed, uint64_t round, KI& best) {
  const int64_t v0 = 4 * g;
  float ztv[4], zdv[4];
  if (vec_ok && v0 + 3 < V) {
    if (DT == SV_F32) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(rt) + g);
      ztv[0] = a.x; ztv[1] = a.y; ztv[2] = a.z; ztv[3] = a.w;
      if (RESID) {
        const float4 d = __ldg(reinterpret_cast<const float4*>(rd) + g);
        zdv[0] = d.x; zdv[1] = d.y; zdv[2] = d.z; zdv[3] = d.w;
      }
    } else {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(rt) + g);
      ztv[0] = bf16lo(a.x); ztv[1] = bf16hi(a.x); ztv[2] = bf16lo(a.y); ztv[3] = bf16hi(a.y);
      if (RESID) {
        const uint2 d = __ldg(reinterpret_cast<const uint2*>(rd) + g);
        zdv[0] = bf16lo(d.x); zdv[1] = bf16hi(d.x); zdv[2] = bf16lo(d.y); zdv[3] = bf16hi(d.y);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t v = v0 + e;
      ztv[e] = (v < V) ? load_logit<DT>(rt, v) : -kInf;
      if (RESID) zdv[e] = (v < V) ? load_logit<DT>(rd, v) : 0.0f;
    }
  }
  const uint4 rnd = philox4x32_10(sv_counter((uint32_t)g, 1u, (uint32_t)st.pos, b, round),
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float key;
    bool cand;
    const float et = ex2(fmaf(ztv[e], st.c, -st.mct));
    if (RESID) {
      // log2(q/p) for this entry; p > q iff x < 0
      const float x = fmaf(zdv[e] - ztv[e], st.c, st.K);
      cand = x < 0.0f;
      key = __fdividef(et * -expm1f(x * kLn2), sv_neglog_u(rr[e]));
    } else {
      cand = ztv[e] > -kInf;
      key = __fdividef(et, sv_neglog_u(rr[e]));
    }
    if (cand && key > best.k) {
      best.k = key;
      best.i = (int)(v0 + e);
    }
  }
}

// Double-precision key with the oracle-level definition, for the refinement.
template <int DT>
__device__ double draw_key_f64(const char* rt, const char* rd, int64_t v, const DrawState& st,
                               bool resid, uint32_t b, uint64_t seed, uint64_t round) {
  const uint4 rnd = philox4x32_10(sv_counter((uint32_t)(v >> 2), 1u, (uint32_t)st.pos, b, round),
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  const double lnE = log(sv_neglog_u_f64(rr[v & 3]));
  const double zt = (double)load_logit<DT>(rt, v);
  if (!resid) return zt * (double)st.invT - lnE;
  const double zd = (double)load_logit<DT>(rd, v);
  const double P = exp2(zt * (double)st.c - (double)st.mct) / st.st;
  const double Q = exp2(zd * (double)st.c - (double)st.mcd) / st.sd;
  const double r = P - Q;
  return (r > 0.0) ? log(r) - lnE : -CUDART_INF;
}

template <int DT, bool RESID>
__device__ __forceinline__ KI draw_range(const char* rt, const char* rd, int64_t g0, int64_t g1,
                                         int64_t V, bool vec_ok, const DrawState& st, uint32_t b,
                                         uint64_t seed, uint64_t round) {
  KI best{-kInf, -1};
  for (int64_t g = g0 + threadIdx.x; g < g1; g += blockDim.x)
    draw_group<DT, RESID>(rt, rd, g, V, vec_ok, st, b, seed, round, best);
  return best;
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

template <int DT>
__global__ void __launch_bounds__(kThreads) k_draw(DrawArgs a) {
  const int b = (int)(blockIdx.x / (unsigned)a.nsplit);
  const int split = (int)(blockIdx.x - (unsigned)b * (unsigned)a.nsplit);
  const DrawState st = a.state[b];
  if (st.mode == kDrawDone) return;
  const bool resid = (st.mode == kDrawResidual);
  const int gamma = a.gamma;
  const int64_t V = a.V;
  const char* rt = row_ptr<DT>(a.zt, a.zd, b, st.pos, gamma, V);
  const char* rd = resid ? row_ptr<DT>(a.zt, a.zd, b, gamma + 1 + st.pos, gamma, V) : nullptr;
  // 4-entry groups are vector-loadable when rows start on a group boundary
  const bool vec_ok = (V % 4) == 0;
  const int64_t ngroups = ceil_div(V, 4);
  const int64_t gpc = kChunkDraw / 4;
  const int64_t g0 = (int64_t)split * gpc, g1 = min(ngroups, g0 + gpc);

  KI mine = resid ? draw_range<DT, true>(rt, rd, g0, g1, V, vec_ok, st, b, a.seed, a.round)
                  : draw_range<DT, false>(rt, rd, g0, g1, V, vec_ok, st, b, a.seed, a.round);
  Top2 t = block_top2(mine);

  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    a.part[(int64_t)b * a.nsplit + split] = t;
    __threadfence();
    const uint32_t prev = atomicAdd(a.counter + b, 1u);
    s_last = (prev == (uint32_t)a.nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last CTA of batch row b: merge the per-CTA top-2
  Top2 m{KI{-kInf, -1}, KI{-kInf, -1}};
  for (int j = threadIdx.x; j < a.nsplit; j += blockDim.x) {
    // other CTAs' partials: read through L2 (never cached in this SM's L1)
    const float4 raw = __ldcg(reinterpret_cast<const float4*>(a.part + (int64_t)b * a.nsplit + j));
    Top2 p;
    p.a.k = raw.x;
    p.a.i = __float_as_int(raw.y);
    p.b.k = raw.z;
    p.b.i = __float_as_int(raw.w);
    m = top2_merge(m, p);
  }
  __shared__ Top2 sm2[kThreads / 32];
  m = warp_reduce_top2(m);
  if ((threadIdx.x & 31) == 0) sm2[threadIdx.x >> 5] = m;
  __syncthreads();
  __shared__ int s_tok;
  __shared__ int s_fallback;
  if (threadIdx.x == 0) {
    Top2 r{KI{-kInf, -1}, KI{-kInf, -1}};
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = top2_merge(r, sm2[w]);
    const int tok = refine<DT>(r, rt, rd, st, resid, (uint32_t)b, a.seed, a.round);
    s_tok = tok;
    s_fallback = (tok < 0 && resid) ? 1 : 0;
    a.counter[b] = 0u;  // leave the workspace ready for the next call
  }
  __syncthreads();
  if (s_fallback) {
    // the residual had no positive entry in floating point: draw from p_n itself
    DrawState sp = st;
    sp.mode = kDrawSampleRow;
    KI f = draw_range<DT, false>(rt, nullptr, 0, ngroups, V, vec_ok, sp, b, a.seed, a.round);
    Top2 tf = block_top2(f);
    if (threadIdx.x == 0) s_tok = refine<DT>(tf, rt, nullptr, sp, false, (uint32_t)b, a.seed,
                                             a.round);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int tok = s_tok;
    uint8_t fl = 0;
    if (s_fallback) fl |= SV_FLAG_RESIDUAL_FALLBACK;
    if (tok < 0) {
      tok = 0;
      fl |= SV_FLAG_ZERO_MASS;
    }
    a.out_tokens[(int64_t)b * (gamma + 1) + st.pos] = tok;
    if (a.out_flags && fl) a.out_flags[b] |= fl;
  }
}

// --------------------------------------------------------------------------
// k_alpha: beta_i = sum_v min(p_i(v), q_i(v)); alpha_b = mean_i beta_i.
// --------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads)
k_alpha(const void* __restrict__ zt, const void* __restrict__ zd, int gamma, int64_t V,
        float temperature, const float* __restrict__ row_T, int nsplit,
        const RowStat* __restrict__ rowstat, float* __restrict__ part,
        uint32_t* __restrict__ counter, float* __restrict__ out_alpha) {
  const int64_t per_b = (int64_t)gamma * nsplit;
  const int b = (int)(blockIdx.x / per_b);
  const int rem = (int)(blockIdx.x - b * per_b);
  const int i = rem / nsplit, split = rem - i * nsplit;
  const int R1 = 2 * gamma + 1;
  const float T = row_T ? __ldg(row_T + b) : temperature;
  const float c = log2_scale(inv_temperature(T));
  const RowStat rs_t = rowstat[(int64_t)b * R1 + i];
  const RowStat rs_d = rowstat[(int64_t)b * R1 + gamma + 1 + i];
  const float it = (rs_t.s > 0.0) ? (float)(1.0 / rs_t.s) : 0.0f;
  const float id = (rs_d.s > 0.0) ? (float)(1.0 / rs_d.s) : 0.0f;
  const char* rt = row_ptr<DT>(zt, zd, b, i, gamma, V);
  const char* rd = row_ptr<DT>(zt, zd, b, gamma + 1 + i, gamma, V);
  const int64_t lo = (int64_t)split * kChunkSweep, hi = min(V, lo + kChunkSweep);
  float acc = 0.0f;
  for (int64_t v = lo + threadIdx.x; v < hi; v += blockDim.x) {
    const float pt = (it > 0.0f) ? ex2(fmaf(load_logit<DT>(rt, v), c, -rs_t.mc)) * it : 0.0f;
    const float pd = (id > 0.0f) ? ex2(fmaf(load_logit<DT>(rd, v), c, -rs_d.mc)) * id : 0.0f;
    acc += fminf(pt, pd);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ float sm[kThreads / 32];
  __shared__ bool s_last;
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += sm[w];
    part[((int64_t)b * gamma + i) * nsplit + split] = s;
    __threadfence();
    const uint32_t prev = atomicAdd(counter + b, 1u);
    s_last = (prev == (uint32_t)(gamma * nsplit) - 1);
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  double tot = 0.0;
  const float* pp = part + (int64_t)b * gamma * nsplit;
  for (int j = 0; j < gamma * nsplit; ++j) tot += (double)__ldcg(pp + j);
  out_alpha[b] = (float)(tot / gamma);
  counter[b] = 0u;
}

// --------------------------------------------------------------------------
// Host-side launcher.
// --------------------------------------------------------------------------
static cudaEvent_t g_events[4] = {nullptr, nullptr, nullptr, nullptr};

void set_timing_events(void* const* ev, int n) {
  for (int i = 0; i < 4; ++i) g_events[i] = (ev && i < n) ? (cudaEvent_t)ev[i] : nullptr;
}

static inline void mark(int i, cudaStream_t s) {
  if (g_events[i]) cudaEventRecord(g_events[i], s);
}

template <int DT>
static cudaError_t launch_sample_t(const void* zt, const void* zd, const int32_t* xt, int B,
                                   int gamma, int64_t V, float temperature, const float* row_T,
                                   uint64_t seed, uint64_t round, int32_t* out_tokens,
                                   int32_t* out_counts, float* out_p, float* out_q,
                                   float* out_alpha, uint8_t* out_flags, char* ws,
                                   const SamplePlan& pl, cudaStream_t stream) {
  const int R1 = pl.R1;
  float2* part1 = reinterpret_cast<float2*>(ws + pl.off_part1);
  RowStat* rowstat = reinterpret_cast<RowStat*>(ws + pl.off_rowstat);
  DrawState* state = reinterpret_cast<DrawState*>(ws + pl.off_state);
  Top2* part3 = reinterpret_cast<Top2*>(ws + pl.off_part3);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + pl.off_cnt);
  float* apart = reinterpret_cast<float*>(ws + pl.off_alpha);

  const unsigned g1 = (unsigned)((int64_t)pl.nsplit1 * B * R1);
  mark(0, stream);
  k_sweep<DT><<<g1, kThreads, 0, stream>>>(zt, zd, gamma, V, temperature, row_T, pl.nsplit1,
                                            part1);
  mark(1, stream);
  k_decide<DT><<<B, 128, 0, stream>>>(zt, zd, xt, gamma, V, temperature, row_T, seed, round,
                                       pl.nsplit1, part1, rowstat, state, cnt, B, out_tokens,
                                       out_counts, out_p, out_q, out_flags);
  mark(2, stream);
  DrawArgs da{zt, zd, gamma, V, seed, round, pl.nsplit3, state, part3, cnt, out_tokens, out_flags};
  k_draw<DT><<<(unsigned)((int64_t)pl.nsplit3 * B), kThreads, 0, stream>>>(da);
  mark(3, stream);
  if (out_alpha) {
    k_alpha<DT><<<(unsigned)((int64_t)pl.nsplit1 * gamma * B), kThreads, 0, stream>>>(
        zt, zd, gamma, V, temperature, row_T, pl.nsplit1, rowstat, apart, cnt + B, out_alpha);
  }
  return cudaGetLastError();
}

cudaError_t launch_sample(const void* zt, const void* zd, const int32_t* xt, int B, int gamma,
                          int64_t V, int dtype, float temperature, const float* row_T,
                          uint64_t seed, uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                          float* out_p, float* out_q, float* out_alpha, uint8_t* out_flags,
                          void* ws, const SamplePlan& pl, cudaStream_t stream) {
  char* w = reinterpret_cast<char*>(ws);
  if (dtype == SV_F32)
    return launch_sample_t<SV_F32>(zt, zd, xt, B, gamma, V, temperature, row_T, seed, round,
                                   out_tokens, out_counts, out_p, out_q, out_alpha, out_flags, w,
                                   pl, stream);
  return launch_sample_t<SV_BF16>(zt, zd, xt, B, gamma, V, temperature, row_T, seed, round,
                                  out_tokens, out_counts, out_p, out_q, out_alpha, out_flags, w,
                                  pl, stream);
}

}  // namespace sv
