// sv_sweep.cuh -- per-lane and per-warp pieces of the softmax-statistics sweep:
// online (max, sum of 2^(y - max)) over a 4 KB block held in registers, and the
// warp combine.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"

namespace sv {

// Per-lane online (max, sum) update with a chunk maximum m of raw logits.
__device__ __forceinline__ void lane_raise_max(float m, float c, float& zmax, float& mc,
                                               float& sacc) {
  if (m > zmax) {
    const float mcn = m * c;
    sacc = (zmax == -kInf) ? 0.0f : sacc * ex2(mc - mcn);
    mc = mcn;
    zmax = m;
  }
}

// One full 4 KB block, each lane holding 8 of its 256 vectors in registers.
// The maximum is a packed tree over the raw words, then one exp2 per logit.
// With TOPK, logits below tau (the row's top-k threshold) add nothing to the sum.
template <int DT, bool TOPK = false>
__device__ __forceinline__ void chunk_update_full(const uint4 (&v)[8], float c, float tau,
                                                  float& zmax, float& mc, float& sacc) {
  float m;
  if constexpr (DT == SV_BF16) {
    uint32_t a[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint32_t p, q;
      asm("max.bf16x2 %0, %1, %2;" : "=r"(p) : "r"(v[u].x), "r"(v[u].y));
      asm("max.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(v[u].z), "r"(v[u].w));
      asm("max.bf16x2 %0, %1, %2;" : "=r"(a[u]) : "r"(p), "r"(q));
    }
#pragma unroll
    for (int k = 4; k > 0; k >>= 1)
#pragma unroll
      for (int u = 0; u < k; ++u) asm("max.bf16x2 %0, %1, %2;" : "=r"(a[u]) : "r"(a[u]), "r"(a[u + k]));
    m = fmaxf(bf16lo(a[0]), bf16hi(a[0]));
  } else {
    float a[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      a[u] = fmaxf(fmaxf(__uint_as_float(v[u].x), __uint_as_float(v[u].y)),
                   fmaxf(__uint_as_float(v[u].z), __uint_as_float(v[u].w)));
#pragma unroll
    for (int k = 4; k > 0; k >>= 1)
#pragma unroll
      for (int u = 0; u < k; ++u) a[u] = fmaxf(a[u], a[u + k]);
    m = a[0];
  }
  lane_raise_max(m, c, zmax, mc, sacc);
  if (!(zmax > -kInf)) return;
  const float nm = -mc;
  // pairs (even, odd element) in packed fp32x2: the same sums, in the same
  // order, as two scalar accumulators s0 (even) and s1 (odd) folded into
  // s2, s3 every second vector
  const uint64_t c2 = pack2(c, c), nm2 = pack2(nm, nm), zero2 = pack2(0.0f, 0.0f);
  uint64_t s01 = zero2, s23 = zero2;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int q = 0; q < 4; q += (DT == SV_BF16) ? 1 : 2) {
      const float za = (DT == SV_BF16) ? bf16lo(w[q]) : __uint_as_float(w[q]);
      const float zb = (DT == SV_BF16) ? bf16hi(w[q]) : __uint_as_float(w[q + 1]);
      const uint64_t z2 = pack2(za, zb);
      float y0, y1;
      unpack2(ffma2(z2, c2, nm2), y0, y1);
      if (TOPK) {
        y0 = (za < tau) ? -kInf : y0;
        y1 = (zb < tau) ? -kInf : y1;
      }
      s01 = fadd2(s01, pack2(ex2(y0), ex2(y1)));
    }
    if (u & 1) {
      s23 = fadd2(s23, s01);
      s01 = zero2;
    }
  }
  float s0, s1, s2, s3;
  unpack2(s01, s0, s1);
  unpack2(s23, s2, s3);
  sacc += (s0 + s1) + (s2 + s3);
}

// A chunk shorter than 4 KB (the end of a row): lanes hold vectors lane + 32u
// for lane + 32u < nv; the same arithmetic as a full chunk otherwise.
template <int DT, bool TOPK = false>
__device__ __forceinline__ void chunk_update_part(const uint4 (&v)[8], int nv, float c, float tau,
                                                  float& zmax, float& mc, float& sacc) {
  const int lane = threadIdx.x & 31;
  float m = -kInf;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    if (lane + 32 * u < nv) m = fmaxf(m, vmax<DT>(v[u]));
  lane_raise_max(m, c, zmax, mc, sacc);
  if (!(zmax > -kInf)) return;
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    if (lane + 32 * u < nv) {
      float f[VecInfo<DT>::kElems];
      unpack<DT>(v[u], f);
#pragma unroll
      for (int e = 0; e < VecInfo<DT>::kElems; e += 2) {
        s0 += (TOPK && f[e] < tau) ? 0.0f : ex2(fmaf(f[e], c, -mc));
        s1 += (TOPK && f[e + 1] < tau) ? 0.0f : ex2(fmaf(f[e + 1], c, -mc));
      }
    }
  }
  sacc += s0 + s1;
}

// The chunk's partial from the lanes' (largest logit, scaled max, sum): the
// largest logit z of the chunk as given, and the sum of 2^(y - z c) (z c is the
// largest of the lanes' scaled maxima, bit for bit: scaling is monotone).
__device__ __forceinline__ float2 warp_chunk_partial(float zmax, float mc, float sacc, float c) {
  const float Z = warp_max(zmax);
  const float M = Z * c;
  float s = (mc > -kInf) ? sacc * ex2(mc - M) : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return make_float2(Z, (M > -kInf) ? s : 0.0f);
}

// Chunks of the vector sweep: row k of batch row b is cut into nck chunks of
// 4 KB from its start, unit g = (b R1 + k) nck + j.  A warp walks g, g + W,
// g + 2W, ...; the cursor (b, k, j) advances by fixed increments (no division
// in the loop: the next chunk's address is ready before its loads are due).
struct UnitCursor {
  int b, k, j;
};
struct UnitWalk {
  int R1, nck, dj, dk, db;
  __device__ __forceinline__ void init(int R1_, int nck_, int W) {
    R1 = R1_;
    nck = nck_;
    dj = W % nck;
    const int dr = W / nck;
    dk = dr % R1;
    db = dr / R1;
  }
  __device__ __forceinline__ UnitCursor at(int64_t g) const {
    const int64_t r = g / nck;
    return UnitCursor{(int)(r / R1), (int)(r % R1), (int)(g - r * nck)};
  }
  __device__ __forceinline__ void step(UnitCursor& c) const {
    c.j += dj;
    int k = c.k + dk;
    if (c.j >= nck) {
      c.j -= nck;
      ++k;
    }
    c.b += db;
    if (k >= R1) {
      k -= R1;
      ++c.b;
    }
    c.k = k;
  }
};

// Warp max of m, then one rescale per lane and a warp sum.
__device__ __forceinline__ MS warp_reduce_ms_fast(MS v) {
  const float M = warp_max(v.m);
  float s = (v.m > -kInf) ? v.s * ex2(v.m - M) : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return MS{M, (M > -kInf) ? s : 0.0f};
}

}  // namespace sv
