// sv_units.cuh -- the vector sweep's loop over the 4 KB chunks of every row.
//
// Row k of batch row b (target rows k = 0..gamma, then the draft rows) is cut
// into nck chunks of 4 KB counted from the row's start; the last chunk of a
// row may be shorter.  Chunks are numbered in batch-row order, g = (b R1 + k)
// nck + j, and warp w of W takes g = w, w + W, w + 2W, ...: the whole GPU walks
// the batch rows in order, so each batch row's chunks are complete at a known
// point of the loop.  A warp holds two chunks in registers, reducing one while
// the other's 16-byte loads are in flight, and the address of the chunk after
// next is formed while the current one is reduced.  Each chunk leaves one
// partial: its largest logit as given and the sum of 2^(y - max y) (y = z T^-1
// log2 e), every lane holding vectors lane + 32u of the chunk.  The partials
// depend only on the values and the shapes, not on where the arrays sit.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_decide.cuh"
#include "sv_device.cuh"
#include "sv_plan.h"
#include "sv_sweep.cuh"

namespace sv {

// A partial as one 64-bit word that is never zero (a zeroed slot reads as "not
// written yet"): the largest logit's bits low, the sum's bits with the sign bit
// flipped high (a sum is never -0).
__device__ __forceinline__ uint64_t part_word(float2 p) {
  return ((uint64_t)(__float_as_uint(p.y) ^ 0x80000000u) << 32) | (uint64_t)__float_as_uint(p.x);
}
__device__ __forceinline__ float2 part_unword(uint64_t w) {
  return make_float2(__uint_as_float((uint32_t)w), __uint_as_float((uint32_t)(w >> 32) ^ 0x80000000u));
}

__device__ __forceinline__ uint64_t ld_relaxed64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Where a chunk is and how it is reduced.
struct UnitInfo {
  const uint4* p;
  int nv;     // 16-byte vectors in the chunk (256 for a full one)
  float c;    // the batch row's scale fl32(1/T) log2 e
  float tau;  // top-k threshold of the row (-inf: none)
};

template <int DT, bool TOPK>
__device__ __forceinline__ UnitInfo unit_info(const SweepCtx& x, const UnitCursor& u, int64_t RB,
                                              float c_all) {
  UnitInfo r;
  const int64_t off = (int64_t)u.j * kSweepChunkBytes;
  const int64_t nb = RB - off;
  r.nv = (nb >= kSweepChunkBytes) ? 256 : (int)(nb >> 4);
  r.p = reinterpret_cast<const uint4*>(row_ptr<DT>(x.zt, x.zd, u.b, u.k, x.gamma, x.V) + off);
  r.c = x.row_T ? log2_scale(inv_temperature(__ldg(x.row_T + u.b))) : c_all;
  r.tau = TOPK ? __ldg(x.thr + (int64_t)u.b * (2 * x.gamma + 1) + u.k) : -kInf;
  return r;
}

__device__ __forceinline__ void unit_load(uint4 (&v)[8], const UnitInfo& u) {
  const int lane = threadIdx.x & 31;
  if (u.nv == 256) {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = ld_stream16(u.p + lane + 32 * q);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      v[q] = (lane + 32 * q < u.nv) ? ld_stream16(u.p + lane + 32 * q) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int DT, bool TOPK>
__device__ __forceinline__ float2 unit_reduce(const uint4 (&v)[8], const UnitInfo& u) {
  float zmax = -kInf, mc = -kInf, sacc = 0.0f;
  if (u.nv == 256)
    chunk_update_full<DT, TOPK>(v, u.c, u.tau, zmax, mc, sacc);
  else
    chunk_update_part<DT, TOPK>(v, u.nv, u.c, u.tau, zmax, mc, sacc);
  return warp_chunk_partial(zmax, mc, sacc, u.c);
}

// The loop of one warp over its chunks, and over the iterations after them up
// to `it_end`.  After the chunk of iteration `it` (if any) is reduced, its
// partial goes to `emit(g, partial)` and `tasks(it)` runs (the other chunk's
// loads still in flight).
template <int DT, bool TOPK, class Emit, class Tasks>
__device__ __forceinline__ void unit_loop(const SweepCtx& x, int nck, int64_t it_end, Emit&& emit,
                                          Tasks&& tasks) {
  const int warp = threadIdx.x >> 5;
  const int W = (int)gridDim.x * (int)(blockDim.x >> 5);
  const int w = (int)blockIdx.x * (int)(blockDim.x >> 5) + warp;
  const int R1 = 2 * x.gamma + 1;
  const int64_t NU = (int64_t)x.B * R1 * nck;
  const int64_t RB = x.V * ((DT == SV_F32) ? 4 : 2);
  const float c_all = log2_scale(inv_temperature(x.temperature));
  UnitWalk walk;
  walk.init(R1, nck, W);
  UnitCursor cn = walk.at(w);
  uint4 va[8], vb[8];
  UnitInfo ia{}, inx{};
  if (w < NU) {
    ia = unit_info<DT, TOPK>(x, cn, RB, c_all);
    unit_load(va, ia);
  }
  walk.step(cn);  // unit w + W
  if (w + W < NU) inx = unit_info<DT, TOPK>(x, cn, RB, c_all);
  walk.step(cn);  // unit w + 2W
  // one iteration: the chunk in `cur` (described by ia), the next one's loads into `nxt`
  auto iteration = [&](int64_t it, uint4 (&cur)[8], uint4 (&nxt)[8]) {
    const int64_t g = w + it * W;
    if (g < NU) {
      if (g + W < NU) unit_load(nxt, inx);
      UnitInfo after{};
      if (g + 2 * (int64_t)W < NU) after = unit_info<DT, TOPK>(x, cn, RB, c_all);
      walk.step(cn);
      emit(g, unit_reduce<DT, TOPK>(cur, ia));
      ia = inx;
      inx = after;
    }
    tasks(it);
  };
  for (int64_t it = 0; it <= it_end; it += 2) {
    iteration(it, va, vb);
    if (it + 1 > it_end) break;
    iteration(it + 1, vb, va);
  }
}

}  // namespace sv
