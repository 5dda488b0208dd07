// sv_units.cuh -- the vector sweep's loop over the 4 KB chunks of every row.
//
// Row k of batch row b (target rows k = 0..gamma, then the draft rows) is cut
// into nck chunks of 4 KB counted from the row's start; the last chunk of a
// row may be shorter.  Chunks are numbered in batch-row order, g = (b R1 + k)
// nck + j, and warp w of W takes g = w, w + W, w + 2W, ...: the whole GPU walks
// the batch rows in order, so each batch row's chunks complete one after
// another.  A warp stages its chunks in NBUF shared-memory buffers of its own
// (cp.async with an L2 evict-first hint, 16 bytes per lane and vector, no
// registers held while the copies are in flight): NBUF - 1 chunks in flight while one is reduced; lane l
// copies and later reads vectors l + 32u of a chunk.  The address of each
// chunk comes from a cursor stepped by fixed increments (no division in the
// loop).  Each chunk leaves one partial: its
// largest logit as given and the sum of 2^(y - max y) (y = z T^-1 log2 e).  The
// partials depend only on the values and the shapes, not on where the arrays
// sit in memory.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_decide.cuh"
#include "sv_device.cuh"
#include "sv_plan.h"
#include "sv_sweep.cuh"

namespace sv {

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

// One chunk into a warp's shared-memory buffer [8][32] of 16-byte vectors: lane
// l copies vectors l + 32u (past the chunk's end: zero fill, nothing read).
// The logits are read once, so their L2 lines are marked evict-first: the
// stream does not push out what the next kernel reads (the partials, the
// counters, its code), and the sweep itself runs faster (28.2 against 29.9 us
// for 148 MB).
__device__ __forceinline__ void unit_copy(uint4* buf, const UnitInfo& u) {
  const int lane = threadIdx.x & 31;
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(buf + 32 * q + lane);
    const bool in = lane + 32 * q < u.nv;  // past the end: the chunk's start, 0 bytes read
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
                 "l"(in ? u.p + lane + 32 * q : u.p), "r"(in ? 16 : 0), "l"(pol)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

// The loop of sweep warp w of W over its chunks g = w + it W, it = 0..it_end
// (iterations past the last chunk only commit empty copy groups).  `wbuf` is
// the warp's NBUF x 4 KB of shared memory.  At iteration `it` the copies of
// chunk it + NBUF - 1 are issued and chunk it is reduced; its partial goes to
// `emit(g, partial)`.
template <int DT, bool TOPK, int NBUF, class Emit>
__device__ __forceinline__ void unit_loop(const SweepCtx& x, int nck, int64_t it_end, uint4* wbuf,
                                          int w, int W, Emit&& emit) {
  const int lane = threadIdx.x & 31;
  const int R1 = 2 * x.gamma + 1;
  const int64_t NU = (int64_t)x.B * R1 * nck;
  const int64_t RB = x.V * ((DT == SV_F32) ? 4 : 2);
  const float c_all = log2_scale(inv_temperature(x.temperature));
  UnitWalk walk;
  walk.init(R1, nck, W);
  UnitCursor cn = walk.at(w);
  UnitInfo info[NBUF];
#pragma unroll
  for (int i = 0; i < NBUF - 1; ++i) {
    if (w + (int64_t)i * W < NU) {
      info[i] = unit_info<DT, TOPK>(x, cn, RB, c_all);
      unit_copy(wbuf + 256 * i, info[i]);
    }
    cp_async_commit();
    walk.step(cn);
  }
  for (int64_t it0 = 0; it0 <= it_end; it0 += NBUF) {
#pragma unroll
    for (int i = 0; i < NBUF; ++i) {
      const int64_t it = it0 + i;
      if (it > it_end) break;
      const int64_t g = w + it * W;
      // the chunk NBUF - 1 iterations ahead goes into the slot freed last iteration
      constexpr int kAhead = NBUF - 1;
      const int sl = (i + kAhead) % NBUF;
      if (g + (int64_t)kAhead * W < NU) {
        info[sl] = unit_info<DT, TOPK>(x, cn, RB, c_all);
        unit_copy(wbuf + 256 * sl, info[sl]);
      }
      cp_async_commit();
      walk.step(cn);
      if (g < NU) {
        cp_async_wait<NBUF - 1>();  // this chunk's copies (this lane's) have landed
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = wbuf[256 * i + 32 * q + lane];
        emit(g, unit_reduce<DT, TOPK>(v, info[i]));
      }
    }
  }
}

}  // namespace sv
