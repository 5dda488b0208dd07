// sv_greedy.cu -- greedy verify on sm_103a.
//
// The argmax limit of the accept rule ("Fast Inference from Transformers via
// Speculative Decoding", section "Speculative sampling: the accept/reject
// rule": at low temperature the rule becomes argmax decoding with a verify
// step) and the greedy comparison of the lihaoran.work essay ("What does
// unchanged output mean?"): keep the longest prefix where the draft token is
// the target's argmax, then append the target's argmax at the stop position.
//
// k_greedy: one cluster of kGreedyCluster CTAs per batch row.  CTA r of the
// cluster takes the r-th slice of every target row of the batch row, one warp
// per row: 16-byte loads, a packed-bf16 max per vector and a scalar scan only
// when the vector beats the running maximum.  After a cluster barrier, CTA 0
// reads every CTA's per-row (max, index) from its shared memory (distributed
// shared memory), takes each row's argmax (ties to the lowest index), does the
// prefix match and writes the outputs.  No global counter: a call needs no
// workspace contents and no memset.
#include <cuda_runtime.h>

#include <cooperative_groups.h>

#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"

namespace sv {

constexpr int kGreedyCluster = 8;

template <int DT>
__global__ void __cluster_dims__(kGreedyCluster, 1, 1) __launch_bounds__(kThreads, 4)
k_greedy(const void* __restrict__ zt, const int32_t* __restrict__ xt, int gamma, int64_t V,
         int64_t slice, int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_counts) {
  namespace cg = cooperative_groups;
  constexpr int VE = VecInfo<DT>::kElems;
  constexpr int kBytes = (DT == SV_F32) ? 4 : 2;
  constexpr int kWarps = kThreads / 32;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = (int)(blockIdx.x / kGreedyCluster);
  const int G1 = gamma + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ KI s_part[33];  // this CTA's (max, index) of its slice of each row
  __shared__ int s_t[33];
  const int64_t lo = (int64_t)rank * slice;
  const int64_t hi = min(V, lo + slice);
  for (int i = warp; i < G1; i += kWarps) {
    const char* row = reinterpret_cast<const char*>(zt) + ((int64_t)b * G1 + i) * V * kBytes;
    // running (value, index); NaN counts as -inf; index -1 = nothing above -inf yet
    float best = -kInf;
    int bi = -1;
    if (lo < hi) {
      const uintptr_t addr_lo = reinterpret_cast<uintptr_t>(row) + lo * kBytes;
      int64_t a0 = lo + (int64_t)(((16 - (addr_lo & 15)) & 15) / kBytes);
      if (a0 > hi) a0 = hi;
      const int64_t nvec = (hi - a0) / VE;
      const int64_t a1 = a0 + nvec * VE;
      for (int64_t v = lo + lane; v < a0; v += 32) {
        const float z = load_logit<DT>(row, v);
        if (z > best) { best = z; bi = (int)v; }
      }
      const uint4* vp = reinterpret_cast<const uint4*>(row + a0 * kBytes);
      constexpr int U = 4;
      for (int64_t j = lane; j < nvec; j += (int64_t)U * 32) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t jj = j + (int64_t)u * 32;
          if (jj < nvec) buf[u] = ld_stream16(vp + jj);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t jj = j + (int64_t)u * 32;
          if (jj < nvec) {
            const float m = vmax<DT>(buf[u]);
            if (m > best) {  // rare: locate the first element equal to the new max
              float f[VE];
              unpack<DT>(buf[u], f);
              int e = VE - 1;
#pragma unroll
              for (int k = VE - 1; k >= 0; --k)
                if (f[k] == m) e = k;
              best = m;
              bi = (int)(a0 + jj * VE + e);
            }
          }
        }
      }
      for (int64_t v = a1 + lane; v < hi; v += 32) {
        const float z = load_logit<DT>(row, v);
        if (z > best) { best = z; bi = (int)v; }
      }
    }
    const KI t = warp_reduce_ki(KI{best, bi});
    if (lane == 0) s_part[i] = t;
  }
  cluster.sync();  // every CTA's partials are in its shared memory
  if (rank == 0) {
    // each row's argmax over the cluster's slices (lower ranks hold lower indices)
    for (int i = warp; i < G1; i += kWarps) {
      KI t{-kInf, -1};
      if (lane < kGreedyCluster) t = cluster.map_shared_rank(s_part, lane)[i];
      t = warp_reduce_ki(t);
      if (lane == 0) s_t[i] = (t.i < 0) ? 0 : t.i;  // all -inf/NaN row: index 0
    }
    __syncthreads();
    if (warp == 0) {
      const int32_t x = (lane < gamma) ? __ldg(xt + (int64_t)b * gamma + lane) : 0;
      const unsigned match = __ballot_sync(0xffffffffu, lane < gamma && x == s_t[lane]);
      const unsigned miss = ~match;
      const int n = (miss == 0u) ? 32 : min(__ffs((int)miss) - 1, gamma);
      int32_t* tok = out_tokens + (int64_t)b * G1;
      for (int i = lane; i < G1; i += 32) {
        if (i < n) tok[i] = __ldg(xt + (int64_t)b * gamma + i);
        else if (i == n) tok[i] = s_t[n];
        else tok[i] = -1;
      }
      if (lane == 0) out_counts[b] = n;
    }
  }
  cluster.sync();  // no CTA leaves while CTA 0 may still read its shared memory
}

cudaError_t launch_greedy(const void* zt, const int32_t* xt, int B, int gamma, int64_t V,
                          int dtype, int32_t* out_tokens, int32_t* out_counts, void*,
                          const GreedyPlan&, cudaStream_t stream) {
  // slices of whole 16-byte vectors of 8 entries
  const int64_t slice = ceil_div(ceil_div(V, (int64_t)kGreedyCluster), (int64_t)8) * 8;
  const unsigned grid = (unsigned)((int64_t)B * kGreedyCluster);
  if (dtype == SV_F32)
    k_greedy<SV_F32><<<grid, kThreads, 0, stream>>>(zt, xt, gamma, V, slice, out_tokens,
                                                     out_counts);
  else
    k_greedy<SV_BF16><<<grid, kThreads, 0, stream>>>(zt, xt, gamma, V, slice, out_tokens,
                                                      out_counts);
  return cudaGetLastError();
}

}  // namespace sv
