// sv_greedy.cu -- greedy verify on sm_103a.
//
// The argmax limit of the accept rule ("Fast Inference from Transformers via
// Speculative Decoding", section "Speculative sampling: the accept/reject
// rule": at low temperature the rule becomes argmax decoding with a verify
// step) and the greedy comparison of the lihaoran.work essay ("What does
// unchanged output mean?"): keep the longest prefix where the draft token is
// the target's argmax, then append the target's argmax at the stop position.
//
// k_greedy: each CTA takes one chunk of one target row, 16-byte loads, a
// packed-bf16 max per vector and a scalar scan only when the vector beats the
// running maximum; the last CTA of a batch row combines the partials of its
// gamma+1 rows, does the prefix match and writes the outputs.
#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"

namespace sv {

template <int DT>
__global__ void __launch_bounds__(kThreads, 4)
k_greedy(const void* __restrict__ zt, const int32_t* __restrict__ xt, int gamma, int64_t V,
         int nsplit, KI* __restrict__ part, uint32_t* __restrict__ counter,
         int32_t* __restrict__ out_tokens, int32_t* __restrict__ out_counts) {
  constexpr int VE = VecInfo<DT>::kElems;
  constexpr int kBytes = (DT == SV_F32) ? 4 : 2;
  const int G1 = gamma + 1;
  const int64_t r = blockIdx.x / (unsigned)nsplit;  // target row over B*(gamma+1)
  const int split = (int)(blockIdx.x - r * nsplit);
  const int b = (int)(r / G1);
  const char* row = reinterpret_cast<const char*>(zt) + (int64_t)r * V * kBytes;
  const int64_t lo = (int64_t)split * kChunkSweep;
  const int64_t hi = min(V, lo + kChunkSweep);
  const int tid = threadIdx.x;

  // running (value, index); NaN counts as -inf; index -1 = nothing above -inf yet
  float best = -kInf;
  int bi = -1;

  const uintptr_t addr_lo = reinterpret_cast<uintptr_t>(row) + lo * kBytes;
  int64_t a0 = lo + (int64_t)(((16 - (addr_lo & 15)) & 15) / kBytes);
  if (a0 > hi) a0 = hi;
  const int64_t nvec = (hi - a0) / VE;
  const int64_t a1 = a0 + nvec * VE;
  for (int64_t v = lo + tid; v < a0; v += blockDim.x) {
    const float z = load_logit<DT>(row, v);
    if (z > best) { best = z; bi = (int)v; }
  }
  const uint4* vp = reinterpret_cast<const uint4*>(row + a0 * kBytes);
  constexpr int U = 4;
  for (int64_t j = tid; j < nvec; j += (int64_t)U * blockDim.x) {
    uint4 buf[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t jj = j + (int64_t)u * blockDim.x;
      if (jj < nvec) buf[u] = ld_stream16(vp + jj);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t jj = j + (int64_t)u * blockDim.x;
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
  for (int64_t v = a1 + tid; v < hi; v += blockDim.x) {
    const float z = load_logit<DT>(row, v);
    if (z > best) { best = z; bi = (int)v; }
  }

  KI mine{best, bi};
  mine = warp_reduce_ki(mine);
  __shared__ KI sm[kThreads / 32];
  __shared__ bool s_last;
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) sm[warp] = mine;
  __syncthreads();
  if (tid == 0) {
    KI t = sm[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (ki_better(sm[w], t)) t = sm[w];
    part[(int64_t)r * nsplit + split] = t;
    __threadfence();
    const uint32_t prev = atomicAdd(counter + b, 1u);
    s_last = (prev == (uint32_t)(G1 * nsplit) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last CTA of batch row b: argmax of each of its gamma+1 rows, then the prefix
  __shared__ int s_t[33];
  for (int i = warp; i < G1; i += (int)(blockDim.x >> 5)) {
    KI t{-kInf, -1};
    const KI* pr = part + ((int64_t)b * G1 + i) * nsplit;
    for (int j = lane; j < nsplit; j += 32) {
      const float2 raw = __ldcg(reinterpret_cast<const float2*>(pr + j));
      const KI x{raw.x, __float_as_int(raw.y)};
      if (ki_better(x, t)) t = x;
    }
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

cudaError_t launch_greedy(const void* zt, const int32_t* xt, int B, int gamma, int64_t V,
                          int dtype, int32_t* out_tokens, int32_t* out_counts, void* ws,
                          const GreedyPlan& pl, cudaStream_t stream) {
  char* w = reinterpret_cast<char*>(ws);
  KI* part = reinterpret_cast<KI*>(w + pl.off_part);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(w + pl.off_cnt);
  const unsigned grid = (unsigned)((int64_t)pl.nsplit * B * (gamma + 1));
  // the last-CTA handoff counts CTAs per batch row from zero
  cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * (size_t)B, stream);
  if (e != cudaSuccess) return e;
  if (dtype == SV_F32)
    k_greedy<SV_F32><<<grid, kThreads, 0, stream>>>(zt, xt, gamma, V, pl.nsplit, part, cnt,
                                                     out_tokens, out_counts);
  else
    k_greedy<SV_BF16><<<grid, kThreads, 0, stream>>>(zt, xt, gamma, V, pl.nsplit, part, cnt,
                                                      out_tokens, out_counts);
  return cudaGetLastError();
}

}  // namespace sv
