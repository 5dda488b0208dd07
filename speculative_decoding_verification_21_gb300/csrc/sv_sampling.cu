// sv_sampling.cu -- the sampling verify's separate kernels on sm_103a.
//
// One round for B independent batch rows, after Algorithm 1 of "Fast Inference
// from Transformers via Speculative Decoding" (section "The loop: draft, verify
// in one pass, keep a prefix") and the course notes "Speculative Decoding"
// ("The algorithm"), as kernels chained by programmatic dependent launch:
//
//   sweep     online softmax statistics of every chunk of all 2*gamma+1 logit
//             rows, counted from each row's start: the largest logit and the
//             sum of 2^(y - max y), y = z * T^-1 * log2 e.  k_sweep_vec (rows a
//             multiple of 16 bytes): the persistent loop over 4 KB chunks of
//             sv_units.cuh.  k_sweep (any shape): one CTA per 8192-logit split.
//   top-k / top-p thresholds (k_topk_cand, k_topk, k_topp), then a thresholded
//             sweep where needed.
//   k_race    the default draw: one thread-block cluster per batch row, one CTA
//             per share of its slices; every CTA takes its batch row's decision
//             from the partials (accept test, first rejection by a warp ballot),
//             races its slices by Gumbel-max (sv_gumbel.cuh), and the cluster's
//             first CTA merges the CTAs' best two over distributed shared memory
//             and emits.
//   k_draw    the opt-in inverse-transform draw (sv_draw.cuh), same structure.
//   k_alpha   optional overlap sum_v min(p_i, q_i) ("The acceptance rate is the
//             overlap of p and q").
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>
#include <mutex>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_plan.h"
#include "sv_tma.cuh"
#include "sv_decide.cuh"
#include "sv_draw.cuh"
#include "sv_gumbel.cuh"
#include "sv_sweep.cuh"
#include "sv_units.cuh"
#include "sv_launch.h"

namespace cg = cooperative_groups;

namespace sv {

// --------------------------------------------------------------------------
// Generic sweep (any V): one CTA per (row, 8192-logit chunk).
// --------------------------------------------------------------------------
// Visit elements [lo, hi) of a row: an unaligned head as scalars, then 16-byte
// vectors, then the tail.
template <int DT, int UNROLL, class FV, class FS>
__device__ __forceinline__ void for_each_in_chunk(const char* row, int64_t lo, int64_t hi,
                                                  FV&& f_vec, FS&& f_one) {
  constexpr int VE = VecInfo<DT>::kElems;
  constexpr int kBytes = (DT == SV_F32) ? 4 : 2;
  const int tid = threadIdx.x;
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

// The inverse-transform draw's per-batch-row arrival counters and the race's
// shared bounds start at 0 in every call; the draw touches them only after this
// grid has completed.
__device__ __forceinline__ void zero_draw_counters(const SweepCtx& x) {
  if (blockIdx.x == 0 && x.done)
    for (int i = threadIdx.x; i < x.B; i += blockDim.x) x.done[i] = 0u;
  if (blockIdx.x == 0 && x.thw)
    for (int i = threadIdx.x; i < x.B; i += blockDim.x) x.thw[(int64_t)i * kThwStride] = 0u;
}

template <int DT, bool TOPK>
__global__ void __launch_bounds__(kThreads, 4) k_sweep(SweepCtx x) {
  pdl_launch_dependents();
  zero_draw_counters(x);
  const int R1 = 2 * x.gamma + 1;
  const int64_t item = blockIdx.x;  // (row, chunk) flattened, rows in batch-row order
  const int64_t r = item / x.np;
  const int split = (int)(item - r * x.np);
  const int b = (int)(r / R1), k = (int)(r - (int64_t)b * R1);
  const float T = x.row_T ? __ldg(x.row_T + b) : x.temperature;
  const float c = log2_scale(inv_temperature(T));
  const char* row = row_ptr<DT>(x.zt, x.zd, b, k, x.gamma, x.V);
  const int64_t lo = (int64_t)split * kChunkSweep;
  const int64_t hi = min(x.V, lo + kChunkSweep);
  const float tau = TOPK ? x.thr[r] : -kInf;  // logits below the top-k threshold add nothing

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
          for (int e = 0; e < VecInfo<DT>::kElems; ++e)
            acc += (TOPK && f[e] < tau) ? 0.0f : ex2(fmaf(f[e], c, -mc));
          s += acc;
        }
      },
      [&](int64_t, float z) {
        raise_max(z);
        if (zmax > -kInf && !(TOPK && z < tau)) s += ex2(fmaf(z, c, -mc));
      });

  MS v = warp_reduce_ms(MS{mc, s});
  const float zw = warp_max(zmax);
  __shared__ MS sm[kThreads / 32];
  __shared__ float sz[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sm[warp] = v;
    sz[warp] = zw;
  }
  __syncthreads();
  if (warp == 0) {
    v = (lane < (int)(blockDim.x >> 5)) ? sm[lane] : MS{-kInf, 0.0f};
    v = warp_reduce_ms(v);
    // the split's largest logit as given (its scaled max is v.m, bit for bit)
    const float Z = warp_max((lane < (int)(blockDim.x >> 5)) ? sz[lane] : -kInf);
    if (lane == 0) x.part[item] = make_float2(Z, v.s);
  }
}

// --------------------------------------------------------------------------
// Vector sweep (rows a multiple of 16 bytes): persistent, one resident wave, the
// 4 KB chunks of every row counted from the row's start (sv_units.cuh); one
// partial per chunk, part[(b R1 + k) nck + j].
// --------------------------------------------------------------------------
template <int DT, bool TOPK>
__global__ void __launch_bounds__(kSweepWarps * 32, kSweepCtasPerSm) k_sweep_vec(SweepCtx x) {
  extern __shared__ uint4 sweep_buf[];  // [kSweepWarps][kSweepBufs][256]
  pdl_launch_dependents();  // the next kernel may be scheduled now; it waits for us
  zero_draw_counters(x);
  const int64_t NU = (int64_t)x.B * (2 * x.gamma + 1) * x.np;
  const int64_t W = (int64_t)gridDim.x * kSweepWarps;
  unit_loop<DT, TOPK, kSweepBufs>(
      x, x.np, (NU - 1) / W, sweep_buf + (threadIdx.x >> 5) * kSweepBufs * 256,
      (int)(blockIdx.x * kSweepWarps + (threadIdx.x >> 5)), (int)W,
      [&](int64_t g, float2 p) {
        if ((threadIdx.x & 31) == 0) x.part[g] = p;
      });
}

// --------------------------------------------------------------------------
// Top-k thresholds ("Fast Inference from Transformers via Speculative
// Decoding", section "The loop": top-k zeroes the tail of p and q and
// renormalises; every entry at or above the k-th largest logit is kept).
// --------------------------------------------------------------------------
// Order-preserving key of a float: a larger float has a larger key (-0 sorts
// just below +0; the two compare equal as floats, so either gives the same cut).
__device__ __forceinline__ uint32_t fkey(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Histogram digits of the top-k radix select: bf16 values fill only the top 16
// bits of the key (digits of 10 and 6 bits; the wide first digit spreads
// logits, which crowd into a few exponents), fp32 values all 32 (four of 8).
template <int DT>
struct RadixDigits {
  static constexpr int kPasses = (DT == SV_BF16) ? 2 : 4;
  static constexpr int kMaxBins = (DT == SV_BF16) ? 1024 : 256;
  __device__ static int width(int pass) { return (DT == SV_BF16) ? (pass == 0 ? 10 : 6) : 8; }
};

// The k-th largest of the values that `visit` hands this CTA (each thread calls
// its argument for each of its values; NaN is not ranked), repeats counted;
// -inf when there are fewer than k.  A most-significant-digit radix select over
// fkey with per-warp shared-memory histograms hist[kWarps][kMaxBins] (fewer
// lanes collide on one counter).  Called by all threads; returns in all.
template <int DT, class Visit>
__device__ float radix_kth(Visit&& visit, int k, uint32_t* hist, uint32_t* s_sel) {
  constexpr int kWarps = kThreads / 32;
  using Dg = RadixDigits<DT>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t prefix = 0, mask = 0, remaining = (uint32_t)k;
  int shift = 32;
  bool few = false;
  for (int pass = 0; pass < Dg::kPasses && !few; ++pass) {
    const int width = Dg::width(pass);
    shift -= width;
    const uint32_t dmask = (1u << width) - 1u;
    const int nbins = 1 << width;
    for (int i = threadIdx.x; i < kWarps * Dg::kMaxBins; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    uint32_t* h = hist + warp * Dg::kMaxBins;
    visit([&](float z) {
      if (z != z) return;  // NaN is not ranked
      const uint32_t key = fkey(z);
      if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & dmask], 1u);
    });
    __syncthreads();
    for (int d = threadIdx.x; d < nbins; d += blockDim.x) {  // sum the warps' copies
      uint32_t n = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) n += hist[w * Dg::kMaxBins + d];
      hist[d] = n;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds `per` digits from top - l*per down; counts accumulate from the top
      const int per = nbins / 32;
      const int top = nbins - 1 - per * lane;
      uint32_t cl = 0;
      for (int j = 0; j < per; ++j) cl += hist[top - j];
      uint32_t incl = cl;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t excl = incl - cl;
      const bool mine = excl < remaining && remaining <= incl;
      if (__ballot_sync(0xffffffffu, mine) == 0u) {
        if (lane == 0) s_sel[2] = 1u;  // fewer than k ranked values
      } else if (mine) {
        uint32_t above = excl;
        int d = top;
        for (int j = 0; j < per; ++j, --d) {
          const uint32_t n = hist[d];
          if (above + n >= remaining) break;
          above += n;
        }
        s_sel[0] = prefix | ((uint32_t)d << shift);
        s_sel[1] = remaining - above;
        s_sel[2] = 0u;
      }
    }
    __syncthreads();
    few = s_sel[2] != 0u;
    prefix = s_sel[0];
    remaining = s_sel[1];
    mask |= dmask << shift;
    __syncthreads();
  }
  if (few) return -kInf;
  // bf16 keys leave the low 16 bits to the sign: 0 for a positive value, 1s otherwise
  const uint32_t key =
      (DT == SV_BF16) ? (prefix | ((prefix & 0x80000000u) ? 0u : 0xFFFFu)) : prefix;
  return fkey_inv(key);
}

// Every value of one logit row, for radix_kth (16-byte vectors where aligned).
template <int DT>
struct RowVisit {
  const char* base;
  int64_t V;
  template <class F>
  __device__ void operator()(F&& f) const {
    for_each_in_chunk<DT, 4>(
        base, 0, V,
        [&](int64_t, const uint4& vec) {
          float v[VecInfo<DT>::kElems];
          unpack<DT>(vec, v);
#pragma unroll
          for (int e = 0; e < VecInfo<DT>::kElems; ++e) f(v[e]);
        },
        [&](int64_t, float z) { f(z); });
  }
};

// One CTA per logit row: thr[row] = the k-th largest of the row's non-NaN
// values (repeats counted), -inf when it has fewer than k of them.
template <int DT>
__global__ void __launch_bounds__(kThreads) k_topk(const void* zt, const void* zd, int gamma,
                                                  int64_t V, int k, float* __restrict__ thr) {
  __shared__ uint32_t hist[(kThreads / 32) * RadixDigits<DT>::kMaxBins];
  __shared__ uint32_t s_sel[3];
  const int R1 = 2 * gamma + 1;
  const int row = blockIdx.x;
  const int b = row / R1, kk = row - b * R1;
  const float tau = radix_kth<DT>(RowVisit<DT>{row_ptr<DT>(zt, zd, b, kk, gamma, V), V}, k,
                                  hist, s_sel);
  if (threadIdx.x == 0) thr[row] = tau;
}

// Shared-memory candidates of the top-k select that follows a plain sweep.
constexpr int kTopkCandCap = 4096;

// Dynamic shared memory of k_topk_cand: per-warp histograms, then candidates.
static size_t topk_cand_smem_bytes(int dtype) {
  return (size_t)(kThreads / 32) * (dtype == SV_BF16 ? 1024 : 256) * sizeof(uint32_t) +
         (size_t)kTopkCandCap * sizeof(float);
}

// Top-k after a plain sweep, from candidates (one CTA per logit row).  The k-th
// largest logit is at least the k-th largest of the row's chunk maxima (k
// chunks each hold a value at or above that), so only entries whose scaled
// value reaches that bound can be kept: they are gathered into shared memory,
// the threshold is their k-th largest, and the kept mass is summed over them.
// The row's chunk partials are then replaced by one partial of the kept
// entries, so the round needs no second sweep.  With more than kTopkCandCap
// candidates, or k above the number of chunks, the threshold comes from radix
// passes over the whole row and the kept mass from one more pass.  A row with a
// NaN or timed-out partial is left as it is (no cut).
template <int DT>
__global__ void __launch_bounds__(kThreads) k_topk_cand(SweepCtx x, int k,
                                                       float* __restrict__ thr) {
  constexpr int kWarps = kThreads / 32;
  extern __shared__ uint32_t dsm[];
  uint32_t* hist = dsm;  // [kWarps][RadixDigits<DT>::kMaxBins]
  float* cand = reinterpret_cast<float*>(dsm + kWarps * RadixDigits<DT>::kMaxBins);
  __shared__ uint32_t s_sel[3];
  __shared__ uint32_t s_n;
  __shared__ int s_bad;
  __shared__ float s_max;
  __shared__ float s_red[kWarps];
  const int R1 = 2 * x.gamma + 1;
  const int row = blockIdx.x;
  const int b = row / R1, kk = row - b * R1;
  const int64_t V = x.V;
  const RowParts rp = row_parts<DT>(x, row);
  const int nch = rp.n;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowVisit<DT> rowv{row_ptr<DT>(x.zt, x.zd, b, kk, x.gamma, V), V};
  const float T = x.row_T ? __ldg(x.row_T + b) : x.temperature;
  const float c = log2_scale(inv_temperature(T));
  if (threadIdx.x == 0) {
    s_n = 0u;
    s_bad = 0;
  }
  __syncthreads();
  // the row's largest logit and whether it is usable
  float m = -kInf;
  int bad = 0;
  for (int j = threadIdx.x; j < nch; j += blockDim.x) {
    const float2 p = __ldcg(rp.at(j));
    if (p.x != p.x || p.y < 0.0f) bad = 1;
    m = fmaxf(m, p.x);
  }
  m = warp_max(m);
  const bool any_bad = __any_sync(0xffffffffu, bad) != 0;
  if (lane == 0) {
    s_red[warp] = m;
    if (any_bad) atomicOr(&s_bad, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = -kInf;
    for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_red[w]);
    s_max = mm;
  }
  __syncthreads();
  if (s_bad || !(s_max > -kInf)) {  // not finite, timed out or empty: no cut
    if (threadIdx.x == 0) thr[row] = -kInf;
    return;
  }
  const float Mz = s_max;     // the row's largest logit
  const float M = Mz * c;     // its scaled max, bit for bit the sweep's
  // lower bound of the threshold: the k-th largest chunk max
  const float bound = (k <= nch) ? radix_kth<SV_F32>(
                                       [&](auto&& f) {
                                         for (int j = threadIdx.x; j < nch; j += blockDim.x)
                                           f(__ldcg(rp.at(j)).x);
                                       },
                                       k, hist, s_sel)
                                 : -kInf;
  if (bound > -kInf) {
    rowv([&](float z) {
      if (z == z && z >= bound) {
        const uint32_t i = atomicAdd(&s_n, 1u);
        if (i < (uint32_t)kTopkCandCap) cand[i] = z;
      }
    });
  }
  __syncthreads();
  const uint32_t n = s_n;
  const bool from_cand = bound > -kInf && n <= (uint32_t)kTopkCandCap;
  float tau;
  if (from_cand) {
    tau = radix_kth<DT>(
        [&](auto&& f) {
          for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) f(cand[i]);
        },
        k, hist, s_sel);
  } else {
    tau = radix_kth<DT>(rowv, k, hist, s_sel);
  }
  // the kept mass, relative to the row's max
  float sum = 0.0f;
  auto add = [&](float z) {
    if (z >= tau) sum += ex2(fmaf(z, c, -M));
  };
  if (from_cand) {
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) add(cand[i]);
  } else {
    rowv(add);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncthreads();
  if (lane == 0) s_red[warp] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float S = 0.0f;
    for (int w = 0; w < kWarps; ++w) S += s_red[w];
    thr[row] = tau;
    *rp.at(0) = make_float2(Mz, S);
  }
  for (int j = 1 + (int)threadIdx.x; j < nch; j += blockDim.x) *rp.at(j) = make_float2(-kInf, 0.0f);
}

// Nucleus (top-p) threshold of one logit row (same passage: nucleus zeroes the
// tail and renormalises).  The row keeps the smallest set of largest-logit
// entries whose probability reaches top_p, entries equal to the last one kept
// as well: thr = the largest logit t such that the mass of {z >= t} reaches
// top_p of the row's mass.  One CTA per row, after a sweep that gave the row's
// max; entries below the row's top-k threshold (thr on entry, when has_k) do
// not count.  Masses 2^(z c - max) are summed as 40-bit fixed point, so the
// sums are exact and independent of order.  The first pass bins every entry
// by its log2 mass, z c - max, in steps of 1/32 (1024 bins; masses below 2^-32
// share the lowest), a digit that never decreases as z grows and that spreads
// the logits over hundreds of bins (bins over the float's leading bits would
// crowd them into a few exponents, and lanes adding to one counter serialise).
// Most-significant-digit passes over order-preserving keys (bf16: digits of 10
// and 6 bits; fp32: four of 8) then refine among the entries of the chosen
// mass bin only: every entry of a higher bin has a larger logit than all of
// them, every entry of a lower bin a smaller one, so the cut is the same as a
// select over the keys of the whole row.  Each mass goes in three 14-bit parts
// to three 32-bit per-warp histograms (native shared-memory atomics; a warp
// adds at most 2^18 entries, so no part overflows for V <= 2^21), combined in
// 64 bits per digit afterwards.  Empty or non-finite rows keep thr as it was.  Empty or non-finite rows keep thr as it was.
template <int DT>
__global__ void __launch_bounds__(kThreads) k_topp(SweepCtx x, float top_p, int has_k,
                                                  float* __restrict__ thr) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kPasses = 1 + ((DT == SV_BF16) ? 2 : 4);
  constexpr int kMaxBins = 1024;
  extern __shared__ unsigned long long hist64[];  // [kMaxBins] combined, then parts
  __shared__ RowStat s_rs;
  __shared__ uint32_t s_sel[2];       // prefix, no-cut flag
  __shared__ double s_target;
  const int R1 = 2 * x.gamma + 1;
  const int row = blockIdx.x;
  const int b = row / R1, kk = row - b * R1;
  const int64_t V = x.V;
  const char* base = row_ptr<DT>(x.zt, x.zd, b, kk, x.gamma, V);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float T = x.row_T ? __ldg(x.row_T + b) : x.temperature;
  const float c = log2_scale(inv_temperature(T));
  const float tk = has_k ? thr[row] : -kInf;
  if (!has_k && threadIdx.x == 0) thr[row] = -kInf;  // no cut unless one is found below
  if (warp == 0) {
    const RowStat rs = combine_parts(row_parts<DT>(x, row), nullptr, c);
    if (lane == 0) s_rs = rs;
  }
  __syncthreads();
  const RowStat rs = s_rs;
  if ((rs.bits & (kRowNaN | kRowTimeout)) || !(rs.s > 0.0f) || !(rs.s < kInf) ||
      !(fabsf(rs.mc) < kInf))
    return;  // empty or not finite: no cut (uniform over the CTA)
  const float mc = rs.mc;
  // mass bin of an entry from its scaled logit u = z c - max (<= 0 up to rounding)
  auto mass_bin = [](float u) -> uint32_t {
    return 1023u - (uint32_t)fminf(fmaxf(-32.0f * u, 0.0f), 1023.0f);
  };
  uint32_t bin0 = 0, prefix = 0, mask = 0;
  int shift = 32;
  double target = 0.0;  // fixed-point mass still to reach inside the current prefix
  for (int pass = 0; pass < kPasses; ++pass) {
    const int width = pass == 0 ? 10 : (DT == SV_BF16) ? (pass == 1 ? 10 : 6) : 8;
    if (pass > 0) shift -= width;
    const uint32_t dmask = (1u << width) - 1u;
    const int nbins = 1 << width;
    uint32_t* parts = reinterpret_cast<uint32_t*>(hist64 + kMaxBins);  // [3][kWarps][kMaxBins]
    for (int i = threadIdx.x; i < 3 * kWarps * kMaxBins; i += blockDim.x) parts[i] = 0u;
    __syncthreads();
    uint32_t* h0 = parts + warp * kMaxBins;
    uint32_t* h1 = h0 + kWarps * kMaxBins;
    uint32_t* h2 = h1 + kWarps * kMaxBins;
    auto add = [&](float z) {
      if (!(z >= tk)) return;  // NaN, or below the top-k threshold
      const float u = fmaf(z, c, -mc);
      const uint32_t mb = mass_bin(u);
      uint32_t d = mb;
      if (pass > 0) {
        const uint32_t key = fkey(z);
        if (mb != bin0 || (key & mask) != prefix) return;
        d = (key >> shift) & dmask;
      }
      const float m = ex2(u);  // <= 1
      // m 2^40 rounded to the nearest integer (ties to even), from the float's bits: the
      // conversion instruction to a 64-bit integer runs on the slow fp64 pipe
      const unsigned long long f = to_fix(m, 40);
      atomicAdd(&h0[d], (uint32_t)(f & 0x3FFFu));
      atomicAdd(&h1[d], (uint32_t)((f >> 14) & 0x3FFFu));
      atomicAdd(&h2[d], (uint32_t)(f >> 28));
    };
    for_each_in_chunk<DT, 4>(
        base, 0, V,
        [&](int64_t, const uint4& vec) {
          float f[VecInfo<DT>::kElems];
          unpack<DT>(vec, f);
#pragma unroll
          for (int e = 0; e < VecInfo<DT>::kElems; ++e) add(f[e]);
        },
        [&](int64_t, float z) { add(z); });
    __syncthreads();
    for (int d = threadIdx.x; d < nbins; d += blockDim.x) {  // sum the warps' copies
      unsigned long long n = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int i = w * kMaxBins + d;
        n += (unsigned long long)parts[i] +
             ((unsigned long long)parts[kWarps * kMaxBins + i] << 14) +
             ((unsigned long long)parts[2 * kWarps * kMaxBins + i] << 28);
      }
      hist64[d] = n;
    }
    __syncthreads();
    if (warp == 0) {
      const int per = nbins / 32;
      const int top = nbins - 1 - per * lane;
      unsigned long long cl = 0;
      for (int j = 0; j < per; ++j) cl += hist64[top - j];
      unsigned long long incl = cl;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (pass == 0) {
        // the whole kept mass is the last lane's total
        const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
        target = (double)top_p * (double)total;
      } else {
        target = s_target;
      }
      const unsigned long long excl = incl - cl;
      const bool mine = (double)excl < target && target <= (double)incl;
      if (__ballot_sync(0xffffffffu, mine) == 0u) {
        if (lane == 0) s_sel[1] = 1u;  // nothing to cut (no mass, or rounding at the end)
      } else if (mine) {
        unsigned long long above = excl;
        int d = top;
        for (int j = 0; j < per; ++j, --d) {
          const unsigned long long n = hist64[d];
          if ((double)(above + n) >= target) break;
          above += n;
        }
        s_sel[0] = (uint32_t)d;
        s_sel[1] = 0u;
        s_target = target - (double)above;
      }
    }
    __syncthreads();
    if (s_sel[1]) return;  // keep thr as it was
    if (pass == 0) {
      bin0 = s_sel[0];
    } else {
      prefix |= s_sel[0] << shift;
      mask |= dmask << shift;
    }
    target = s_target;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // bf16 keys leave the low 16 bits to the sign: 0 for a positive value, 1s otherwise
    const uint32_t key =
        (DT == SV_BF16) ? (prefix | ((prefix & 0x80000000u) ? 0u : 0xFFFFu)) : prefix;
    thr[row] = fkey_inv(key);
  }
}

// --------------------------------------------------------------------------
// Draw of the target's own token.
// --------------------------------------------------------------------------
// One CTA per (batch row, spc segments of 256 entries).  Every CTA of a batch
// row first takes the batch row's decision itself from the sweep's partials:
// one warp per logit row combines its partials, then one warp runs the accept
// test (the same arithmetic on the same numbers in every CTA, so all agree).
// The first CTA of the batch row also writes the row statistics, the accepted
// prefix, p, q, the count and the draw state.  Then the CTA writes the weight
// sums of its segments; the CTA that finishes last (a counter per batch row)
// draws the token from all of them by the inverse transform, falls back to p_n
// when the residual has no positive weight, and emits.
// The decision of batch row b taken by one CTA of the draw: the draft tokens and
// the logits at them (read before waiting for the previous kernel), the row
// statistics (one warp per logit row), then the accept test by warp 0.  Every
// CTA of the batch row computes the same numbers; the lead CTA writes the
// outputs of the decision.  The draw set-up lands in *s_st.
template <int DT, bool TOPK>
__device__ __forceinline__ void decide_in_cta(const SweepCtx& x, int b, bool lead,
                                              uint32_t* alpha_cnt, RowStat* srs, DraftAt* sda,
                                              DrawState* s_st) {
  const int gamma = x.gamma;
  const int R1 = 2 * gamma + 1;
  const int64_t V = x.V;
  constexpr int kWarps = kThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kWarps - 1 && lane < gamma) {
    // independent of the sweep: read before waiting for it
    DraftAt d;
    d.x = __ldg(x.xt + (int64_t)b * gamma + lane);
    d.zt = d.zd = 0.0f;
    if (d.x >= 0 && (int64_t)d.x < V) {
      d.zt = load_logit<DT>(row_ptr<DT>(x.zt, x.zd, b, lane, gamma, V), d.x);
      d.zd = load_logit<DT>(row_ptr<DT>(x.zt, x.zd, b, gamma + 1 + lane, gamma, V), d.x);
    }
    sda[lane] = d;
  }
  pdl_wait();  // the sweep's partials (and the top-k thresholds)
  pdl_launch_dependents();
  if (TOPK && warp == kWarps - 1 && lane < gamma) {
    // a draft token outside a row's top-k has probability 0 there
    DraftAt d = sda[lane];
    if (d.x >= 0 && (int64_t)d.x < V) {
      if (d.zt < __ldcg(x.thr + (int64_t)b * R1 + lane)) d.zt = -kInf;
      if (d.zd < __ldcg(x.thr + (int64_t)b * R1 + gamma + 1 + lane)) d.zd = -kInf;
    }
    sda[lane] = d;
  }
  if (lead && threadIdx.x == 0) alpha_cnt[b] = 0u;
  const float c_b = log2_scale(inv_temperature(x.row_T ? __ldg(x.row_T + b) : x.temperature));
  for (int k = warp; k < R1; k += 2 * kWarps) {
    // rows k and k + kWarps together: one round of partial loads for R1 <= 16
    const int k2 = k + kWarps;
    const int64_t r0 = (int64_t)b * R1 + k, r2 = (int64_t)b * R1 + k2;
    RowStat rs0, rs2;
    RowParts p2 = row_parts<DT>(x, k2 < R1 ? r2 : r0);
    if (k2 >= R1) p2.n = 0;
    combine_parts2(row_parts<DT>(x, r0), p2, lead ? x.rowstat + r0 : nullptr,
                   lead ? x.rowstat + r2 : nullptr, rs0, rs2, c_b);
    if (lane == 0) {
      srs[k] = rs0;
      if (k2 < R1) srs[k2] = rs2;
    }
  }
  __syncthreads();
  if (warp == 0) decide_batch_row<DT>(x, b, srs, sda, lead, s_st);
  __syncthreads();
}

template <int DT, bool TOPK>
__global__ void __launch_bounds__(kThreads, kDrawCtasPerSm) k_draw(SweepCtx x, DrawArgs a) {
  const int b = (int)(blockIdx.x / (unsigned)a.nsplit);
  const int split = (int)(blockIdx.x - (unsigned)b * (unsigned)a.nsplit);
  const int gamma = a.gamma;
  const int64_t V = a.V;
  const bool lead = (split == 0);
  constexpr int kWarps = kThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ RowStat srs[65];
  __shared__ DraftAt sda[32];
  __shared__ DrawState s_st;
  __shared__ int s_last;
  decide_in_cta<DT, TOPK>(x, b, lead, a.alpha_cnt, srs, sda, &s_st);
  const DrawState st = s_st;
  if (st.mode == kDrawDone) return;  // the same in every CTA of the batch row
  const bool resid = (st.mode == kDrawResidual);
  const char* rt = row_ptr<DT>(a.zt, a.zd, b, st.pos, gamma, V);
  const char* rd = resid ? row_ptr<DT>(a.zt, a.zd, b, gamma + 1 + st.pos, gamma, V) : nullptr;
  uint64_t* seg = a.segsum + (int64_t)b * a.nseg;
  const int s0 = split * a.spc, s1 = min(a.nseg, s0 + a.spc);
  __shared__ uint64_t s_wtot[kWarps];
  __shared__ int s_tok;
  const uint64_t wt =
      resid ? segment_sums<DT, true, TOPK>(rt, rd, V, a.vec, st, s0, s1, warp, kWarps, a.fsh, seg)
            : segment_sums<DT, false, TOPK>(rt, nullptr, V, a.vec, st, s0, s1, warp, kWarps,
                                            a.fsh, seg);
  if (lane == 0) s_wtot[warp] = wt;
  __threadfence();  // this CTA's segment sums before its arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t ct = 0;
    for (int w = 0; w < kWarps; ++w) ct += s_wtot[w];
    a.ctot[(int64_t)b * a.nsplit + split] = ct;
    __threadfence();
    s_last = (atomicAdd(a.done + b, 1u) == (unsigned)(a.nsplit - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // every other CTA's sums are visible from here
  const uint64_t k53 = draw_uniform53(a.seed, (uint32_t)st.pos, (uint32_t)b, a.round);
  const uint64_t* ctot = a.ctot + (int64_t)b * a.nsplit;
  int fl = st.flags;
  if (warp == 0) {
    const int t = resid ? draw_select_warp<DT, true, TOPK>(rt, rd, V, a.vec, st, seg, a.nseg,
                                                           ctot, a.nsplit, a.spc, a.fsh, k53)
                        : draw_select_warp<DT, false, TOPK>(rt, nullptr, V, a.vec, st, seg,
                                                            a.nseg, ctot, a.nsplit, a.spc,
                                                            a.fsh, k53);
    if (lane == 0) s_tok = t;
  }
  __syncthreads();
  int tok = s_tok;
  if (resid && tok < 0) {
    // the residual had no positive entry in floating point: draw from p_n itself
    fl |= SV_FLAG_RESIDUAL_FALLBACK;
    DrawState sp = st;
    sp.mode = kDrawSampleRow;
    segment_sums<DT, false, TOPK>(rt, nullptr, V, a.vec, sp, 0, a.nseg, warp, kWarps, a.fsh,
                                  seg);
    __syncthreads();
    if (warp == 0) {
      const int t = draw_select_warp<DT, false, TOPK>(rt, nullptr, V, a.vec, sp, seg, a.nseg,
                                                      nullptr, 0, 0, a.fsh, k53);
      if (lane == 0) s_tok = t;
    }
    __syncthreads();
    tok = s_tok;
  }
  if (threadIdx.x == 0) {
    if (tok < 0) {
      tok = 0;
      fl |= SV_FLAG_ZERO_MASS;
    }
    a.out_tokens[(int64_t)b * (gamma + 1) + st.pos] = tok;
    if (a.out_flags) a.out_flags[b] = (uint8_t)fl;
  }
}

// --------------------------------------------------------------------------
// k_race: the target's own token by Gumbel-max (the default sampler) after a
// separate sweep.  nsplit CTAs per batch row, one resident wave.  Every CTA
// takes its batch row's decision (decide_in_cta); each warp then races one
// eighth of the CTA's share of the slices (kRaceSlice entries each) in one
// contiguous piece, its rounds of loads staged in shared memory with the next
// rounds in flight.  The warps racing one draw share their bound on the
// second-best key through a word per batch row (zeroed by the sweep).  The
// batch row's CTAs form one thread-block cluster: each keeps its best two in
// shared memory, and after a cluster barrier the first reads the others' over
// distributed shared memory, merges and emits (no global counter, fence or
// candidate words on the way; a second barrier keeps the others resident while
// it reads).
// --------------------------------------------------------------------------
struct RaceArgs {
  uint32_t* alpha_cnt;    // [B] counters of the optional overlap kernel, zeroed here
  int nsplit;             // CTAs per batch row: the cluster size, 1..kRaceMaxCluster
  bool vec;               // 16-byte loads of 8 entries are aligned in every row
};
constexpr int kRaceMaxCluster = 8;  // the portable cluster size
constexpr size_t kRaceSmemBytes = (kThreads / 32) * kRaceWarpSmem;

template <int DT, bool TOPK>
__global__ void __launch_bounds__(kThreads, kRaceCtasPerSm) k_race(SweepCtx x, RaceArgs a) {
  const int b = (int)(blockIdx.x / (unsigned)a.nsplit);
  const int split = (int)(blockIdx.x - (unsigned)b * (unsigned)a.nsplit);
  const int64_t V = x.V;
  constexpr int kWarps = kThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  extern __shared__ uint4 race_smem[];  // [kWarps][kRaceWarpSmem / 16]
  uint4* sb = race_smem + warp * (kRaceWarpSmem / sizeof(uint4));
  __shared__ RowStat srs[65];
  __shared__ DraftAt sda[32];
  __shared__ DrawState s_st;
  __shared__ KeyTop2 s_t[kWarps];
  __shared__ KeyTop2 s_best;  // the CTA's best two, read by the cluster's first CTA
  decide_in_cta<DT, TOPK>(x, b, split == 0, a.alpha_cnt, srs, sda, &s_st);
  const DrawState st = s_st;
  // the same in every CTA of the batch row, so the whole cluster leaves together
  if (st.mode == kDrawDone) return;
  const bool resid = st.mode == kDrawResidual;
  // the CTA's share of the batch row's slices, one contiguous piece per warp (a
  // multiple of 8 entries each), so that a warp's rounds follow one another
  const int S = (int)race_slices(V);
  const int spc = (S + a.nsplit - 1) / a.nsplit;
  const int64_t clo = (int64_t)split * spc * kRaceSlice;
  const int64_t chi = min(V, clo + (int64_t)spc * kRaceSlice);
  const int64_t wlen = ceil_div(ceil_div(chi - clo, (int64_t)kWarps), (int64_t)8) * 8;
  const int64_t wlo = clo + warp * wlen;
  const int64_t whi = min(chi, wlo + wlen);
  KeyTop2 t = key_top2_empty();
  float th = -kInf;
  if (wlo < whi) race_draw<DT, TOPK>(x, b, st, resid, wlo, whi, a.vec, t, th,
                                       x.thw + (int64_t)b * kThwStride, sb);
  t = key_warp(t);
  if (lane == 0) s_t[warp] = t;
  __syncthreads();
  if (warp == 0) {
    KeyTop2 r = (lane < kWarps) ? s_t[lane] : key_top2_empty();
    r = key_warp(r);
    if (lane == 0) s_best = r;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every CTA's best two are in its shared memory
  if (split == 0 && warp == 0) {
    // the batch row's best two over its CTAs (lane j: CTA j's), then the emit
    KeyTop2 T = (lane < a.nsplit) ? *cluster.map_shared_rank(&s_best, lane) : key_top2_empty();
    T = key_warp(T);
    if (resid && T.a.i < 0)
      race_fallback_emit<DT, TOPK>(x, b, st, a.vec, st.flags, sb);
    else
      race_emit<DT>(x, b, st, T, resid, st.flags);
  }
  cluster.sync();  // no CTA leaves while the first may still read its shared memory
}

// --------------------------------------------------------------------------
// k_alpha: beta_i = sum_v min(p_i(v), q_i(v)); alpha_b = mean_i beta_i.
// --------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads)
k_alpha(const void* __restrict__ zt, const void* __restrict__ zd, int gamma, int64_t V,
        float temperature, const float* __restrict__ row_T, int nsplit,
        const RowStat* __restrict__ rowstat, const float* __restrict__ thr,
        float* __restrict__ part, uint32_t* __restrict__ counter,
        float* __restrict__ out_alpha) {
  const int64_t per_b = (int64_t)gamma * nsplit;
  const int b = (int)(blockIdx.x / per_b);
  const int rem = (int)(blockIdx.x - b * per_b);
  const int i = rem / nsplit, split = rem - i * nsplit;
  const int R1 = 2 * gamma + 1;
  const float T = row_T ? __ldg(row_T + b) : temperature;
  const float c = log2_scale(inv_temperature(T));
  const RowStat rs_t = rowstat[(int64_t)b * R1 + i];
  const RowStat rs_d = rowstat[(int64_t)b * R1 + gamma + 1 + i];
  const float it = (rs_t.s > 0.0f) ? 1.0f / rs_t.s : 0.0f;
  const float id = (rs_d.s > 0.0f) ? 1.0f / rs_d.s : 0.0f;
  const char* rt = row_ptr<DT>(zt, zd, b, i, gamma, V);
  const char* rd = row_ptr<DT>(zt, zd, b, gamma + 1 + i, gamma, V);
  const int64_t lo = (int64_t)split * kChunkSweep, hi = min(V, lo + kChunkSweep);
  // top-k thresholds of the two rows (-inf: no adjustment)
  const float tt = thr ? thr[(int64_t)b * R1 + i] : -kInf;
  const float td = thr ? thr[(int64_t)b * R1 + gamma + 1 + i] : -kInf;
  float acc = 0.0f;
  for (int64_t v = lo + threadIdx.x; v < hi; v += blockDim.x) {
    const float zt = load_logit<DT>(rt, v), zd = load_logit<DT>(rd, v);
    const float pt = (it > 0.0f && !(zt < tt)) ? ex2(fmaf(zt, c, -rs_t.mc)) * it : 0.0f;
    const float pd = (id > 0.0f && !(zd < td)) ? ex2(fmaf(zd, c, -rs_d.mc)) * id : 0.0f;
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
    s_last = is_last(atomicAdd(counter + b, 1u), (uint32_t)(gamma * nsplit));
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  double tot = 0.0;
  const float* pp = part + (int64_t)b * gamma * nsplit;
  for (int j = 0; j < gamma * nsplit; ++j) tot += (double)__ldcg(pp + j);
  out_alpha[b] = (float)(tot / gamma);
}

// --------------------------------------------------------------------------
// Host side.
// --------------------------------------------------------------------------
// Per-device launch facts for the persistent sweep, looked up once per device.
struct DeviceInfo {
  int sms = 0;
  int sweep_ctas_per_sm[2][2] = {{0, 0}, {0, 0}};  // by dtype, then top-k variant
  // k_race clusters of c CTAs that can be resident at once, c = 1..kRaceMaxCluster
  int race_clusters[2][2][kRaceMaxCluster + 1] = {};
  bool ready = false;
};

// Dynamic shared memory of k_topp: the combined 64-bit histogram, then three
// 32-bit per-warp histograms of the mass parts (1024 bins: the widest digit).
static size_t topp_smem_bytes() {
  const size_t bins = 1024;
  return bins * sizeof(unsigned long long) + 3 * (size_t)(kThreads / 32) * bins * sizeof(uint32_t);
}

template <int DT, bool TOPK>
static cudaError_t sweep_setup(DeviceInfo& d) {
  cudaError_t e = cudaFuncSetAttribute(k_sweep_vec<DT, TOPK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSweepSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.sweep_ctas_per_sm[DT][TOPK ? 1 : 0],
                                                    k_sweep_vec<DT, TOPK>, kSweepWarps * 32,
                                                    kSweepSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_race<DT, TOPK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kRaceSmemBytes);
  if (e != cudaSuccess) return e;
  for (int c = 1; c <= kRaceMaxCluster; ++c) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)c);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kRaceSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&d.race_clusters[DT][TOPK ? 1 : 0][c], k_race<DT, TOPK>,
                                       &cfg);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
static std::mutex g_dev_mu;
static DeviceInfo g_dev[64];

static cudaError_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_topp<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)topp_smem_bytes());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_topp<SV_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)topp_smem_bytes());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_topk_cand<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)topk_cand_smem_bytes(SV_BF16));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_topk_cand<SV_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)topk_cand_smem_bytes(SV_F32));
    if (e != cudaSuccess) return e;
    if ((e = sweep_setup<SV_F32, false>(d)) != cudaSuccess) return e;
    if ((e = sweep_setup<SV_BF16, false>(d)) != cudaSuccess) return e;
    if ((e = sweep_setup<SV_F32, true>(d)) != cudaSuccess) return e;
    if ((e = sweep_setup<SV_BF16, true>(d)) != cudaSuccess) return e;

    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

template <int DT>
static cudaError_t launch_sample_t(const void* zt, const void* zd, const int32_t* xt, int B,
                                   int gamma, int64_t V, float temperature, const float* row_T,
                                   uint64_t seed, uint64_t round, int32_t* out_tokens,
                                   int32_t* out_counts, float* out_p, float* out_q,
                                   float* out_alpha, uint8_t* out_flags, char* ws,
                                   const SamplePlan& pl, cudaStream_t stream, float lenience,
                                   int top_k, float top_p, int sampler) {
  const int R1 = pl.R1;
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + pl.off_cnt);
  float2* part1 = reinterpret_cast<float2*>(ws + pl.off_part1);
  RowStat* rowstat = reinterpret_cast<RowStat*>(ws + pl.off_rowstat);
  DrawState* state = reinterpret_cast<DrawState*>(ws + pl.off_state);
  uint64_t* segsum = reinterpret_cast<uint64_t*>(ws + pl.off_segsum);
  uint64_t* ctot = reinterpret_cast<uint64_t*>(ws + pl.off_ctot);
  float* apart = reinterpret_cast<float*>(ws + pl.off_alpha);
  float* thr = reinterpret_cast<float*>(ws + pl.off_thr);
  uint32_t* alpha_cnt = cnt;
  uint32_t* done = cnt + B;
  DeviceInfo* di = nullptr;
  {
    const cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
  }
  // top-k adjusts the rows only when it cuts something: k < V; top-p when p < 1
  const bool topk = top_k > 0 && (int64_t)top_k < V;
  const bool topp = top_p < 1.0f;
  const bool masked = topk || topp;  // the round runs on thresholded rows
  const int tk = masked ? 1 : 0;
  const bool vec_sweep = use_vec_sweep(DT, V) && di->sweep_ctas_per_sm[DT][tk] > 0;
  // partials per row: 4 KB chunks (vector sweep) or kChunkSweep-logit splits
  const int nch = (int)ceil_div(V, kChunkSweep);
  SweepCtx sx{};
  sx.zt = zt;
  sx.zd = zd;
  sx.xt = xt;
  sx.B = B;
  sx.gamma = gamma;
  sx.V = V;
  sx.temperature = temperature;
  sx.row_T = row_T;
  sx.seed = seed;
  sx.round = round;
  sx.np = vec_sweep ? (int)vec_sweep_chunks(DT, V) : nch;
  sx.part = part1;
  sx.rowstat = rowstat;
  sx.state = state;
  sx.out_tokens = out_tokens;
  sx.out_counts = out_counts;
  sx.out_p = out_p;
  sx.out_q = out_q;
  sx.out_flags = out_flags;
  sx.inv_lenience = 1.0f / lenience;
  sx.thr = masked ? thr : nullptr;
  sx.done = done;
  sx.thw = reinterpret_cast<uint32_t*>(ws + pl.off_thw);
  const auto alpha = [&]() -> cudaError_t {
    if (!out_alpha) return cudaSuccess;
    const int ns = (int)ceil_div(V, kChunkSweep);
    k_alpha<DT><<<(unsigned)((int64_t)ns * gamma * B), kThreads, 0, stream>>>(
        zt, zd, gamma, V, temperature, row_T, ns, rowstat, sx.thr, apart, alpha_cnt, out_alpha);
    return cudaGetLastError();
  };
  auto sweep = [&](bool with_thr, const SweepCtx& ctx) {
    if (vec_sweep) {
      // one resident wave of warps, chunks dealt round-robin
      const int64_t nc = (int64_t)B * R1 * ctx.np;
      const int64_t full = (int64_t)di->sms * di->sweep_ctas_per_sm[DT][with_thr ? 1 : 0];
      const int64_t need = ceil_div(nc, kSweepWarps);
      const int64_t g = full < need ? full : need;
      const dim3 grid((unsigned)(g < 1 ? 1 : g));
      if (with_thr)
        k_sweep_vec<DT, true><<<grid, kSweepWarps * 32, kSweepSmemBytes, stream>>>(ctx);
      else
        k_sweep_vec<DT, false><<<grid, kSweepWarps * 32, kSweepSmemBytes, stream>>>(ctx);
    } else {
      const dim3 grid((unsigned)((int64_t)nch * B * R1));
      if (with_thr)
        k_sweep<DT, true><<<grid, kThreads, 0, stream>>>(ctx);
      else
        k_sweep<DT, false><<<grid, kThreads, 0, stream>>>(ctx);
    }
  };
  mark(0, stream);
  if (topk && !topp) {
    // top-k alone: a plain sweep, then the threshold and the kept mass from the
    // entries at or above the k-th largest chunk max (no second sweep)
    sweep(false, sx);
    k_topk_cand<DT><<<(unsigned)((int64_t)B * R1), kThreads, topk_cand_smem_bytes(DT), stream>>>(
        sx, top_k, thr);
    mark(1, stream);
  }
  if (topk && topp)
    k_topk<DT><<<(unsigned)((int64_t)B * R1), kThreads, 0, stream>>>(zt, zd, gamma, V, top_k,
                                                                        thr);
  if (topp) {
    // the row maxima (after top-k) for the nucleus masses, then the nucleus cut
    SweepCtx s0 = sx;
    s0.thr = topk ? thr : nullptr;
    sweep(topk, s0);
    k_topp<DT><<<(unsigned)((int64_t)B * R1), kThreads, topp_smem_bytes(), stream>>>(
        sx, top_p, topk ? 1 : 0, thr);
  }
  if (!(topk && !topp)) {
    sweep(masked, sx);
    mark(1, stream);
  }
  const int64_t vec_elems = (DT == SV_F32) ? 4 : 8;
  const bool vec = (V % vec_elems) == 0 && (reinterpret_cast<uintptr_t>(zt) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(zd) % 16) == 0;
  const int64_t slots = (int64_t)di->sms * kDrawCtasPerSm;
  cudaError_t e = cudaSuccess;
  if (sampler == SV_SAMPLER_INVERSE) {
    // One resident wave of draw CTAs when the batch allows: every CTA takes its
    // batch row's decision before drawing, so a second wave would pay that
    // latency again.  At least kChunkDraw entries per CTA.
    const int64_t nseg = ceil_div(V, kDrawSegEntries);
    int64_t nsplit = pl.nsplit3;
    if ((int64_t)B * nsplit > slots) nsplit = (slots / B > 1) ? slots / B : 1;
    const int64_t spc = ceil_div(nseg, nsplit);
    nsplit = ceil_div(nseg, spc);  // no CTA without segments
    DrawArgs da{zt, zd, B, gamma, V, seed, round, alpha_cnt, done, segsum, ctot, fix_shift(V),
                (int)nseg, (int)nsplit, (int)spc, vec, out_tokens, out_flags};
    e = masked ? launch_pdl(k_draw<DT, true>, dim3((unsigned)(nsplit * B)), dim3(kThreads), 0,
                            stream, sx, da)
               : launch_pdl(k_draw<DT, false>, dim3((unsigned)(nsplit * B)), dim3(kThreads), 0,
                            stream, sx, da);
  } else {
    // Gumbel-max: one cluster of race CTAs per batch row, all clusters resident
    // at once (every CTA takes its batch row's decision, so a second wave would
    // pay that latency again), at most one slice per warp
    const int64_t S = race_slices(V);
    const int* ncl = di->race_clusters[DT][masked ? 1 : 0];
    int nsplit = (int)min((int64_t)kRaceMaxCluster, ceil_div(S, (int64_t)(kThreads / 32)));
    while (nsplit > 1 && B > ncl[nsplit]) --nsplit;
    RaceArgs ra{alpha_cnt, nsplit, vec};
    e = masked ? launch_pdl_cluster(k_race<DT, true>, dim3((unsigned)(nsplit * B)),
                                    dim3(kThreads), kRaceSmemBytes, (unsigned)nsplit, stream, sx,
                                    ra)
               : launch_pdl_cluster(k_race<DT, false>, dim3((unsigned)(nsplit * B)),
                                    dim3(kThreads), kRaceSmemBytes, (unsigned)nsplit, stream, sx,
                                    ra);
  }
  if (e != cudaSuccess) return e;
  mark(2, stream);
  return alpha();
}

cudaError_t launch_sample(const void* zt, const void* zd, const int32_t* xt, int B, int gamma,
                          int64_t V, int dtype, float temperature, const float* row_T,
                          uint64_t seed, uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                          float* out_p, float* out_q, float* out_alpha, uint8_t* out_flags,
                          void* ws, const SamplePlan& pl, cudaStream_t stream, float lenience,
                          int top_k, float top_p, int sampler) {
  char* w = reinterpret_cast<char*>(ws);
  if (dtype == SV_F32)
    return launch_sample_t<SV_F32>(zt, zd, xt, B, gamma, V, temperature, row_T, seed, round,
                                   out_tokens, out_counts, out_p, out_q, out_alpha, out_flags, w,
                                   pl, stream, lenience, top_k, top_p, sampler);
  return launch_sample_t<SV_BF16>(zt, zd, xt, B, gamma, V, temperature, row_T, seed, round,
                                  out_tokens, out_counts, out_p, out_q, out_alpha, out_flags, w,
                                  pl, stream, lenience, top_k, top_p, sampler);
}

}  // namespace sv
