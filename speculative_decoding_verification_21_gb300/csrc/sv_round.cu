// sv_round.cu -- the sampling round as one persistent kernel on sm_103a.
//
// One round for B independent batch rows ("Fast Inference from Transformers
// via Speculative Decoding", section "The loop: draft, verify in one pass, keep
// a prefix", Algorithm 1 steps 3-4; the course notes "Speculative Decoding",
// "The algorithm").  Every warp of one resident wave runs the vector sweep over
// the 4 KB chunks of all 2*gamma+1 rows of every batch row, in batch-row order
// (sv_units.cuh), and takes on three kinds of task for the batch rows whose
// chunks are done, at fixed iterations of its loop:
//
//   decision  (one warp per batch row, `lag` iterations after the batch row's
//             last chunk): the row statistics from the chunk partials, p(x_i),
//             q(x_i), u_i, accept iff u_i <= p/q, the first rejection by a warp
//             ballot; writes the prefix, the count, p, q and publishes the draw
//             set-up.
//   race      (one warp per slice of kRaceSlice vocabulary entries, one
//             iteration later): the Gumbel-max race over the slice for the
//             residual max(0, p_n - q_n) (and p_n, its fallback) or for the
//             bonus row p_gamma; publishes the slice's best two of each.
//   merge     (one warp per batch row, one iteration later): the best two over
//             the slices, re-decided in double near a tie (sv_gumbel.cuh); emits
//             the token and the flags.
//
// Tasks hand over through 64-bit words that are never zero once written (the
// partials, the decision, the slices' candidates), zeroed before the launch:
// a consumer reads a word until it is non-zero.  Each word carries its whole
// value, so no fence is needed (relaxed 64-bit accesses are single-copy
// atomic).  Every wait is bounded (a deadline per task, and the first wait
// that gives up ends all others); a wait that gives up marks the batch row
// SV_FLAG_TIMEOUT.  A task only waits for work of earlier iterations, and the
// kernel is a cooperative launch (all CTAs resident), so every wait ends.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>

#include "specverify.h"
#include "sv_decide.cuh"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_gumbel.cuh"
#include "sv_launch.h"
#include "sv_plan.h"
#include "sv_sweep.cuh"
#include "sv_units.cuh"

namespace sv {

namespace {

struct RoundArgs {
  SweepCtx x;         // inputs, outputs; x.part unused (the partials are words here)
  uint32_t* abort;    // set by the first wait that gives up: every other wait ends at once
  uint64_t* dword;    // [B][3] the decision of each batch row
  uint64_t* cword;    // [B][S][4] per race slice: residual best two, p_n best two
  uint64_t* pword;    // [B][R1][nck] the chunk partials
  int nck;            // chunks per row
  int S;              // race slices per batch row
  int lag;            // iterations between a batch row's last chunk and its decision
};

// A task's waits share one deadline (20 ms after the task starts: the whole
// round takes tens of microseconds), and the first wait of the launch that gives
// up sets a word that ends every other wait at once.
constexpr uint64_t kTaskBudgetNs = 20000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct Waiter {
  uint64_t deadline;
  uint32_t* abort;
  __device__ __forceinline__ explicit Waiter(uint32_t* a) : deadline(global_ns() + kTaskBudgetNs), abort(a) {}
  // *p once it is non-zero; 0 when the wait gives up.
  __device__ __forceinline__ uint64_t poll(const uint64_t* p) const {
    uint64_t v = ld_relaxed64(p);
    while (v == 0) {
      if (*reinterpret_cast<volatile uint32_t*>(abort) != 0u) return 0;
      if (global_ns() > deadline) {
        atomicExch(abort, 1u);
        return 0;
      }
      __nanosleep(200);
      v = ld_relaxed64(p);
    }
    return v;
  }
};

// The decision of a batch row in three words (each never zero).
__device__ __forceinline__ void publish_state(uint64_t* d, const DrawState& st) {
  const uint32_t info = 0x80000000u | (uint32_t)st.mode | ((uint32_t)st.pos << 2) |
                        ((uint32_t)(st.flags & 0xFF) << 16);
  st_relaxed64(d + 0, ((uint64_t)__float_as_uint(st.zmt) << 32) | info);
  st_relaxed64(d + 1, ((uint64_t)(__float_as_uint(st.K) ^ 0x80000000u) << 32) |
                          __float_as_uint(st.zmd));
  st_relaxed64(d + 2, ((uint64_t)(__float_as_uint(st.sd) ^ 0x80000000u) << 32) |
                          __float_as_uint(st.st));
}

// The draw set-up of batch row b (false when the wait gave up).
__device__ __forceinline__ bool read_state(const RoundArgs& a, int b, DrawState& st,
                                           const Waiter& wt) {
  const uint64_t* d = a.dword + (int64_t)b * 3;
  const uint64_t w0 = wt.poll(d), w1 = wt.poll(d + 1), w2 = wt.poll(d + 2);
  if (!w0 || !w1 || !w2) return false;
  const uint32_t info = (uint32_t)w0;
  st = DrawState{};
  st.mode = (int)(info & 3u);
  st.pos = (int)((info >> 2) & 0x3FFFu);
  st.flags = (int)((info >> 16) & 0xFFu);
  st.zmt = __uint_as_float((uint32_t)(w0 >> 32));
  st.zmd = __uint_as_float((uint32_t)w1);
  st.K = __uint_as_float((uint32_t)(w1 >> 32) ^ 0x80000000u);
  st.st = __uint_as_float((uint32_t)w2);
  st.sd = __uint_as_float((uint32_t)(w2 >> 32) ^ 0x80000000u);
  const float T = a.x.row_T ? __ldg(a.x.row_T + b) : a.x.temperature;
  st.invT = inv_temperature(T);
  st.c = log2_scale(st.invT);
  st.mct = st.zmt * st.c;  // bit for bit the row statistics' scaled max
  st.mcd = st.zmd * st.c;
  st.tt = st.td = -kInf;
  return true;
}

// ---- decision ----------------------------------------------------------------
// Rows combine in groups of kRowGroup with kWordsInFlight partials per lane and
// row in flight; lane l adds the row's partials j = l, l + 32, ... in order
// (the combine of every other path).
constexpr int kRowGroup = 4;
constexpr int kWordsInFlight = 2;

template <int DT>
__device__ void round_decide(const RoundArgs& a, int b, RowStat* srs, DraftAt* sda,
                             DrawState* sst) {
  const SweepCtx& x = a.x;
  const int lane = threadIdx.x & 31;
  const int gamma = x.gamma, R1 = 2 * gamma + 1, nck = a.nck;
  const int64_t V = x.V;
  const float T = x.row_T ? __ldg(x.row_T + b) : x.temperature;
  const float c = log2_scale(inv_temperature(T));
  if (lane < gamma) {  // inputs: no wait
    DraftAt d;
    d.x = __ldg(x.xt + (int64_t)b * gamma + lane);
    d.zt = d.zd = 0.0f;
    if (d.x >= 0 && (int64_t)d.x < V) {
      d.zt = load_logit<DT>(row_ptr<DT>(x.zt, x.zd, b, lane, gamma, V), d.x);
      d.zd = load_logit<DT>(row_ptr<DT>(x.zt, x.zd, b, gamma + 1 + lane, gamma, V), d.x);
    }
    sda[lane] = d;
  }
  const uint64_t* pw = a.pword + (int64_t)b * R1 * nck;
  const Waiter wt(a.abort);
  for (int k0 = 0; k0 < R1; k0 += kRowGroup) {
    RowAcc acc[kRowGroup];
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) acc[r] = row_acc_init();
    for (int j0 = 0; j0 < nck; j0 += 32 * kWordsInFlight) {
      uint64_t wv[kRowGroup][kWordsInFlight];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int u = 0; u < kWordsInFlight; ++u) {
          const int j = j0 + lane + 32 * u;
          wv[r][u] = (k0 + r < R1 && j < nck) ? ld_relaxed64(pw + (int64_t)(k0 + r) * nck + j) : 1ull;
        }
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int u = 0; u < kWordsInFlight; ++u) {
          const int j = j0 + lane + 32 * u;
          if (k0 + r < R1 && j < nck) {
            uint64_t v = wv[r][u];
            if (v == 0) v = wt.poll(pw + (int64_t)(k0 + r) * nck + j);
            // a partial that never came: the row is not usable (timed out)
            row_acc_add(acc[r], v ? part_unword(v) : make_float2(CUDART_NAN_F, -1.0f), c);
          }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowGroup; ++r) {
      if (k0 + r >= R1) break;
      const RowStat rs = row_acc_finish(acc[r], x.rowstat + (int64_t)b * R1 + k0 + r);
      if (lane == 0) srs[k0 + r] = rs;
    }
  }
  __syncwarp();
  decide_batch_row<DT>(x, b, srs, sda, true, sst);
  __syncwarp();
  if (lane == 0) publish_state(a.dword + (int64_t)b * 3, *sst);
}

// ---- race over one slice -----------------------------------------------------
template <int DT>
__device__ void round_race(const RoundArgs& a, int b, int s) {
  const SweepCtx& x = a.x;
  DrawState st;
  const Waiter wt(a.abort);
  if (!read_state(a, b, st, wt) || st.mode == kDrawDone) return;
  const int gamma = x.gamma;
  const int64_t V = x.V;
  const bool resid = st.mode == kDrawResidual;
  const char* rt = row_ptr<DT>(x.zt, x.zd, b, st.pos, gamma, V);
  const char* rd = resid ? row_ptr<DT>(x.zt, x.zd, b, gamma + 1 + st.pos, gamma, V) : rt;
  const int64_t lo = (int64_t)s * kRaceSlice;
  const int64_t hi = (lo + kRaceSlice < V) ? lo + kRaceSlice : V;
  RaceTop2 tr = race_top2_empty(), tp = race_top2_empty();
  if (resid)
    race_range<DT, true, false>(rt, rd, lo, hi, V, true, st, __fsub_rn(st.K, st.mct), x.seed,
                                x.round, b, tr, tp);
  else
    race_range<DT, false, false>(rt, rd, lo, hi, V, true, st, 0.0f, x.seed, x.round, b, tr, tp);
  tr = race_warp(tr);
  tp = race_warp(tp);
  if ((threadIdx.x & 31) == 0) {
    uint64_t* o = a.cword + ((int64_t)b * a.S + s) * 4;
    st_relaxed64(o + 0, key_word(race_key(tr.a)));
    st_relaxed64(o + 1, key_word(race_key(tr.b)));
    st_relaxed64(o + 2, key_word(race_key(tp.a)));
    st_relaxed64(o + 3, key_word(race_key(tp.b)));
  }
}

// ---- merge -------------------------------------------------------------------
template <int DT>
__device__ void round_merge(const RoundArgs& a, int b) {
  const SweepCtx& x = a.x;
  const int lane = threadIdx.x & 31;
  DrawState st;
  const Waiter wt(a.abort);
  if (!read_state(a, b, st, wt)) {
    if (lane == 0 && x.out_flags) x.out_flags[b] = (uint8_t)(SV_FLAG_TIMEOUT | SV_FLAG_NONFINITE);
    return;
  }
  if (st.mode == kDrawDone) return;  // the decision emitted the row
  KeyTop2 R{KeyIdx{-1.0f, -1}, KeyIdx{-1.0f, -1}}, P = R;
  bool lost = false;
  const uint64_t* cw = a.cword + (int64_t)b * a.S * 4;
  for (int s = lane; s < a.S; s += 32) {
    uint64_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = ld_relaxed64(cw + (int64_t)s * 4 + q);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (w[q] == 0) w[q] = wt.poll(cw + (int64_t)s * 4 + q);
    lost |= !w[0] || !w[1] || !w[2] || !w[3];
    if (w[0]) key_insert(R, key_unword(w[0]));
    if (w[1]) key_insert(R, key_unword(w[1]));
    if (w[2]) key_insert(P, key_unword(w[2]));
    if (w[3]) key_insert(P, key_unword(w[3]));
  }
  R = key_warp(R);
  P = key_warp(P);
  lost = __any_sync(0xffffffffu, lost);
  race_emit<DT>(x, b, st, R, P, lost);
}

// ---- the kernel --------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kSweepWarps * 32, kSweepCtasPerSm) k_round(RoundArgs a) {
  __shared__ RowStat s_rs[kSweepWarps][2 * 32 + 1];
  __shared__ DraftAt s_da[kSweepWarps][32];
  __shared__ DrawState s_st[kSweepWarps];
  const SweepCtx& x = a.x;
  const int warp = threadIdx.x >> 5;
  const int G = (int)gridDim.x, W = G * kSweepWarps;
  const int cta = (int)blockIdx.x;
  const int B = x.B, R1 = 2 * x.gamma + 1;
  const int64_t U = (int64_t)R1 * a.nck;  // chunks per batch row
  const int64_t NU = (int64_t)B * U;
  // batch rows whose last chunk comes at iteration q: [rows_from(q), rows_from(q + 1))
  auto rows_from = [&](int64_t q) -> int {
    if (q <= 0) return 0;
    const int64_t r = q * W / U;
    return (int)(r < B ? r : B);
  };
  const int64_t it_last = (NU - 1) / W;
  const int64_t it_end = it_last + a.lag + 2;
  // this warp's share of each kind of task: index i goes to CTA (i + off) mod G,
  // warp (i / G) mod 8 of it (reversed for decisions and merges)
  const int idx_race = warp * G + cta;
  const int idx_dec = (kSweepWarps - 1 - warp) * G + cta;
  const int idx_merge = (kSweepWarps - 1 - warp) * G + (cta + G - G / 2) % G;
  unit_loop<DT, false>(
      x, a.nck, it_end,
      [&](int64_t g, float2 p) {
        if ((threadIdx.x & 31) == 0) st_relaxed64(a.pword + g, part_word(p));
      },
      [&](int64_t it) {
        int b0 = rows_from(it - a.lag), b1 = rows_from(it - a.lag + 1);
        if (it - a.lag >= 0)
          for (int i = idx_dec; i < b1 - b0; i += W)
            round_decide<DT>(a, b0 + i, s_rs[warp], s_da[warp], &s_st[warp]);
        b0 = rows_from(it - a.lag - 1);
        b1 = rows_from(it - a.lag);
        if (it - a.lag - 1 >= 0) {
          const int n = (b1 - b0) * a.S;
          for (int i = idx_race; i < n; i += W) round_race<DT>(a, b0 + i / a.S, i % a.S);
        }
        b0 = rows_from(it - a.lag - 2);
        b1 = rows_from(it - a.lag - 1);
        if (it - a.lag - 2 >= 0)
          for (int i = idx_merge; i < b1 - b0; i += W) round_merge<DT>(a, b0 + i);
      });
}

}  // namespace

// Per-device facts of the fused round, looked up once per device.
struct RoundDevice {
  int sms = 0, ctas[2] = {0, 0};
  bool ready = false;
};
static RoundDevice g_round_dev[64];

static cudaError_t round_device(RoundDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  RoundDevice& d = g_round_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.ctas[SV_F32], k_round<SV_F32>,
                                                           kSweepWarps * 32, 0)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.ctas[SV_BF16], k_round<SV_BF16>,
                                                           kSweepWarps * 32, 0)) != cudaSuccess)
      return e;
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

// The fused round: zero its words, then one cooperative launch.  Needs the
// vector sweep's shapes (rows a multiple of 16 bytes) and no top-k / top-p.
cudaError_t launch_round(const SweepCtx& x, int dtype, char* ws, const SamplePlan& pl,
                         cudaStream_t stream) {
  RoundDevice* d = nullptr;
  cudaError_t e = round_device(&d);
  if (e != cudaSuccess) return e;
  const int nck = (int)vec_sweep_chunks(dtype, x.V);
  const int B = x.B, R1 = 2 * x.gamma + 1;
  mark(0, stream);
  e = cudaMemsetAsync(ws + pl.off_abort, 0, pl.fused_zero_bytes(B, nck), stream);
  if (e != cudaSuccess) return e;
  mark(1, stream);
  RoundArgs a;
  a.x = x;
  a.abort = reinterpret_cast<uint32_t*>(ws + pl.off_abort);
  a.dword = reinterpret_cast<uint64_t*>(ws + pl.off_dword);
  a.cword = reinterpret_cast<uint64_t*>(ws + pl.off_cword);
  a.pword = reinterpret_cast<uint64_t*>(ws + pl.off_part1);
  a.nck = nck;
  a.S = pl.nrace;
  a.lag = 1;
  const int64_t units = (int64_t)B * R1 * nck;
  int64_t grid = (int64_t)d->sms * d->ctas[dtype];
  const int64_t need = ceil_div(units, (int64_t)kSweepWarps);
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kSweepWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = (dtype == SV_F32) ? cudaLaunchKernelEx(&cfg, k_round<SV_F32>, a)
                        : cudaLaunchKernelEx(&cfg, k_round<SV_BF16>, a);
  if (e != cudaSuccess) return e;
  mark(2, stream);
  return cudaSuccess;
}

}  // namespace sv
