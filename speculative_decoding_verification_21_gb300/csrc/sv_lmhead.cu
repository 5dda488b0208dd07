// sv_lmhead.cu -- fused LM heads + sampling verify on the 5th-generation tensor
// cores (tcgen05, tensor memory, 2-D tensor copies) of sm_103a.
//
// The logits are the final projections of the two models' passes, z = h W with
// bf16 operands and fp32 accumulation ("Fast Inference from Transformers via
// Speculative Decoding", section "The loop: draft, verify in one pass, keep a
// prefix": one target pass over the gamma+1 positions gives p_1..p_{gamma+1},
// the draft gives q_i).  They are consumed tile by tile in the epilogue of the
// GEMM and never written to HBM.  Four kernels per call:
//
//   k_lm<1>      persistent, one CTA per SM.  Vocabulary tiles of 128 entries
//                are dealt round-robin; for each tile the CTA computes the
//                target block (B(gamma+1) token rows x 128) and then the draft
//                block (B gamma rows x 128).  Warps 0 and 2 stream W (from
//                HBM) and h (from L2) with tensor copies into two shared-
//                memory rings, a 128-wide hidden block per stage, warp 1 issues
//                tcgen05.mma into one of two tensor-memory accumulators, and
//                warps 3-10 drain the other (tcgen05.ld): per-row online
//                softmax statistics carried over the CTA's tiles and z at each
//                draft token; one partial per row and CTA.
//   k_lm_finish  one CTA per batch row: row combine and the decision exactly as
//                for given logits, then a compact copy of the hidden rows of
//                the row to draw from: the residual at the first rejection,
//                or p_gamma after a clean sweep.
//   k_lm<2>      the same GEMM for the compact rows only (tiles in reverse
//                order), target and draft blocks side by side in tensor
//                memory.  The compact rows are copied into the row tile twice
//                (B <= 64) so that two lane quadrants share the epilogue: the
//                Gumbel-max race of the draw (Philox tag 1 at the draw
//                position), the best two keys of the residual max(0, p_n - q_n)
//                and of p_n per row and CTA, with the logits at them.
//   k_lm_merge   one warp per compact row: the best two over the CTAs,
//                re-decided in double near a tie from the logits the keys came
//                from; p_n for an empty residual; emit.
//
// Draft sampling (spec_lmhead_draft) is a third use of the GEMM (k_lm<3>) with
// Gumbel-max keys y_v - log2(-log2 u_v), y = z / T * log2 e, on Philox tag 2.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <cstdint>
#include <mutex>

#include "specverify.h"
#include "sv_decide.cuh"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_launch.h"
#include "sv_plan.h"
#include "sv_tma.cuh"
#include "sv_umma.cuh"

namespace sv {

namespace {

constexpr int kTileM = 128;   // token rows per MMA (tensor-memory lanes)
constexpr int kKAtom = 64;    // hidden entries of one 128-byte swizzle span
constexpr int kKBlock = 128;  // hidden entries per stage: two spans
constexpr int kWHalf = (kLmTileN / 2) * kKBlock * 2;  // W box: 64 vocab x 128 hidden, 16 KB
constexpr int kWBytes = 2 * kWHalf;                    // one W tile per stage, 32 KB
constexpr int kEpiWarps = 8;     // two per tensor-memory lane quadrant, each half the columns
constexpr int kLmThreads = 32 * (3 + kEpiWarps);  // W producer, MMA issuer, h producer, epilogue
constexpr int kTmemCols = 512;   // two accumulators of 256 columns
constexpr uint32_t kWaitLimit = 1u << 22;
// The wait limit and the withheld hand-over of the next launches (a failure
// test sets them through sv_test_lmhead_stall; host-side, not thread-safe).
uint32_t g_lm_wait_limit = kWaitLimit;
int g_lm_stall_job = -1;
constexpr int kMaxWStages = 8;  // W-ring slots
constexpr int kHStagesPass2 = 3;  // h-ring slots of the recompute pass (small h tiles)
constexpr int kMaxRep = 2;      // copies of the compact rows in the recompute pass
constexpr size_t kSmemBudget = 227 * 1024;  // dynamic shared memory of one CTA
constexpr size_t kSmemFixed = 1024 + 512;   // 1024-byte alignment slack + barriers

constexpr uint32_t kIdesc = umma_idesc_bf16(kTileM, kLmTileN, /*a_mn=*/false, /*b_mn=*/true);

struct LmArgs {
  const int32_t* xt;
  int B, gamma, V, nvt;
  int nslot;           // CTAs of the GEMM passes: partials per row and column half
  int Mt, Md;          // token rows of the target and draft sides
  int kbt, kbd;        // hidden blocks of 64
  int Ht, Hd;
  int box_t, box_d;    // h rows per tensor copy: rows rounded up to 8 (pass 2: compact rows)
  int perm_t;          // target rows in smem are position-major (row i*B + b), else b*(gamma+1) + i
  int rep, rstride;    // passes 2, 3: copies of the rows in the row tile, rows apart
  int draft_pos;       // pass 3: position of the draft tokens being sampled
  const float* dlse;   // [B][gamma] draft rows' log-normalisers from the draft step, or null
  const float* dlogit; // [B][gamma] draft logits at the drafted tokens (with dlse)
  int nw, nh;          // W-ring and h-ring slots (nw >= nh)
  int a_half;          // bytes of the h tile of one 64-wide span (rows x 128)
  float temperature;
  uint64_t seed, round;
  float2* part;        // [B*R1][nslot][2] (max, sum) per row, CTA and column half
  float* zat;          // [B*R1] logit at the row's draft token
  LmCand* res;         // pass 3: [B][nslot][2] top-2 Gumbel keys per batch row and CTA
  LmCand* res2;        // pass 2: [B][nslot][4] per compact row and CTA: the best two keys
                       // of the residual race, then of p_n
  DrawState* state;    // [B]
  int* slot_b;         // [B] batch row of each compact row
  uint32_t* ctl;       // count, pass-1 error, pass-2 error
  const uint16_t* h_t;
  const uint16_t* h_d;
  uint16_t* c_t;       // compact hidden rows [B][Ht]
  uint16_t* c_d;       // [B][Hd]
  float* dbg;          // [B*R1][V] or null
  int32_t* out_tokens;
  int32_t* out_counts;
  float* out_p;
  float* out_q;
  uint8_t* out_flags;
  uint32_t wait_limit;  // tries of every bounded wait (kWaitLimit unless a test set it)
  int stall_job;        // test only: the job of CTA 0's first pass whose accumulator is
                        // never handed to the epilogue (-1: none)
};

__device__ __forceinline__ bool cand_better(const LmCand& a, const LmCand& b) {
  if (a.idx < 0) return false;
  if (b.idx < 0) return true;
  return a.key > b.key || (a.key == b.key && a.idx < b.idx);
}

struct Cand2 {
  LmCand a, b;
};

__device__ __forceinline__ LmCand cand_empty() { return LmCand{-kInf, -1, 0.0f, 0.0f}; }

__device__ __forceinline__ void cand_insert(Cand2& t, const LmCand& c) {
  if (cand_better(c, t.a)) {
    t.b = t.a;
    t.a = c;
  } else if (cand_better(c, t.b)) {
    t.b = c;
  }
}

__device__ __forceinline__ LmCand cand_shfl(const LmCand& c, int o) {
  LmCand r;
  r.key = __shfl_xor_sync(0xffffffffu, c.key, o);
  r.idx = __shfl_xor_sync(0xffffffffu, c.idx, o);
  r.zt = __shfl_xor_sync(0xffffffffu, c.zt, o);
  r.zd = __shfl_xor_sync(0xffffffffu, c.zd, o);
  return r;
}

__device__ __forceinline__ Cand2 warp_cand2(Cand2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const LmCand a = cand_shfl(t.a, o), b = cand_shfl(t.b, o);
    cand_insert(t, a);
    cand_insert(t, b);
  }
  return t;
}

// Top-2 over the CTA (valid in thread 0).
__device__ Cand2 block_cand2(Cand2 t, Cand2* sm /* [32] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  t = warp_cand2(t);
  __syncthreads();
  if (lane == 0) sm[warp] = t;
  __syncthreads();
  Cand2 r{cand_empty(), cand_empty()};
  if (warp == 0) {
    if (lane < nw) r = sm[lane];
    r = warp_cand2(r);
  }
  return r;
}

// Bounded wait (`limit` tries) that also gives up when another role of the CTA
// has aborted.
__device__ __forceinline__ bool lm_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// The same for a whole warp: lane 0 polls, the others wait at the shuffle.
__device__ __forceinline__ bool lm_wait_warp(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, uint32_t limit) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = lm_wait(bar, parity, abort_flag, limit);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// The double-precision Gumbel noise -ln(-ln u) of entry v at Philox position
// pos (tag 2: draft sampling), for the re-decision of a near tie.
__device__ __forceinline__ double gumbel_f64(int64_t v, int pos, int b, uint64_t seed,
                                             uint64_t round, uint32_t tag) {
  const uint4 rnd = philox4x32_10(sv_counter((uint32_t)(v >> 2), tag, (uint32_t)pos, (uint32_t)b, round),
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
  const uint32_t lanes[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  return -log(sv_neglog_u_f64(lanes[v & 3]));
}

// The best of a top-2, re-decided in double when the two fp32 keys are within
// 2^-10 (log2 units).  `key_f64` gives the definition-level key of a candidate.
template <class F>
__device__ int redecide(const Cand2& t, F key_f64) {
  if (t.a.idx < 0) return -1;
  if (t.b.idx < 0 || !(t.a.key - t.b.key <= 0x1p-10f)) return t.a.idx;
  const double ka = key_f64(t.a), kb = key_f64(t.b);
  if (kb > ka || (kb == ka && t.b.idx < t.a.idx)) return t.b.idx;
  return t.a.idx;
}

// ---------------------------------------------------------------------------
// The persistent GEMM + epilogue kernel.  PASS 1: all token rows; PASS 2: the
// compact rows.  Maps: mA0/mB0 target h and W, mA1/mB1 draft h and W.
// ---------------------------------------------------------------------------
struct Seg {
  const CUtensorMap* amap;
  const CUtensorMap* bmap;
  int kblocks;
  int mtiles;  // 1 or 2 MMA row tiles
  int start1;  // first h row of the second tile (rows start1 .. start1+127)
  int col;     // tensor-memory column of the block within the accumulator
  int box;     // h rows per copy (rounded up to 8)
  int rows;    // rows a copy delivers (its transaction bytes / 128)
  bool perm;   // a 3-D copy: position-major target rows
};

// The second 128-row tile of a side with 128 < M <= 256 rows ends at the last
// row (rounded up to 8) and overlaps the first; the overlap is computed twice
// and kept once, so no row of a copy is padding.
__device__ __forceinline__ Seg side_seg(const CUtensorMap* am, const CUtensorMap* bm, int kb, int M,
                                        int box, int col, bool perm) {
  const bool two = M > kTileM;
  // a 2-D box always delivers `box` rows (zero-filled past M); the 3-D box exactly M
  return Seg{am, bm, kb, two ? 2 : 1, two ? box - kTileM : 0, col, box, perm ? M : box, perm};
}

template <int PASS>
struct Jobs;

// Pass 1: per vocabulary tile, job 0 = target block, job 1 = draft block.
template <>
struct Jobs<1> {
  static constexpr int kPerTile = 2;
  __device__ static int nseg(int) { return 1; }
  __device__ static Seg seg(int job, int, const CUtensorMap* a0, const CUtensorMap* b0,
                            const CUtensorMap* a1, const CUtensorMap* b1, const LmArgs& a) {
    if (job == 0) return side_seg(a0, b0, a.kbt, a.Mt, a.box_t, 0, a.perm_t != 0);
    return side_seg(a1, b1, a.kbd, a.Md, a.box_d, 0, false);
  }
};

// Pass 2: one job per tile, target block at column 0 and draft block at 128.
template <>
struct Jobs<2> {
  static constexpr int kPerTile = 1;
  __device__ static int nseg(int) { return 2; }
  __device__ static Seg seg(int, int s, const CUtensorMap* a0, const CUtensorMap* b0,
                            const CUtensorMap* a1, const CUtensorMap* b1, const LmArgs& a) {
    if (s == 0) return Seg{a0, b0, a.kbt, 1, 0, 0, a.box_t, a.box_t, false};
    return Seg{a1, b1, a.kbd, 1, 0, kLmTileN, a.box_d, a.box_d, false};
  }
};

// Pass 4 (the first pass of a drafted round): the target block only.
template <>
struct Jobs<4> {
  static constexpr int kPerTile = 1;
  __device__ static int nseg(int) { return 1; }
  __device__ static Seg seg(int, int, const CUtensorMap* a0, const CUtensorMap* b0,
                            const CUtensorMap*, const CUtensorMap*, const LmArgs& a) {
    return side_seg(a0, b0, a.kbt, a.Mt, a.box_t, 0, a.perm_t != 0);
  }
};

// Pass 3 (draft sampling): one job per tile, the draft rows' block at column 0.
template <>
struct Jobs<3> {
  static constexpr int kPerTile = 1;
  __device__ static int nseg(int) { return 1; }
  __device__ static Seg seg(int, int, const CUtensorMap* a0, const CUtensorMap* b0,
                            const CUtensorMap*, const CUtensorMap*, const LmArgs& a) {
    return Seg{a0, b0, a.kbd, 1, 0, 0, a.box_d, a.box_d, false};
  }
};

// Vocabulary tile of the CTA's tile counter t.  The recompute pass walks the
// tiles in the reverse order, so that its first tiles are the ones the first
// pass read last (still in L2).
template <int PASS>
__device__ __forceinline__ int vocab_tile(int t, int nvt) {
  return PASS == 2 ? nvt - 1 - t : t;
}

// Slot index and phase of a ring of n slots, advanced stage by stage (no
// division in the issue loops).
struct Slot {
  uint32_t i = 0, ph = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// Wait (bounded, `limit` tries per slot) until every copy issued into a ring
// has landed.
__device__ void drain_ring(uint64_t* full, uint32_t n, uint32_t issued, uint32_t limit) {
  for (uint32_t s = 0; s < n; ++s) {
    if (issued <= s) continue;
    const uint32_t last = (issued - 1u) - ((issued - 1u - s) % n);
    mbar_wait_bounded(full + s, (last / n) & 1u, limit);
  }
}

// Online (max, sum) update of one row with 32 logits (invalid ones -inf).
__device__ __forceinline__ void fold32(const float* f, float c, float& mc, float& s) {
  float m8[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    m8[j] = fmaxf(fmaxf(f[4 * j], f[4 * j + 1]), fmaxf(f[4 * j + 2], f[4 * j + 3]));
  const float cm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
  const float nm = fmaxf(mc, cm * c);
  if (!(nm > -kInf)) return;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = ex2(fmaf(f[j], c, -nm));
#pragma unroll
  for (int e = 8; e < 32; ++e) acc[e & 7] += ex2(fmaf(f[e], c, -nm));
  const float old = (mc == -kInf) ? 0.0f : s * ex2(mc - nm);
  mc = nm;
  s = old + (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7])));
}

__device__ __forceinline__ Cand2 merge2(const Cand2* t) {
  Cand2 r = t[0];
  cand_insert(r, t[1].a);
  cand_insert(r, t[1].b);
  return r;
}

// Row of a side handled by this thread in row tile m (-1: none).  Tile m holds
// rows start .. start+127; rows below 128 of the second tile belong to the first.
__device__ __forceinline__ int side_row(const LmArgs& a, int side, int m, int quad, int lane) {
  const int M = side ? a.Md : a.Mt;
  const int box = side ? a.box_d : a.box_t;
  if (m == 1 && M <= kTileM) return -1;
  const int r = (m ? box - kTileM : 0) + 32 * quad + lane;
  return (r < M && r >= m * kTileM) ? r : -1;
}

// Batch row b, logit row k within it (0..gamma target, gamma+1.. draft) and the
// draft token at the row (-1: none) of token row r of a side.
struct RowId {
  int b, k, x;
};
__device__ __forceinline__ RowId row_id(const LmArgs& a, int side, int r) {
  const int gamma = a.gamma;
  RowId id;
  if (side == 0) {
    int i;
    if (a.perm_t) {
      i = r / a.B;
      id.b = r - i * a.B;
    } else {
      id.b = r / (gamma + 1);
      i = r - id.b * (gamma + 1);
    }
    id.k = i;
    id.x = (i < gamma) ? __ldg(a.xt + (int64_t)id.b * gamma + i) : -1;
  } else {
    id.b = r / gamma;
    id.k = gamma + 1 + (r - id.b * gamma);
    id.x = __ldg(a.xt + r);
  }
  return id;
}

// What a pass-1 epilogue thread carries over the vocabulary tiles of its CTA:
// the online (max, sum) of each of its rows.
struct Pass1Carry {
  float mc[2][2], s[2][2];  // [side][row tile]
};

__device__ __forceinline__ void carry_init(Pass1Carry& cy) {
#pragma unroll
  for (int sd = 0; sd < 2; ++sd)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      cy.mc[sd][m] = -kInf;
      cy.s[sd][m] = 0.0f;
    }
}

// Pass-1 epilogue of one job (SIDE 0 target rows, 1 draft rows) for this warp's
// lane quadrant and column half (two 32-column chunks of the tile).
template <int SIDE>
__device__ __forceinline__ void epilogue_pass1(const LmArgs& a, int t, uint32_t tacc, int quad,
                                               int half, Pass1Carry& cy) {
  const int lane = threadIdx.x & 31;
  const int R1 = 2 * a.gamma + 1, V = a.V;
  const int M = SIDE ? a.Md : a.Mt;
  const int box = SIDE ? a.box_d : a.box_t;
  const int v0 = t * kLmTileN;
  const float c = log2_scale(inv_temperature(a.temperature));
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    if (m == 1 && M <= kTileM) break;
    const int rb = (m ? box - kTileM : 0) + 32 * quad;
    if (rb >= M || rb + 31 < m * kTileM) continue;  // warp-uniform
    uint32_t raw[2][32];
    const uint32_t ta = tacc + ((uint32_t)(32 * quad) << 16) + (uint32_t)(m * kTileM + half * 64);
    tmem_ld32_async(ta, raw[0]);
    tmem_ld32_async(ta + 32, raw[1]);
    tmem_wait_ld();
    const int r = side_row(a, SIDE, m, quad, lane);
    if (r < 0) continue;
    const RowId id = row_id(a, SIDE, r);
    const int64_t grow = (int64_t)id.b * R1 + id.k;
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const int vb = v0 + half * 64 + c2 * 32;
      if (vb >= V) break;
      float f[32];
      const int nvalid = min(32, V - vb);
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = (e < nvalid) ? __uint_as_float(raw[c2][e]) : -kInf;
      if (a.dbg) {
        float4* d = reinterpret_cast<float4*>(a.dbg + grow * V + vb);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (4 * j < nvalid) d[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
      }
      fold32(f, c, cy.mc[SIDE][m], cy.s[SIDE][m]);
      if ((unsigned)(id.x - vb) < 32u) {
        float g = 0.0f;
#pragma unroll
        for (int e = 0; e < 32; ++e) g = (e == id.x - vb) ? f[e] : g;
        a.zat[grow] = g;
      }
    }
  }
}

// One partial per row, CTA and column half: slot (row * nslot + cta) * 2 + half.
// NSIDES 1: the target rows only (the draft rows' statistics come from the
// draft step).
template <int NSIDES>
__device__ __forceinline__ void pass1_flush(const LmArgs& a, const Pass1Carry& cy, int quad,
                                            int half) {
  const int lane = threadIdx.x & 31;
  const int R1 = 2 * a.gamma + 1;
#pragma unroll
  for (int sd = 0; sd < NSIDES; ++sd)
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int r = side_row(a, sd, m, quad, lane);
      if (r < 0) continue;
      const RowId id = row_id(a, sd, r);
      const int64_t grow = (int64_t)id.b * R1 + id.k;
      a.part[(grow * a.nslot + blockIdx.x) * 2 + half] = make_float2(cy.mc[sd][m], cy.s[sd][m]);
    }
}

// Where a pass-2 epilogue warp works.  The compact rows sit in the row tile
// `rep` times (copy c at lanes c*rstride ..), so that up to four lane quadrants
// hold rows; copy c covers the tile's columns [c*128/rep, (c+1)*128/rep), split
// between the quadrant's two warps.  Quadrants past the last copy stay idle.
struct P2Slice {
  int copy, row0, ncol, col0;
};
__device__ __forceinline__ P2Slice pass2_slice(const LmArgs& a, int quad, int half) {
  P2Slice sl;
  sl.copy = (32 * quad) / a.rstride;
  sl.row0 = 32 * quad - sl.copy * a.rstride;
  sl.ncol = 64 / a.rep;
  sl.col0 = sl.copy * (kLmTileN / a.rep) + half * sl.ncol;
  return sl;
}

// What a pass-2 epilogue thread carries over the CTA's tiles: the best two keys
// of its compact row's residual race and of p_n over its column slice (two
// interleaved top-2s each, merged at the end).
struct Pass2Carry {
  Cand2 r[2], p[2];
};

// Pass-2 epilogue of one job (compact rows; target at column 0, draft at 128):
// the Gumbel-max race of this thread's row over its column slice, keys
// log2 w_v - log2 E_v with E_v = -log2 u_v (u_v from Philox tag 1 at the draw
// position of the row's batch row), w = p_n for every entry and w = max(0, p_n -
// q_n) for a residual row, both up to the row's factor 2^-mct / St.  No logit
// leaves the tensor memory: the candidates carry their two logits.
__device__ __forceinline__ void epilogue_pass2(const LmArgs& a, int t, uint32_t tacc, int quad,
                                               int half, int rows, const PhiloxKeys& pk,
                                               Pass2Carry& cy) {
  const int lane = threadIdx.x & 31;
  const int V = a.V;
  const P2Slice sl = pass2_slice(a, quad, half);
  if (sl.copy >= a.rep || sl.row0 >= rows) return;  // warp-uniform
  const int r = sl.row0 + lane;
  const bool rv = r < rows;
  DrawState st{};
  int b = 0;
  if (rv) {
    b = a.slot_b[r];
    st = a.state[b];
  }
  const bool resid = st.mode == kDrawResidual;
  const float kd = __fsub_rn(st.K, st.mct);
  const uint32_t ta = tacc + ((uint32_t)(32 * quad) << 16) + (uint32_t)sl.col0;
#pragma unroll 1
  for (int c16 = 0; c16 < sl.ncol; c16 += 16) {
    uint32_t rt[16], rd[16];
    __syncwarp();
    tmem_ld16_async(ta + (uint32_t)c16, rt);
    tmem_ld16_async(ta + (uint32_t)(kLmTileN + c16), rd);
    tmem_wait_ld();
    const int vb = t * kLmTileN + sl.col0 + c16;  // a multiple of 16
    if (rv && vb < V) {
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const int v = vb + 4 * g4;
        if (v >= V) break;  // columns past V hold no logit
        const uint4 rnd =
            philox_rk(sv_counter((uint32_t)(v >> 2), 1u, (uint32_t)st.pos, (uint32_t)b, a.round), pk);
        const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float zt = __uint_as_float(rt[4 * g4 + e]);
          const float zd = __uint_as_float(rd[4 * g4 + e]);
          if (!(zt > -kInf)) continue;  // weight 0 (or not a number)
          const float lE = __log2f(neglog2_u(rr[e]));
          const float yt = __fmaf_rn(zt, st.c, -st.mct);
          cand_insert(cy.p[e & 1], LmCand{yt - lE, v + e, zt, zd});
          if (resid) {
            const float et = ex2(yt), ed = ex2(__fmaf_rn(zd, st.c, kd));
            if (et > ed) cand_insert(cy.r[e & 1], LmCand{__log2f(__fsub_rn(et, ed)) - lE, v + e, zt, zd});
          }
        }
      }
    }
  }
}

// What a pass-3 (draft sampling) epilogue thread carries over the CTA's tiles:
// its row's online (max, sum) over its column slice and the top-2 Gumbel-max
// keys z c - log2(-log2 u) (Philox tag 2 at the draft position).
struct Pass3Carry {
  float mc, s;
  Cand2 t[2];
};

// Pass-3 epilogue of one tile: rows are batch rows (copied into the row tile
// as in pass 2); the draft logits of the tile's columns in this warp's slice.
__device__ __forceinline__ void epilogue_pass3(const LmArgs& a, int t, uint32_t tacc, int quad,
                                               int half, const PhiloxKeys& pk, Pass3Carry& cy) {
  const int lane = threadIdx.x & 31;
  const int V = a.V, B = a.B;
  const P2Slice sl = pass2_slice(a, quad, half);
  if (sl.copy >= a.rep || sl.row0 >= B) return;  // warp-uniform
  const int r = sl.row0 + lane;  // batch row
  const bool rv = r < B;
  const float c = log2_scale(inv_temperature(a.temperature));
  const uint32_t ta = tacc + ((uint32_t)(32 * quad) << 16) + (uint32_t)sl.col0;
#pragma unroll 1
  for (int c16 = 0; c16 < sl.ncol; c16 += 16) {
    uint32_t raw[16];
    __syncwarp();
    tmem_ld16_async(ta + (uint32_t)c16, raw);
    tmem_wait_ld();
    const int vb = t * kLmTileN + sl.col0 + c16;
    if (rv && vb < V) {
      const int nvalid = min(16, V - vb);
      float f[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) f[e] = (e < nvalid) ? __uint_as_float(raw[e]) : -kInf;
      if (a.dbg) {
        float4* d = reinterpret_cast<float4*>(a.dbg + (int64_t)r * V + vb);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (4 * j < nvalid) d[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
      }
      // online (max, sum of 2^(z c - max))
      float m4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        m4[j] = fmaxf(fmaxf(f[4 * j], f[4 * j + 1]), fmaxf(f[4 * j + 2], f[4 * j + 3]));
      const float nm = fmaxf(cy.mc, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c);
      if (nm > -kInf) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e & 3] += ex2(fmaf(f[e], c, -nm));
        const float old = (cy.mc == -kInf) ? 0.0f : cy.s * ex2(cy.mc - nm);
        cy.mc = nm;
        cy.s = old + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
      }
      // Gumbel-max keys
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const int v = vb + 4 * g4;
        if (v >= V) break;
        const uint4 rnd =
            philox_rk(sv_counter((uint32_t)(v >> 2), 2u, (uint32_t)a.draft_pos, (uint32_t)r,
                                 a.round),
                      pk);
        const uint32_t rr[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float z = f[4 * g4 + e];
          if (z > -kInf)
            cand_insert(cy.t[e & 1], LmCand{fmaf(z, c, -__log2f(neglog2_u(rr[e]))), v + e, z, 0.0f});
        }
      }
    }
  }
}

// One (max, sum) partial and one top-2 per batch row and CTA: the slices of a
// row are merged through shared memory (the ring, idle after the last job).
__device__ __forceinline__ void pass3_flush(const LmArgs& a, int quad, int half,
                                            const Pass3Carry& cy, unsigned char* smem) {
  const int B = a.B;
  const int nsl = 2 * a.rep;
  const P2Slice sl = pass2_slice(a, quad, half);
  const int r = sl.row0 + (threadIdx.x & 31);
  LmCand* sc = reinterpret_cast<LmCand*>(smem);                         // [B][nsl][2]
  float2* sm = reinterpret_cast<float2*>(sc + (size_t)B * nsl * 2);     // [B][nsl]
  if (sl.copy < a.rep && r < B) {
    const Cand2 t2 = merge2(cy.t);
    LmCand* o = sc + ((size_t)r * nsl + sl.copy * 2 + half) * 2;
    o[0] = t2.a;
    o[1] = t2.b;
    sm[(size_t)r * nsl + sl.copy * 2 + half] = make_float2(cy.mc, cy.s);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
  for (int rr = (int)threadIdx.x - 3 * 32; rr < B; rr += 32 * kEpiWarps) {
    Cand2 x{cand_empty(), cand_empty()};
    MS ms{-kInf, 0.0f};
    for (int j = 0; j < nsl; ++j) {
      const LmCand* q = sc + ((size_t)rr * nsl + j) * 2;
      cand_insert(x, q[0]);
      cand_insert(x, q[1]);
      const float2 p = sm[(size_t)rr * nsl + j];
      ms = ms_combine(ms, MS{p.x, p.y});
    }
    a.part[(int64_t)rr * a.nslot + blockIdx.x] = make_float2(ms.m, ms.s);
    LmCand* o = a.res + ((int64_t)rr * a.nslot + blockIdx.x) * 2;
    o[0] = x.a;
    o[1] = x.b;
  }
}

// One set of candidates per compact row and CTA (the residual's best two, then
// p_n's): the row's column slices are merged through shared memory (the ring,
// idle after the last job).
__device__ __forceinline__ void pass2_flush(const LmArgs& a, int quad, int half, int rows,
                                            const Pass2Carry& cy, unsigned char* smem) {
  const int nsl = 2 * a.rep;
  const P2Slice sl = pass2_slice(a, quad, half);
  const int r = sl.row0 + (threadIdx.x & 31);
  LmCand* sc = reinterpret_cast<LmCand*>(smem);  // [rows][nsl][4]
  if (sl.copy < a.rep && r < rows) {
    const Cand2 tr = merge2(cy.r), tp = merge2(cy.p);
    LmCand* o = sc + ((size_t)r * nsl + sl.copy * 2 + half) * 4;
    o[0] = tr.a;
    o[1] = tr.b;
    o[2] = tp.a;
    o[3] = tp.b;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
  for (int rr = (int)threadIdx.x - 3 * 32; rr < rows; rr += 32 * kEpiWarps) {
    Cand2 xr{cand_empty(), cand_empty()}, xp = xr;
    for (int j = 0; j < nsl; ++j) {
      const LmCand* q = sc + ((size_t)rr * nsl + j) * 4;
      cand_insert(xr, q[0]);
      cand_insert(xr, q[1]);
      cand_insert(xp, q[2]);
      cand_insert(xp, q[3]);
    }
    LmCand* o = a.res2 + ((int64_t)rr * a.nslot + blockIdx.x) * 4;
    o[0] = xr.a;
    o[1] = xr.b;
    o[2] = xp.a;
    o[3] = xp.b;
  }
}

template <int PASS>
__global__ void __launch_bounds__(kLmThreads, 1)
    k_lm(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mB0,
         const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mB1,
         LmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  int rows2 = 0;
  if (PASS == 2) {
    pdl_wait();  // the compact rows and their draw states
    rows2 = (int)*reinterpret_cast<volatile uint32_t*>(a.ctl);
    if (rows2 <= 0) return;  // nothing rejected this round (uniform over the grid)
  }
  pdl_launch_dependents();
  // Shared memory: the h ring (nh slots of [span 0 | span 1]), the W ring (nw
  // slots of [vocab half 0 | vocab half 1]), then barriers.  Stage k of the
  // K loop uses h slot k % nh and W slot k % nw, and the W slot's barriers serve
  // the stage: `full` completes when the copies of both producers have landed,
  // `empty` when the MMAs that read the stage are done (the h producer reuses
  // slot k % nh once stage k - nh is empty).  An MMA reads a 128-row window from
  // the start of its h span; rows past the copied box only feed accumulator rows
  // that are never read.
  const uint32_t nw = (uint32_t)a.nw, nh = (uint32_t)a.nh;
  const size_t hslot = (size_t)2 * a.a_half;
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* hring = smem_raw + (((base_u32 + 1023u) & ~1023u) - base_u32);
  uint8_t* wring = hring + (size_t)nh * hslot;
  uint64_t* full = reinterpret_cast<uint64_t*>(wring + (size_t)nw * kWBytes);
  uint64_t* empty = full + kMaxWStages;
  uint64_t* accf = empty + kMaxWStages;  // [2]
  uint64_t* acce = accf + 2;             // [2]
  uint64_t* fin = acce + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < nw; ++s) {
      mbar_init(full + s, 2);  // both producers
      mbar_init(empty + s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(accf + j, 1);
      mbar_init(acce + j, kEpiWarps);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int nvt = a.nvt;
  const int G = (int)gridDim.x;

  if (warp == 0 || warp == 2) {
    // ---------------- producers: W tiles (warp 0), h tiles (warp 2) ----------------
    if (lane == 0) {
      const bool isw = (warp == 0);
      const uint64_t pol = isw ? l2_policy_evict_first() : l2_policy_evict_last();
      uint32_t k = 0;  // stage counter
      Slot w, hs, lag;  // W slot of stage k, h slot of stage k, W slot of stage k - nh
      bool ok = true;
      for (int t = blockIdx.x; ok && t < nvt; t += G) {
        const int v0 = vocab_tile<PASS>(t, nvt) * kLmTileN;
        for (int job = 0; ok && job < Jobs<PASS>::kPerTile; ++job) {
          for (int sg = 0; ok && sg < Jobs<PASS>::nseg(job); ++sg) {
            const Seg q = Jobs<PASS>::seg(job, sg, &mA0, &mB0, &mA1, &mB1, a);
            for (int kb = 0; kb < q.kblocks; ++kb, ++k) {
              const uint32_t ws = w.i;
              const int k0 = kb * kKBlock;  // spans past the hidden size read as zeros
              if (isw) {
                if (!lm_wait(empty + ws, w.ph ^ 1u, abort_flag, a.wait_limit)) {
                  ok = false;
                  break;
                }
                uint8_t* wst = wring + (size_t)ws * kWBytes;
                mbar_arrive_expect_tx(full + ws, (uint32_t)kWBytes);
                tma_load_2d_hint(wst, q.bmap, v0, k0, full + ws, pol);
                tma_load_2d_hint(wst + kWHalf, q.bmap, v0 + kLmTileN / 2, k0, full + ws, pol);
              } else {
                if (k >= nh) {
                  // stage k - nh, the last to use this h slot, is done
                  if (!lm_wait(empty + lag.i, lag.ph, abort_flag, a.wait_limit)) {
                    ok = false;
                    break;
                  }
                  lag.next(nw);
                }
                uint8_t* hst = hring + (size_t)hs.i * hslot;
                // passes 2 and 3: `rep` copies of the rows, `rstride` rows apart
                const int rep = (PASS == 2 || PASS == 3) ? a.rep : 1;
                mbar_arrive_expect_tx(full + ws, (uint32_t)(rep * 2 * q.rows * kKAtom * 2));
                for (int h = 0; h < 2; ++h) {
                  for (int cp = 0; cp < rep; ++cp) {
                    uint8_t* dst = hst + (size_t)h * a.a_half + (size_t)cp * a.rstride * (kKAtom * 2);
                    if (q.perm)
                      tma_load_3d_hint(dst, q.amap, k0 + h * kKAtom, 0, 0, full + ws, pol);
                    else
                      tma_load_2d_hint(dst, q.amap, k0 + h * kKAtom, 0, full + ws, pol);
                  }
                }
              }
              w.next(nw);
              hs.next(nh);
            }
          }
        }
      }
      drain_ring(full, nw, k, a.wait_limit);  // every issued copy has landed before the CTA may exit
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      Slot w, hs;
      int jobi = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < nvt; t += G) {
        for (int job = 0; ok && job < Jobs<PASS>::kPerTile; ++job, ++jobi) {
          const int buf = jobi & 1;
          const uint32_t ap = (uint32_t)(jobi >> 1) & 1u;
          if (!lm_wait(acce + buf, ap ^ 1u, abort_flag, a.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int sg = 0; ok && sg < Jobs<PASS>::nseg(job); ++sg) {
            const Seg q = Jobs<PASS>::seg(job, sg, &mA0, &mB0, &mA1, &mB1, a);
            const uint32_t dcol = tbase + (uint32_t)(buf * 256 + q.col);
            for (int kb = 0; kb < q.kblocks; ++kb) {
              const uint32_t ws = w.i;
              // one wait per stage: the copies of both producers have landed
              if (!lm_wait(full + ws, w.ph, abort_flag, a.wait_limit)) {
                ok = false;
                break;
              }
              const uint32_t sa = smem_u32(hring + (size_t)hs.i * hslot);
              const uint64_t bdesc =
                  umma_smem_desc(smem_u32(wring + (size_t)ws * kWBytes), kWHalf, 1024);
              for (int m = 0; m < q.mtiles; ++m) {
                const uint32_t row0 = m ? (uint32_t)q.start1 : 0u;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint64_t adesc =
                      umma_smem_desc(sa + (uint32_t)(h * a.a_half) + row0 * (kKAtom * 2), 16, 1024);
#pragma unroll
                  for (int kk = 0; kk < kKAtom / 16; ++kk)
                    umma_bf16(dcol + (uint32_t)(m * kTileM), adesc + (uint64_t)(2 * kk),
                              bdesc + (uint64_t)(128 * (h * (kKAtom / 16) + kk)), kIdesc,
                              (kb | h | kk) != 0);
                }
              }
              umma_commit(empty + ws);
              w.next(nw);
              hs.next(nh);
            }
          }
          // (a test may withhold one hand-over: the epilogue's wait then runs out)
          if (ok && !(PASS == 1 && blockIdx.x == 0 && jobi == a.stall_job)) umma_commit(accf + buf);
        }
      }
      // all MMAs of this CTA complete before tensor memory is released
      umma_commit(fin);
      mbar_wait_bounded(fin, 0);
    }
    __syncwarp();
  } else {
    // ---------- epilogue (warps 3..10: lane quadrant warp%4, column half (warp-3)/4) ----------
    const int quad = warp & 3, half = (warp - 3) >> 2;
    const PhiloxKeys pk = philox_keys(a.seed);
    Pass1Carry cy;
    Pass2Carry cy2;
    Pass3Carry cy3;
    if (PASS == 1 || PASS == 4) {
      carry_init(cy);
    } else if (PASS == 2) {
      cy2.r[0] = cy2.r[1] = cy2.p[0] = cy2.p[1] = Cand2{cand_empty(), cand_empty()};
    } else if (PASS == 3) {
      cy3.mc = -kInf;
      cy3.s = 0.0f;
      cy3.t[0] = cy3.t[1] = Cand2{cand_empty(), cand_empty()};
    }
    int jobi = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < nvt; t += G) {
#pragma unroll
      for (int job = 0; job < Jobs<PASS>::kPerTile; ++job) {
        const int buf = (jobi + job) & 1;
        const uint32_t ap = (uint32_t)((jobi + job) >> 1) & 1u;
        if (!lm_wait_warp(accf + buf, ap, abort_flag, a.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tacc = tbase + (uint32_t)(buf * 256);
        const int tv = vocab_tile<PASS>(t, nvt);
        if (PASS == 1 || PASS == 4) {
          if (job == 0)
            epilogue_pass1<0>(a, tv, tacc, quad, half, cy);
          else
            epilogue_pass1<1>(a, tv, tacc, quad, half, cy);
        } else if (PASS == 2) {
          epilogue_pass2(a, tv, tacc, quad, half, rows2, pk, cy2);
        } else {
          epilogue_pass3(a, tv, tacc, quad, half, pk, cy3);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce + buf);
      }
      jobi += Jobs<PASS>::kPerTile;
    }
    // partials of this CTA (also after an abort: the error flag marks them)
    if (PASS == 1)
      pass1_flush<2>(a, cy, quad, half);
    else if (PASS == 4)
      pass1_flush<1>(a, cy, quad, half);
    else if (PASS == 2)
      pass2_flush(a, quad, half, rows2, cy2, hring);
    else if (PASS == 3)
      pass3_flush(a, quad, half, cy3, hring);
  }

  tc_fence_before();
  __syncthreads();  // every role is done: an abort by any of them is in the flag
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(a.ctl + ((PASS == 1 || PASS == 4) ? 1 : 2), 1u);
  if (warp == 1) tmem_dealloc(tbase, kTmemCols);
}

// ---------------------------------------------------------------------------
// k_lm_finish: one CTA per batch row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_lm_finish(LmArgs a) {
  const int b = blockIdx.x;
  const int gamma = a.gamma, R1 = 2 * gamma + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (int)(blockDim.x >> 5);
  __shared__ RowStat srs[2 * 32 + 1];
  __shared__ DraftAt sda[32];
  __shared__ int s_slot;
  pdl_wait();  // partials of the GEMM pass
  pdl_launch_dependents();
  const bool err = *reinterpret_cast<volatile uint32_t*>(a.ctl + 1) != 0u;
  if (warp < nw - 1) {
    for (int k = warp; k < R1; k += nw - 1) {
      RowStat rs;
      if (a.dlse && k > gamma) {
        // a drafted round: the draft row's statistics are its log-normaliser,
        // as max = lse log2 e with sum 1
        const float lse = __ldg(a.dlse + (int64_t)b * gamma + (k - gamma - 1));
        rs.mc = lse * kLog2e;
        rs.bits = (lse != lse) ? kRowNaN : 0;
        rs.s = (lse != lse) ? CUDART_NAN_F : ((lse == -kInf) ? 0.0f : 1.0f);
      } else {
        rs = combine_row(a.part + ((int64_t)b * R1 + k) * a.nslot * 2, a.nslot * 2, nullptr, 1.0f);
      }
      if (err) {
        rs.bits |= kRowTimeout | kRowNaN;
        rs.s = CUDART_NAN_F;
      }
      if (lane == 0) srs[k] = rs;
    }
  } else {
    for (int i = lane; i < gamma; i += 32) {
      const int32_t x = __ldg(a.xt + (int64_t)b * gamma + i);
      const bool ok = x >= 0 && x < a.V;
      const float* za = a.zat + (int64_t)b * R1;
      const float zd = a.dlogit ? __ldg(a.dlogit + (int64_t)b * gamma + i) : __ldcg(za + gamma + 1 + i);
      sda[i] = DraftAt{x, ok ? __ldcg(za + i) : 0.0f, ok ? zd : 0.0f};
    }
  }
  __syncthreads();
  if (warp == 0) {
    SweepCtx sx{};
    sx.xt = a.xt;
    sx.B = a.B;
    sx.gamma = gamma;
    sx.V = a.V;
    sx.temperature = a.temperature;
    sx.row_T = nullptr;
    sx.seed = a.seed;
    sx.round = a.round;
    sx.state = a.state;
    sx.out_tokens = a.out_tokens;
    sx.out_counts = a.out_counts;
    sx.out_p = a.out_p;
    sx.out_q = a.out_q;
    sx.out_flags = a.out_flags;
    sx.inv_lenience = 1.0f;
    sx.thr = nullptr;
    decide_batch_row<SV_F32>(sx, b, srs, sda);
  }
  __syncthreads();
  const DrawState st = a.state[b];
  if (st.mode == kDrawDone) return;
  // a draw over a full row at position n (the residual at the first rejection,
  // or p_gamma after a clean sweep): queue its hidden rows for pass 2
  if (threadIdx.x == 0) {
    const int slot = (int)atomicAdd(a.ctl, 1u);
    a.slot_b[slot] = b;
    s_slot = slot;
  }
  __syncthreads();
  const int slot = s_slot;
  const int n = st.pos;
  const uint4* srct = reinterpret_cast<const uint4*>(a.h_t + ((int64_t)b * (gamma + 1) + n) * a.Ht);
  uint4* dt = reinterpret_cast<uint4*>(a.c_t + (int64_t)slot * a.Ht);
  uint4* dd = reinterpret_cast<uint4*>(a.c_d + (int64_t)slot * a.Hd);
  for (int j = threadIdx.x; j < a.Ht / 8; j += blockDim.x) dt[j] = __ldg(srct + j);
  if (n < gamma) {
    const uint4* srcd = reinterpret_cast<const uint4*>(a.h_d + ((int64_t)b * gamma + n) * a.Hd);
    for (int j = threadIdx.x; j < a.Hd / 8; j += blockDim.x) dd[j] = __ldg(srcd + j);
  } else {
    // p_gamma has no draft row: zeros (its draft logits are never read)
    for (int j = threadIdx.x; j < a.Hd / 8; j += blockDim.x) dd[j] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------------------
// k_lm_merge: one warp per compact row.  The best two keys of the residual
// race over the recompute pass's CTAs (p_n's when the residual had no positive
// entry: the fallback), re-decided in double when within 2^-10 (log2 units):
// log(p_n - q_n) + g with p_n = 2^(z c - mct) / St, q_n likewise, or z / T + g
// for a draw from p_n, on the logits the candidates carry.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) k_lm_merge(LmArgs a) {
  const int slot = blockIdx.x;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const int rows = (int)*reinterpret_cast<volatile uint32_t*>(a.ctl);
  if (slot >= rows) return;
  const bool err = *reinterpret_cast<volatile uint32_t*>(a.ctl + 2) != 0u;
  const int b = a.slot_b[slot];
  const DrawState st = a.state[b];
  Cand2 R{cand_empty(), cand_empty()}, P = R;
  for (int j = lane; j < a.nslot; j += 32) {
    const LmCand* q = a.res2 + ((int64_t)slot * a.nslot + j) * 4;
    cand_insert(R, q[0]);
    cand_insert(R, q[1]);
    cand_insert(P, q[2]);
    cand_insert(P, q[3]);
  }
  R = warp_cand2(R);
  P = warp_cand2(P);
  int fl = st.flags;
  bool use_r = false;
  Cand2 T = P;
  if (st.mode == kDrawResidual) {
    if (R.a.idx >= 0) {
      T = R;
      use_r = true;
    } else {
      fl |= SV_FLAG_RESIDUAL_FALLBACK;  // no positive residual entry: p_n, the same noise
    }
  }
  const double c = (double)st.c, invT = (double)st.invT;
  int tk = redecide(T, [&](const LmCand& q) -> double {
    const double g = gumbel_f64(q.idx, st.pos, b, a.seed, a.round, 1u);
    if (!use_r) return (double)q.zt * invT + g;
    const double p = exp2((double)q.zt * c - (double)st.mct) / (double)st.st;
    const double pq = (q.zd > -kInf) ? exp2((double)q.zd * c - (double)st.mcd) / (double)st.sd : 0.0;
    const double w = p - pq;
    return (w > 0.0) ? log(w) + g : -HUGE_VAL;
  });
  if (lane != 0) return;
  if (err) fl |= SV_FLAG_TIMEOUT | SV_FLAG_NONFINITE;
  if (tk < 0 || tk >= a.V) {
    tk = 0;
    if (!err) fl |= SV_FLAG_ZERO_MASS;
  }
  a.out_tokens[(int64_t)b * (a.gamma + 1) + st.pos] = tk;
  if (a.out_flags) a.out_flags[b] = (uint8_t)fl;
}

// ---------------------------------------------------------------------------
// k_lm_draft_merge: one CTA per batch row of a draft-sampling call: the row's
// (max, sum) from the per-CTA partials, the token from the per-CTA top-2 keys
// (re-decided in double near a tie), q(x) and the log-normaliser.
// ---------------------------------------------------------------------------
struct DraftOut {
  int32_t* tokens;
  float* q;
  float* lse;
  float* logit;
};

__global__ void __launch_bounds__(256) k_lm_draft_merge(LmArgs a, DraftOut out) {
  const int b = blockIdx.x;
  __shared__ Cand2 scand[32];
  __shared__ RowStat s_rs;
  pdl_wait();
  const bool err = *reinterpret_cast<volatile uint32_t*>(a.ctl + 2) != 0u;
  if (threadIdx.x < 32) {
    const RowStat rs = combine_row(a.part + (int64_t)b * a.nslot, a.nslot, nullptr, 1.0f);
    if (threadIdx.x == 0) s_rs = rs;
  }
  Cand2 t{cand_empty(), cand_empty()};
  const LmCand* rp = a.res + (int64_t)b * a.nslot * 2;
  for (int j = threadIdx.x; j < a.nslot; j += blockDim.x) {
    cand_insert(t, rp[2 * j]);
    cand_insert(t, rp[2 * j + 1]);
  }
  t = block_cand2(t, scand);
  if (threadIdx.x != 0) return;
  const RowStat rs = s_rs;
  const float invT_f = inv_temperature(a.temperature);
  const double invT = (double)invT_f;
  int tk = redecide(t, [&](const LmCand& q) {
    return (double)q.zt * invT + gumbel_f64(q.idx, a.draft_pos, b, a.seed, a.round, 2u);
  });
  float zt = 0.0f;
  if (tk >= 0) {
    zt = (tk == t.a.idx) ? t.a.zt : t.b.zt;
  }
  const bool ok = !err && tk >= 0 && rs.s > 0.0 && !(rs.bits & kRowNaN);
  if (tk < 0 || err) tk = 0;
  out.tokens[b] = tk;
  const double c = (double)log2_scale(invT_f);
  if (out.q) out.q[b] = ok ? (float)(exp2((double)zt * c - (double)rs.mc) / rs.s) : 0.0f;
  if (out.lse)
    out.lse[b] = (rs.s > 0.0) ? (float)(((double)rs.mc + log2(rs.s)) * 0.6931471805599453)
                              : -CUDART_INF_F;
  if (out.logit) out.logit[b] = ok ? zt : -CUDART_INF_F;
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct LmDevice {
  int sms = 0;
  bool ready = false;
};
std::mutex g_lm_mu;
LmDevice g_lm_dev[64];
EncodeTiled g_encode = nullptr;

cudaError_t lm_device(LmDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_lm_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<EncodeTiled>(fn);
  }
  LmDevice& d = g_lm_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_lm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_lm<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_lm<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_lm<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    d.ready = true;
  }
  *out = &d;
  return cudaSuccess;
}

// Row-major bf16 matrix [rows][cols] as a 2-D tensor map with a box of
// box_cols x box_rows and 128-byte swizzle (out-of-range elements read as 0).
bool encode_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// h [B][P][H] bf16 read as a 3-D box (64 hidden, B, P) with the position
// dimension outermost: smem row i*B + b holds h[b][i].
bool encode_bf16_pos_major(CUtensorMap* map, const void* base, int B, int P, int H) {
  const cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)B, (cuuint64_t)P};
  const cuuint64_t strides[2] = {(cuuint64_t)P * H * 2, (cuuint64_t)H * 2};
  const cuuint32_t box[3] = {kKAtom, (cuuint32_t)B, (cuuint32_t)P};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned_to(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

int round8(int x) { return (x + 7) & ~7; }

// The rings of one pass: h slots of two spans of `span_rows` rows, and 32 KB W
// slots.  nh = 0 gives both rings the same depth (as many stages as fit: the
// h tiles of the first pass are as large as the W tiles and come from L2 at
// about the same latency); otherwise nh h slots and as many W slots as the
// rest of the shared memory holds.  Spans are whole 1 KB swizzle atoms (rows
// are a multiple of 8).
bool ring_config(LmArgs& a, int span_rows, int nh, size_t* smem) {
  a.a_half = span_rows * kKAtom * 2;
  const size_t hslot = (size_t)2 * a.a_half;
  const size_t room = kSmemBudget - kSmemFixed;
  int nw;
  if (nh == 0) {
    nh = nw = (int)(room / (hslot + kWBytes));
  } else {
    if ((size_t)nh * hslot > room) return false;
    nw = (int)((room - (size_t)nh * hslot) / kWBytes);
  }
  nw = nw > kMaxWStages ? kMaxWStages : nw;
  nh = nh > nw ? nw : nh;
  if (nh < 2) return false;
  a.nh = nh;
  a.nw = nw;
  *smem = kSmemFixed + (size_t)nh * hslot + (size_t)nw * kWBytes;
  return true;
}

}  // namespace

size_t lmhead_workspace_bytes(int B, int gamma, int64_t V) {
  return make_lm_plan(B, gamma, V).total;
}

int lmhead_verify(const void* h_target, const void* W_target, int Ht, const void* h_draft,
                  const void* W_draft, int Hd, const int32_t* draft_tokens, int B, int gamma,
                  int64_t V, float temperature, uint64_t seed, uint64_t round,
                  int32_t* out_tokens, int32_t* out_counts, float* out_p, float* out_q,
                  uint8_t* out_flags, float* debug_logits, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream, const float* draft_lse,
                  const float* draft_logit) {
  const bool drafted = draft_lse != nullptr;  // the draft rows' statistics are given
  if (drafted && (!draft_logit || !aligned_to(draft_lse, 4) || !aligned_to(draft_logit, 4)))
    return draft_logit ? SV_ERR_ALIGN : SV_ERR_ARG;
  if (!h_target || !W_target || !h_draft || !W_draft || !draft_tokens || !out_tokens ||
      !out_counts)
    return SV_ERR_ARG;
  if (Ht < 64 || Hd < 64 || Ht % 64 || Hd % 64 || Ht > kLmMaxHidden || Hd > kLmMaxHidden ||
      (int64_t)B * (gamma + 1) > kLmMaxRows || V % 8 != 0 || V > ((int64_t)1 << 31) - 256)
    return SV_ERR_UNSUPPORTED;
  if (!aligned_to(h_target, 16) || !aligned_to(W_target, 16) || !aligned_to(h_draft, 16) ||
      !aligned_to(W_draft, 16) || !aligned_to(draft_tokens, 4) || !aligned_to(out_tokens, 4) ||
      !aligned_to(out_counts, 4) || (out_p && !aligned_to(out_p, 4)) ||
      (out_q && !aligned_to(out_q, 4)) || (debug_logits && !aligned_to(debug_logits, 16)))
    return SV_ERR_ALIGN;
  const LmPlan pl = make_lm_plan(B, gamma, V);
  if (!workspace || workspace_bytes < pl.total) return SV_ERR_WORKSPACE;
  if (!aligned_to(workspace, kAlign)) return SV_ERR_ALIGN;
  LmDevice* dev = nullptr;
  if (lm_device(&dev) != cudaSuccess) return SV_ERR_CUDA;

  char* ws = reinterpret_cast<char*>(workspace);
  LmArgs a{};
  a.wait_limit = g_lm_wait_limit;
  a.stall_job = g_lm_stall_job;
  a.xt = draft_tokens;
  a.B = B;
  a.gamma = gamma;
  a.V = (int)V;
  a.nvt = pl.nvt;
  a.Mt = B * (gamma + 1);
  a.Md = B * gamma;
  a.kbt = (Ht + kKBlock - 1) / kKBlock;
  a.kbd = (Hd + kKBlock - 1) / kKBlock;
  a.Ht = Ht;
  a.Hd = Hd;
  a.temperature = temperature;
  a.seed = seed;
  a.round = round;
  a.part = reinterpret_cast<float2*>(ws + pl.off_part);
  a.zat = reinterpret_cast<float*>(ws + pl.off_zat);
  a.res2 = reinterpret_cast<LmCand*>(ws + pl.off_res2);
  a.state = reinterpret_cast<DrawState*>(ws + pl.off_state);
  a.slot_b = reinterpret_cast<int*>(ws + pl.off_slot);
  a.ctl = reinterpret_cast<uint32_t*>(ws + pl.off_ctl);
  a.h_t = reinterpret_cast<const uint16_t*>(h_target);
  a.h_d = reinterpret_cast<const uint16_t*>(h_draft);
  a.c_t = reinterpret_cast<uint16_t*>(ws + pl.off_ct);
  a.c_d = reinterpret_cast<uint16_t*>(ws + pl.off_cd);
  a.dbg = debug_logits;
  a.out_tokens = out_tokens;
  a.out_counts = out_counts;
  a.out_p = out_p;
  a.out_q = out_q;
  a.out_flags = out_flags;
  a.dlse = draft_lse;
  a.dlogit = draft_logit;

  // pass 1: all token rows (a drafted round: the target rows only); pass 2: the
  // compact rows (at most B per side)
  LmArgs a2 = a;
  a.box_t = round8(a.Mt);
  a.box_d = round8(a.Md);
  size_t smem1 = 0, smem2 = 0;
  a2.box_t = a2.box_d = round8(B);
  // copies of the compact rows: one per 32-row-aligned block that fits in 128 lanes
  a2.rstride = (B + 31) & ~31;
  a2.rep = kTileM / a2.rstride;
  a2.rep = a2.rep > kMaxRep ? kMaxRep : a2.rep;
  if (!ring_config(a, (drafted || a.box_t > a.box_d) ? a.box_t : a.box_d, 0, &smem1) ||
      !ring_config(a2, a2.rep > 1 ? a2.rep * a2.rstride : a2.box_t, kHStagesPass2, &smem2))
    return SV_ERR_UNSUPPORTED;

  CUtensorMap hT, WT, hD, WD, cT, cD;
  // target rows position-major (all batch rows of position 0, then 1, ...);
  // the plain order if the map is refused
  a.perm_t = encode_bf16_pos_major(&hT, h_target, B, gamma + 1, Ht) ? 1 : 0;
  if (!a.perm_t &&
      !encode_bf16(&hT, h_target, (uint64_t)a.Mt, (uint64_t)Ht, kKAtom, (uint32_t)a.box_t))
    return SV_ERR_CUDA;
  if (!encode_bf16(&hD, h_draft, (uint64_t)a.Md, (uint64_t)Hd, kKAtom, (uint32_t)a.box_d) ||
      !encode_bf16(&WT, W_target, (uint64_t)Ht, (uint64_t)V, kLmTileN / 2, kKBlock) ||
      !encode_bf16(&WD, W_draft, (uint64_t)Hd, (uint64_t)V, kLmTileN / 2, kKBlock) ||
      !encode_bf16(&cT, a.c_t, (uint64_t)B, (uint64_t)Ht, kKAtom, (uint32_t)a2.box_t) ||
      !encode_bf16(&cD, a.c_d, (uint64_t)B, (uint64_t)Hd, kKAtom, (uint32_t)a2.box_d))
    return SV_ERR_CUDA;

  cudaError_t e = cudaMemsetAsync(a.ctl, 0, 4 * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  const unsigned grid = (unsigned)(pl.nvt < dev->sms ? pl.nvt : dev->sms);
  a.nslot = a2.nslot = (int)grid;
  mark(0, stream);
  if (drafted)
    k_lm<4><<<grid, kLmThreads, smem1, stream>>>(hT, WT, hT, WT, a);
  else
    k_lm<1><<<grid, kLmThreads, smem1, stream>>>(hT, WT, hD, WD, a);
  mark(1, stream);
  const int fw = ((2 * gamma + 1) < 31 ? (2 * gamma + 1) : 31) + 1;
  e = launch_pdl(k_lm_finish, dim3((unsigned)B), dim3(32 * fw), 0, stream, a);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  mark(2, stream);
  e = launch_pdl(k_lm<2>, dim3(grid), dim3(kLmThreads), smem2, stream, cT, WT, cD, WD, a2);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  mark(3, stream);
  e = launch_pdl(k_lm_merge, dim3((unsigned)B), dim3(32), 0, stream, a);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  mark(4, stream);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

size_t lmhead_draft_workspace_bytes(int B, int64_t V) { return make_draft_plan(B, V).total; }

// Draft sampling of one position: z = h_draft W_draft (tensor cores), x ~
// softmax(z / T) by Gumbel-max on Philox tag 2, q(x) and the log-normaliser.
int lmhead_draft(const void* h_draft, const void* W_draft, int Hd, int B, int64_t V,
                 float temperature, uint64_t seed, uint64_t round, int pos, int32_t* out_tokens,
                 float* out_q, float* out_lse, float* out_logit, float* debug_logits,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!h_draft || !W_draft || !out_tokens || pos < 0 || pos > 0xFFFFFF) return SV_ERR_ARG;
  if (Hd < 64 || Hd % 64 || Hd > kLmMaxHidden || B > kTileM || V % 8 != 0 ||
      V > ((int64_t)1 << 31) - 256)
    return SV_ERR_UNSUPPORTED;
  if (!aligned_to(h_draft, 16) || !aligned_to(W_draft, 16) || !aligned_to(out_tokens, 4) ||
      (out_q && !aligned_to(out_q, 4)) || (out_lse && !aligned_to(out_lse, 4)) ||
      (out_logit && !aligned_to(out_logit, 4)) || (debug_logits && !aligned_to(debug_logits, 16)))
    return SV_ERR_ALIGN;
  const DraftPlan pl = make_draft_plan(B, V);
  if (!workspace || workspace_bytes < pl.total) return SV_ERR_WORKSPACE;
  if (!aligned_to(workspace, kAlign)) return SV_ERR_ALIGN;
  LmDevice* dev = nullptr;
  if (lm_device(&dev) != cudaSuccess) return SV_ERR_CUDA;

  char* ws = reinterpret_cast<char*>(workspace);
  LmArgs a{};
  a.wait_limit = g_lm_wait_limit;
  a.stall_job = g_lm_stall_job;
  a.B = B;
  a.gamma = 1;
  a.V = (int)V;
  a.nvt = pl.nvt;
  a.Md = B;
  a.kbd = (Hd + kKBlock - 1) / kKBlock;
  a.Hd = Hd;
  a.temperature = temperature;
  a.seed = seed;
  a.round = round;
  a.draft_pos = pos;
  a.ctl = reinterpret_cast<uint32_t*>(ws + pl.off_ctl);
  a.part = reinterpret_cast<float2*>(ws + pl.off_part);
  a.res = reinterpret_cast<LmCand*>(ws + pl.off_cand);
  a.dbg = debug_logits;
  a.box_d = round8(B);
  // copies of the rows: one per 32-row-aligned block that fits in 128 lanes
  a.rstride = (B + 31) & ~31;
  a.rep = kTileM / a.rstride;
  a.rep = a.rep > kMaxRep ? kMaxRep : a.rep;
  size_t smem = 0;
  if (!ring_config(a, a.rep > 1 ? a.rep * a.rstride : a.box_d, kHStagesPass2, &smem))
    return SV_ERR_UNSUPPORTED;
  CUtensorMap hD, WD;
  if (!encode_bf16(&hD, h_draft, (uint64_t)B, (uint64_t)Hd, kKAtom, (uint32_t)a.box_d) ||
      !encode_bf16(&WD, W_draft, (uint64_t)Hd, (uint64_t)V, kLmTileN / 2, kKBlock))
    return SV_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(a.ctl, 0, 4 * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  const unsigned grid = (unsigned)(pl.nvt < dev->sms ? pl.nvt : dev->sms);
  a.nslot = (int)grid;
  mark(0, stream);
  k_lm<3><<<grid, kLmThreads, smem, stream>>>(hD, WD, hD, WD, a);
  mark(1, stream);
  e = launch_pdl(k_lm_draft_merge, dim3((unsigned)B), dim3(256), 0, stream, a,
                 DraftOut{out_tokens, out_q, out_lse, out_logit});
  if (e != cudaSuccess) return SV_ERR_CUDA;
  mark(2, stream);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv

// Test only: the next fused LM-head launches withhold the first pass's hand-over
// of accumulator `job` in CTA 0 (job < 0: none), so that the epilogue's wait runs
// out, and every bounded wait gives up after `wait_limit` tries (0: the default).
extern "C" int sv_test_lmhead_stall(int job, uint32_t wait_limit) {
  sv::g_lm_stall_job = job < 0 ? -1 : job;
  sv::g_lm_wait_limit = wait_limit ? wait_limit : sv::kWaitLimit;
  return 0;
}

