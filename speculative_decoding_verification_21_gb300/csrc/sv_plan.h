// sv_plan.h -- launch geometry and workspace layout shared by the entry points.
#pragma once

#include <cstddef>
#include <cstdint>

#if defined(__CUDACC__)
#define SV_HD __host__ __device__
#else
#define SV_HD
#endif

namespace sv {

constexpr int kThreads = 256;          // threads per CTA for the streaming kernels
constexpr int64_t kChunkSweep = 8192;  // logits per CTA in the softmax/argmax sweeps
constexpr int64_t kChunkDraw = 8192;   // least vocabulary entries per CTA in the draw pass
constexpr int kDrawCtasPerSm = 4;      // resident draw CTAs per SM (its launch bounds)
constexpr int kRaceCtasPerSm = 2;      // resident race CTAs per SM (its launch bounds)
constexpr size_t kAlign = 256;

// Persistent vector sweep: warps per CTA, resident CTAs per SM (its launch bounds),
// bytes per chunk, chunks in flight per warp (each in a 4 KB shared-memory buffer).
constexpr int kSweepWarps = 8;
constexpr int kSweepCtasPerSm = 2;
constexpr int kSweepChunkBytes = 4096;
constexpr int kSweepBufs = 2;
constexpr size_t kSweepSmemBytes = (size_t)kSweepWarps * kSweepBufs * kSweepChunkBytes;

// The vector sweep cuts every row into chunks of 4 KB counted from the row's
// start (the last one may be shorter) and loads 16-byte vectors, so every row
// must start on a 16-byte boundary: rows whose byte length is a multiple of 16
// (the bases are 16-byte aligned).  Results do not depend on where the arrays
// sit in memory, only on the values and the shapes.
SV_HD inline bool use_vec_sweep(int dtype, int64_t V) {
  const int64_t rb = V * (dtype == 0 ? 4 : 2);
  return rb % 16 == 0;
}

SV_HD inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
SV_HD inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Partials per logit row: one per 4 KB chunk of the row (vector sweep) or per
// kChunkSweep-logit split (generic sweep).  A workspace is sized for the most
// of either over both element types: one per 1024 logits.
SV_HD inline int64_t vec_sweep_chunks(int dtype, int64_t V) {
  return ceil_div(V * (dtype == 0 ? 4 : 2), (int64_t)kSweepChunkBytes);
}
SV_HD inline int64_t max_row_partials(int64_t V) { return ceil_div(V, (int64_t)1024); }

// The race's slices: kRaceSlice vocabulary entries.
constexpr int kRaceSlice = 1024;
SV_HD inline int64_t race_slices(int64_t V) { return ceil_div(V, (int64_t)kRaceSlice); }


// Per-row softmax statistics after the chunk combine: max (scaled, log2 units),
// row condition bits, the sum of 2^(y - max) and the largest logit as given.
struct RowStat {
  float mc;
  int bits;  // kRowNaN | kRowTimeout
  float s;   // sum of 2^(y - mc) over the row (fp32 throughout: GB300 runs fp64 slowly)
  float z;   // the row's largest logit as given (mc = z * scale), where the partials carry it
};
constexpr int kRowNaN = 1, kRowTimeout = 2;

// Counters start at zero; an add's old value tells the caller it was the n-th
// (last) arrival when old + 1 == n.
SV_HD inline bool is_last(uint32_t old, uint32_t n) { return old + 1u == n; }

// What the draw pass must do for one batch row.
enum DrawMode : int { kDrawDone = 0, kDrawSampleRow = 1, kDrawResidual = 2 };

struct DrawState {
  int mode;      // DrawMode
  int pos;       // position n of the draw (tag-1 Philox position)
  float c;       // fl32(fl32(1/T) * log2 e), the per-element scale
  float invT;    // fl32(1/T)
  float mct;     // target row n: scaled max
  float mcd;     // draft row n: scaled max (residual only)
  float K;       // (mct + log2 St) - (mcd + log2 Sd), log2 of q/p offset
  int flags;     // SV_FLAG_* gathered by the decision
  float tt;      // top-k threshold of target row n: logits below it have weight 0 (-inf: off)
  float td;      // top-k threshold of draft row n (residual only)
  float st;      // target row n: sum
  float sd;      // draft row n: sum (residual only)
  float zmt;     // target row n: largest logit as given (mct = zmt * c)
  float zmd;     // draft row n: largest logit as given (residual only)
};

// The race's shared bound of a batch row sits alone in a 128-byte line (every
// warp racing the row adds to it and reads it each round; rows packed into one
// line would make all warps of the GPU queue on the same L2 line).
constexpr int kThwStride = 32;  // 32-bit words between the bounds of consecutive rows

struct SamplePlan {
  int R1 = 0;          // logit rows per batch row, 2*gamma+1
  int npmax = 0;       // partials per row the workspace holds (one per 1024 logits)
  int nsplit3 = 0;     // most CTAs per batch row in the inverse-transform draw
  // the race's shared bound per batch row [B][kThwStride] (zeroed by the sweep), then the
  // sweep's partials [B][R1][partials per row] as float2 pairs
  size_t off_thw = 0, off_part1 = 0;
  // counters: [B] overlap CTAs (zeroed by the first draw CTA of each batch row),
  // then [B] inverse-transform draw CTAs that finished (zeroed by the sweep)
  size_t off_cnt = 0, cnt_bytes = 0, off_rowstat = 0, off_state = 0, off_segsum = 0,
         off_ctot = 0, off_alpha = 0, off_thr = 0, total = 0;
};

inline SamplePlan make_sample_plan(int B, int gamma, int64_t V) {
  SamplePlan p;
  if (B <= 0) return p;
  p.R1 = 2 * gamma + 1;
  p.npmax = (int)max_row_partials(V);
  p.nsplit3 = (int)ceil_div(V, kChunkDraw);
  size_t o = 0;
  p.off_thw = o;      o += sizeof(uint32_t) * kThwStride * (size_t)B;
  p.off_part1 = o;    o = align_up(o + 8 * (size_t)B * p.R1 * (size_t)p.npmax);
  p.cnt_bytes = 2 * sizeof(uint32_t) * (size_t)B;
  p.off_cnt = o;      o = align_up(o + p.cnt_bytes);
  p.off_rowstat = o;  o = align_up(o + sizeof(RowStat) * (size_t)B * p.R1);
  p.off_state = o;    o = align_up(o + sizeof(DrawState) * (size_t)B);
  // inverse-transform draw: one fixed-point weight sum per 256-entry segment
  p.off_segsum = o;   o = align_up(o + sizeof(uint64_t) * (size_t)B * (size_t)ceil_div(V, 256));
  p.off_ctot = o;     o = align_up(o + sizeof(uint64_t) * (size_t)B * p.nsplit3);  // per draw CTA
  p.off_alpha = o;    o = align_up(o + sizeof(float) * (size_t)B * gamma * ceil_div(V, kChunkSweep));
  p.off_thr = o;      o = align_up(o + sizeof(float) * (size_t)B * p.R1);  // top-k thresholds
  p.total = o;
  return p;
}

struct GreedyPlan {
  int nsplit = 0;
  size_t off_cnt = 0, off_part = 0, total = 0;
};

inline GreedyPlan make_greedy_plan(int B, int gamma, int64_t V) {
  GreedyPlan p;
  if (B <= 0) return p;
  p.nsplit = (int)ceil_div(V, kChunkSweep);
  size_t o = 0;
  p.off_cnt = o;   o = align_up(o + sizeof(uint32_t) * (size_t)B);
  p.off_part = o;  o = align_up(o + 8 * (size_t)B * (gamma + 1) * p.nsplit);
  p.total = o;
  return p;
}


// Fused LM head: vocabulary tile width, the largest hidden size whose compact
// row copies the workspace holds, and the largest token-row count per side.
constexpr int kLmTileN = 128;
constexpr int kLmMaxHidden = 16384;
constexpr int kLmMaxRows = 256;

// One candidate of a Gumbel-max: key (log2 units), vocabulary index, and the
// target / draft logits there (for the double-precision re-decision).
struct LmCand {
  float key;
  int idx;
  float zt, zd;
};

struct LmPlan {
  int R1 = 0;   // 2*gamma+1 logit rows per batch row
  int nvt = 0;  // vocabulary tiles
  // ctl: [0] compact-row count, [1] pass-1 error, [2] pass-2 error (zeroed per call)
  size_t off_ctl = 0, off_part = 0, off_zat = 0, off_state = 0, off_slot = 0, off_res2 = 0,
         off_ct = 0, off_cd = 0, total = 0;
};

inline LmPlan make_lm_plan(int B, int gamma, int64_t V) {
  LmPlan p;
  if (B <= 0) return p;
  p.R1 = 2 * gamma + 1;
  p.nvt = (int)ceil_div(V, kLmTileN);
  const size_t rows = (size_t)B * p.R1;
  size_t o = 0;
  p.off_ctl = o;    o = align_up(o + 4 * sizeof(uint32_t));
  // two partials per row and CTA of the GEMM passes (the two column halves of
  // the epilogue); there are at most as many CTAs as vocabulary tiles
  p.off_part = o;   o = align_up(o + 8 * rows * p.nvt * 2);
  p.off_zat = o;    o = align_up(o + sizeof(float) * rows);
  p.off_state = o;  o = align_up(o + sizeof(DrawState) * (size_t)B);
  p.off_slot = o;   o = align_up(o + sizeof(int) * (size_t)B);
  // the draw: per compact row and GEMM CTA (at most one per vocabulary tile) the
  // best two race candidates of the residual and of p_n
  p.off_res2 = o;   o = align_up(o + 4 * sizeof(LmCand) * (size_t)B * p.nvt);
  p.off_ct = o;     o = align_up(o + 2 * (size_t)B * kLmMaxHidden);
  p.off_cd = o;     o = align_up(o + 2 * (size_t)B * kLmMaxHidden);
  p.total = o;
  return p;
}

// Workspace of a draft-sampling call (spec_lmhead_draft): per (batch row, CTA)
// one (max, sum) partial and a top-2 of keys; control words.
struct DraftPlan {
  int nvt = 0;
  size_t off_ctl = 0, off_part = 0, off_cand = 0, total = 0;
};

inline DraftPlan make_draft_plan(int B, int64_t V) {
  DraftPlan p;
  if (B <= 0) return p;
  p.nvt = (int)ceil_div(V, kLmTileN);
  size_t o = 0;
  p.off_ctl = o;   o = align_up(o + 4 * sizeof(uint32_t));
  p.off_part = o;  o = align_up(o + 8 * (size_t)B * p.nvt);
  p.off_cand = o;  o = align_up(o + 2 * sizeof(LmCand) * (size_t)B * p.nvt);
  p.total = o;
  return p;
}

}  // namespace sv
