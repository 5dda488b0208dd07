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
constexpr size_t kAlign = 256;

// Persistent vector sweep: warps per CTA, resident CTAs per SM (its launch bounds),
// bytes per chunk.
constexpr int kSweepWarps = 8;
constexpr int kSweepCtasPerSm = 2;
constexpr int kSweepChunkBytes = 4096;

// The vector sweep needs every row to start on a 16-byte boundary (the bases are)
// and rows of at least one chunk, so that a chunk touches at most two rows.
SV_HD inline bool use_vec_sweep(int dtype, int64_t V) {
  const int64_t rb = V * (dtype == 0 ? 4 : 2);
  return rb % 16 == 0 && rb >= kSweepChunkBytes;
}

SV_HD inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
SV_HD inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Partials of a sweep, at most: one per 4 KB block of the target and draft arrays of
// fp32 rows (either base may sit anywhere in its first block: one more block each),
// the two edge pieces of every row, or one per kChunkSweep-logit split of every row.
SV_HD inline int64_t vec_sweep_blocks(int B, int gamma, int64_t V) {
  const int64_t rb = V * 4;
  return ceil_div((int64_t)B * (gamma + 1) * rb, 4096) + 1 + ceil_div((int64_t)B * gamma * rb, 4096) + 1;
}
SV_HD inline int64_t vec_sweep_partials(int B, int gamma, int64_t V) {
  const int64_t rows = (int64_t)B * (2 * gamma + 1);
  const int64_t vec = vec_sweep_blocks(B, gamma, V) + 2 * rows;
  const int64_t gen = rows * ceil_div(V, kChunkSweep);
  return vec > gen ? vec : gen;
}

// Per-row softmax statistics after the chunk combine: max (scaled, log2 units),
// row condition bits, and the sum of 2^(y - max) in double.
struct RowStat {
  float mc;
  int bits;  // kRowNaN | kRowTimeout
  float s;   // sum of 2^(y - mc) over the row (fp32 throughout: GB300 runs fp64 slowly)
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
};

struct SamplePlan {
  int R1 = 0;          // logit rows per batch row, 2*gamma+1
  int nsplit1 = 0;     // 8192-logit chunks per row (generic sweep, overlap pass)
  int nsplit3 = 0;     // most CTAs per batch row in the draw pass
  // counters: [B] overlap CTAs (zeroed by the first draw CTA of each batch row),
  // then [B] draw CTAs that finished their segment sums (zeroed by the sweep)
  size_t off_cnt = 0, cnt_bytes = 0, off_part1 = 0, off_rowstat = 0, off_state = 0,
         off_segsum = 0, off_ctot = 0, off_alpha = 0, off_thr = 0, total = 0;
};

inline SamplePlan make_sample_plan(int B, int gamma, int64_t V) {
  SamplePlan p;
  if (B <= 0) return p;
  p.R1 = 2 * gamma + 1;
  p.nsplit1 = (int)ceil_div(V, kChunkSweep);
  p.nsplit3 = (int)ceil_div(V, kChunkDraw);
  // chunk partials: [row][8192-logit split] (generic sweep), or one per 4 KB block of
  // the two logit arrays plus [row][2] edge pieces (vector sweep; fp32 has the most)
  const int64_t nparts = vec_sweep_partials(B, gamma, V);
  const int64_t nch_max = ceil_div(nparts, (int64_t)B * p.R1);
  size_t o = 0;
  p.cnt_bytes = 2 * sizeof(uint32_t) * (size_t)B;
  p.off_cnt = o;      o = align_up(o + p.cnt_bytes);
  p.off_rowstat = o;  o = align_up(o + sizeof(RowStat) * (size_t)B * p.R1);
  p.off_part1 = o;    o = align_up(o + 8 * (size_t)B * p.R1 * (size_t)nch_max);
  p.off_state = o;    o = align_up(o + sizeof(DrawState) * (size_t)B);
  // draw: one fixed-point weight sum per 256-entry segment of the row drawn from
  p.off_segsum = o;   o = align_up(o + sizeof(uint64_t) * (size_t)B * (size_t)ceil_div(V, 256));
  p.off_ctot = o;     o = align_up(o + sizeof(uint64_t) * (size_t)B * p.nsplit3);  // per draw CTA
  p.off_alpha = o;    o = align_up(o + sizeof(float) * (size_t)B * gamma * p.nsplit1);
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
  size_t off_ctl = 0, off_part = 0, off_zat = 0, off_state = 0, off_slot = 0,
         off_csr = 0, off_csp = 0, off_tsr = 0, off_tsp = 0,
         off_gsr = 0, off_gsp = 0, off_ct = 0, off_cd = 0, total = 0;
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
  // the draw: weight sums per 16-entry chunk, per tile and per group of 32 tiles
  const size_t nchunk = (size_t)ceil_div(V, 16);
  p.off_csr = o;    o = align_up(o + sizeof(float) * (size_t)B * nchunk);
  p.off_csp = o;    o = align_up(o + sizeof(float) * (size_t)B * nchunk);
  p.off_tsr = o;    o = align_up(o + sizeof(uint64_t) * (size_t)B * p.nvt);
  p.off_tsp = o;    o = align_up(o + sizeof(uint64_t) * (size_t)B * p.nvt);
  p.off_gsr = o;    o = align_up(o + sizeof(uint64_t) * (size_t)B * ((p.nvt + 31) / 32));
  p.off_gsp = o;    o = align_up(o + sizeof(uint64_t) * (size_t)B * ((p.nvt + 31) / 32));
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
