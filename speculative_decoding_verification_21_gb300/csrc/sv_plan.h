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
constexpr int64_t kChunkDraw = 4096;   // vocabulary entries per CTA in the draw pass
constexpr size_t kAlign = 256;

SV_HD inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
SV_HD inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Per-row softmax statistics after the split combine: max (scaled, log2 units)
// and the sum of 2^(y - max) in double.
struct RowStat {
  float mc;
  float pad;
  double s;
};

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
  int pad;
  double st;     // target row n: sum
  double sd;     // draft row n: sum (residual only)
};

struct SamplePlan {
  int R1 = 0;          // logit rows per batch row, 2*gamma+1
  int nsplit1 = 0;     // CTAs per row in the sweep
  int nsplit3 = 0;     // CTAs per batch row in the draw pass
  size_t off_cnt = 0, off_part1 = 0, off_rowstat = 0, off_state = 0, off_part3 = 0,
         off_alpha = 0, total = 0;
};

inline SamplePlan make_sample_plan(int B, int gamma, int64_t V) {
  SamplePlan p;
  if (B <= 0) return p;
  p.R1 = 2 * gamma + 1;
  p.nsplit1 = (int)ceil_div(V, kChunkSweep);
  p.nsplit3 = (int)ceil_div(V, kChunkDraw);
  size_t o = 0;
  p.off_cnt = o;      o = align_up(o + sizeof(uint32_t) * 2 * (size_t)B);
  p.off_part1 = o;    o = align_up(o + 8 * (size_t)B * p.R1 * p.nsplit1);
  p.off_rowstat = o;  o = align_up(o + sizeof(RowStat) * (size_t)B * p.R1);
  p.off_state = o;    o = align_up(o + sizeof(DrawState) * (size_t)B);
  p.off_part3 = o;    o = align_up(o + 16 * (size_t)B * p.nsplit3);
  p.off_alpha = o;    o = align_up(o + sizeof(float) * (size_t)B * gamma * p.nsplit1);
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

}  // namespace sv
