// sv_abi.cu -- the extern "C" entry points of libspecverify: argument checks,
// workspace layout and kernel launches.  Declarations and contracts are in
// include/specverify.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "specverify.h"
#include "sv_plan.h"
#include "sv_launch.h"

namespace sv {
cudaError_t launch_sample(const void* zt, const void* zd, const int32_t* xt, int B, int gamma,
                          int64_t V, int dtype, float temperature, const float* row_T,
                          uint64_t seed, uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                          float* out_p, float* out_q, float* out_alpha, uint8_t* out_flags,
                          void* ws, const SamplePlan& pl, cudaStream_t stream,
                          float lenience, int top_k, float top_p, int sampler);
cudaError_t launch_greedy(const void* zt, const int32_t* xt, int B, int gamma, int64_t V,
                          int dtype, int32_t* out_tokens, int32_t* out_counts, void* ws,
                          const GreedyPlan& pl, cudaStream_t stream);
int lmhead_verify(const void* h_target, const void* W_target, int Ht, const void* h_draft,
                  const void* W_draft, int Hd, const int32_t* draft_tokens, int B, int gamma,
                  int64_t V, float temperature, uint64_t seed, uint64_t round,
                  int32_t* out_tokens, int32_t* out_counts, float* out_p, float* out_q,
                  uint8_t* out_flags, float* debug_logits, void* workspace,
                  size_t workspace_bytes, cudaStream_t stream, const float* draft_lse,
                  const float* draft_logit);
size_t lmhead_workspace_bytes(int B, int gamma, int64_t V);
int lmhead_draft(const void* h_draft, const void* W_draft, int Hd, int B, int64_t V,
                 float temperature, uint64_t seed, uint64_t round, int pos, int32_t* out_tokens,
                 float* out_q, float* out_lse, float* out_logit, float* debug_logits,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t lmhead_draft_workspace_bytes(int B, int64_t V);
}  // namespace sv

namespace sv {
static cudaEvent_t g_events[kMaxTimingEvents] = {};

void set_timing_events(void* const* ev, int n) {
  for (int i = 0; i < kMaxTimingEvents; ++i)
    g_events[i] = (ev && i < n) ? (cudaEvent_t)ev[i] : nullptr;
}

void mark(int i, cudaStream_t s) {
  if (i >= 0 && i < kMaxTimingEvents && g_events[i]) cudaEventRecord(g_events[i], s);
}
}  // namespace sv

namespace {

constexpr int kMaxGamma = 32;
constexpr int64_t kMaxV = (int64_t)1 << 31;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int B, int gamma, int64_t V) {
  if (B < 0 || gamma < 1 || gamma > kMaxGamma || V < 1 || V >= kMaxV) return SV_ERR_ARG;
  return SV_OK;
}

int check_workspace(const void* ws, size_t have, size_t need) {
  if (need == 0) return SV_OK;
  if (!ws || have < need) return SV_ERR_WORKSPACE;
  if (!aligned(ws, sv::kAlign)) return SV_ERR_ALIGN;
  return SV_OK;
}

}  // namespace

extern "C" {

size_t sv_workspace_bytes(int B, int gamma, int64_t V, int mode) {
  if (check_shape(B, gamma, V) != SV_OK || B == 0) return 0;
  switch (mode) {
    case SV_MODE_SAMPLE: return sv::make_sample_plan(B, gamma, V).total;
    case SV_MODE_GREEDY: return sv::make_greedy_plan(B, gamma, V).total;
    case SV_MODE_LMHEAD: return sv::lmhead_workspace_bytes(B, gamma, V);
    case SV_MODE_DRAFT: return sv::lmhead_draft_workspace_bytes(B, V);
    default: return 0;
  }
}

int sv_workspace_init(void* workspace, size_t bytes, void* cuda_stream) {
  if (bytes == 0) return SV_OK;
  if (!workspace) return SV_ERR_ARG;
  return cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)cuda_stream) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

int spec_verify(const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, int B, int gamma, int64_t V, int dtype,
                float temperature, const float* row_temperature, uint64_t seed,
                uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                float* out_p_at_draft, float* out_q_at_draft, float* out_alpha,
                uint8_t* out_flags, void* workspace, size_t workspace_bytes,
                void* cuda_stream) {
  return spec_verify_opts(target_logits, draft_logits, draft_tokens, B, gamma, V, dtype,
                          temperature, row_temperature, seed, round, out_tokens, out_counts,
                          out_p_at_draft, out_q_at_draft, out_alpha, out_flags, nullptr,
                          workspace, workspace_bytes, cuda_stream);
}

int spec_verify_opts(const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, int B, int gamma, int64_t V, int dtype,
                     float temperature, const float* row_temperature, uint64_t seed,
                     uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                     float* out_p_at_draft, float* out_q_at_draft, float* out_alpha,
                     uint8_t* out_flags, const sv_options* options, void* workspace,
                     size_t workspace_bytes, void* cuda_stream) {
  float lenience = 1.0f, top_p = 1.0f;
  int top_k = 0, sampler = SV_SAMPLER_GUMBEL;
  if (options) {
    lenience = options->lenience;
    top_k = options->top_k;
    top_p = options->top_p;
    sampler = options->sampler;
    if (!(lenience > 0.0f && lenience <= 1.0f) || top_k < 0 || !(top_p > 0.0f && top_p <= 1.0f) ||
        (sampler != SV_SAMPLER_GUMBEL && sampler != SV_SAMPLER_INVERSE))
      return SV_ERR_ARG;
    if (top_p < 1.0f && V > (int64_t(1) << 21)) return SV_ERR_UNSUPPORTED;  // nucleus sums
  }
  int st = check_shape(B, gamma, V);
  if (st != SV_OK) return st;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (!row_temperature && !(temperature > 0.0f && std::isfinite(temperature))) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !out_tokens || !out_counts)
    return SV_ERR_ARG;
  if (!aligned(target_logits, 16) || !aligned(draft_logits, 16) || !aligned(draft_tokens, 4) ||
      !aligned(out_tokens, 4) || !aligned(out_counts, 4) ||
      (row_temperature && !aligned(row_temperature, 4)) ||
      (out_p_at_draft && !aligned(out_p_at_draft, 4)) ||
      (out_q_at_draft && !aligned(out_q_at_draft, 4)) || (out_alpha && !aligned(out_alpha, 4)))
    return SV_ERR_ALIGN;
  const sv::SamplePlan pl = sv::make_sample_plan(B, gamma, V);
  st = check_workspace(workspace, workspace_bytes, pl.total);
  if (st != SV_OK) return st;
  const cudaError_t e = sv::launch_sample(
      target_logits, draft_logits, draft_tokens, B, gamma, V, dtype, temperature, row_temperature,
      seed, round, out_tokens, out_counts, out_p_at_draft, out_q_at_draft, out_alpha, out_flags,
      workspace, pl, (cudaStream_t)cuda_stream, lenience, top_k, top_p, sampler);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B,
                       int gamma, int64_t V, int dtype, int32_t* out_tokens,
                       int32_t* out_counts, void* workspace, size_t workspace_bytes,
                       void* cuda_stream) {
  int st = check_shape(B, gamma, V);
  if (st != SV_OK) return st;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (B == 0) return SV_OK;
  if (!target_logits || !draft_tokens || !out_tokens || !out_counts) return SV_ERR_ARG;
  if (!aligned(target_logits, 16) || !aligned(draft_tokens, 4) || !aligned(out_tokens, 4) ||
      !aligned(out_counts, 4))
    return SV_ERR_ALIGN;
  const sv::GreedyPlan pl = sv::make_greedy_plan(B, gamma, V);
  st = check_workspace(workspace, workspace_bytes, pl.total);
  if (st != SV_OK) return st;
  const cudaError_t e = sv::launch_greedy(target_logits, draft_tokens, B, gamma, V, dtype,
                                          out_tokens, out_counts, workspace, pl,
                                          (cudaStream_t)cuda_stream);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int spec_lmhead_verify(const void* h_target, const void* W_target, int Ht, const void* h_draft,
                       const void* W_draft, int Hd, const int32_t* draft_tokens, int B,
                       int gamma, int64_t V, float temperature, uint64_t seed, uint64_t round,
                       int32_t* out_tokens, int32_t* out_counts, float* out_p_at_draft,
                       float* out_q_at_draft, uint8_t* out_flags, float* debug_logits,
                       void* workspace, size_t workspace_bytes, void* cuda_stream) {
  int st = check_shape(B, gamma, V);
  if (st != SV_OK) return st;
  if (!(temperature > 0.0f && std::isfinite(temperature))) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  return sv::lmhead_verify(h_target, W_target, Ht, h_draft, W_draft, Hd, draft_tokens, B, gamma,
                           V, temperature, seed, round, out_tokens, out_counts, out_p_at_draft,
                           out_q_at_draft, out_flags, debug_logits, workspace, workspace_bytes,
                           (cudaStream_t)cuda_stream, nullptr, nullptr);
}

int spec_lmhead_verify_drafted(const void* h_target, const void* W_target, int Ht,
                               const void* h_draft, const void* W_draft, int Hd,
                               const int32_t* draft_tokens, const float* draft_lse,
                               const float* draft_logit, int B, int gamma, int64_t V,
                               float temperature, uint64_t seed, uint64_t round,
                               int32_t* out_tokens, int32_t* out_counts, float* out_p_at_draft,
                               float* out_q_at_draft, uint8_t* out_flags, float* debug_logits,
                               void* workspace, size_t workspace_bytes, void* cuda_stream) {
  int st = check_shape(B, gamma, V);
  if (st != SV_OK) return st;
  if (!(temperature > 0.0f && std::isfinite(temperature))) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  if (!draft_lse || !draft_logit) return SV_ERR_ARG;
  return sv::lmhead_verify(h_target, W_target, Ht, h_draft, W_draft, Hd, draft_tokens, B, gamma,
                           V, temperature, seed, round, out_tokens, out_counts, out_p_at_draft,
                           out_q_at_draft, out_flags, debug_logits, workspace, workspace_bytes,
                           (cudaStream_t)cuda_stream, draft_lse, draft_logit);
}

int spec_lmhead_draft(const void* h_draft, const void* W_draft, int Hd, int B, int64_t V,
                      float temperature, uint64_t seed, uint64_t round, int pos,
                      int32_t* out_tokens, float* out_q, float* out_lse, float* out_logit,
                      float* debug_logits, void* workspace, size_t workspace_bytes,
                      void* cuda_stream) {
  if (B < 0 || V < 1 || V >= ((int64_t)1 << 31)) return SV_ERR_ARG;
  if (!(temperature > 0.0f && std::isfinite(temperature))) return SV_ERR_ARG;
  if (B == 0) return SV_OK;
  return sv::lmhead_draft(h_draft, W_draft, Hd, B, V, temperature, seed, round, pos, out_tokens,
                          out_q, out_lse, out_logit, debug_logits, workspace, workspace_bytes,
                          (cudaStream_t)cuda_stream);
}

int sv_set_timing_events(void* const* events, int n) {
  if (events && n < 1) return SV_ERR_ARG;
  sv::set_timing_events(events, n);
  return SV_OK;
}

const char* sv_status_string(int status) {
  switch (status) {
    case SV_OK: return "SV_OK";
    case SV_ERR_ARG: return "SV_ERR_ARG: invalid argument";
    case SV_ERR_DTYPE: return "SV_ERR_DTYPE: unsupported dtype";
    case SV_ERR_ALIGN: return "SV_ERR_ALIGN: misaligned pointer";
    case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing or too small";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: CUDA runtime or launch failure";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: unsupported device or shape";
    default: return "unknown status";
  }
}

int sv_version(void) { return 100; }

}  // extern "C"
