// sv_noalloc.cu -- spec_verify_noalloc: the sampling verify for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running inside a
// memory-pool-less runtime, a plugin that is handed only its input and output
// buffers, or an allocator that must not be touched on the hot path (for
// instance because it would synchronise the device or fragment a reserved
// pool).  This entry point takes the same inputs and outputs as spec_verify but
// no workspace: the scratch memory its kernels need lives in one file-scope
// device array, reserved when the library is loaded on a GPU and held by every
// GPU that loads the library until the process exits.
//
// Contract (also in include/specverify.h):
//   - the scratch array has a fixed size, kNoAllocScratchBytes (4 MiB); calls
//     whose sizes need more than that (sv_workspace_bytes(B, gamma, V,
//     SV_MODE_SAMPLE) > 4 MiB) are rejected with SV_ERR_WORKSPACE before any
//     work is queued;
//   - nothing here calls cudaMalloc, cudaFree or any allocating routine;
//   - the first call on a device, with that device current, looks up the
//     array's device address (cudaGetSymbolAddress) and caches it; make that
//     first call before any stream capture;
//   - every call shares the one array, which keeps whatever the last call left
//     in it.  Each call first resets, on its stream, the counters and markers
//     it relies on.  Calls that overlap on the GPU (other streams, other host
//     threads) race on the array: serialise them.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "specverify.h"
#include "sv_plan.h"

namespace sv {
cudaError_t launch_sample(const void* zt, const void* zd, const int32_t* xt, int B, int gamma,
                          int64_t V, int dtype, float temperature, const float* row_T,
                          uint64_t seed, uint64_t round, int32_t* out_tokens, int32_t* out_counts,
                          float* out_p, float* out_q, float* out_alpha, uint8_t* out_flags,
                          void* ws, const SamplePlan& pl, cudaStream_t stream,
                          float lenience, int top_k, float top_p, int sampler);
}  // namespace sv

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

// The scratch memory: one array per device that loads the library.  In host
// code `g_scratch` names a host-side stand-in, not device memory; only the
// address from cudaGetSymbolAddress may be handed to a kernel.
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) return SV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                   const int32_t* draft_tokens, int B, int gamma, int64_t V,
                                   int dtype, float temperature, const float* row_temperature,
                                   uint64_t seed, uint64_t round, int32_t* out_tokens,
                                   int32_t* out_counts, float* out_p_at_draft,
                                   float* out_q_at_draft, float* out_alpha, uint8_t* out_flags,
                                   void* cuda_stream) {
  if (B < 0 || gamma < 1 || gamma > 32 || V < 1 || V >= ((int64_t)1 << 31)) return SV_ERR_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
  if (!row_temperature && !(temperature > 0.0f && temperature < __builtin_huge_valf()))
    return SV_ERR_ARG;
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
  if (pl.total > kNoAllocScratchBytes) return SV_ERR_WORKSPACE;  // beyond the static scratch
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != SV_OK) return st;
  const cudaError_t e = sv::launch_sample(
      target_logits, draft_logits, draft_tokens, B, gamma, V, dtype, temperature, row_temperature,
      seed, round, out_tokens, out_counts, out_p_at_draft, out_q_at_draft, out_alpha, out_flags,
      scratch, pl, (cudaStream_t)cuda_stream, 1.0f, 0, 1.0f, SV_SAMPLER_GUMBEL);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
