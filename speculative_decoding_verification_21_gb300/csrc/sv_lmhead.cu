// sv_lmhead.cu -- fused LM head + verify (tcgen05).  Placeholder until the
// tensor-core kernel lands: reports SV_ERR_UNSUPPORTED.
#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"

namespace sv {

size_t lmhead_workspace_bytes(int, int, int64_t) { return 0; }

int lmhead_verify(const void*, const void*, int, const void*, const void*, int, const int32_t*,
                  int, int, int64_t, float, uint64_t, uint64_t, int32_t*, int32_t*, float*,
                  float*, uint8_t*, float*, void*, size_t, cudaStream_t) {
  return SV_ERR_UNSUPPORTED;
}

}  // namespace sv
