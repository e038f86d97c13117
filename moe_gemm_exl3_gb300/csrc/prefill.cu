// prefill.cu -- large-M (prefill) path.  Placeholder until the tensor-core kernel lands:
// reports "not launched" so the caller keeps the decode-mode passes.
#include <cuda_runtime.h>

#include "internal.h"

namespace exl3 {

bool prefill_supported() { return false; }

cudaError_t launch_prefill(const uint16_t *, const uint16_t *, int64_t, int, int, const uint16_t *,
                           const uint16_t *, uint16_t *, int64_t, int32_t *, cudaStream_t, bool *launched) {
    *launched = false;
    return cudaSuccess;
}

}  // namespace exl3
