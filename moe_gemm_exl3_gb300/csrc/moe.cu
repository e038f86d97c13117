// moe.cu -- grouped MoE over an EXL3 expert bank (bank.py layout).
#include <cuda_runtime.h>

#include "../../include/exl3.h"
#include "internal.h"

namespace exl3 {
exl3_status fail(exl3_status st, const char *fmt, ...);
}
using namespace exl3;

extern "C" {

exl3_status exl3_moe_topk_softmax(const float *, int32_t, int32_t, int32_t, int32_t *, float *, exl3_stream) {
    return fail(EXL3_EUNSUPPORTED, "moe_topk_softmax: not built yet");
}

size_t exl3_moe_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

exl3_status exl3_moe_grouped(const uint16_t *, int32_t, int32_t, int32_t, int32_t, int32_t, const int32_t *,
                             const float *, const exl3_moe_bank *, uint16_t *, void *, size_t, exl3_stream) {
    return fail(EXL3_EUNSUPPORTED, "moe_grouped: not built yet");
}

}  // extern "C"
