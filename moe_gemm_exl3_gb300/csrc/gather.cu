// gather.cu -- int8 embedding rows with a per-row fp16 scale, gathered and
// dequantized on the gathered rows only (vllm-quantpack exl3/embedding.py,
// embedding()).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace exl3 {

// A thread takes kGatherChunks 16-byte chunks of one gathered row (16 int8 ->
// 16 bf16 = two 16-byte stores each): one row id and scale read, then all of its
// row loads in flight at once.  Chunk k of thread j of a row is j + k * tpr (tpr
// threads per row), so at every step a warp's loads and stores cover consecutive
// 16-byte chunks of a row (coalesced).  The table is streamed once per gathered
// row, the output streamed out of L2 first.
constexpr int kGatherChunks = 4;

__global__ void __launch_bounds__(256) gather_kernel(const int8_t *__restrict__ q,
                                                     const uint16_t *__restrict__ scale,
                                                     int64_t V, int H,
                                                     const int32_t *__restrict__ ids,
                                                     int64_t N, uint16_t *__restrict__ out,
                                                     int32_t *n_bad) {
    const int chunks = H / 16;
    const int tpr = (chunks + kGatherChunks - 1) / kGatherChunks;   // threads per row
    const unsigned t = blockIdx.x * blockDim.x + threadIdx.x;       // N * tpr < 2^31 (checked on launch)
    const unsigned iu = t / (unsigned)tpr;
    const int64_t i = iu;                          // gathered row
    if (i >= N) return;
    const int j = (int)(t - iu * (unsigned)tpr);
    const int64_t id = __ldg(ids + i);
    uint4 *dst = reinterpret_cast<uint4 *>(out + i * H);
    if (id < 0 || id >= V) {
#pragma unroll
        for (int k = 0; k < kGatherChunks; k++) {
            const int ch = j + k * tpr;
            if (ch < chunks) {
                dst[2 * ch] = make_uint4(0, 0, 0, 0);
                dst[2 * ch + 1] = make_uint4(0, 0, 0, 0);
            }
        }
        if (j == 0 && n_bad) atomicAdd(n_bad, 1);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(q + id * H);
    uint4 raw[kGatherChunks];
#pragma unroll
    for (int k = 0; k < kGatherChunks; k++) {
        const int ch = j + k * tpr;
        if (ch < chunks) raw[k] = __ldcs(src + ch);
    }
    const float s = f16_bits_to_f32(__ldg(scale + id));
#pragma unroll
    for (int k = 0; k < kGatherChunks; k++) {
        const int ch = j + k * tpr;
        if (ch >= chunks) break;
        const uint32_t words[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
        uint32_t o[8];
#pragma unroll
        for (int w = 0; w < 4; w++) {
#pragma unroll
            for (int h = 0; h < 2; h++) {
                // int8 * fp16 scale is exact in fp32 (8 + 11 significant bits): one rounding
                const float x0 = (float)(int8_t)(words[w] >> (16 * h));
                const float x1 = (float)(int8_t)(words[w] >> (16 * h + 8));
                o[2 * w + h] = (uint32_t)f32_to_bf16_bits(x0 * s) | ((uint32_t)f32_to_bf16_bits(x1 * s) << 16);
            }
        }
        __stcs(dst + 2 * ch, make_uint4(o[0], o[1], o[2], o[3]));
        __stcs(dst + 2 * ch + 1, make_uint4(o[4], o[5], o[6], o[7]));
    }
}

cudaError_t launch_gather(const int8_t *q, const uint16_t *scale, int64_t V, int H,
                          const int32_t *ids, int64_t N, uint16_t *out, int32_t *n_bad,
                          cudaStream_t s) {
    const int64_t tpr = (H / 16 + kGatherChunks - 1) / kGatherChunks;
    const int64_t threads = N * tpr;
    if (threads >= 0x7FFFFF00LL) return cudaErrorInvalidValue;   // thread index must fit 31 bits
    const int64_t grid = (threads + 255) / 256;
    gather_kernel<<<(unsigned)grid, 256, 0, s>>>(q, scale, V, H, ids, N, out, n_bad);
    return cudaGetLastError();
}

}  // namespace exl3
