// gather.cu -- int8 embedding rows with a per-row fp16 scale, gathered and
// dequantized on the gathered rows only (vllm-quantpack exl3/embedding.py,
// embedding()).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace exl3 {

// One warp per gathered row: the id and the scale are read once (broadcast),
// then each lane converts 16-byte chunks (16 int8 -> 16 bf16 = two 16-byte
// stores) at a stride of 32 chunks, with up to four chunk loads in flight per
// lane before the first conversion.  The table is streamed once per gathered
// row; reads and writes are coalesced across the warp.
__global__ void __launch_bounds__(256) gather_kernel(const int8_t *__restrict__ q,
                                                     const uint16_t *__restrict__ scale,
                                                     int64_t V, int H,
                                                     const int32_t *__restrict__ ids,
                                                     int64_t N, uint16_t *__restrict__ out,
                                                     int32_t *n_bad) {
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (i >= N) return;
    const int chunks = H / 16;
    const int64_t id = __ldg(ids + i);
    uint4 *dst = reinterpret_cast<uint4 *>(out + i * H);
    if (id < 0 || id >= V) {
        for (int ch = lane; ch < chunks; ch += 32) {
            dst[2 * ch] = make_uint4(0, 0, 0, 0);
            dst[2 * ch + 1] = make_uint4(0, 0, 0, 0);
        }
        if (lane == 0 && n_bad) atomicAdd(n_bad, 1);
        return;
    }
    const float s = f16_bits_to_f32(__ldg(scale + id));
    const uint4 *src = reinterpret_cast<const uint4 *>(q + id * H);
    for (int ch0 = lane; ch0 < chunks; ch0 += 32 * U) {
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; u++)
            if (ch0 + 32 * u < chunks) raw[u] = __ldcs(src + ch0 + 32 * u);
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int ch = ch0 + 32 * u;
            if (ch >= chunks) break;
            const uint32_t words[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
            uint32_t o[8];
#pragma unroll
            for (int k = 0; k < 4; k++) {
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    // int8 * fp16 scale is exact in fp32 (8 + 11 significant bits): one rounding
                    const float a = (float)(int8_t)(words[k] >> (16 * h));
                    const float b = (float)(int8_t)(words[k] >> (16 * h + 8));
                    o[2 * k + h] = (uint32_t)f32_to_bf16_bits(a * s) | ((uint32_t)f32_to_bf16_bits(b * s) << 16);
                }
            }
            __stcs(dst + 2 * ch, make_uint4(o[0], o[1], o[2], o[3]));
            __stcs(dst + 2 * ch + 1, make_uint4(o[4], o[5], o[6], o[7]));
        }
    }
}

cudaError_t launch_gather(const int8_t *q, const uint16_t *scale, int64_t V, int H,
                          const int32_t *ids, int64_t N, uint16_t *out, int32_t *n_bad,
                          cudaStream_t s) {
    const int64_t grid = (N + 7) / 8;     // 8 rows (warps) per 256-thread CTA
    gather_kernel<<<(unsigned)grid, 256, 0, s>>>(q, scale, V, H, ids, N, out, n_bad);
    return cudaGetLastError();
}

}  // namespace exl3
