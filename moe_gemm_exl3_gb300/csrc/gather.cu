// gather.cu -- int8 embedding rows with a per-row fp16 scale, gathered and
// dequantized on the gathered rows only (vllm-quantpack exl3/embedding.py,
// embedding()).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace exl3 {

// One thread per 16-byte chunk of a gathered row (16 int8 -> 16 bf16 = two
// 16-byte stores): every load of the job is independent and in flight at once,
// so the kernel streams at the memory system's rate rather than a loop's.  The
// row id and scale are read per thread (broadcast within a warp: a warp covers
// 512 consecutive bytes of one row when H >= 512).  Reads and writes are
// coalesced across the warp; the table is streamed once per gathered row.
__global__ void __launch_bounds__(256) gather_kernel(const int8_t *__restrict__ q,
                                                     const uint16_t *__restrict__ scale,
                                                     int64_t V, int H,
                                                     const int32_t *__restrict__ ids,
                                                     int64_t N, uint16_t *__restrict__ out,
                                                     int32_t *n_bad) {
    const unsigned chunks = (unsigned)H / 16;
    const unsigned t = blockIdx.x * blockDim.x + threadIdx.x;   // N * H / 16 < 2^31 (checked on launch)
    const unsigned iu = t / chunks;
    const int64_t i = iu;                          // gathered row
    if (i >= N) return;
    const int ch = (int)(t - iu * chunks);
    const int64_t id = __ldg(ids + i);
    uint4 *dst = reinterpret_cast<uint4 *>(out + i * H) + 2 * ch;
    if (id < 0 || id >= V) {
        dst[0] = make_uint4(0, 0, 0, 0);
        dst[1] = make_uint4(0, 0, 0, 0);
        if (ch == 0 && n_bad) atomicAdd(n_bad, 1);
        return;
    }
    const uint4 raw = __ldcs(reinterpret_cast<const uint4 *>(q + id * H) + ch);
    const float s = f16_bits_to_f32(__ldg(scale + id));
    const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; k++) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            // int8 * fp16 scale is exact in fp32 (8 + 11 significant bits): one rounding
            const float x0 = (float)(int8_t)(words[k] >> (16 * h));
            const float x1 = (float)(int8_t)(words[k] >> (16 * h + 8));
            o[2 * k + h] = (uint32_t)f32_to_bf16_bits(x0 * s) | ((uint32_t)f32_to_bf16_bits(x1 * s) << 16);
        }
    }
    __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

cudaError_t launch_gather(const int8_t *q, const uint16_t *scale, int64_t V, int H,
                          const int32_t *ids, int64_t N, uint16_t *out, int32_t *n_bad,
                          cudaStream_t s) {
    const int64_t threads = N * (H / 16);
    if (threads >= 0x7FFFFF00LL) return cudaErrorInvalidValue;   // thread index must fit 31 bits
    const int64_t grid = (threads + 255) / 256;
    gather_kernel<<<(unsigned)grid, 256, 0, s>>>(q, scale, V, H, ids, N, out, n_bad);
    return cudaGetLastError();
}

}  // namespace exl3
