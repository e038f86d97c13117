// a8.cu -- the 8-bit activation variant (radiance_escha.py, escha_linear_into:
// the uint8 activation buffer A [M][IC] with a float32 scale As [M] taken from a
// per-row amax).  The activations are pre-transformed as in the 16-bit path,
// then quantized per row:
//     As = amax / 127,  q = round_half_even(u / As) clamped to [-127, 127],
//     code = q + 128 (q = 0 for an all-zero row).
// The GEMM multiplies q exactly (q and the decoded weights are fp16-exact) and
// the epilogue multiplies each row by As.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace exl3 {

namespace {

constexpr int kQRun = 4;   // 128-channel blocks a warp loads before transforming them

// One CTA per (shard, row): CTA b serves row b % M with shard b / M's scales and
// writes row b of dst and As.  8 warps: warp w transforms blocks w, w + 8, ... of the row
// into shared memory (fp32, loads of up to kQRun blocks issued together), the
// CTA reduces amax, then every thread quantizes 4 consecutive channels at a
// time.  F16 = false writes codes (uint8), true the exact fp16 value of q.
template <bool F16>
__global__ void __launch_bounds__(256) quantize_a8_kernel(const uint16_t *__restrict__ x, int64_t M, int IC,
                                                          const __grid_constant__ PretransformShards p,
                                                          void *__restrict__ dst, float *__restrict__ As) {
    extern __shared__ __align__(16) float su[];   // [IC]
    __shared__ float s_amax[8];
    // wait for the preceding kernel, then let a dependent launch be scheduled (it
    // waits for this grid before reading; a reconstruct may run alongside)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t m = blockIdx.x;                 // row of dst and As
    const int sh = (int)(m / M);
    const uint16_t *s_in = p.s_in[sh], *rin = p.rin[sh];
    const int blocks = IC / kHad;
    const uint16_t *xr = x + (m - sh * M) * IC;
    float amax = 0.f;
    for (int b0 = warp; b0 < blocks; b0 += 8 * kQRun) {
        uint2 xv[kQRun], sv[kQRun], rv[kQRun];
#pragma unroll
        for (int k = 0; k < kQRun; k++) {
            const int b = b0 + 8 * k;
            if (b < blocks) {
                const int c0 = b * kHad + 4 * lane;
                xv[k] = *reinterpret_cast<const uint2 *>(xr + c0);
                sv[k] = __ldg(reinterpret_cast<const uint2 *>(s_in + c0));
                rv[k] = __ldg(reinterpret_cast<const uint2 *>(rin + c0));
            }
        }
#pragma unroll
        for (int k = 0; k < kQRun; k++) {
            const int b = b0 + 8 * k;
            if (b >= blocks) break;   // warp-uniform
            const uint32_t xs[2] = {xv[k].x, xv[k].y}, ss[2] = {sv[k].x, sv[k].y}, rs[2] = {rv[k].x, rv[k].y};
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int bs = 16 * (i & 1);
                v[i] = (bf16_bits_to_f32((xs[i >> 1] >> bs) & 0xFFFFu) * f16_bits_to_f32((uint16_t)(ss[i >> 1] >> bs))) *
                       f16_bits_to_f32((uint16_t)(rs[i >> 1] >> bs));
            }
            warp_fwht128(v, lane);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                v[i] *= kHadNorm;
                amax = fmaxf(amax, fabsf(v[i]));
            }
            *reinterpret_cast<float4 *>(su + b * kHad + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    if (lane == 0) s_amax[warp] = amax;
    __syncthreads();   // also publishes su
    amax = s_amax[0];
#pragma unroll
    for (int w = 1; w < 8; w++) amax = fmaxf(amax, s_amax[w]);
    const float s = amax / 127.f;
    if (threadIdx.x == 0) As[m] = s;
    for (int c = 4 * threadIdx.x; c < IC; c += 4 * 256) {
        const float4 v4 = *reinterpret_cast<const float4 *>(su + c);
        const float v[4] = {v4.x, v4.y, v4.z, v4.w};
        int q[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            q[i] = 0;
            if (s > 0.f) {
                q[i] = __float2int_rn(__fdiv_rn(v[i], s));   // round half to even
                q[i] = q[i] > 127 ? 127 : (q[i] < -127 ? -127 : q[i]);
            }
        }
        if constexpr (F16) {
            // |q| <= 127: exact in fp16
            uint2 o;
            o.x = (uint32_t)f32_to_f16_bits((float)q[0]) | ((uint32_t)f32_to_f16_bits((float)q[1]) << 16);
            o.y = (uint32_t)f32_to_f16_bits((float)q[2]) | ((uint32_t)f32_to_f16_bits((float)q[3]) << 16);
            *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(dst) + m * IC + c) = o;
        } else {
            const uint32_t w = (uint32_t)(q[0] + 128) | ((uint32_t)(q[1] + 128) << 8) |
                               ((uint32_t)(q[2] + 128) << 16) | ((uint32_t)(q[3] + 128) << 24);
            *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(dst) + m * IC + c) = w;
        }
    }
}

// 8 codes -> 8 exact fp16 values per thread.
__global__ void __launch_bounds__(256) codes_to_f16_kernel(const uint8_t *__restrict__ A, int64_t n8,
                                                           uint16_t *__restrict__ dst) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint2 c = __ldg(reinterpret_cast<const uint2 *>(A) + i);
        const uint32_t cw[2] = {c.x, c.y};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; h++) {
#pragma unroll
            for (int p = 0; p < 2; p++) {
                const float q0 = (float)(int)((cw[h] >> (16 * p)) & 0xFFu) - 128.f;
                const float q1 = (float)(int)((cw[h] >> (16 * p + 8)) & 0xFFu) - 128.f;
                o[2 * h + p] = (uint32_t)f32_to_f16_bits(q0) | ((uint32_t)f32_to_f16_bits(q1) << 16);
            }
        }
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

size_t quantize_a8_smem_bytes(int IC) { return (size_t)IC * sizeof(float); }

cudaError_t launch_quantize_a8(const uint16_t *x, int64_t M, int IC, const PretransformShards &p, void *dst,
                               bool f16_out, float *As, cudaStream_t s) {
    if (M <= 0 || IC <= 0 || IC % kHad || p.n < 1 || p.n > 4 || p.n * M > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = quantize_a8_smem_bytes(IC);
    const void *fn = f16_out ? (const void *)quantize_a8_kernel<true> : (const void *)quantize_a8_kernel<false>;
    cudaError_t e = kernel_smem_optin(fn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n * M));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (f16_out) return cudaLaunchKernelEx(&cfg, quantize_a8_kernel<true>, x, M, IC, p, dst, As);
    return cudaLaunchKernelEx(&cfg, quantize_a8_kernel<false>, x, M, IC, p, dst, As);
}

cudaError_t launch_codes_to_f16(const uint8_t *A, int64_t n, uint16_t *dst, cudaStream_t s) {
    if (n <= 0 || n % 8) return cudaErrorInvalidValue;
    const int64_t n8 = n / 8;
    int64_t grid = (n8 + 255) / 256;
    const int64_t cap = (int64_t)device_info().sm_count * 8;
    if (grid > cap) grid = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, codes_to_f16_kernel, A, n8, dst);
}

}  // namespace exl3
