// lm_head.cu -- the int8 table as the output projection (vllm-quantpack
// exl3/embedding.py, Exl3EmbeddingMethod.apply: the weight is the int8 table
// times its per-row scale and the head computes x @ weight^T):
//     out[m][v] = bf16( s[v] * sum_h x[m][h] * q[v][h] )
// with the row scale factored out of the sum and one rounding.
//
// Few rows (decode): the table is streamed once and converted in registers.
// A warp owns 16 vocabulary rows (one MMA's M) over the whole hidden width and
// takes such tiles from a counter in the workspace (one tile ahead, so its
// loads run on across tiles); a tile's result is computed by one warp alone, so
// the output does not depend on the schedule.  int8 converts to fp16 exactly
// (1024 + byte trick); the bf16 activations are converted to fp16 once per call
// (exact within fp16's normal range) and multiply as the
// m16n8k16 B operand (read from the workspace: small and cache-resident), fp32
// accumulation.  The last warp to finish resets the counters.
//
// Many rows (prefill): chunks of the table are converted to fp16 in the
// workspace and multiplied by the persistent tcgen05 GEMM with a row-scale
// epilogue (prefill.cu).
#include <cuda_runtime.h>

#include "../../include/exl3.h"
#include "common.cuh"
#include "internal.h"

namespace exl3 {
exl3_status fail(exl3_status st, const char *fmt, ...);
exl3_status cuda_fail(cudaError_t e, const char *where);
void trace(const char *fmt, ...);
size_t fixed_workspace_bytes();
int32_t *workspace_err(void *base);
int32_t *workspace_counters(void *base);

namespace {

constexpr int kLhWarps = 8;
constexpr int kLhStepCh = 64;     // channels per warp step (4 MMA K-slices)
constexpr int kLhPF = 4;          // steps of table bytes in flight per warp (H % (kLhPF * kLhStepCh) == 0)

// Four int8 weights (one little-endian word) -> two fp16x2 words (ch 0,1 | ch 2,3), exact.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;                       // b + 128 as an unsigned byte
    const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);   // fp16 1024 + u, two lanes
    const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 off = __half2half2(__ushort_as_half(0x6480));   // 1152
    const __half2 rl = __hsub2(*reinterpret_cast<const __half2 *>(&l), off);
    const __half2 rh = __hsub2(*reinterpret_cast<const __half2 *>(&h), off);
    lo = *reinterpret_cast<const uint32_t *>(&rl);
    hi = *reinterpret_cast<const uint32_t *>(&rh);
}

// The table is read once: its loads skip L1, which keeps the activations cached.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Row stride (halves) of the activation rows in shared memory: 16 bytes of
// padding put the rows of one warp access on different banks.
__host__ __device__ inline int lh_row_halves(int H) { return H + 8; }

// XS: the activations are copied to shared memory (when 8 * NB rows fit);
// otherwise they are read from the workspace through L1.
template <int NB, bool XS>
__global__ void __launch_bounds__(kLhWarps * 32, 2)
lm_head_decode_kernel(const uint16_t *__restrict__ x16, int M, int H, const int8_t *__restrict__ q,
                      const uint16_t *__restrict__ scale, int64_t V, uint16_t *__restrict__ out, int64_t ldo,
                      int32_t *ctr) {
    extern __shared__ __align__(16) uint16_t sx[];   // XS: fp16 [8 * NB][H + 8]
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, qd = lane & 3;
    const int RS = lh_row_halves(H);
    // x16 (fp16 [M][H], converted by the preceding kernel) and the counters
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (XS) {
        for (int i = threadIdx.x; i < 8 * NB * (H / 8); i += blockDim.x) {
            const int n = i / (H / 8), c = (i - n * (H / 8)) * 8;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n < M) v = *reinterpret_cast<const uint4 *>(x16 + (int64_t)n * H + c);
            *reinterpret_cast<uint4 *>(sx + n * RS + c) = v;
        }
        __syncthreads();
    }
    const int64_t ntiles = (V + 15) / 16;
    const int steps = H / kLhStepCh;
    auto grab = [&]() -> int64_t {
        int64_t t = 0;
        if (lane == 0) t = atomicAdd(ctr, 1);
        return __shfl_sync(kFull, t, 0);
    };
    // table rows of a tile for this lane (rows g and g + 8, clamped to the table)
    auto rows_of = [&](int64_t t, const int8_t *&r0, const int8_t *&r1) {
        int64_t v0 = 16 * t + g, v1 = v0 + 8;
        if (v0 >= V) v0 = V - 1;
        if (v1 >= V) v1 = V - 1;
        r0 = q + v0 * H + 16 * qd;
        r1 = q + v1 * H + 16 * qd;
    };
    int64_t tile = grab();
    int64_t next = tile < ntiles ? grab() : ntiles;
    // the stream of (tile, step) loads, kLhPF steps ahead
    uint4 qa[kLhPF], qb[kLhPF];
    int64_t lt = tile;   // tile and step of the next load
    int ls = 0;
    const int8_t *lr0 = nullptr, *lr1 = nullptr;
    if (lt < ntiles) rows_of(lt, lr0, lr1);
    auto issue = [&](int slot) {
        if (lt >= ntiles) return;
        qa[slot] = ld_stream(lr0 + ls * kLhStepCh);
        qb[slot] = ld_stream(lr1 + ls * kLhStepCh);
        if (++ls == steps) {
            ls = 0;
            lt = next;
            if (lt < ntiles) rows_of(lt, lr0, lr1);
        }
    };
#pragma unroll
    for (int d = 0; d < kLhPF; d++) issue(d);
    while (tile < ntiles) {
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; nb++)
#pragma unroll
            for (int r = 0; r < 4; r++) acc[nb][r] = 0.f;
        // steps in groups of kLhPF, so every ring slot index is known at compile time
        // (steps is a multiple of kLhPF: step s of any tile sits in slot s % kLhPF)
        for (int s0 = 0; s0 < steps; s0 += kLhPF) {
#pragma unroll
            for (int d = 0; d < kLhPF; d++) {
                const uint32_t wa[4] = {qa[d].x, qa[d].y, qa[d].z, qa[d].w};
                const uint32_t wb[4] = {qb[d].x, qb[d].y, qb[d].z, qb[d].w};
                // refill this slot with the load kLhPF steps ahead (it crosses into the
                // next tile, already taken, near the end of this one)
                issue(d);
                const int ch = (s0 + d) * kLhStepCh + 16 * qd;
#pragma unroll
                for (int nb = 0; nb < NB; nb++) {
                    // activations of token 8 nb + g (zeros past M): small, cache-resident
                    uint4 xv0 = make_uint4(0u, 0u, 0u, 0u), xv1 = xv0;
                    if constexpr (XS) {
                        xv0 = *reinterpret_cast<const uint4 *>(sx + (8 * nb + g) * RS + ch);
                        xv1 = *reinterpret_cast<const uint4 *>(sx + (8 * nb + g) * RS + ch + 8);
                    } else if (8 * nb + g < M) {
                        xv0 = __ldg(reinterpret_cast<const uint4 *>(x16 + (int64_t)(8 * nb + g) * H + ch));
                        xv1 = __ldg(reinterpret_cast<const uint4 *>(x16 + (int64_t)(8 * nb + g) * H + ch + 8));
                    }
                    const uint32_t xw[8] = {xv0.x, xv0.y, xv0.z, xv0.w, xv1.x, xv1.y, xv1.z, xv1.w};
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        uint32_t a0, a2, a1, a3;
                        i8x4_to_f16(wa[j], a0, a2);
                        i8x4_to_f16(wb[j], a1, a3);
                        mma_16816(acc[nb], a0, a1, a2, a3, xw[2 * j], xw[2 * j + 1]);
                    }
                }
            }
        }
        // epilogue: rows v = 16 tile + g (+ 8), tokens n = 8 nb + 2 qd (+ 1)
        const int64_t va = 16 * tile + g, vb = va + 8;
        const float sa = va < V ? f16_bits_to_f32(scale[va]) : 0.f;
        const float sb = vb < V ? f16_bits_to_f32(scale[vb]) : 0.f;
#pragma unroll
        for (int nb = 0; nb < NB; nb++) {
            const int n0 = 8 * nb + 2 * qd;
            if (n0 < M) {
                if (va < V) out[(int64_t)n0 * ldo + va] = f32_to_bf16_bits(acc[nb][0] * sa);
                if (vb < V) out[(int64_t)n0 * ldo + vb] = f32_to_bf16_bits(acc[nb][2] * sb);
            }
            if (n0 + 1 < M) {
                if (va < V) out[(int64_t)(n0 + 1) * ldo + va] = f32_to_bf16_bits(acc[nb][1] * sa);
                if (vb < V) out[(int64_t)(n0 + 1) * ldo + vb] = f32_to_bf16_bits(acc[nb][3] * sb);
            }
        }
        tile = next;
        if (tile < ntiles) next = grab();
    }
    // the last warp of the grid to finish resets the counters for the next call
    if (lane == 0) {
        const int total = gridDim.x * kLhWarps;
        if (atomicAdd(ctr + 1, 1) == total - 1) {
            ctr[0] = 0;
            ctr[1] = 0;
        }
    }
}

__global__ void i8_to_f16_kernel(const int8_t *__restrict__ q, int64_t n16, uint16_t *__restrict__ dst) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(q) + i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; k++) i8x4_to_f16(ws[k], o[2 * k], o[2 * k + 1]);
        reinterpret_cast<uint4 *>(dst)[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<uint4 *>(dst)[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

__global__ void bf16_to_f16_kernel(const uint16_t *__restrict__ x, int64_t n8, uint16_t *__restrict__ dst) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = *(reinterpret_cast<const uint4 *>(x) + i);
        const uint32_t vs[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; k++)
            o[k] = (uint32_t)f32_to_f16_bits(bf16_bits_to_f32(vs[k] & 0xFFFFu)) |
                   ((uint32_t)f32_to_f16_bits(bf16_bits_to_f32(vs[k] >> 16)) << 16);
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_i8_to_f16(const int8_t *q, int64_t n, uint16_t *dst, cudaStream_t s) {
    if (n % 16) return cudaErrorInvalidValue;
    const int64_t n16 = n / 16;
    int64_t grid = (n16 + 255) / 256;
    if (grid > 8 * (int64_t)device_info().sm_count) grid = 8 * (int64_t)device_info().sm_count;
    i8_to_f16_kernel<<<(unsigned)grid, 256, 0, s>>>(q, n16, dst);
    return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(const uint16_t *x, int64_t n, uint16_t *dst, cudaStream_t s) {
    if (n % 8) return cudaErrorInvalidValue;
    const int64_t n8 = n / 8;
    int64_t grid = (n8 + 255) / 256;
    if (grid > 8 * (int64_t)device_info().sm_count) grid = 8 * (int64_t)device_info().sm_count;
    bf16_to_f16_kernel<<<(unsigned)grid, 256, 0, s>>>(x, n8, dst);
    return cudaGetLastError();
}

cudaError_t launch_lm_head_decode(const uint16_t *x16, int M, int H, const int8_t *q, const uint16_t *scale, int64_t V,
                                  uint16_t *out, int64_t ldo, int32_t *ctr, cudaStream_t s) {
    const int nb = (M + 7) / 8;
    // the load stream runs kLhPF steps ahead, in whole groups of kLhPF steps
    if (nb < 1 || nb > 4 || H % (kLhPF * kLhStepCh)) return cudaErrorInvalidValue;
    const int nbk = nb == 3 ? 4 : nb;
    // activations in shared memory when two CTAs per SM still fit
    const size_t xs_bytes = sizeof(uint16_t) * 8 * nbk * lh_row_halves(H);
    const bool xs = xs_bytes <= 100 * 1024;
    const size_t smem = xs ? xs_bytes : 0;
    const void *fn = xs ? (nbk == 1 ? (const void *)lm_head_decode_kernel<1, true>
                                    : nbk == 2 ? (const void *)lm_head_decode_kernel<2, true>
                                               : (const void *)lm_head_decode_kernel<4, true>)
                        : (nbk == 1 ? (const void *)lm_head_decode_kernel<1, false>
                                    : nbk == 2 ? (const void *)lm_head_decode_kernel<2, false>
                                               : (const void *)lm_head_decode_kernel<4, false>);
    int occ = 1;
    cudaError_t e = kernel_occupancy(fn, kLhWarps * 32, smem, &occ);
    if (e != cudaSuccess) return e;
    int64_t grid = (int64_t)device_info().sm_count * occ;
    const int64_t ntiles = (V + 15) / 16;
    if (grid * kLhWarps > ntiles) grid = (ntiles + kLhWarps - 1) / kLhWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kLhWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {(void *)&x16, (void *)&M, (void *)&H, (void *)&q, (void *)&scale, (void *)&V, (void *)&out,
                    (void *)&ldo, (void *)&ctr};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace exl3

// ------------------------------------------------------------------ C ABI
namespace exl3 {
namespace {

constexpr int64_t kLhDecodeMaxRows = 32;    // rows one streaming pass serves (4 blocks of 8)
constexpr int64_t kLhChunkRows = 16384;     // table rows converted per tensor-core pass

inline size_t lh_align256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace: fixed header (error word, counters) | fp16 x [M][H] | fp16 table chunk
// [kLhChunkRows][H] (the chunk only when some M > kLhDecodeMaxRows takes the
// tensor-core path).
size_t lh_layout(int64_t max_M, int32_t H, int64_t V, size_t *x16_off, size_t *chunk_off) {
    size_t off = fixed_workspace_bytes();
    *x16_off = off;
    off = lh_align256(off + sizeof(uint16_t) * (size_t)max_M * H);
    *chunk_off = 0;
    if (max_M > kLhDecodeMaxRows && prefill_supported()) {
        *chunk_off = off;
        const int64_t rows = V < kLhChunkRows ? V : kLhChunkRows;
        off = lh_align256(off + sizeof(uint16_t) * (size_t)rows * H);
    }
    return off;
}

}  // namespace
}  // namespace exl3

using namespace exl3;

extern "C" {

size_t exl3_lm_head_workspace_bytes(int64_t max_M, int32_t H, int64_t V) {
    if (max_M < 0 || H <= 0 || H % 256 || V <= 0) return 0;
    size_t a, b;
    return lh_layout(max_M, H, V, &a, &b);
}

exl3_status exl3_lm_head_int8(const uint16_t *x, int64_t M, int32_t H, const int8_t *q, const uint16_t *scale,
                              int64_t V, uint16_t *out, int64_t ldo, void *ws, size_t ws_bytes, exl3_stream stream) {
    const char *fn = "lm_head_int8";
    if (M < 0 || H <= 0 || H % 256 || V <= 0 || V > ((int64_t)1 << 31) * 16 - 16)
        return fail(EXL3_EINVAL, "%s: M = %lld, H = %d (a positive multiple of 256), V = %lld", fn, (long long)M, H,
                    (long long)V);
    if (ldo < V) return fail(EXL3_EINVAL, "%s: ldo = %lld < V = %lld", fn, (long long)ldo, (long long)V);
    if (M == 0) return EXL3_OK;
    if (!x || !q || !scale || !out) return fail(EXL3_EINVAL, "%s: null pointer", fn);
    if (((uintptr_t)x | (uintptr_t)q) & 15u)
        return fail(EXL3_EINVAL, "%s: x (%p) and q (%p) must be 16-byte aligned", fn, x, q);
    if ((uintptr_t)scale & 1u || (uintptr_t)out & 1u) return fail(EXL3_EINVAL, "%s: misaligned scale or out", fn);
    size_t x16_off, chunk_off;
    const size_t need = lh_layout(M, H, V, &x16_off, &chunk_off);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < need)
        return fail(EXL3_EWORKSPACE, "%s: workspace %p of %zu bytes; this call needs %zu bytes, 256-byte aligned", fn,
                    ws, ws_bytes, need);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    char *b = static_cast<char *>(ws);
    uint16_t *x16 = reinterpret_cast<uint16_t *>(b + x16_off);
    // the activations as fp16, once (exact within fp16's normal range)
    if ((e = launch_bf16_to_f16(x, M * H, x16, s)) != cudaSuccess) return cuda_fail(e, fn);
    if (M <= kLhDecodeMaxRows || !prefill_supported()) {
        // streaming passes of up to 32 rows; the table is read once per pass
        for (int64_t r0 = 0; r0 < M; r0 += kLhDecodeMaxRows) {
            const int rows = (int)(M - r0 < kLhDecodeMaxRows ? M - r0 : kLhDecodeMaxRows);
            e = launch_lm_head_decode(x16 + r0 * H, rows, H, q, scale, V, out + r0 * ldo, ldo, workspace_counters(ws),
                                      s);
            if (e != cudaSuccess) return cuda_fail(e, fn);
        }
        trace("%s M=%lld H=%d V=%lld streaming", fn, (long long)M, H, (long long)V);
        return EXL3_OK;
    }
    // tensor cores: the table in chunks converted to fp16
    uint16_t *w16 = reinterpret_cast<uint16_t *>(b + chunk_off);
    for (int64_t v0 = 0; v0 < V; v0 += kLhChunkRows) {
        const int64_t nv = V - v0 < kLhChunkRows ? V - v0 : kLhChunkRows;
        if ((e = launch_i8_to_f16(q + v0 * H, nv * H, w16, s)) != cudaSuccess) return cuda_fail(e, fn);
        bool launched = false;
        e = launch_prefill(x16, w16, M, H, (int)nv, scale + v0, nullptr, out + v0, ldo, workspace_err(ws), s, &launched,
                           1);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        if (!launched) return fail(EXL3_EUNSUPPORTED, "%s: tensor-core path unavailable", fn);
    }
    trace("%s M=%lld H=%d V=%lld tensor cores", fn, (long long)M, H, (long long)V);
    return EXL3_OK;
}

}  // extern "C"
