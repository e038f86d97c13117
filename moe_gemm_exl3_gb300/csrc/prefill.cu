// prefill.cu -- large-M (prefill) path of the EXL3 linear on the 5th-generation
// tensor cores: y = (Had128(u @ W) * rout) * s_out for u fp16 [M][IC] and the
// decoded weights W^T fp16 [OC][IC] (K-major), in 128 x 256 output tiles
// accumulated in tensor memory by a persistent grid (one CTA per SM).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: u and W^T tiles (64-element K slices, 128-byte
//               swizzle) into a 4-stage shared-memory ring
//   warp 1      TMEM allocation; one elected lane issues tcgen05.mma
//               (M=128, N=256, K=16, fp16 in, fp32 accumulate)
//   warps 2..5  epilogue: tcgen05.ld of one row per thread, in-register
//               128-point Hadamard, rout then s_out, bf16 stores into the slice
// Every mbarrier wait is bounded: on timeout the kernel records an error in the
// workspace error word, drains what it issued (again bounded), frees its tensor
// memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace exl3 {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;                 // 16 KB
constexpr int B_BYTES = BN * BK * 2;                 // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /* alignment */ + 256 /* barriers */;
constexpr uint32_t kIdesc = make_idesc_f16(BM, BN);

// ------------------------------------------------------------ kernel
// Tile order: groups of kGroupN column tiles; within a group the column tile
// varies fastest, then the row tile, so the CTAs running at one time share a
// few activation and weight panels in L2.
constexpr int kGroupN = 16;

__device__ __forceinline__ void tile_coords(int t, int MT, int NT, int &mt, int &nt) {
    const int per_group = kGroupN * MT;
    const int g = t / per_group;
    const int r = t % per_group;
    const int gsize = NT - g * kGroupN < kGroupN ? NT - g * kGroupN : kGroupN;
    nt = g * kGroupN + r % gsize;
    mt = r / gsize;
}

// Persistent: one CTA per SM walks tiles blockIdx.x, + gridDim.x, ...  Two TMEM
// accumulators (2 x 256 columns) let the epilogue of one tile overlap the MMAs of
// the next.  EPI 0: y = (Had128(v) * rout) * s_out (the EXL3 output transform);
// EPI 1: y = v * rout per column (the int8 output head's row scale; s_out unused).
template <int EPI>
__global__ void __launch_bounds__(192, 1)
prefill_gemm_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_w,
                    int M, int IC, int OC, const uint16_t *__restrict__ rout, const uint16_t *__restrict__ s_out,
                    uint16_t *__restrict__ out, int64_t ldo, int32_t *err, const float *__restrict__ row_scale) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *sbase = smem_raw + (base - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + STAGES * STAGE_BYTES);
    // bars[0..S) full, [S..2S) empty, [2S..2S+2) accumulator full, [2S+2..2S+4) accumulator empty, [2S+4] MMA done
    uint64_t *acc_full = bars + 2 * STAGES, *acc_empty = bars + 2 * STAGES + 2, *mma_done = bars + 2 * STAGES + 4;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_issued = const_cast<int *>(reinterpret_cast<volatile int *>(s_tmem + 2));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = IC / BK;
    const int MT = (M + BM - 1) / BM, NT = (OC + BN - 1) / BN;
    const int ntiles = MT * NT;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; i++) {
            mbar_init(smem_u32(&bars[i]), 1);
            mbar_init(smem_u32(&bars[STAGES + i]), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);     // one arrival per epilogue warp
        }
        mbar_init(smem_u32(mma_done), 1);
        *s_abort = 0;
        *s_issued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                     "r"(2 * TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: every k-slice of every tile of this CTA
        int g = 0;   // global k-slice counter of this CTA
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            int mt, nt;
            tile_coords(t, MT, NT, mt, nt);
            for (int kb = 0; kb < nk; kb++, g++) {
                const int s = g % STAGES;
                const uint32_t ph = (g / STAGES) & 1;
                if (!mbar_wait(smem_u32(&bars[STAGES + s]), ph ^ 1, err, s_abort)) { ok = false; break; }
                const uint32_t full = smem_u32(&bars[s]);
                mbar_expect_tx(full, STAGE_BYTES);
                const uint32_t sa = base + s * STAGE_BYTES;
                tma_load_2d(sa, &tm_u, kb * BK, mt * BM, full);
                tma_load_2d(sa + A_BYTES, &tm_w, kb * BK, nt * BN, full);
            }
        }
        *s_issued = g;
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        int g = 0, i = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, i++) {
            const int b = i & 1;
            if (!mbar_wait(smem_u32(&acc_empty[b]), ((i >> 1) & 1) ^ 1, err, s_abort)) break;
            tc_fence_after();
            const uint32_t acc = tmem + b * TMEM_COLS;
            for (int kb = 0; kb < nk; kb++, g++) {
                const int s = g % STAGES;
                const uint32_t ph = (g / STAGES) & 1;
                if (!mbar_wait(smem_u32(&bars[s]), ph, err, s_abort)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = base + s * STAGE_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; k++) {
                    const uint64_t da = smem_desc_sw128(sa + k * 32);
                    const uint64_t db = smem_desc_sw128(sa + A_BYTES + k * 32);
                    umma_f16(acc, da, db, kIdesc, (kb | k) != 0);
                }
                umma_commit(smem_u32(&bars[STAGES + s]));   // frees the stage when these MMAs finish
            }
            if (ok) umma_commit(smem_u32(&acc_full[b]));   // this tile's accumulator is complete
        }
        umma_commit(smem_u32(mma_done));                   // every MMA this thread issued has finished
        mbar_drain(smem_u32(mma_done), 0);                 // even after an abort: TMEM is freed below
    } else if (warp >= 2) {
        // ---------------- epilogue: one output row per thread
        const int quarter = warp & 3;                    // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, i++) {
            int mt, nt;
            tile_coords(t, MT, NT, mt, nt);
            const int b = i & 1;
            if (!mbar_wait(smem_u32(&acc_full[b]), (i >> 1) & 1, err, s_abort)) break;
            tc_fence_after();
            const int m = mt * BM + row;
            for (int h = 0; h < BN / kHad; h++) {
                const int col = nt * BN + h * kHad;
                if (col >= OC) break;
                float v[128];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    float tt[32];
                    tmem_ld32(tmem + b * TMEM_COLS + ((uint32_t)(quarter * 32) << 16) + h * kHad + c * 32, tt);
#pragma unroll
                    for (int q = 0; q < 32; q++) v[c * 32 + q] = tt[q];
                }
                tmem_ld_wait();
                if (m >= M) continue;
                uint16_t *dst = out + (int64_t)m * ldo + col;
                // the Hadamard scale, times the row's activation scale when there is one
                const float hn = row_scale ? kHadNorm * __ldg(row_scale + m) : kHadNorm;
                if constexpr (EPI == 1) {
                    // per-column scale, no transform; a partial last block stores its columns one by one
                    const int ncol = OC - col < kHad ? OC - col : kHad;
                    if (ncol == kHad && ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(rout + col)) & 15u) == 0) {
#pragma unroll
                        for (int c8 = 0; c8 < 16; c8++) {
                            const uint4 sc = __ldg(reinterpret_cast<const uint4 *>(rout + col) + c8);
                            const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
                            uint32_t o[4];
#pragma unroll
                            for (int qq = 0; qq < 4; qq++) {
                                const int c = c8 * 8 + 2 * qq;
                                const float y0 = v[c] * f16_bits_to_f32((uint16_t)(sw[qq] & 0xFFFFu));
                                const float y1 = v[c + 1] * f16_bits_to_f32((uint16_t)(sw[qq] >> 16));
                                o[qq] = (uint32_t)f32_to_bf16_bits(y0) | ((uint32_t)f32_to_bf16_bits(y1) << 16);
                            }
                            reinterpret_cast<uint4 *>(dst)[c8] = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < kHad; c++)
                            if (c < ncol) dst[c] = f32_to_bf16_bits(v[c] * f16_bits_to_f32(__ldg(rout + col + c)));
                    }
                    continue;
                }
#pragma unroll
                for (int hs = 1; hs < 128; hs <<= 1) {
#pragma unroll
                    for (int q = 0; q < 128; q++) {
                        if (q & hs) continue;
                        const float a = v[q], c2 = v[q + hs];
                        v[q] = a + c2;
                        v[q + hs] = a - c2;
                    }
                }
#pragma unroll
                for (int c8 = 0; c8 < 16; c8++) {
                    // scale vectors are only 8-byte aligned
                    const uint2 r0 = __ldg(reinterpret_cast<const uint2 *>(rout + col) + 2 * c8);
                    const uint2 r1 = __ldg(reinterpret_cast<const uint2 *>(rout + col) + 2 * c8 + 1);
                    const uint2 q0 = __ldg(reinterpret_cast<const uint2 *>(s_out + col) + 2 * c8);
                    const uint2 q1 = __ldg(reinterpret_cast<const uint2 *>(s_out + col) + 2 * c8 + 1);
                    const uint32_t rw[4] = {r0.x, r0.y, r1.x, r1.y}, sw[4] = {q0.x, q0.y, q1.x, q1.y};
                    uint32_t o[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int c = c8 * 8 + 2 * q;
                        float y0 = (v[c] * hn) * f16_bits_to_f32((uint16_t)(rw[q] & 0xFFFFu));
                        float y1 = (v[c + 1] * hn) * f16_bits_to_f32((uint16_t)(rw[q] >> 16));
                        y0 *= f16_bits_to_f32((uint16_t)(sw[q] & 0xFFFFu));
                        y1 *= f16_bits_to_f32((uint16_t)(sw[q] >> 16));
                        o[q] = (uint32_t)f32_to_bf16_bits(y0) | ((uint32_t)f32_to_bf16_bits(y1) << 16);
                    }
                    reinterpret_cast<uint4 *>(dst)[c8] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            // the accumulator buffer may be overwritten by the tile after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&acc_empty[b])) : "memory");
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && *s_abort) {
        // drain: wait (bounded) for the copies this CTA issued into stages nobody consumed
        const int issued = *s_issued;
        for (int g = issued - STAGES > 0 ? issued - STAGES : 0; g < issued; g++) {
            mbar_drain(smem_u32(&bars[g % STAGES]), (g / STAGES) & 1);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * TMEM_COLS));
    }
}

}  // namespace

bool prefill_supported() { return tma_encode_available(); }

cudaError_t launch_prefill(const uint16_t *u, const uint16_t *wt, int64_t M, int IC, int OC, const uint16_t *rout,
                           const uint16_t *s_out, uint16_t *out, int64_t ldo, int32_t *err, cudaStream_t s,
                           bool *launched, int epi, const float *row_scale) {
    *launched = false;
    if (M <= 0 || IC % BK || (epi == 0 && OC % kHad) || M > INT32_MAX || (epi != 0 && row_scale))
        return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(wt)) & 15u) return cudaErrorInvalidValue;
    CUtensorMap tm_u, tm_w;
    if (!make_map_f16(&tm_u, u, M, IC, BM) || !make_map_f16(&tm_w, wt, OC, IC, BN)) return cudaErrorInvalidValue;
    const void *fn = epi == 0 ? (const void *)prefill_gemm_kernel<0> : (const void *)prefill_gemm_kernel<1>;
    cudaError_t ea = kernel_smem_optin(fn, SMEM_BYTES);
    if (ea != cudaSuccess) return ea;
    const int64_t tiles = ((M + BM - 1) / BM) * (int64_t)((OC + BN - 1) / BN);
    int64_t grid = device_info().sm_count;   // persistent: one CTA per SM
    if (grid > tiles) grid = tiles;
    if (epi == 0)
        prefill_gemm_kernel<0><<<(unsigned)grid, 192, SMEM_BYTES, s>>>(tm_u, tm_w, (int)M, IC, OC, rout, s_out, out,
                                                                       ldo, err, row_scale);
    else
        prefill_gemm_kernel<1><<<(unsigned)grid, 192, SMEM_BYTES, s>>>(tm_u, tm_w, (int)M, IC, OC, rout, s_out, out,
                                                                       ldo, err, nullptr);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace exl3
