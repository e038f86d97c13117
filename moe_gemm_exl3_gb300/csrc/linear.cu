// linear.cu -- EXL3 linear: activation pre-transform, trellis reconstruct,
// codebook table and the decode-mode (small M) fused trellis GEMM.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace exl3 {

// --------------------------------------------------------------------------
// Activation pre-transform: u = Had128((x * s_in) * rin) per 128-channel
// block (radiance_escha.py, module docstring "THE FORWARD", first factor).
// One warp per (row, block); lane l holds channels 4l..4l+3 of the block.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pretransform_kernel(const uint16_t *__restrict__ x,
                                                           int64_t M, int IC,
                                                           const uint16_t *__restrict__ s_in,
                                                           const uint16_t *__restrict__ rin,
                                                           uint16_t *__restrict__ u) {
    const int lane = threadIdx.x & 31;
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int blocks = IC / kHad;
    if (wid >= M * blocks) return;
    const int64_t m = wid / blocks;
    const int c0 = (int)(wid % blocks) * kHad + 4 * lane;
    const uint2 xv = *reinterpret_cast<const uint2 *>(x + m * IC + c0);
    const uint2 sv = __ldg(reinterpret_cast<const uint2 *>(s_in + c0));
    const uint2 rv = __ldg(reinterpret_cast<const uint2 *>(rin + c0));
    const uint32_t xs[2] = {xv.x, xv.y}, ss[2] = {sv.x, sv.y}, rs[2] = {rv.x, rv.y};
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t xb = (xs[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
        const float s = f16_bits_to_f32((uint16_t)(ss[i >> 1] >> (16 * (i & 1))));
        const float r = f16_bits_to_f32((uint16_t)(rs[i >> 1] >> (16 * (i & 1))));
        v[i] = (bf16_bits_to_f32(xb) * s) * r;
    }
    warp_fwht128(v, lane);
    uint2 o;
    o.x = (uint32_t)f32_to_f16_bits(v[0] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[1] * kHadNorm) << 16);
    o.y = (uint32_t)f32_to_f16_bits(v[2] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[3] * kHadNorm) << 16);
    *reinterpret_cast<uint2 *>(u + m * IC + c0) = o;
}

cudaError_t launch_pretransform(const uint16_t *x, int64_t M, int IC, const uint16_t *s_in,
                                const uint16_t *rin, uint16_t *u, cudaStream_t s) {
    const int64_t warps = M * (IC / kHad);
    const int64_t grid = (warps + 7) / 8;
    pretransform_kernel<<<(unsigned)grid, 256, 0, s>>>(x, M, IC, s_in, rin, u);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------
// Reconstruct: decode every tile to dense fp16.  One thread per tile quarter
// (4 rows x 16 columns); the 4 quarters of a tile sit in 4 consecutive lanes.
// transposed = false: W [IC][OC]; true: W^T [OC][IC] (K-major operand).
// --------------------------------------------------------------------------
template <int K>
__global__ void __launch_bounds__(256) reconstruct_kernel(const int16_t *__restrict__ code,
                                                          int IC, int OC,
                                                          uint16_t *__restrict__ W,
                                                          bool transposed) {
    const int lane = threadIdx.x & 31;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int TO = OC / kTile;
    const int64_t quarters = (int64_t)(IC / kTile) * TO * 4;
    const bool active = tid < quarters;
    const int64_t qid = active ? tid : (tid & 3);   // idle lanes still join the shuffle
    const int q = (int)(qid & 3);
    const int64_t tile = qid >> 2;
    const int a = (int)(tile / TO), b = (int)(tile % TO);
    uint32_t w[2 * K];
    load_quarter<K>(w, reinterpret_cast<const uint32_t *>(code + tile * 16 * K) + q * 2 * K);
    QuarterStream<K> st;
    st.build(w, quarter_prev_word(w[2 * K - 1], lane));
    if (!active) return;
    if (!transposed) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            uint32_t pk[8];
#pragma unroll
            for (int c = 0; c < 16; c += 2)
                pk[c / 2] = trellis_weight_pair(trellis_hash(st.state(16 * r + c)),
                                                trellis_hash(st.state(16 * r + c + 1)));
            uint4 *dst = reinterpret_cast<uint4 *>(W + (int64_t)(16 * a + 4 * q + r) * OC + 16 * b);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 16; c++) {
            uint32_t p0 = trellis_weight_pair(trellis_hash(st.state(c)), trellis_hash(st.state(16 + c)));
            uint32_t p1 = trellis_weight_pair(trellis_hash(st.state(32 + c)), trellis_hash(st.state(48 + c)));
            *reinterpret_cast<uint2 *>(W + (int64_t)(16 * b + c) * IC + 16 * a + 4 * q) = make_uint2(p0, p1);
        }
    }
}

cudaError_t launch_reconstruct(const int16_t *code, int IC, int OC, int K, uint16_t *W,
                               bool transposed, cudaStream_t s) {
    const int64_t quarters = (int64_t)(IC / kTile) * (OC / kTile) * 4;
    const unsigned grid = (unsigned)((quarters + 255) / 256);
    switch (K) {
        case 2: reconstruct_kernel<2><<<grid, 256, 0, s>>>(code, IC, OC, W, transposed); break;
        case 3: reconstruct_kernel<3><<<grid, 256, 0, s>>>(code, IC, OC, W, transposed); break;
        case 4: reconstruct_kernel<4><<<grid, 256, 0, s>>>(code, IC, OC, W, transposed); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

__global__ void codebook_table_kernel(uint16_t *table) {
    const uint32_t s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s < 65536u) table[s] = __half_as_ushort(trellis_weight(trellis_hash(s)));
}

cudaError_t launch_codebook_table(uint16_t *table, cudaStream_t s) {
    codebook_table_kernel<<<256, 256, 0, s>>>(table);
    return cudaGetLastError();
}

// --------------------------------------------------------------------------
// Decode-mode fused trellis GEMM (M <= 32 rows per pass).
//
// v = u @ W with W decoded on the fly from the code words, then the epilogue
// y = (Had128(v) * rout) * s_out written as bf16 into the caller's columns.
//
// Mapping.  A warp owns one column group G (8 tiles = 128 output columns) and
// one tile row a (16 input channels) per step.  Lane (g, q) = (lane/4, lane%4)
// loads quarter q (tile rows 4q..4q+3) of tile (a, 8G + g): the warp's 8 tiles
// are contiguous in memory, so one step is one coalesced 512-byte (K=2) read.
// The decoded weights go straight into the A operand of m16n8k16 MMAs with the
// roles swapped (A = W^T: output columns on the MMA's M, tokens on its N):
// A row g <-> column 16(8G+g)+2j, row g+8 <-> the next column, and each A
// register holds the two fp16 halves (lo, hi) of one weight's codebook sum
// against a B register holding the same activation twice, so the tensor core
// forms u*(lo+hi) and no per-weight add is issued on the ALUs.
//
// Split-K.  The (G, a) units are split evenly over a persistent grid; a CTA's
// range covers parts of one or two column groups.  Warps reduce through shared
// memory in fixed order; CTAs sharing a group write their partial to a slab
// slot and bump the group's counter; the last to arrive sums the partials in
// CTA order (deterministic), runs the epilogue and resets the counter.  No CTA
// waits on another (radiance_escha.py: split-K partial slab + block counter).
// --------------------------------------------------------------------------
template <int NB>
struct DecodeSmem {
    float red[8 * NB * 4 * 32];   // CTA partial in MMA fragment order
    int last;
};

// Fragment-order index of (token n, group-local column oc).
template <int NB>
__device__ __forceinline__ int frag_index(int n, int oc) {
    const int g = oc >> 4, j = (oc & 15) >> 1, rrow = oc & 1;
    const int nb = n >> 3, q = (n & 7) >> 1, c = n & 1;
    return ((j * NB + nb) * 4 + (2 * rrow + c)) * 32 + (4 * g + q);
}

template <int K, int NB>
__global__ void __launch_bounds__(256) decode_gemm_kernel(const DecodeGemmArgs a) {
    __shared__ DecodeSmem<NB> sm;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int A = a.IC / kTile;
    const int NG = a.OC / kHad;
    const int TO = a.OC / kTile;
    const int64_t total = (int64_t)NG * A;
    const int nCTA = gridDim.x, c = blockIdx.x;
    int64_t f = (int64_t)c * total / nCTA;
    const int64_t f_end = (int64_t)(c + 1) * total / nCTA;
    constexpr int FRAG = 8 * NB * 4 * 32;

    while (f < f_end) {
        const int G = (int)(f / A);
        const int a_lo = (int)(f % A);
        const int a_hi = (int)((int64_t)A < a_lo + (f_end - f) ? (int64_t)A : a_lo + (f_end - f));

        float acc[8][NB][4];
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int nb = 0; nb < NB; nb++)
#pragma unroll
                for (int r = 0; r < 4; r++) acc[j][nb][r] = 0.f;

        const uint32_t *tile0 = reinterpret_cast<const uint32_t *>(a.code) +
                                ((int64_t)(8 * G + g) * 16 * K) / 2 + q * 2 * K;
        const int64_t row_words = (int64_t)TO * 8 * K;   // uint32 words per tile row
        int ar = a_lo + warp;
        uint32_t w[2 * K];
        if (ar < a_hi) load_quarter<K>(w, tile0 + ar * row_words);
        for (; ar < a_hi; ar += kDecodeWarps) {
            uint32_t wn[2 * K];
            const int an = ar + kDecodeWarps;
            if (an < a_hi) load_quarter<K>(wn, tile0 + an * row_words);

            // activations for k = 16a + 4q + 0..3, each duplicated into a half2
            uint32_t b[NB][4];
#pragma unroll
            for (int nb = 0; nb < NB; nb++) {
                const int n = 8 * nb + g;
                uint2 v = make_uint2(0u, 0u);
                if (n < a.M)
                    v = __ldg(reinterpret_cast<const uint2 *>(a.u + (int64_t)n * a.IC + 16 * ar + 4 * q));
                b[nb][0] = dup_half_lo(v.x);
                b[nb][1] = dup_half_hi(v.x);
                b[nb][2] = dup_half_lo(v.y);
                b[nb][3] = dup_half_hi(v.y);
            }

            QuarterStream<K> st;
            st.build(w, quarter_prev_word(w[2 * K - 1], lane));
#pragma unroll
            for (int rp = 0; rp < 2; rp++) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int i0 = 32 * rp + 2 * j;
                    const uint32_t z0 = trellis_hash(st.state(i0));
                    const uint32_t z1 = trellis_hash(st.state(i0 + 1));
                    const uint32_t z2 = trellis_hash(st.state(i0 + 16));
                    const uint32_t z3 = trellis_hash(st.state(i0 + 17));
#pragma unroll
                    for (int nb = 0; nb < NB; nb++)
                        mma_16816(acc[j][nb], z0, z1, z2, z3, b[nb][2 * rp], b[nb][2 * rp + 1]);
                }
            }
#pragma unroll
            for (int i = 0; i < 2 * K; i++) w[i] = wn[i];
        }

        // ---- CTA reduction in fixed warp order (fragment order, conflict-free)
        for (int wv = 0; wv < kDecodeWarps; wv++) {
            if (warp == wv) {
#pragma unroll
                for (int j = 0; j < 8; j++)
#pragma unroll
                    for (int nb = 0; nb < NB; nb++)
#pragma unroll
                        for (int r = 0; r < 4; r++) {
                            float &dst = sm.red[((j * NB + nb) * 4 + r) * 32 + lane];
                            dst = (wv == 0) ? acc[j][nb][r] : dst + acc[j][nb][r];
                        }
            }
            __syncthreads();
        }

        // ---- split-K across CTAs
        const int64_t x0 = (int64_t)G * A, x1 = (int64_t)(G + 1) * A - 1;
        const int c_first = (int)(((x0 + 1) * nCTA - 1) / total);
        const int c_last = (int)(((x1 + 1) * nCTA - 1) / total);
        bool do_epilogue = true;
        if (c_first != c_last) {
            float *slot = a.partials + (int64_t)(c + G) * FRAG;
            for (int i = threadIdx.x; i < FRAG; i += blockDim.x) slot[i] = sm.red[i];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                const int prev = atomicAdd(a.counters + G, 1);
                sm.last = (prev == c_last - c_first);
            }
            __syncthreads();
            do_epilogue = sm.last;
            if (do_epilogue) {
                __threadfence();
                for (int i = threadIdx.x; i < FRAG; i += blockDim.x) {
                    float s = 0.f;
                    for (int cc = c_first; cc <= c_last; cc++)
                        s += __ldcg(a.partials + (int64_t)(cc + G) * FRAG + i);
                    sm.red[i] = s;
                }
                if (threadIdx.x == 0) a.counters[G] = 0;
                __syncthreads();
            }
        }

        // ---- epilogue: y = (Had128(v) * rout) * s_out -> bf16, one warp per token
        if (do_epilogue) {
            const int oc0 = G * kHad + 4 * lane;
            const uint2 rv = __ldg(reinterpret_cast<const uint2 *>(a.rout + oc0));
            const uint2 sv = __ldg(reinterpret_cast<const uint2 *>(a.s_out + oc0));
            const uint32_t rs[2] = {rv.x, rv.y}, ss[2] = {sv.x, sv.y};
            for (int n = warp; n < a.M; n += kDecodeWarps) {
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; i++) v[i] = sm.red[frag_index<NB>(n, 4 * lane + i)];
                warp_fwht128(v, lane);
                uint32_t o[2];
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    float y0 = (v[2 * h] * kHadNorm) * f16_bits_to_f32((uint16_t)(rs[h] & 0xFFFFu));
                    float y1 = (v[2 * h + 1] * kHadNorm) * f16_bits_to_f32((uint16_t)(rs[h] >> 16));
                    y0 *= f16_bits_to_f32((uint16_t)(ss[h] & 0xFFFFu));
                    y1 *= f16_bits_to_f32((uint16_t)(ss[h] >> 16));
                    o[h] = (uint32_t)f32_to_bf16_bits(y0) | ((uint32_t)f32_to_bf16_bits(y1) << 16);
                }
                *reinterpret_cast<uint2 *>(a.out + (int64_t)n * a.ldo + oc0) = make_uint2(o[0], o[1]);
            }
        }
        __syncthreads();   // sm.red is reused by the next segment
        f += a_hi - a_lo;
    }
}

template <int K, int NB>
static cudaError_t launch_decode_t(const DecodeGemmArgs &a, cudaStream_t s) {
    static int occ = -1;
    if (occ < 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_gemm_kernel<K, NB>, 256, 0);
        if (e != cudaSuccess) return e;
        if (occ < 1) occ = 1;
    }
    const int64_t total = (int64_t)(a.OC / kHad) * (a.IC / kTile);
    int64_t grid = (int64_t)device_info().sm_count * occ;
    if (grid > kDecodeMaxCtas) grid = kDecodeMaxCtas;
    if (grid > total) grid = total;
    decode_gemm_kernel<K, NB><<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <int K>
static cudaError_t launch_decode_k(const DecodeGemmArgs &a, cudaStream_t s) {
    const int nb = (a.M + 7) / 8;
    switch (nb) {
        case 1: return launch_decode_t<K, 1>(a, s);
        case 2: return launch_decode_t<K, 2>(a, s);
        case 3: return launch_decode_t<K, 3>(a, s);
        case 4: return launch_decode_t<K, 4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_gemm(const DecodeGemmArgs &a, cudaStream_t s) {
    switch (a.K) {
        case 2: return launch_decode_k<2>(a, s);
        case 3: return launch_decode_k<3>(a, s);
        case 4: return launch_decode_k<4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace exl3
