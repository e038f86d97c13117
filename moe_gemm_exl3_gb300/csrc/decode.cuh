// decode.cuh -- the register-resident trellis decode + mma.sync core of the
// decode-mode GEMM (linear.cu): dense projections, the grouped MoE GEMMs and the
// 8-bit activation variant.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace exl3 {

// Fragment-order index of (row n, group-local column oc).
template <int NB>
__device__ __forceinline__ int frag_index(int n, int oc) {
    const int g = oc >> 4, j = (oc & 15) >> 1, rrow = oc & 1;
    const int nb = n >> 3, q = (n & 7) >> 1, c = n & 1;
    return ((j * NB + nb) * 4 + (2 * rrow + c)) * 32 + (4 * g + q);
}

// CTAs per SM the register budget is sized for.  NB = 1 runs two CTAs (16 warps)
// of up to 128 registers: measured faster than three CTAs at 80 registers (the
// extra registers buy prefetch depth and instruction-level parallelism).
template <int NB>
struct DecodeOcc { static constexpr int value = NB <= 2 ? 2 : 1; };

// Shared memory of the grouped GEMM: per accumulator set (two when paired) the
// warps' fragments, then the entries, then the arrival flag.
template <int NB, bool PAIR = false>
constexpr size_t group_smem_bytes() {
    return (PAIR ? 2 : 1) * (sizeof(float) * kDecodeWarps * 8 * NB * 4 * 32 + sizeof(GroupEntry)) + 16;
}


// Accumulate tile rows [a_lo, a_hi) of one column group into acc (one warp,
// rows a_lo + warp, a_lo + warp + STEP, ...: STEP warps share the range).  wait_u: the kernel has not yet
// waited for the kernel before it (a programmatic dependent launch); the first
// code words, weights that no kernel writes, are requested before the wait,
// the activations after it.
// Where the activation rows come from (USRC, one 8-row block per entry for the
// last two):
//   kUGlobal  rows e.u_row0 + g of u (row stride IC)
//   kUGather  row gather_rows[r0 + g] of half j of u (j = e.u_row0 >= R_half,
//             r0 = e.u_row0 - j * R_half): activations stored per (token, route)
//             pair rather than per routed row
//   kUCodes   8-bit activation codes (uint8 q + 128, rows e.u_row0 + g of u read
//             as bytes); the MMA multiplies q exactly, the row scale is applied by
//             the epilogue
enum USrc { kUGlobal = 0, kUGather = 1, kUCodes = 2 };

// Four 8-bit activation codes (q + 128) -> each q (exact) duplicated into a half2.
__device__ __forceinline__ void codes_to_dup_f16(uint32_t w, uint32_t (&b)[4]) {
    const __half2 off = __half2half2(__ushort_as_half(0x6480));   // 1152 = 1024 + 128
    const uint32_t sel[4] = {0x4040u, 0x4141u, 0x4242u, 0x4343u};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t h = __byte_perm(w, 0x64646464u, sel[i]);   // fp16 1024 + code, twice
        const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), off);
        b[i] = *reinterpret_cast<const uint32_t *>(&r);
    }
}

template <int K, int NB, int USRC = kUGlobal, int STEP = kDecodeWarps>
__device__ __forceinline__ void group_accumulate(float (&acc)[8][NB][4], const GroupEntry &e, const uint16_t *u,
                                                 int IC, int G, int a_lo, int a_hi, int lane, int warp,
                                                 uint32_t hx, const uint32_t *pow2,
                                                 const int32_t *gather_rows = nullptr, int R_half = 0,
                                                 bool wait_u = false) {
    static_assert(USRC == kUGlobal || NB == 1, "gathered and 8-bit activation rows serve one 8-row block");
    const int g = lane >> 2, q = lane & 3;
    const int TO = e.OC / kTile;
    const uint32_t *tile0 = reinterpret_cast<const uint32_t *>(e.code) + (int64_t)(8 * G + g) * 8 * K + q * 2 * K;
    const int64_t row_words = (int64_t)TO * 8 * K;   // uint32 words per tile row
    const uint16_t *ub = u + (int64_t)e.u_row0 * IC;
    // activations of row 8nb+g, channels 16a + 4q .. +3 (zeros past the entry's rows)
    auto load_u = [&](uint2 (&v)[NB], int ar) {
#pragma unroll
        for (int nb = 0; nb < NB; nb++) {
            v[nb] = make_uint2(0u, 0u);
            if (8 * nb + g < e.nrows && ar < a_hi)
                v[nb] = __ldg(reinterpret_cast<const uint2 *>(ub + (int64_t)(8 * nb + g) * IC + 16 * ar + 4 * q));
        }
    };
    // this row's activations, each duplicated into a half2
    auto dup_u = [&](uint32_t (&b)[NB][4], const uint2 (&v)[NB]) {
#pragma unroll
        for (int nb = 0; nb < NB; nb++) {
            b[nb][0] = dup_half_lo(v[nb].x);
            b[nb][1] = dup_half_hi(v[nb].x);
            b[nb][2] = dup_half_lo(v[nb].y);
            b[nb][3] = dup_half_hi(v[nb].y);
        }
    };
    // the 64 weights of this lane's quarter: hash, then MMAs against the activations
    auto mma_row = [&](const QuarterStream<K> &st, const uint32_t (&b)[NB][4]) {
#pragma unroll
        for (int rp = 0; rp < 2; rp++) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int i0 = 32 * rp + 2 * j;
                const uint32_t z0 = trellis_hash_x(st.state(i0, pow2), hx);
                const uint32_t z1 = trellis_hash_x(st.state(i0 + 1, pow2), hx);
                const uint32_t z2 = trellis_hash_x(st.state(i0 + 16, pow2), hx);
                const uint32_t z3 = trellis_hash_x(st.state(i0 + 17, pow2), hx);
#pragma unroll
                for (int nb = 0; nb < NB; nb++)
                    mma_16816(acc[j][nb], z0, z1, z2, z3, b[nb][2 * rp], b[nb][2 * rp + 1]);
            }
        }
    };
    int ar = a_lo + warp;
    uint2 un[NB];
    if constexpr (NB == 1) {
        // two tile-row buffers used in turn, each refilled with the row two steps
        // ahead as soon as its words are realigned (no register copies); the code
        // and activation pointers advance by increments only
        if (ar >= a_hi) return;
        const int n = (a_hi - ar + STEP - 1) / STEP;
        const int64_t stride = row_words * STEP;
        const uint32_t *p = tile0 + ar * row_words;
        const bool urow = g < e.nrows;
        int64_t urow_index = (int64_t)e.u_row0 + g;
        if constexpr (USRC == kUGather) {
            const int j = e.u_row0 >= R_half ? 1 : 0;
            urow_index = urow ? (int64_t)j * R_half + gather_rows[e.u_row0 - j * R_half + g] : 0;
        }
        // codes: one byte per channel, addressed through the same pointer type (in
        // units of two channels, hence the halved offsets)
        const uint16_t *up = USRC == kUCodes ? reinterpret_cast<const uint16_t *>(
                                                  reinterpret_cast<const uint8_t *>(u) + urow_index * IC + 16 * ar + 4 * q)
                                            : u + urow_index * IC + 16 * ar + 4 * q;
        constexpr int kUS = (USRC == kUCodes ? 8 : 16) * STEP;   // activation step per warp step
        auto ldu = [&](const uint16_t *pu) -> uint2 {
            if constexpr (USRC == kUCodes) return make_uint2(__ldg(reinterpret_cast<const uint32_t *>(pu)), 0u);
            else return __ldg(reinterpret_cast<const uint2 *>(pu));
        };
        uint32_t wa[2 * K], wb[2 * K];
        // rows past the entry multiply zeros (codes: 128 is q = 0)
        const uint32_t zero = USRC == kUCodes ? 0x80808080u : 0u;
        uint2 ua = make_uint2(zero, zero), ubv = make_uint2(zero, zero);
        load_quarter<K>(wa, p);
        if (n > 1) load_quarter<K>(wb, p + stride);
        if (wait_u) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (urow) ua = ldu(up);
        if (n > 1 && urow) ubv = ldu(up + kUS);
        auto row = [&](uint32_t (&w)[2 * K], uint2 &uv, bool refill, const uint32_t *pn, const uint16_t *upn) {
            QuarterStream<K> st;
            st.build(w, quarter_prev_word(w[2 * K - 1], lane));
            uint32_t b[NB][4];
            if constexpr (USRC == kUCodes) {
                codes_to_dup_f16(uv.x, b[0]);
            } else {
                b[0][0] = dup_half_lo(uv.x);
                b[0][1] = dup_half_hi(uv.x);
                b[0][2] = dup_half_lo(uv.y);
                b[0][3] = dup_half_hi(uv.y);
            }
            if (refill) {
                load_quarter<K>(w, pn);
                if (urow) uv = ldu(upn);
            }
            mma_row(st, b);
        };
        for (int i = 0; i < n; i += 2) {
            row(wa, ua, i + 2 < n, p + 2 * stride, up + 2 * kUS);
            if (i + 1 >= n) break;
            row(wb, ubv, i + 3 < n, p + 3 * stride, up + 3 * kUS);
            p += 2 * stride;
            up += 2 * kUS;
        }
    } else {
        // one rotating prefetch queue (fewer live registers with more rows)
        constexpr int PF = 2;   // tile rows of code words in flight per warp
        uint32_t wq[PF][2 * K];
#pragma unroll
        for (int d = 0; d < PF; d++)
            if (ar + d * STEP < a_hi) load_quarter<K>(wq[d], tile0 + (ar + d * STEP) * row_words);
        if (wait_u) asm volatile("griddepcontrol.wait;" ::: "memory");
        load_u(un, ar);
        for (; ar < a_hi; ar += STEP) {
            uint32_t w[2 * K];
#pragma unroll
            for (int i = 0; i < 2 * K; i++) w[i] = wq[0][i];
#pragma unroll
            for (int d = 0; d + 1 < PF; d++)
#pragma unroll
                for (int i = 0; i < 2 * K; i++) wq[d][i] = wq[d + 1][i];
            if (ar + PF * STEP < a_hi) load_quarter<K>(wq[PF - 1], tile0 + (ar + PF * STEP) * row_words);
            uint32_t b[NB][4];
            dup_u(b, un);
            load_u(un, ar + STEP);
            QuarterStream<K> st;
            st.build(w, quarter_prev_word(w[2 * K - 1], lane));
            mma_row(st, b);
        }
    }
}


// The output transform of one column group for entry rows [0, nrows): Had128
// of each row's 128 accumulated columns (red, fragment order), times the
// row's scale row_scale[n] if given, then post (and post2 if given);
// f(n, oc0, y[4]) stores row n's 4 columns oc0..oc0+3 (one warp per row, lane
// l holds columns 4l..4l+3).
template <int NB, class Store>
__device__ __forceinline__ void group_epilogue(const float *red, int nrows, const float *row_scale,
                                               const uint16_t *post, const uint16_t *post2,
                                               int G, int lane, int warp, Store f) {
    const int oc0 = G * kHad + 4 * lane;
    const uint2 rv = __ldg(reinterpret_cast<const uint2 *>(post + oc0));
    uint2 sv = make_uint2(0x3C003C00u, 0x3C003C00u);
    if (post2) sv = __ldg(reinterpret_cast<const uint2 *>(post2 + oc0));
    const uint32_t rs[2] = {rv.x, rv.y}, ss[2] = {sv.x, sv.y};
    for (int n = warp; n < nrows; n += kDecodeWarps) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; i++) v[i] = red[frag_index<NB>(n, 4 * lane + i)];
        warp_fwht128(v, lane);
        const float hn = row_scale ? kHadNorm * __ldg(row_scale + n) : kHadNorm;
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int h = i >> 1, sh = 16 * (i & 1);
            y[i] = (v[i] * hn) * f16_bits_to_f32((uint16_t)(rs[h] >> sh));
            if (post2) y[i] *= f16_bits_to_f32((uint16_t)(ss[h] >> sh));
        }
        f(n, oc0, y);
    }
}

}  // namespace exl3
