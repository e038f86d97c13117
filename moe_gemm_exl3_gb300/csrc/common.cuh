// common.cuh -- device helpers shared by the EXL3 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/exl3.h"

namespace exl3 {

constexpr int kHad = 128;        // incoherence transform block
constexpr int kTile = 16;        // weight tile edge
constexpr unsigned kFull = 0xFFFFFFFFu;
// 1/sqrt(128): the orthonormal Had128 scale, applied in fp32.
constexpr float kHadNorm = 0.08838834764831845f;

// Device error codes recorded in the workspace error word (first one wins).
enum DeviceError : int32_t {
    kErrNone = 0,
    kErrWaitTimeout = 1,     // a bounded mbarrier wait gave up
    kErrBadExpertId = 2,     // a MoE route named an expert outside [0, E)
    kErrRouteOverflow = 3,   // more routed rows than the workspace was sized for
};

__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- formats
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
    return __uint_as_float(b16 << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}
__device__ __forceinline__ uint16_t f32_to_f16_bits(float v) {
    return __half_as_ushort(__float2half_rn(v));
}

// ---------------------------------------------------------------- trellis
// 3INST hash of a 16-bit trellis state: returns the two fp16 halves z' whose
// sum is the decoded weight (low half in bits 0..15, high half in 16..31).
constexpr uint32_t kHashMul = 89226354u, kHashAdd = 64248484u;
constexpr uint32_t kHashMask = 0x8FFF8FFFu, kHashXor = 0x3B603B60u;
__device__ __forceinline__ uint32_t trellis_hash(uint32_t state) {
    uint32_t z = state * kHashMul + kHashAdd;
    return (z & kHashMask) ^ kHashXor;
}

// The same hash with the xor constant held in a register: one LOP3 instead of
// two (a LOP3 takes at most one 32-bit immediate).  Hot loops pass kHashXor
// through a kernel argument so the compiler cannot fold it back into an
// immediate.
__device__ __forceinline__ uint32_t trellis_hash_x(uint32_t state, uint32_t xor_reg) {
    uint32_t z = state * kHashMul + kHashAdd;
    return (z & kHashMask) ^ xor_reg;
}

// The decoded fp16 weight of one hashed state: lo + hi, rounded once.
__device__ __forceinline__ __half trellis_weight(uint32_t zp) {
    __half2 h = *reinterpret_cast<const __half2 *>(&zp);
    return __hadd(__low2half(h), __high2half(h));
}

// Pack the decoded weights of two hashed states into one half2 (a, b).
__device__ __forceinline__ uint32_t trellis_weight_pair(uint32_t za, uint32_t zb) {
    uint32_t lo = __byte_perm(za, zb, 0x5410);   // (lo_a, lo_b)
    uint32_t hi = __byte_perm(za, zb, 0x7632);   // (hi_a, hi_b)
    __half2 s = __hadd2(*reinterpret_cast<__half2 *>(&lo), *reinterpret_cast<__half2 *>(&hi));
    return *reinterpret_cast<uint32_t *>(&s);
}

// Multipliers 1 << o for the state extraction, passed to kernels by value.
struct Pow2Table {
    uint32_t v[17];
};
inline Pow2Table make_pow2_table() {
    Pow2Table t;
    for (int i = 0; i < 17; i++) t.v[i] = 1u << i;
    return t;
}

// A quarter of a tile: 4 tile rows x 16 columns = 64 weights, 64K stream bits
// held as 2K little-endian uint32 words (int16 word 2j in bits 0..15 of word j).
// `prev` is the uint32 word preceding the quarter in the circular tile stream;
// only its high int16 (the stream word just before the quarter) is used.
//
// Let S be the quarter's bits preceded by those 16 bits.  E[j] = S bits
// [32j, 32j + 32) and F[j] = S bits [32j + 16, 32j + 48), as big-endian 32-bit
// values; the state of quarter weight i (0..63) is the 16 bits of S starting
// at bit (i+1)K, which always lie within one E or one F word at an offset
// o in [0, 16] from its top.
template <int K>
struct QuarterStream {
    uint32_t E[2 * K + 1];
    uint32_t F[2 * K];

    __device__ __forceinline__ void build(const uint32_t (&w)[2 * K], uint32_t prev) {
        E[0] = __byte_perm(w[0], prev, 0x7610);
#pragma unroll
        for (int j = 1; j < 2 * K; j++) E[j] = __byte_perm(w[j], w[j - 1], 0x7610);
        E[2 * K] = w[2 * K - 1] & 0xFFFF0000u;
#pragma unroll
        for (int j = 0; j < 2 * K; j++) F[j] = __byte_perm(w[j], 0, 0x1032);
    }

    // 16-bit trellis state of quarter weight i (compile-time i after unrolling).
    // Windows on a byte boundary take one byte permute.  The general case shifts
    // the window to the top of the word with a multiply by 2^o and then down by
    // 16: the multiply runs on the FMA pipe, which balances the integer ALU pipe
    // that the hash's LOP3 and the shift occupy.
    // pow2[o] must hold 1 << o; it is read from a kernel argument so that the
    // compiler cannot turn the multiply back into an ALU shift.
    __device__ __forceinline__ uint32_t state(int i, const uint32_t *pow2) const {
        const int p = (i + 1) * K;
        const int j = p >> 5, o = p & 31;
        const uint32_t R = o <= 16 ? E[j] : F[j];
        const int oo = o <= 16 ? o : o - 16;
        if (oo == 0) return R >> 16;
        if (oo == 16) return R & 0xFFFFu;
        if (oo == 8) return __byte_perm(R, 0, 0x4421);   // bytes 1..2: one permute
        return (R * pow2[oo]) >> 16;
    }
};

// Word preceding a quarter inside its tile (tail-biting): lanes are laid out
// as 4 consecutive quarters q = lane % 4 of one tile; quarter 0 takes the last
// word of quarter 3.
__device__ __forceinline__ uint32_t quarter_prev_word(uint32_t last_word, int lane) {
    const int q = lane & 3;
    const int src = q == 0 ? lane + 3 : lane - 1;
    return __shfl_sync(kFull, last_word, src);
}

// Load one quarter (2K uint32 words) with loads as wide as its alignment allows.
template <int K>
__device__ __forceinline__ void load_quarter(uint32_t (&w)[2 * K], const uint32_t *p) {
    if constexpr (K == 2) {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (K == 4) {
        uint4 v0 = __ldg(reinterpret_cast<const uint4 *>(p));
        uint4 v1 = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
    } else {
#pragma unroll
        for (int j = 0; j < K; j++) {
            uint2 v = __ldg(reinterpret_cast<const uint2 *>(p) + j);
            w[2 * j] = v.x; w[2 * j + 1] = v.y;
        }
    }
}

// ---------------------------------------------------------------- Hadamard
// In-warp unnormalised Had128 of 128 values held 4 per lane as v[i] = value
// (4*lane + i): two register stages (index bits 0, 1) then five shuffle stages
// (index bits 2..6 = lane bits 0..4).  Sylvester order: H[i][j] = (-1)^popc(i&j).
__device__ __forceinline__ void warp_fwht128(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[1] = a1 + a3; v[2] = a0 - a2; v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        // upper lane: p - v, lower lane: v + p, as one FMA with a sign of +-1
        // (exact product, the same single rounding)
        const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float p = __shfl_xor_sync(kFull, v[i], m);
            v[i] = fmaf(sgn, v[i], p);
        }
    }
}

// Unnormalised Had128 of 128 values held 16 per lane by a group of 8 lanes
// (sub = lane % 8): v[i] = value (16 * sub + i).  Four register stages (index
// bits 0..3), then three shuffle stages within the group (bits 4..6 = sub bits
// 0..2).  Every lane of the warp must take part (the shuffles span the warp).
__device__ __forceinline__ void group8_fwht128(float (&v)[16], int sub) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            if (i & h) continue;
            const float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        // upper lane o - v, lower lane v + o: one FMA with an exact sign of +-1
        const float sgn = (sub & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const float o = __shfl_xor_sync(kFull, v[i], m);
            v[i] = fmaf(sgn, v[i], o);
        }
    }
}

// 16 consecutive 16-bit values: two 16-byte loads when V16, else four 8-byte
// loads (scale vectors need only 8-byte alignment).
template <bool V16>
__device__ __forceinline__ void load16x16(uint4 (&v)[2], const uint16_t *p) {
    if constexpr (V16) {
        v[0] = __ldg(reinterpret_cast<const uint4 *>(p));
        v[1] = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
    } else {
        const uint2 a = __ldg(reinterpret_cast<const uint2 *>(p)), b = __ldg(reinterpret_cast<const uint2 *>(p) + 1);
        const uint2 c = __ldg(reinterpret_cast<const uint2 *>(p) + 2), d = __ldg(reinterpret_cast<const uint2 *>(p) + 3);
        v[0] = make_uint4(a.x, a.y, b.x, b.y);
        v[1] = make_uint4(c.x, c.y, d.x, d.y);
    }
}

// Half i (0..15) of 16 consecutive 16-bit values held in two uint4.
__device__ __forceinline__ uint32_t half_bits(const uint4 (&v)[2], int i) {
    const uint4 &q = v[i >> 3];
    const uint32_t w = (i & 4) ? ((i & 2) ? q.w : q.z) : ((i & 2) ? q.y : q.x);
    return (w >> (16 * (i & 1))) & 0xFFFFu;
}

// ---------------------------------------------------------------- MMA
// D += A * B, m16n8k16, fp16 operands, fp32 accumulate (legacy warp-level MMA).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t dup_half_lo(uint32_t h2) { return __byte_perm(h2, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_half_hi(uint32_t h2) { return __byte_perm(h2, 0, 0x3232); }

}  // namespace exl3
