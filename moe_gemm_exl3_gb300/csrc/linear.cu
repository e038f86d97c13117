// linear.cu -- EXL3 linear: activation pre-transform, trellis reconstruct,
// codebook table and the decode-mode (small M) fused trellis GEMM.
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode.cuh"
#include "internal.h"

namespace exl3 {

// --------------------------------------------------------------------------
// Activation pre-transform: u = Had128((x * s_in) * rin) per 128-channel
// block (radiance_escha.py, module docstring "THE FORWARD", first factor).
// Eight lanes serve one block, 16 consecutive channels each (32-byte loads and
// stores); a warp covers four blocks of the flattened (shard, row, block)
// order per step and kPtSteps steps, issuing all of its loads first.  The
// transform: four register stages over a lane's 16 channels (index bits 0..3),
// three shuffle stages across the 8-lane group (bits 4..6).
// --------------------------------------------------------------------------
constexpr int kPtSteps = 2;

// V16: x and u are 16-byte aligned (16-byte loads and stores of the activations)
template <bool V16>
__global__ void __launch_bounds__(256) pretransform_kernel(const uint16_t *__restrict__ x,
                                                           int64_t M, int IC,
                                                           const __grid_constant__ PretransformShards p,
                                                           uint16_t *__restrict__ u, int steps) {
    // this launch may itself start before the preceding kernel has finished (a
    // programmatic dependent launch): wait for it before reading x or writing u
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // then let a dependent launch be scheduled: the GEMM that reads u (it waits for
    // this grid), or the reconstruct, which writes only the staging buffer and may
    // run alongside (every kernel before this one has completed by now)
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31, sub = lane & 7;
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int nb = IC / kHad;
    const int64_t total = (int64_t)p.n * M * nb;
    uint4 xv[kPtSteps][2], sv[kPtSteps][2], rv[kPtSteps][2];
    int64_t row[kPtSteps];
    int c0[kPtSteps];
#pragma unroll
    for (int k = 0; k < kPtSteps; k++) {
        const int64_t B = (wid * steps + k) * 4 + (lane >> 3);   // this lane group's block
        row[k] = -1;
        if (k < steps && B < total) {
            const int64_t r = B / nb;                 // shard * M + m
            const int sh = (int)(r / M);
            c0[k] = (int)(B - r * nb) * kHad + 16 * sub;
            row[k] = r;
            load16x16<V16>(xv[k], x + (r - sh * M) * IC + c0[k]);
            load16x16<false>(sv[k], p.s_in[sh] + c0[k]);
            load16x16<false>(rv[k], p.rin[sh] + c0[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < kPtSteps; k++) {
        if (k >= steps) break;                       // warp-uniform
        // lanes of a group past the end transform zeros and store nothing (every
        // lane joins the shuffles)
        const bool live = row[k] >= 0;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; i++)
            v[i] = live ? (bf16_bits_to_f32(half_bits(xv[k], i)) * f16_bits_to_f32((uint16_t)half_bits(sv[k], i))) *
                              f16_bits_to_f32((uint16_t)half_bits(rv[k], i))
                        : 0.f;
        group8_fwht128(v, sub);
        if (!live) continue;
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; i++)
            o[i] = (uint32_t)f32_to_f16_bits(v[2 * i] * kHadNorm) |
                   ((uint32_t)f32_to_f16_bits(v[2 * i + 1] * kHadNorm) << 16);
        if constexpr (V16) {
            uint4 *dst = reinterpret_cast<uint4 *>(u + row[k] * IC + c0[k]);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
            uint2 *dst = reinterpret_cast<uint2 *>(u + row[k] * IC + c0[k]);
#pragma unroll
            for (int i = 0; i < 4; i++) dst[i] = make_uint2(o[2 * i], o[2 * i + 1]);
        }
    }
}

cudaError_t launch_pretransform_shards(const uint16_t *x, int64_t M, int IC, const PretransformShards &p,
                                       uint16_t *u, cudaStream_t s) {
    const int64_t blocks = (int64_t)p.n * M * (IC / kHad);
    // kPtSteps steps per warp once the blocks fill several waves of warps; one
    // step otherwise (more warps, shorter latency)
    const int steps = blocks >= (int64_t)device_info().sm_count * 64 * 4 * kPtSteps ? kPtSteps : 1;
    const int64_t warps = (blocks + 4 * steps - 1) / (4 * steps);
    const int64_t grid = (warps + 7) / 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(u)) & 15u) == 0)
        return cudaLaunchKernelEx(&cfg, pretransform_kernel<true>, x, M, IC, p, u, steps);
    return cudaLaunchKernelEx(&cfg, pretransform_kernel<false>, x, M, IC, p, u, steps);
}

cudaError_t launch_pretransform(const uint16_t *x, int64_t M, int IC, const uint16_t *s_in,
                                const uint16_t *rin, uint16_t *u, cudaStream_t s) {
    PretransformShards p = {};
    p.s_in[0] = s_in;
    p.rin[0] = rin;
    p.n = 1;
    return launch_pretransform_shards(x, M, IC, p, u, s);
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
                                                          bool transposed, const Pow2Table p2) {
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
                pk[c / 2] = trellis_weight_pair(trellis_hash(st.state(16 * r + c, p2.v)),
                                                trellis_hash(st.state(16 * r + c + 1, p2.v)));
            uint4 *dst = reinterpret_cast<uint4 *>(W + (int64_t)(16 * a + 4 * q + r) * OC + 16 * b);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 16; c++) {
            uint32_t p0 = trellis_weight_pair(trellis_hash(st.state(c, p2.v)), trellis_hash(st.state(16 + c, p2.v)));
            uint32_t p1 = trellis_weight_pair(trellis_hash(st.state(32 + c, p2.v)), trellis_hash(st.state(48 + c, p2.v)));
            *reinterpret_cast<uint2 *>(W + (int64_t)(16 * b + c) * IC + 16 * a + 4 * q) = make_uint2(p0, p1);
        }
    }
    // launched as a programmatic dependent of the pre-transform, this grid runs
    // alongside it; it completes only once the pre-transform has, so the GEMM that
    // waits for this grid sees both u and W (a no-op without the dependency)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

cudaError_t launch_reconstruct(const int16_t *code, int IC, int OC, int K, uint16_t *W,
                               bool transposed, cudaStream_t s, bool pdl) {
    const int64_t quarters = (int64_t)(IC / kTile) * (OC / kTile) * 4;
    const Pow2Table p2 = make_pow2_table();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((quarters + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (K) {
        case 2: return cudaLaunchKernelEx(&cfg, reconstruct_kernel<2>, code, IC, OC, W, transposed, p2);
        case 3: return cudaLaunchKernelEx(&cfg, reconstruct_kernel<3>, code, IC, OC, W, transposed, p2);
        case 4: return cudaLaunchKernelEx(&cfg, reconstruct_kernel<4>, code, IC, OC, W, transposed, p2);
        default: return cudaErrorInvalidValue;
    }
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
// Grouped decode-mode fused trellis GEMM (rows per problem <= 8 * NB <= 32).
//
// Each problem ("entry") is one code tensor applied to a block of activation
// rows: v = u @ W with W decoded on the fly from the code words, followed by
// the output transform.  The dense linear is one entry per shard; the MoE
// layer is one entry per (expert, row block) with each expert's own K.
//
// Mapping.  A warp owns one column group G (8 tiles = 128 output columns) and
// one tile row a (16 input channels) per step.  Lane (g, q) = (lane/4, lane%4)
// loads quarter q (tile rows 4q..4q+3) of tile (a, 8G + g): the warp's 8 tiles
// are contiguous in memory, so one step is one coalesced read of 512 K bytes.
// The decoded weights go straight into the A operand of m16n8k16 MMAs with the
// roles swapped (A = W^T: output columns on the MMA's M, rows on its N):
// A row g <-> column 16(8G+g)+2j, row g+8 <-> the next column, and each A
// register holds the two fp16 halves (lo, hi) of one weight's codebook sum
// against a B register holding the same activation twice, so the tensor core
// forms u*(lo+hi) and no per-weight add is issued on the ALUs.
//
// Split-K.  The (group, a) units of all entries are split evenly over a
// persistent grid; a CTA's range covers parts of one or two column groups.
// Warps reduce through shared memory in fixed order; CTAs sharing a group write
// their partial to a slab slot and bump the group's counter; the last to arrive
// sums the partials in CTA order (deterministic), runs the epilogue and resets
// the counter.  No CTA waits on another (radiance_escha.py: split-K partial slab
// + block counter).
// --------------------------------------------------------------------------

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Parts per column group when the groups fit the grid: as many as the grid
// allows, but each part keeps at least kMinRowsPerWarp tile rows per warp (a
// part's fixed costs, the load ramp and the split-K handshake, outweigh a few
// rows of decode).
constexpr int kMinRowsPerWarp = 4;
__host__ __device__ __forceinline__ int decode_parts(int fit, int A) {
    int cap = A / (kMinRowsPerWarp * kDecodeWarps);
    if (cap < 1) cap = 1;
    int p = fit < cap ? fit : cap;
    return p < 1 ? 1 : p;
}

// Output transform of column group G of entry e from the reduced fragments rr
// (fragment order, NB row blocks): Had128 of each row's 128 columns, then the
// post-scales; rows n0, n0 + nstep, ... < e.nrows, one warp per row.  Dense
// mode stores bf16 into out; rows mode stores fp32 rows and, with the combine
// epilogue, sums each token's routes.
template <int NB>
__device__ __forceinline__ void group_output(const GroupGemmArgs &a, const float *rr, const GroupEntry &e, int G,
                                             int lane, int n0, int nstep) {
    const int oc0 = G * kHad + 4 * lane;
    const uint2 rv = __ldg(reinterpret_cast<const uint2 *>(e.post + oc0));
    uint2 sv = make_uint2(0x3C003C00u, 0x3C003C00u);
    if (a.mode == kModeDense) sv = __ldg(reinterpret_cast<const uint2 *>(e.post2 + oc0));
    const uint32_t rs[2] = {rv.x, rv.y}, ss[2] = {sv.x, sv.y};
    for (int n = n0; n < e.nrows; n += nstep) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; i++) v[i] = rr[frag_index<NB>(n, 4 * lane + i)];
        warp_fwht128(v, lane);
        // the Hadamard scale, times the row's activation scale when there is one
        const float hn = a.row_scale ? kHadNorm * __ldg(a.row_scale + e.u_row0 + n) : kHadNorm;
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int h = i >> 1, sh = 16 * (i & 1);
            y[i] = (v[i] * hn) * f16_bits_to_f32((uint16_t)(rs[h] >> sh));
            if (a.mode == kModeDense) y[i] *= f16_bits_to_f32((uint16_t)(ss[h] >> sh));
        }
        if (a.mode == kModeDense) {
            const uint32_t o0 = (uint32_t)f32_to_bf16_bits(y[0]) | ((uint32_t)f32_to_bf16_bits(y[1]) << 16);
            const uint32_t o1 = (uint32_t)f32_to_bf16_bits(y[2]) | ((uint32_t)f32_to_bf16_bits(y[3]) << 16);
            *reinterpret_cast<uint2 *>(a.out + (int64_t)n * a.ldo + e.out_off + oc0) = make_uint2(o0, o1);
        } else {
            *reinterpret_cast<float4 *>(a.out_rows + (e.out_off + n) * (int64_t)e.OC + oc0) =
                make_float4(y[0], y[1], y[2], y[3]);
            if (a.comb) {
                // routed row r = token t's route: the last of t's valid routes to
                // arrive at this column group sums them in route order into y[t]
                __threadfence();
                __syncwarp();
                const int t = a.row_pair[e.out_off + n] / a.topk;
                const int GH = e.OC / kHad;
                int last = 0;
                if (lane == 0) {
                    int nv = 0;
                    for (int k = 0; k < a.topk; k++) nv += a.comb_pos[(int64_t)t * a.topk + k] >= 0;
                    last = atomicAdd(a.comb_counters + (int64_t)t * GH + G, 1) == nv - 1;
                }
                last = __shfl_sync(kFull, last, 0);
                if (last) {
                    __threadfence();
                    float sum[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int k = 0; k < a.topk; k++) {
                        const int rk = a.comb_pos[(int64_t)t * a.topk + k];
                        if (rk < 0) continue;
                        const float wk = a.comb_w[(int64_t)t * a.topk + k];
                        const float4 d = __ldcg(reinterpret_cast<const float4 *>(a.out_rows + (int64_t)rk * e.OC + oc0));
                        sum[0] += wk * d.x;
                        sum[1] += wk * d.y;
                        sum[2] += wk * d.z;
                        sum[3] += wk * d.w;
                    }
                    const uint32_t o0 = (uint32_t)f32_to_bf16_bits(sum[0]) | ((uint32_t)f32_to_bf16_bits(sum[1]) << 16);
                    const uint32_t o1 = (uint32_t)f32_to_bf16_bits(sum[2]) | ((uint32_t)f32_to_bf16_bits(sum[3]) << 16);
                    *reinterpret_cast<uint2 *>(a.comb_y + (int64_t)t * e.OC + oc0) = make_uint2(o0, o1);
                    if (lane == 0) a.comb_counters[(int64_t)t * GH + G] = 0;
                }
            }
        }
    }
}

// KSET: bit k set = the launch may contain entries of bitrate k (2, 3, 4); only
// those decode paths are compiled into the kernel, which keeps registers low.
// USRC: where the activation rows come from (kUGlobal, kUGather or kUCodes; see
// group_accumulate).  PAIR (MoE FC1 with gathered rows): consecutive entries 2i,
// 2i + 1 are an expert row block's w1 and w3; a column group covers both (2A
// units: w1's tile rows, then w3's), and its epilogue produces FC2's input,
// Had((silu(g) * u) * w2_suh[slot]), instead of two fp32 rows.
template <int NB, int KSET, int USRC = kUGlobal, bool PAIR = false>
__global__ void __launch_bounds__(256, DecodeOcc<NB>::value) group_gemm_kernel(const GroupGemmArgs a) {
    static_assert(USRC == kUGlobal || NB == 1, "gathered and 8-bit activation rows serve one 8-row block per entry");
    static_assert(!PAIR || USRC == kUGather, "the paired epilogue serves the gathered FC1");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int FRAG = 8 * NB * 4 * 32;
    constexpr int NSUB = PAIR ? 2 : 1;                                  // accumulator sets: (gate, up) when paired
    float *red = reinterpret_cast<float *>(smem_raw);                   // [NSUB][warps][FRAG]
    GroupEntry *s_ent = reinterpret_cast<GroupEntry *>(red + NSUB * kDecodeWarps * FRAG);
    int *s_last = reinterpret_cast<int *>(s_ent + NSUB);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int A = a.IC / kTile;
    const int AU = NSUB * A;   // units (tile rows) per column group

    // Entries passed by value (dense launches) name only weights and this
    // launch's activations: the first code words are requested before waiting
    // for the preceding kernel in the stream (it may still be writing the
    // activations), the rest after.  So are device entry lists written by an
    // earlier kernel (entries_ready); those written by the preceding kernel
    // itself are read after the wait.
    const bool hoist = (!a.n_entries_dev && !a.entries) || a.entries_ready;
    if (!hoist) grid_dependency_wait();
    // the next kernel in the stream may be scheduled now: it must itself wait for
    // this grid to complete before touching memory (every kernel here does)
    asm volatile("griddepcontrol.launch_dependents;");

    int n_groups;
    const int n_entries = a.n_entries_dev ? *a.n_entries_dev : a.n_inline;
    if (a.n_groups_per_entry > 0) {
        n_groups = (PAIR ? n_entries / 2 : n_entries) * a.n_groups_per_entry;
    } else {
        n_groups = 0;
        for (int i = 0; i < n_entries; i++) n_groups += a.inline_e[i].OC / kHad;
    }
    const int64_t total = (int64_t)n_groups * AU;
    const int c = blockIdx.x;
    // entry lists built on the device (MoE): when the groups fit the grid, whole
    // groups or a few parts of each, as the host does for dense launches
    int parts = a.parts;
    if (parts == 0 && a.n_entries_dev && n_groups > 0 && n_groups <= (int)gridDim.x)
        parts = decode_parts(gridDim.x / n_groups, AU);
    int nCTA;
    int64_t f, f_end;
    if (parts > 0) {
        // item partition: CTA c takes part c % parts of column group c / parts, so a
        // CTA never switches groups and a group's partials come from exactly `parts` CTAs
        nCTA = n_groups * parts;
        if (c >= nCTA) return;
        const int g = c / parts, pp = c - g * parts;
        f = (int64_t)g * AU + (int64_t)pp * AU / parts;
        f_end = (int64_t)g * AU + (int64_t)(pp + 1) * AU / parts;
    } else {
        // stream-K: every CTA of the partition must own at least one unit (an empty
        // range would never arrive at its group's counter): with fewer units than
        // CTAs the extra CTAs leave
        nCTA = (int64_t)gridDim.x < total ? (int)gridDim.x : (int)total;
        if (c >= nCTA) return;
        f = (int64_t)c * total / nCTA;
        f_end = (int64_t)(c + 1) * total / nCTA;
    }
    const uint32_t hx = a.hash_xor;

    while (f < f_end) {
        const int gi = (int)(f / AU);                // global column-group index
        const int a_lo = (int)(f % AU);
        const int a_hi = (int)((int64_t)AU < a_lo + (f_end - f) ? (int64_t)AU : a_lo + (f_end - f));
        // the entry owning group gi (both entries of the pair)
        if (threadIdx.x == 0) {
            if (PAIR) {
                s_ent[0] = a.entries[2 * (gi / a.n_groups_per_entry)];
                s_ent[1] = a.entries[2 * (gi / a.n_groups_per_entry) + 1];
            } else if (a.n_groups_per_entry > 0) {
                *s_ent = a.entries ? a.entries[gi / a.n_groups_per_entry] : a.inline_e[gi / a.n_groups_per_entry];
            } else {
                int i = 0;
                while (i + 1 < n_entries && a.inline_e[i + 1].g0 <= gi) i++;
                *s_ent = a.inline_e[i];
            }
        }
        __syncthreads();
        const GroupEntry e = *s_ent;
        const int G = a.n_groups_per_entry > 0 ? gi % a.n_groups_per_entry : gi - e.g0;

        // one accumulator set per sub-range (paired: w1's tile rows, then w3's),
        // each reduced over the warps in fixed order into its own region of red
#pragma unroll 1
        for (int sub = 0; sub < NSUB; sub++) {
            const int lo = PAIR ? (a_lo > sub * A ? a_lo : sub * A) - sub * A : a_lo;
            const int hi = PAIR ? (a_hi < (sub + 1) * A ? a_hi : (sub + 1) * A) - sub * A : a_hi;
            const GroupEntry es = PAIR ? s_ent[sub] : e;
            float acc[8][NB][4];
#pragma unroll
            for (int j = 0; j < 8; j++)
#pragma unroll
                for (int nb = 0; nb < NB; nb++)
#pragma unroll
                    for (int r = 0; r < 4; r++) acc[j][nb][r] = 0.f;
            if (lo < hi) {
                if ((KSET & 4) && es.K == 2)
                    group_accumulate<2, NB, USRC>(acc, es, a.u, a.IC, G, lo, hi, lane, warp, hx, a.pow2, a.row_pair, a.R,
                                                 hoist);
                if ((KSET & 8) && es.K == 3)
                    group_accumulate<3, NB, USRC>(acc, es, a.u, a.IC, G, lo, hi, lane, warp, hx, a.pow2, a.row_pair, a.R,
                                                 hoist);
                if ((KSET & 16) && es.K == 4)
                    group_accumulate<4, NB, USRC>(acc, es, a.u, a.IC, G, lo, hi, lane, warp, hx, a.pow2, a.row_pair, a.R,
                                                 hoist);
            }
            // warps without rows in this range: the split-K slab and counters below
            // are shared with the preceding kernel
            if (hoist) grid_dependency_wait();
            float *rs = red + sub * kDecodeWarps * FRAG;
            // ---- CTA reduction in fixed warp order (fragment order, one barrier)
#pragma unroll
            for (int j = 0; j < 8; j++)
#pragma unroll
                for (int nb = 0; nb < NB; nb++)
#pragma unroll
                    for (int r = 0; r < 4; r++) rs[warp * FRAG + ((j * NB + nb) * 4 + r) * 32 + lane] = acc[j][nb][r];
            __syncthreads();
            for (int i = threadIdx.x; i < FRAG; i += blockDim.x) {
                float sum = rs[i];
#pragma unroll
                for (int wv = 1; wv < kDecodeWarps; wv++) sum += rs[wv * FRAG + i];
                rs[i] = sum;
            }
            __syncthreads();
        }
        // element i of the reduced sets (i < NSUB * FRAG) lives at red[ridx(i)]
        auto ridx = [&](int i) { return PAIR ? (i / FRAG) * (kDecodeWarps * FRAG) + i % FRAG : i; };

        // ---- split-K across CTAs
        int c_first, c_last;     // the CTAs that own units of group gi
        if (parts > 0) {
            c_first = gi * parts;
            c_last = c_first + parts - 1;
        } else {
            const int64_t x0 = (int64_t)gi * AU, x1 = (int64_t)(gi + 1) * AU - 1;
            c_first = (int)(((x0 + 1) * nCTA - 1) / total);
            c_last = (int)(((x1 + 1) * nCTA - 1) / total);
        }
        bool do_epilogue = true;
        if (c_first != c_last) {
            float *slot = a.partials + (int64_t)(c + gi) * (NSUB * FRAG);
            for (int i = threadIdx.x; i < NSUB * FRAG; i += blockDim.x) slot[i] = red[ridx(i)];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) {
                const int prev = atomicAdd(a.counters + gi, 1);
                *s_last = (prev == c_last - c_first);
            }
            __syncthreads();
            do_epilogue = *s_last;
            if (do_epilogue) {
                __threadfence();
                // CTA order outermost so each CTA's elements load in parallel; the
                // sum runs in ascending CTA order (deterministic)
                constexpr int PER = (NSUB * FRAG + kDecodeWarps * 32 - 1) / (kDecodeWarps * 32);
                float sum[PER];
#pragma unroll
                for (int k = 0; k < PER; k++) sum[k] = 0.f;
                for (int cc = c_first; cc <= c_last; cc++) {
                    const float *src = a.partials + (int64_t)(cc + gi) * (NSUB * FRAG);
#pragma unroll
                    for (int k = 0; k < PER; k++) {
                        const int i = threadIdx.x + k * kDecodeWarps * 32;
                        if (i < NSUB * FRAG) sum[k] += __ldcg(src + i);
                    }
                }
#pragma unroll
                for (int k = 0; k < PER; k++) {
                    const int i = threadIdx.x + k * kDecodeWarps * 32;
                    if (i < NSUB * FRAG) red[ridx(i)] = sum[k];
                }
                if (threadIdx.x == 0) a.counters[gi] = 0;
                __syncthreads();
            }
        }

        // ---- paired epilogue: g = Had128(v_w1) * svh_w1, u = Had128(v_w3) * svh_w3,
        // then FC2's input h2 = Had128((silu(g) * u) * w2_suh[slot]) -> fp16
        if (PAIR && do_epilogue) {
            const GroupEntry e3 = s_ent[1];
            const int oc0 = G * kHad + 4 * lane;
            const uint2 pg = __ldg(reinterpret_cast<const uint2 *>(e.post + oc0));
            const uint2 pu = __ldg(reinterpret_cast<const uint2 *>(e3.post + oc0));
            const uint2 ps = __ldg(reinterpret_cast<const uint2 *>(a.act_suh + (int64_t)e.slot * e.OC + oc0));
            const uint32_t wg[2] = {pg.x, pg.y}, wu[2] = {pu.x, pu.y}, ws[2] = {ps.x, ps.y};
            for (int n = warp; n < e.nrows; n += kDecodeWarps) {
                float vg[4], vu[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    vg[i] = red[frag_index<NB>(n, 4 * lane + i)];
                    vu[i] = red[kDecodeWarps * FRAG + frag_index<NB>(n, 4 * lane + i)];
                }
                warp_fwht128(vg, lane);
                warp_fwht128(vu, lane);
                float h[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int hh = i >> 1, sh = 16 * (i & 1);
                    const float g = (vg[i] * kHadNorm) * f16_bits_to_f32((uint16_t)(wg[hh] >> sh));
                    const float u = (vu[i] * kHadNorm) * f16_bits_to_f32((uint16_t)(wu[hh] >> sh));
                    const float silu = g / (1.0f + __expf(-g));
                    h[i] = (silu * u) * f16_bits_to_f32((uint16_t)(ws[hh] >> sh));
                }
                warp_fwht128(h, lane);
                uint2 o;
                o.x = (uint32_t)f32_to_f16_bits(h[0] * kHadNorm) | ((uint32_t)f32_to_f16_bits(h[1] * kHadNorm) << 16);
                o.y = (uint32_t)f32_to_f16_bits(h[2] * kHadNorm) | ((uint32_t)f32_to_f16_bits(h[3] * kHadNorm) << 16);
                *reinterpret_cast<uint2 *>(a.act_out + (e.out_off + n) * (int64_t)e.OC + oc0) = o;
            }
        }
        // ---- epilogue: Had128 of each row's 128 columns, then the post-scales
        if (!PAIR && do_epilogue) group_output<NB>(a, red, e, G, lane, warp, kDecodeWarps);
        __syncthreads();   // red and s_ent are reused by the next segment
        f += a_hi - a_lo;
    }
}

// --------------------------------------------------------------------------
// Two dense shards of equal width (a merged gate/up layer) at up to 16 rows
// (one or two 8-row blocks; 8-bit codes: one), with more column groups per
// shard than half the SMs and at most as many as the SMs.  With one group per 8-warp CTA, two CTAs share most SMs: where a
// cheap (smaller K) and an expensive group meet, the cheap CTA ends early and
// the other runs on alone at half the warps; other SMs hold two expensive
// groups, or one group only.  Here one 16-warp CTA per SM takes shard 0's
// group G (warps 0-7) and shard 1's group G (warps 8-15): every SM carries
// one group of each shard.  The halves share nothing; each reduces its group
// in fixed warp order and runs the epilogue (no split-K, deterministic).
// Measured against moving the last tile rows of the costlier group to the
// other half (either way round, 8 to 40 rows): every such split was slower,
// its second load ramp costing more than the balance gains.
// --------------------------------------------------------------------------
constexpr int kPairThreads = 2 * kDecodeWarps * 32;
// floats of one warp's fragments, and the CTA's shared memory (both halves' warps)
template <int NB> __host__ __device__ constexpr size_t pair_frag() { return 8 * NB * 4 * 32; }
template <int NB> constexpr size_t pair_smem() { return 2 * sizeof(float) * kDecodeWarps * pair_frag<NB>(); }

// USRC: fp16 rows of u or 8-bit codes (kUGlobal / kUCodes; see group_accumulate).
// NB: 8-row blocks (up to 16 rows: two, fp16 rows only).
template <int KSET, int USRC, int NB>
__global__ void __launch_bounds__(kPairThreads, 1) group_pair_kernel(const GroupGemmArgs a) {
    static_assert(USRC == kUGlobal || NB == 1, "8-bit activation codes serve one 8-row block");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int FRAG = (int)pair_frag<NB>();
    const int lane = threadIdx.x & 31;
    const int warp = (threadIdx.x >> 5) & (kDecodeWarps - 1);   // warp within the half
    const int ht = threadIdx.x & (kDecodeWarps * 32 - 1);       // thread within the half
    const int A = a.IC / kTile;
    const int G = blockIdx.x;
    const uint32_t hx = a.hash_xor;

    // the first code words (weights) are requested before waiting for the
    // preceding kernel, which may still be writing the activations
    asm volatile("griddepcontrol.launch_dependents;");

    // one half: accumulate all A tile rows of group G of e, reduce over the
    // half's warps into red[0, FRAG), then the dense epilogue
    auto half = [&](const GroupEntry &e, float *red, int bar) {
        float acc[8][NB][4];
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int nb = 0; nb < NB; nb++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[j][nb][q] = 0.f;
        if ((KSET & 4) && e.K == 2) group_accumulate<2, NB, USRC>(acc, e, a.u, a.IC, G, 0, A, lane, warp, hx, a.pow2, nullptr, 0, true);
        if ((KSET & 8) && e.K == 3) group_accumulate<3, NB, USRC>(acc, e, a.u, a.IC, G, 0, A, lane, warp, hx, a.pow2, nullptr, 0, true);
        if ((KSET & 16) && e.K == 4) group_accumulate<4, NB, USRC>(acc, e, a.u, a.IC, G, 0, A, lane, warp, hx, a.pow2, nullptr, 0, true);
        grid_dependency_wait();   // a no-op once waited; the row scales and out follow
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int nb = 0; nb < NB; nb++)
#pragma unroll
                for (int q = 0; q < 4; q++) red[warp * FRAG + ((j * NB + nb) * 4 + q) * 32 + lane] = acc[j][nb][q];
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kDecodeWarps * 32) : "memory");
        for (int i = ht; i < FRAG; i += kDecodeWarps * 32) {
            float sum = red[i];
#pragma unroll
            for (int wv = 1; wv < kDecodeWarps; wv++) sum += red[wv * FRAG + i];
            red[i] = sum;
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kDecodeWarps * 32) : "memory");
        const float *rsc = a.row_scale ? a.row_scale + e.u_row0 : nullptr;
        group_epilogue<NB>(red, e.nrows, rsc, e.post, e.post2, G, lane, warp, [&](int n, int oc0, const float (&y)[4]) {
            const uint32_t o0 = (uint32_t)f32_to_bf16_bits(y[0]) | ((uint32_t)f32_to_bf16_bits(y[1]) << 16);
            const uint32_t o1 = (uint32_t)f32_to_bf16_bits(y[2]) | ((uint32_t)f32_to_bf16_bits(y[3]) << 16);
            *reinterpret_cast<uint2 *>(a.out + (int64_t)n * a.ldo + e.out_off + oc0) = make_uint2(o0, o1);
        });
    };
    float *red = reinterpret_cast<float *>(smem_raw);
    if (threadIdx.x < kDecodeWarps * 32) half(a.inline_e[0], red, 1);
    else half(a.inline_e[1], red + kDecodeWarps * FRAG, 2);
}

// The paired kernel serves this launch: two dense shards of one width and one
// 8-row block (two with fp16 rows), with more column groups per shard than half
// the SMs and at most as many as the SMs.
static bool pair_launch_fits(const GroupGemmArgs &a, int nb) {
    if (nb < 1 || nb > (a.codes ? 1 : 2) || a.gather || a.pair_act || a.mode != kModeDense) return false;
    if (a.n_entries_dev || a.entries || a.n_groups_per_entry != 0 || a.n_inline != 2) return false;
    const GroupEntry &e0 = a.inline_e[0], &e1 = a.inline_e[1];
    if (e0.OC != e1.OC || e0.nrows != e1.nrows || e0.nrows > 8 * nb) return false;
    const int groups = e0.OC / kHad, sms = device_info().sm_count;
    return 2 * groups > sms && groups <= sms;
}

template <int USRC, int NB>
static const void *pair_kernel(int kset) {
    switch (kset) {
        case 4: return (const void *)group_pair_kernel<4, USRC, NB>;
        case 8: return (const void *)group_pair_kernel<8, USRC, NB>;
        case 16: return (const void *)group_pair_kernel<16, USRC, NB>;
        case 12: return (const void *)group_pair_kernel<12, USRC, NB>;
        default: return (const void *)group_pair_kernel<28, USRC, NB>;
    }
}

static cudaError_t launch_group_pair(const GroupGemmArgs &a0, int nb, int kset, bool pdl, cudaStream_t s) {
    GroupGemmArgs a = a0;
    a.hash_xor = kHashXor;
    for (int i = 0; i < 17; i++) a.pow2[i] = 1u << i;
    const void *fn = a.codes ? pair_kernel<kUCodes, 1>(kset)
                             : (nb == 2 ? pair_kernel<kUGlobal, 2>(kset) : pair_kernel<kUGlobal, 1>(kset));
    const size_t smem = nb == 2 ? pair_smem<2>() : pair_smem<1>();
    cudaError_t e = kernel_smem_optin(fn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.inline_e[0].OC / kHad));
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void *args[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// --------------------------------------------------------------------------
// MoE FC1 over w1 and w3 of each expert row block, activation rows gathered
// per (token, route) pair, in 16-warp CTAs: warps 0-7 decode a range of w1's
// tile rows and warps 8-15 the same tile rows of w3, at the same time (in
// group_gemm_kernel's paired mode one set of 8 warps runs w1's rows, then w3's,
// each with its own load ramp and reduction).  Units are (column group, tile
// row); when the groups fit the grid each CTA takes one part of one group,
// otherwise ranges split evenly (stream-K).  Split-K across CTAs, the slab
// slots (both accumulator sets) and the epilogue, Had128((silu(g) * u) *
// w2_suh[slot]) as FC2's input, are those of group_gemm_kernel's paired mode.
// Used for few routed pairs (kPairActMaxPairs): with many groups over the grid,
// two 8-warp CTAs per SM measured faster, one CTA's reduction and epilogue
// overlapping the other's decode.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(2 * kDecodeWarps * 32, 1) group_pair_act_kernel(const GroupGemmArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int FRAG = 8 * 4 * 32;
    constexpr int NT = 2 * kDecodeWarps * 32;
    float *red = reinterpret_cast<float *>(smem_raw);   // [w1, w3][8 warps][FRAG]
    GroupEntry *s_ent = reinterpret_cast<GroupEntry *>(red + 2 * kDecodeWarps * FRAG);
    int *s_last = reinterpret_cast<int *>(s_ent + 2);
    const int lane = threadIdx.x & 31;
    const int sub = threadIdx.x >> 8;                             // 0: w1, 1: w3
    const int warp = (threadIdx.x >> 5) & (kDecodeWarps - 1);     // warp within the half
    const int ht = threadIdx.x & (kDecodeWarps * 32 - 1);
    const int A = a.IC / kTile;

    // the entry lists and the gathered rows are the preceding kernel's output
    grid_dependency_wait();
    asm volatile("griddepcontrol.launch_dependents;");
    const int n_groups = (*a.n_entries_dev / 2) * a.n_groups_per_entry;
    const int64_t total = (int64_t)n_groups * A;
    const int c = blockIdx.x;
    int parts = 0, nCTA;
    int64_t f, f_end;
    if (n_groups > 0 && n_groups <= (int)gridDim.x) {
        parts = decode_parts(gridDim.x / n_groups, A);
        nCTA = n_groups * parts;
        if (c >= nCTA) return;
        const int g = c / parts, pp = c - g * parts;
        f = (int64_t)g * A + (int64_t)pp * A / parts;
        f_end = (int64_t)g * A + (int64_t)(pp + 1) * A / parts;
    } else {
        nCTA = (int64_t)gridDim.x < total ? (int)gridDim.x : (int)total;
        if (c >= nCTA) return;
        f = (int64_t)c * total / nCTA;
        f_end = (int64_t)(c + 1) * total / nCTA;
    }
    const uint32_t hx = a.hash_xor;
    while (f < f_end) {
        const int gi = (int)(f / A);
        const int a_lo = (int)(f % A);
        const int a_hi = (int)((int64_t)A < a_lo + (f_end - f) ? (int64_t)A : a_lo + (f_end - f));
        if (threadIdx.x < 2) s_ent[threadIdx.x] = a.entries[2 * (gi / a.n_groups_per_entry) + threadIdx.x];
        __syncthreads();
        const int G = gi % a.n_groups_per_entry;
        {
            const GroupEntry es = s_ent[sub];
            float acc[8][1][4];
#pragma unroll
            for (int j = 0; j < 8; j++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[j][0][q] = 0.f;
            if (es.K == 2) group_accumulate<2, 1, kUGather>(acc, es, a.u, a.IC, G, a_lo, a_hi, lane, warp, hx, a.pow2, a.row_pair, a.R);
            if (es.K == 3) group_accumulate<3, 1, kUGather>(acc, es, a.u, a.IC, G, a_lo, a_hi, lane, warp, hx, a.pow2, a.row_pair, a.R);
            if (es.K == 4) group_accumulate<4, 1, kUGather>(acc, es, a.u, a.IC, G, a_lo, a_hi, lane, warp, hx, a.pow2, a.row_pair, a.R);
            float *rs = red + sub * kDecodeWarps * FRAG;
#pragma unroll
            for (int j = 0; j < 8; j++)
#pragma unroll
                for (int q = 0; q < 4; q++) rs[warp * FRAG + (j * 4 + q) * 32 + lane] = acc[j][0][q];
            if (sub) asm volatile("bar.sync 2, %0;" ::"r"(kDecodeWarps * 32) : "memory");
            else asm volatile("bar.sync 1, %0;" ::"r"(kDecodeWarps * 32) : "memory");
            for (int i = ht; i < FRAG; i += kDecodeWarps * 32) {
                float sum = rs[i];
#pragma unroll
                for (int wv = 1; wv < kDecodeWarps; wv++) sum += rs[wv * FRAG + i];
                rs[i] = sum;
            }
        }
        __syncthreads();
        // element i < 2 FRAG of the reduced sets lives at red[ridx(i)]
        auto ridx = [&](int i) { return (i / FRAG) * (kDecodeWarps * FRAG) + i % FRAG; };

        // ---- split-K across CTAs
        int c_first, c_last;
        if (parts > 0) {
            c_first = gi * parts;
            c_last = c_first + parts - 1;
        } else {
            const int64_t x0 = (int64_t)gi * A, x1 = (int64_t)(gi + 1) * A - 1;
            c_first = (int)(((x0 + 1) * nCTA - 1) / total);
            c_last = (int)(((x1 + 1) * nCTA - 1) / total);
        }
        bool do_epilogue = true;
        if (c_first != c_last) {
            float *slot = a.partials + (int64_t)(c + gi) * (2 * FRAG);
            for (int i = threadIdx.x; i < 2 * FRAG; i += NT) slot[i] = red[ridx(i)];
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) *s_last = atomicAdd(a.counters + gi, 1) == c_last - c_first;
            __syncthreads();
            do_epilogue = *s_last;
            if (do_epilogue) {
                __threadfence();
                // CTA order outermost (each CTA's elements load together); the sum
                // runs in ascending CTA order (deterministic)
                constexpr int PER = 2 * FRAG / NT;
                float sum[PER];
#pragma unroll
                for (int k = 0; k < PER; k++) sum[k] = 0.f;
                for (int cc = c_first; cc <= c_last; cc++) {
                    const float *src = a.partials + (int64_t)(cc + gi) * (2 * FRAG);
#pragma unroll
                    for (int k = 0; k < PER; k++) sum[k] += __ldcg(src + threadIdx.x + k * NT);
                }
#pragma unroll
                for (int k = 0; k < PER; k++) red[ridx(threadIdx.x + k * NT)] = sum[k];
                if (threadIdx.x == 0) a.counters[gi] = 0;
                __syncthreads();
            }
        }

        // ---- epilogue: g = Had128(v_w1) * svh_w1, u = Had128(v_w3) * svh_w3,
        // then FC2's input h2 = Had128((silu(g) * u) * w2_suh[slot]) -> fp16
        if (do_epilogue) {
            const GroupEntry e = s_ent[0], e3 = s_ent[1];
            const int oc0 = G * kHad + 4 * lane;
            const int w16 = threadIdx.x >> 5;
            if (w16 < e.nrows) {
                const uint2 pg = __ldg(reinterpret_cast<const uint2 *>(e.post + oc0));
                const uint2 pu = __ldg(reinterpret_cast<const uint2 *>(e3.post + oc0));
                const uint2 ps = __ldg(reinterpret_cast<const uint2 *>(a.act_suh + (int64_t)e.slot * e.OC + oc0));
                const uint32_t wg[2] = {pg.x, pg.y}, wu[2] = {pu.x, pu.y}, ws[2] = {ps.x, ps.y};
                const int n = w16;
                float vg[4], vu[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    vg[i] = red[frag_index<1>(n, 4 * lane + i)];
                    vu[i] = red[kDecodeWarps * FRAG + frag_index<1>(n, 4 * lane + i)];
                }
                warp_fwht128(vg, lane);
                warp_fwht128(vu, lane);
                float h[4];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int hh = i >> 1, sh = 16 * (i & 1);
                    const float g = (vg[i] * kHadNorm) * f16_bits_to_f32((uint16_t)(wg[hh] >> sh));
                    const float u = (vu[i] * kHadNorm) * f16_bits_to_f32((uint16_t)(wu[hh] >> sh));
                    const float silu = g / (1.0f + __expf(-g));
                    h[i] = (silu * u) * f16_bits_to_f32((uint16_t)(ws[hh] >> sh));
                }
                warp_fwht128(h, lane);
                uint2 o;
                o.x = (uint32_t)f32_to_f16_bits(h[0] * kHadNorm) | ((uint32_t)f32_to_f16_bits(h[1] * kHadNorm) << 16);
                o.y = (uint32_t)f32_to_f16_bits(h[2] * kHadNorm) | ((uint32_t)f32_to_f16_bits(h[3] * kHadNorm) << 16);
                *reinterpret_cast<uint2 *>(a.act_out + (e.out_off + n) * (int64_t)e.OC + oc0) = o;
            }
        }
        __syncthreads();   // red and s_ent are reused by the next segment
        f += a_hi - a_lo;
    }
}

// Routed pairs up to which the paired FC1 runs in group_pair_act_kernel.
constexpr int kPairActMaxPairs = 32;

static cudaError_t launch_group_pair_act(const GroupGemmArgs &a0, bool pdl, cudaStream_t s) {
    constexpr size_t smem = sizeof(float) * 2 * kDecodeWarps * 8 * 4 * 32 + 2 * sizeof(GroupEntry) + 16;
    cudaError_t e = kernel_smem_optin((const void *)group_pair_act_kernel, smem);
    if (e != cudaSuccess) return e;
    GroupGemmArgs a = a0;
    a.hash_xor = kHashXor;
    for (int i = 0; i < 17; i++) a.pow2[i] = 1u << i;
    int64_t grid = device_info().sm_count;
    if (grid > kDecodeMaxCtas) grid = kDecodeMaxCtas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(2 * kDecodeWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, group_pair_act_kernel, a);
}

// --------------------------------------------------------------------------
// Rows mode over device entry lists with few, short column groups (MoE FC2 at
// a few routed pairs: 48 tile rows a group at I = 768): one 16-warp CTA takes
// whole column groups in turn (gi = blockIdx.x, + gridDim.x, ...), its warps
// splitting each group's tile rows three or so apiece, and reduces the group in
// shared memory in fixed warp order: no split-K, and half the rows per warp of
// one 8-warp CTA per group.  The caller uses it when every group can have its
// own CTA (measured at MoE T = 1: 30.8 -> 28.5 us; at T = 2, two groups on some
// CTAs, 40.5 -> 43.6 us).
// --------------------------------------------------------------------------
constexpr int kWideWarps = 2 * kDecodeWarps;

template <int KSET>
__global__ void __launch_bounds__(kWideWarps * 32, 1) group_wide_kernel(const GroupGemmArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int FRAG = 8 * 4 * 32;
    float *red = reinterpret_cast<float *>(smem_raw);   // [16 warps][FRAG]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int A = a.IC / kTile;
    // entry lists written by an earlier launch than the preceding one: read them,
    // and request the first code words, before waiting for the preceding kernel
    const bool hoist = a.entries_ready != 0;
    if (!hoist) grid_dependency_wait();
    asm volatile("griddepcontrol.launch_dependents;");
    const int n_groups = *a.n_entries_dev * a.n_groups_per_entry;
    const uint32_t hx = a.hash_xor;
    for (int gi = blockIdx.x; gi < n_groups; gi += gridDim.x) {
        const GroupEntry e = a.entries[gi / a.n_groups_per_entry];
        const int G = gi % a.n_groups_per_entry;
        float acc[8][1][4];
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int q = 0; q < 4; q++) acc[j][0][q] = 0.f;
        if ((KSET & 4) && e.K == 2)
            group_accumulate<2, 1, kUGlobal, kWideWarps>(acc, e, a.u, a.IC, G, 0, A, lane, warp, hx, a.pow2, nullptr, 0, hoist);
        if ((KSET & 8) && e.K == 3)
            group_accumulate<3, 1, kUGlobal, kWideWarps>(acc, e, a.u, a.IC, G, 0, A, lane, warp, hx, a.pow2, nullptr, 0, hoist);
        if ((KSET & 16) && e.K == 4)
            group_accumulate<4, 1, kUGlobal, kWideWarps>(acc, e, a.u, a.IC, G, 0, A, lane, warp, hx, a.pow2, nullptr, 0, hoist);
        // the outputs and the combine counters are shared with the preceding kernel
        if (hoist) grid_dependency_wait();
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int q = 0; q < 4; q++) red[warp * FRAG + (j * 4 + q) * 32 + lane] = acc[j][0][q];
        __syncthreads();
        for (int i = threadIdx.x; i < FRAG; i += kWideWarps * 32) {
            float sum = red[i];
#pragma unroll
            for (int wv = 1; wv < kWideWarps; wv++) sum += red[wv * FRAG + i];
            red[i] = sum;
        }
        __syncthreads();
        group_output<1>(a, red, e, G, lane, warp, kWideWarps);
        __syncthreads();   // red is reused by the next group
    }
}

static cudaError_t launch_group_wide(const GroupGemmArgs &a0, bool pdl, cudaStream_t s) {
    constexpr size_t smem = sizeof(float) * kWideWarps * 8 * 4 * 32;
    cudaError_t e = kernel_smem_optin((const void *)group_wide_kernel<28>, smem);
    if (e != cudaSuccess) return e;
    GroupGemmArgs a = a0;
    a.hash_xor = kHashXor;
    for (int i = 0; i < 17; i++) a.pow2[i] = 1u << i;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)device_info().sm_count);
    cfg.blockDim = dim3(kWideWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, group_wide_kernel<28>, a);
}

template <int NB, int KSET, int USRC = kUGlobal, bool PAIR = false>
static cudaError_t launch_group_t(const GroupGemmArgs &a0, bool pdl, int64_t total_hint, cudaStream_t s) {
    constexpr size_t smem = group_smem_bytes<NB, PAIR>();
    int occ = 1;
    cudaError_t e = kernel_occupancy((const void *)group_gemm_kernel<NB, KSET, USRC, PAIR>, 256, smem, &occ);
    if (e != cudaSuccess) return e;
    GroupGemmArgs a = a0;
    a.hash_xor = kHashXor;
    for (int i = 0; i < 17; i++) a.pow2[i] = 1u << i;
    int64_t grid = (int64_t)device_info().sm_count * occ;
    if (grid > kDecodeMaxCtas) grid = kDecodeMaxCtas;
    a.parts = 0;
    const int64_t A = a.IC / kTile;
    if (total_hint > 0 && !a.n_entries_dev && a.n_groups_per_entry == 0) {
        // column groups known on the host: when they fit in one wave, give every CTA
        // one part of one group (no group switches inside a CTA, equal work per CTA)
        const int64_t groups = total_hint / A;
        if (groups > 0 && groups <= grid) {
            const int parts = decode_parts((int)(grid / groups), (int)A);
            a.parts = parts;
            grid = groups * parts;
        }
    }
    if (total_hint > 0 && grid > total_hint) grid = total_hint;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, group_gemm_kernel<NB, KSET, USRC, PAIR>, a);
}

template <int NB>
static cudaError_t launch_group_nb(const GroupGemmArgs &a, int kset, bool pdl, int64_t total, cudaStream_t s) {
    switch (kset) {
        case 4: return launch_group_t<NB, 4>(a, pdl, total, s);
        case 8: return launch_group_t<NB, 8>(a, pdl, total, s);
        case 16: return launch_group_t<NB, 16>(a, pdl, total, s);
        case 12: return launch_group_t<NB, 12>(a, pdl, total, s);
        default: return launch_group_t<NB, 28>(a, pdl, total, s);
    }
}

size_t group_slab_floats(int max_groups, int nb) {
    return (size_t)(kDecodeMaxCtas + max_groups) * (8 * nb * 4 * 32);
}

cudaError_t launch_group_gemm(const GroupGemmArgs &a, int nb, bool pdl, cudaStream_t s) {
    // total units when known on the host (dense): never launch more CTAs than units
    int64_t total = -1;
    int kset = 28;
    if (!a.n_entries_dev) {
        int64_t groups = 0;
        kset = 0;
        for (int i = 0; i < a.n_inline; i++) {
            groups += a.inline_e[i].OC / kHad;
            kset |= 1 << a.inline_e[i].K;
        }
        total = groups * (a.IC / kTile);
    }
    if (a.wide) {
        // whole short groups per 16-warp CTA: rows mode over device entry lists, one 8-row block of fp16 rows
        if (nb != 1 || a.gather || a.pair_act || a.codes || a.mode != kModeRows || !a.entries || !a.n_entries_dev ||
            a.n_groups_per_entry <= 0)
            return cudaErrorInvalidValue;
        return launch_group_wide(a, pdl, s);
    }
    if (a.gather) {
        // grouped MoE with activation rows stored per pair: one 8-row block per entry, any K
        if (nb != 1 || a.codes) return cudaErrorInvalidValue;
        // few routed pairs: w1 and w3 side by side in 16-warp CTAs; many: two 8-warp
        // CTAs per SM, whose reductions and epilogues overlap each other's decode
        // (measured: T = 1 32.2 -> 30.8 us and T = 4 69.6 -> 64.9 us with the first;
        // T = 16 131.0 -> 134.4 us and T = 64 192.4 -> 197.6 us)
        if (a.pair_act)
            return a.R <= kPairActMaxPairs ? launch_group_pair_act(a, pdl, s)
                                           : launch_group_t<1, 28, kUGather, true>(a, pdl, total, s);
        return launch_group_t<1, 28, kUGather>(a, pdl, total, s);
    }
    if (a.pair_act) return cudaErrorInvalidValue;
    if (pair_launch_fits(a, nb)) return launch_group_pair(a, nb, kset, pdl, s);
    if (a.codes) {
        // 8-bit activation codes: one 8-row block per entry
        if (nb != 1) return cudaErrorInvalidValue;
        switch (kset) {
            case 4: return launch_group_t<1, 4, kUCodes>(a, pdl, total, s);
            case 8: return launch_group_t<1, 8, kUCodes>(a, pdl, total, s);
            case 16: return launch_group_t<1, 16, kUCodes>(a, pdl, total, s);
            default: return launch_group_t<1, 28, kUCodes>(a, pdl, total, s);
        }
    }
    if (nb == 3) nb = 4;
    switch (nb) {
        case 1: return launch_group_nb<1>(a, kset, pdl, total, s);
        case 2: return launch_group_nb<2>(a, kset, pdl, total, s);
        case 4: return launch_group_nb<4>(a, kset, pdl, total, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace exl3
