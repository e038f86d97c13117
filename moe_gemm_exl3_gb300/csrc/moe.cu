// moe.cu -- grouped SiLU-gated MoE over an EXL3 expert bank (bank.py layout:
// w13 = [w1 | w3] per K-sorted slot, w2, fp16 suh/svh vectors [E, ...]).
//
// Launch chain, all on the caller's stream, no host synchronization:
//   top-k     (from router logits) ids and softmax weights, one warp per token;
//             for a few tokens inside the routing launch
//   route     ids -> expert-sorted rows (stable counting sort), per-row slot,
//             per-pair row position, and the grouped-GEMM entry lists
//   rotate    u1 = Had(x_t * w13_suh[p][0]), u3 = Had(x_t * w13_suh[p][1]) per
//             routed row, or (one 8-row block per entry) per (token, route) pair
//             in the same launch as the routing
//   FC1       grouped trellis GEMM over (slot, row block) x {w1, w3}, epilogue
//             Had(v) * w13_svh -> fp32 rows
//   act       h = silu(g) * u, then FC2's input transform Had(h * w2_suh[p])
//   FC2       grouped trellis GEMM over (slot, row block), epilogue
//             Had(v) * w2_svh -> fp32 rows; with one 8-row block per entry the
//             epilogue also combines (below)
//   combine   y_t = sum over k (in order) of w[t][k] * d[pos(t,k)] -> bf16: the
//             last of a token's routes to finish a column group sums them
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
}  // namespace exl3

using namespace exl3;

namespace {

constexpr int kMoeMaxE = 1024;
constexpr int kMoeMaxTopk = 32;
// The three-kernel chain's combine counters (one per token and column group of
// y) sit in the upper half of the workspace counters; the grouped GEMMs' split-K
// counters use the lower half.
constexpr int64_t kCombCounterBase = 32768;
// Tokens up to which the small-T chain folds the top-k into its first launch.
constexpr int kFoldTopkTokens = 8;

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Rows per grouped-GEMM entry: an expert gets at most T rows (a token routes to
// an expert at most once), so small batches need only small row blocks.
// Row blocks (of 8) per decode-mode entry, from the mean rows per expert: one
// block costs ~22 % less per code byte than two, and an expert with more rows
// than a block just gets more entries, so wider blocks only pay once most
// experts fill them.
int moe_nb(int R, int E) { return R <= 4 * E ? 1 : (R <= 8 * E ? 2 : 4); }

struct MoeLayout {
    size_t pos, row_pair, row_slot, counts, ent1, ent2, u13, st1, h2, st2, slab, total;
    int R, chunk, max_entries, nb;
    bool fused;   // FC1 and FC2 on the fused tensor-core GEMM (rows mode) instead of the decode-mode GEMM
};

// The fused tensor-core GEMM pays off once experts average 16 or more rows
// (measured on E = 128, H = 2048, I = 768: T = 512 averages 32).
bool moe_fused(int T, int H, int I, int E, int topk) {
    const int force = forced_mode();
    if (force == 1 || !fused_supported()) return false;
    const int64_t R = (int64_t)T * topk;
    if (force != 2 && R < 16 * (int64_t)E) return false;
    const int active = E < R ? E : (int)R;
    const int64_t max_entries = (R + kFusedRowsNT - 1) / kFusedRowsNT + active;
    return fused_rows_fits(2 * max_entries, I / kHad, H) && fused_rows_fits(max_entries, H / kHad, I);
}

// Tokens one pass of the layer serves.  Every grouped-GEMM column group of a
// launch owns one workspace arrival counter; a launch has at most
// G * (ceil(R / 8) + E) groups (G column groups per entry, R = T * topk routed
// rows, row blocks of at least 8), so passes of this many tokens never run out
// of counters.  Longer calls run as several passes.  0: not even one token fits.
int64_t moe_pass_tokens(int H, int I, int E, int topk) {
    const int64_t G = 2 * (I / kHad) > H / kHad ? 2 * (I / kHad) : H / kHad;
    const int64_t entries = (int64_t)kWorkspaceCounters / G - 1 - E;
    return entries > 0 ? entries * 8 / topk : 0;
}

MoeLayout moe_layout(int T, int H, int I, int E, int topk) {
    MoeLayout L = {};
    L.R = T * topk;
    L.nb = moe_nb(L.R, E);
    L.fused = moe_fused(T, H, I, E, topk);
    L.chunk = L.fused ? kFusedRowsNT : 8 * L.nb;
    const int active = E < L.R ? E : L.R;
    L.max_entries = (L.R + L.chunk - 1) / L.chunk + active;
    size_t off = fixed_workspace_bytes();
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    L.pos = take(sizeof(int32_t) * L.R);
    L.row_pair = take(sizeof(int32_t) * L.R);
    L.row_slot = take(sizeof(int32_t) * L.R);
    L.counts = take(sizeof(int32_t) * 4);                     // rows, entries FC1, entries FC2
    L.ent1 = take(sizeof(GroupEntry) * 2 * L.max_entries);
    L.ent2 = take(sizeof(GroupEntry) * L.max_entries);
    L.u13 = take(sizeof(uint16_t) * 2 * (size_t)L.R * H);
    L.st1 = take(sizeof(float) * 2 * (size_t)L.R * I);
    L.h2 = take(sizeof(uint16_t) * (size_t)L.R * I);
    L.st2 = take(sizeof(float) * (size_t)L.R * H);
    const int groups1 = 2 * L.max_entries * (I / kHad), groups2 = L.max_entries * (H / kHad);
    const int gmax = groups1 > groups2 ? groups1 : groups2;
    // one 8-row block per entry: FC1 may run paired, one column group per (expert
    // row block, 128 columns of I) with two accumulator sets per slab slot
    size_t dec_slab = group_slab_floats(gmax, L.nb);
    if (L.nb == 1) {
        const size_t paired = 2 * group_slab_floats(L.max_entries * (I / kHad), 1);
        if (paired > dec_slab) dec_slab = paired;
    }
    L.slab = take(sizeof(float) * (L.fused ? fused_slab_floats(gmax, kFusedRowsNT) : dec_slab));
    L.total = off;
    return L;
}

// ------------------------------------------------------------------ top-k
// One warp per token: each lane holds the logits e = lane, lane + 32, ... (PER of
// them, E <= 32 PER); each of the topk rounds is a warp arg-max (largest logit,
// ties to the lower expert id); then softmax over the selected logits.  Lane
// k < topk ends with the k-th choice's expert id (*id) and weight (*wt).
template <int PER>
__device__ __forceinline__ void topk_warp_n(const float *__restrict__ l, int E, int topk, int lane, int *id,
                                            float *wt) {
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; i++) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(l + e) : -INFINITY;
    }
    uint32_t taken = 0;     // bit i: logit lane + 32 i already selected
    float sel0 = 0.f, den = 0.f, my_sel = 0.f;
    for (int k = 0; k < topk; k++) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < PER; i++) {
            const int e = lane + 32 * i;
            if (e < E && !(taken & (1u << i)) && (v[i] > bv || be == 0x7FFFFFFF)) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, off);
            const int oe = __shfl_xor_sync(kFull, be, off);
            if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (k == 0) sel0 = bv;
        const float ex = expf(bv - sel0);
        den += ex;
        if (lane == k) {
            my_sel = ex;
            *id = be;
        }
    }
    *wt = my_sel / den;
}

// The rounds run over as few logits per lane as E needs (each round is on the
// layer's critical path): 4 per lane for E <= 128.
__device__ __forceinline__ void topk_warp(const float *__restrict__ l, int E, int topk, int lane, int *id,
                                          float *wt) {
    static_assert(kMoeMaxE == 32 * 32, "the widest instance holds 32 logits per lane");
    if (E <= 128)
        topk_warp_n<4>(l, E, topk, lane, id, wt);
    else if (E <= 256)
        topk_warp_n<8>(l, E, topk, lane, id, wt);
    else if (E <= 512)
        topk_warp_n<16>(l, E, topk, lane, id, wt);
    else
        topk_warp_n<32>(l, E, topk, lane, id, wt);
}

__global__ void __launch_bounds__(256) topk_softmax_kernel(const float *__restrict__ logits, int T, int E, int topk,
                                                           int32_t *__restrict__ ids, float *__restrict__ w) {
    // the routing kernel that follows may be scheduled now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");
    // launched as a programmatic dependent itself: wait for the preceding kernel
    // before reading the logits or writing ids and w
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    int id = 0;
    float wt = 0.f;
    topk_warp(logits + (int64_t)t * E, E, topk, lane, &id, &wt);
    if (lane < topk) {
        ids[(int64_t)t * topk + lane] = id;
        w[(int64_t)t * topk + lane] = wt;
    }
}

// One warp per token, as a programmatic dependent of the preceding kernel.
cudaError_t launch_topk(const float *logits, int T, int E, int topk, int32_t *ids, float *w, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((T + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_softmax_kernel, logits, T, E, topk, ids, w);
}

// ------------------------------------------------------------------ route
struct RouteArgs {
    const int32_t *ids;
    int R, topk, E, H, I, chunk;
    exl3_moe_bank bank;
    int32_t *pos, *row_pair, *row_slot, *counts;
    GroupEntry *ent1, *ent2;
    int32_t *err;
    uint16_t *y_zero;   // non-null: write zero rows y[t] for tokens with no valid route
};

constexpr int kRouteParE = 128;   // slots up to which the stable ranking runs on all warps at once
constexpr int kRouteRegPairs = 8; // pairs per lane that the ranking keeps in registers (fast path)

// One CTA of 1024 threads.  Rows of one slot are ordered by pair index (stable),
// so the row -> entry assignment, and with it every partial sum, is the same on
// every run.  With E <= kRouteParE each warp ranks a contiguous chunk of pairs
// starting from its own per-slot cursor (the counts of the chunks before it);
// otherwise one warp walks all pairs.  When a warp's chunk is at most
// 32 * kRouteRegPairs pairs (fast path), its lanes keep the pairs' slots in
// registers from the count to the ranking, read the expert tables from shared
// memory, and write each row's pair and slot as soon as the row is known.
__device__ __forceinline__ void route_body(const RouteArgs &a) {
    __shared__ int cnt[kMoeMaxE], base[kMoeMaxE], ebase[kMoeMaxE], cursor[kMoeMaxE];
    __shared__ int wcur[32][kRouteParE];     // per warp and slot: pairs in the chunk, then its cursor
    __shared__ int s_perm[kRouteParE], s_kgu[kRouteParE], s_kd[kRouteParE];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, W = blockDim.x >> 5;
    const bool par = a.E <= kRouteParE;
    const int C = ((a.R + W - 1) / W + 31) & ~31;              // pairs per warp chunk
    const int c_lo = w * C, c_hi = (w + 1) * C < a.R ? (w + 1) * C : a.R;
    const bool fast = par && C <= 32 * kRouteRegPairs;
    for (int p = tid; p < a.E; p += blockDim.x) { cnt[p] = 0; cursor[p] = 0; }
    if (par) {
        for (int i = tid; i < W * kRouteParE; i += blockDim.x) (&wcur[0][0])[i] = 0;
        for (int e = tid; e < a.E; e += blockDim.x) {
            s_perm[e] = a.bank.perm[e];
            s_kgu[e] = a.bank.k_gu[e];
            s_kd[e] = a.bank.k_d[e];
        }
    }
    __syncthreads();
    // slot of expert id e, or -1 (invalid id, slot or bitrate: recorded, routed nowhere)
    auto slot_of = [&](int e) {
        int p = -1;
        if (e >= 0 && e < a.E) p = par ? s_perm[e] : a.bank.perm[e];
        if (p >= 0 && p < a.E) {
            const int kg = par ? s_kgu[p] : a.bank.k_gu[p], kd = par ? s_kd[p] : a.bank.k_d[p];
            if (kg < 2 || kg > 4 || kd < 2 || kd > 4) p = -1;
        } else {
            p = -1;
        }
        if (p < 0) record_error(a.err, kErrBadExpertId);
        return p;
    };
    int pr[kRouteRegPairs];   // fast path: slot of pair c_lo + 32 k + lane (-2: no pair)
    if (fast) {
#pragma unroll
        for (int k = 0; k < kRouteRegPairs; k++) {
            const int i = c_lo + 32 * k + lane;
            pr[k] = i < c_hi ? a.ids[i] : 0;
        }
#pragma unroll
        for (int k = 0; k < kRouteRegPairs; k++) {
            const int i = c_lo + 32 * k + lane;
            if (i < c_hi) {
                pr[k] = slot_of(pr[k]);
                if (pr[k] >= 0) {
                    atomicAdd(&cnt[pr[k]], 1);
                    atomicAdd(&wcur[w][pr[k]], 1);
                }
            } else {
                pr[k] = -2;
            }
        }
    }
    // pass 1: slot of every pair, counted per slot (and per warp chunk)
    const int i_first = par ? c_lo + lane : tid, i_step = par ? 32 : (int)blockDim.x, i_end = par ? c_hi : a.R;
    for (int i = i_first; i < i_end && !fast; i += i_step) {
        const int p = slot_of(a.ids[i]);
        if (p >= 0) {
            atomicAdd(&cnt[p], 1);
            if (par) atomicAdd(&wcur[w][p], 1);
        }
        a.row_slot[i] = p;   // scratch: slot per pair (overwritten below with slot per row)
    }
    __syncthreads();
    // exclusive scans of rows and row chunks over the slots (E <= 1024 = one value per
    // thread): warp scans, then a scan of the warp totals
    {
        __shared__ int wsum_r[32], wsum_c[32];
        const int vr = tid < a.E ? cnt[tid] : 0;
        const int vc = tid < a.E ? (vr + a.chunk - 1) / a.chunk : 0;
        int ir = vr, ic = vc;   // inclusive within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tr = __shfl_up_sync(kFull, ir, o), tc = __shfl_up_sync(kFull, ic, o);
            if (lane >= o) { ir += tr; ic += tc; }
        }
        if (lane == 31) { wsum_r[w] = ir; wsum_c[w] = ic; }
        __syncthreads();
        if (w == 0) {
            int xr = lane < W ? wsum_r[lane] : 0, xc = lane < W ? wsum_c[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tr = __shfl_up_sync(kFull, xr, o), tc = __shfl_up_sync(kFull, xc, o);
                if (lane >= o) { xr += tr; xc += tc; }
            }
            if (lane < W) { wsum_r[lane] = xr; wsum_c[lane] = xc; }   // inclusive warp prefix
            if (lane == 31) {
                a.counts[0] = xr;
                a.counts[1] = 2 * xc;
                a.counts[2] = xc;
            }
        }
        __syncthreads();
        if (tid < a.E) {
            base[tid] = ir - vr + (w > 0 ? wsum_r[w - 1] : 0);
            ebase[tid] = ic - vc + (w > 0 ? wsum_c[w - 1] : 0);
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    if (par) {
        // each warp's starting cursor per slot: the slot's base plus the earlier chunks' counts
        for (int p = tid; p < a.E; p += blockDim.x) {
            int run = base[p];
            for (int ww = 0; ww < W; ww++) {
                const int t = wcur[ww][p];
                wcur[ww][p] = run;
                run += t;
            }
        }
        __syncthreads();
        if (fast) {
#pragma unroll
            for (int k = 0; k < kRouteRegPairs; k++) {
                const int i = c_lo + 32 * k + lane;
                if (c_lo + 32 * k >= c_hi) break;
                const int p = pr[k];
                const unsigned peers = __match_any_sync(kFull, p);
                const int rank = __popc(peers & lt);
                int position = -1;
                if (p >= 0) position = wcur[w][p] + rank;
                __syncwarp();
                if (p >= 0 && (peers & lt) == 0) wcur[w][p] += __popc(peers);
                __syncwarp();
                if (i < c_hi) a.pos[i] = position;
                if (position >= 0) {
                    a.row_pair[position] = i;
                    a.row_slot[position] = p;
                }
            }
        }
        for (int i0 = c_lo; i0 < c_hi && !fast; i0 += 32) {
            const int i = i0 + lane;
            const int p = i < c_hi ? a.row_slot[i] : -2;
            const unsigned peers = __match_any_sync(kFull, p);
            const int rank = __popc(peers & lt);
            int position = -1;
            if (p >= 0) position = wcur[w][p] + rank;
            __syncwarp();
            if (p >= 0 && (peers & lt) == 0) wcur[w][p] += __popc(peers);
            __syncwarp();
            if (i < c_hi) a.pos[i] = position;
        }
    } else if (tid < 32) {
        // stable positions: warp 0 walks the pairs 32 at a time
        for (int i0 = 0; i0 < a.R; i0 += 32) {
            const int i = i0 + tid;
            const int p = i < a.R ? a.row_slot[i] : -2;
            const unsigned peers = __match_any_sync(kFull, p);
            const int rank = __popc(peers & lt);
            int position = -1;
            if (p >= 0) position = base[p] + cursor[p] + rank;
            __syncwarp();
            if (p >= 0 && (peers & lt) == 0) cursor[p] += __popc(peers);
            __syncwarp();
            if (i < a.R) a.pos[i] = position;
        }
    }
    if (!fast) {
        __syncthreads();
        for (int i = tid; i < a.R; i += blockDim.x) {
            const int r = a.pos[i];
            if (r >= 0) a.row_pair[r] = i;
        }
        __syncthreads();
        // slot per row (after every pair read its slot above)
        for (int i = tid; i < a.R; i += blockDim.x) {
            const int r = a.pos[i];
            const int e = a.ids[i];
            if (r >= 0) a.row_slot[r] = a.bank.perm[e];
        }
    }
    // grouped-GEMM entries: one per (slot, block of `chunk` rows); FC1 has a w1 and a w3 entry
    for (int p = tid; p < a.E; p += blockDim.x) {
        const int n = cnt[p];
        for (int c = 0; c * a.chunk < n; c++) {
            const int r0 = base[p] + c * a.chunk;
            const int nr = n - c * a.chunk < a.chunk ? n - c * a.chunk : a.chunk;
            const int idx = ebase[p] + c;
            for (int j = 0; j < 2; j++) {
                GroupEntry ge = {};
                ge.code = a.bank.w13 + (j == 0 ? a.bank.off_w1[p] : a.bank.off_w3[p]);
                ge.post = a.bank.w13_svh + ((int64_t)p * 2 + j) * a.I;
                ge.post2 = nullptr;
                ge.K = a.bank.k_gu[p];
                ge.OC = a.I;
                ge.u_row0 = j * a.R + r0;
                ge.out_off = j * a.R + r0;
                ge.nrows = nr;
                ge.slot = p;
                a.ent1[2 * idx + j] = ge;
            }
            GroupEntry ge = {};
            ge.code = a.bank.w2 + a.bank.off_w2[p];
            ge.post = a.bank.w2_svh + (int64_t)p * a.H;
            ge.post2 = nullptr;
            ge.K = a.bank.k_d[p];
            ge.OC = a.H;
            ge.u_row0 = r0;
            ge.out_off = r0;
            ge.nrows = nr;
            a.ent2[idx] = ge;
        }
    }
    if (a.y_zero) {
        // tokens whose routes are all invalid get y = 0 (no combine reaches them)
        __syncthreads();
        const int T = a.R / a.topk;
        for (int t = tid; t < T; t += blockDim.x) {
            bool any = false;
            for (int k = 0; k < a.topk; k++) any |= a.pos[(int64_t)t * a.topk + k] >= 0;
            if (!any)
                for (int c = 0; c < a.H; c += 8)
                    *reinterpret_cast<uint4 *>(a.y_zero + (int64_t)t * a.H + c) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

__global__ void __launch_bounds__(1024) route_kernel(const RouteArgs a) { route_body(a); }

// The routing of at most 32 (token, choice) pairs by one warp, lane i holding pair
// i: ranking the keys (slot, pair index) gives route_body's stable slot-major row
// order, and with it the same positions, rows, entry lists and counts, without
// the CTA-wide passes (tables, scans, barriers) that dominate it for a few pairs.
__device__ __forceinline__ void route_small(const RouteArgs &a, int lane) {
    int p = -1;
    if (lane < a.R) {
        const int e = a.ids[lane];
        if (e >= 0 && e < a.E) p = a.bank.perm[e];
        if (p >= 0 && p < a.E) {
            const int kg = a.bank.k_gu[p], kd = a.bank.k_d[p];
            if (kg < 2 || kg > 4 || kd < 2 || kd > 4) p = -1;
        } else {
            p = -1;
        }
        if (p < 0) record_error(a.err, kErrBadExpertId);
    }
    const bool valid = p >= 0;
    const unsigned key = valid ? ((unsigned)p << 5) | (unsigned)lane : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(kFull, valid ? p : -1 - lane);   // lanes of the same slot
    const int n = __popc(peers);                                             // rows of this slot
    const bool leader = valid && (__ffs(peers) - 1) == lane;                 // its lowest pair
    const int nchunks = leader ? (n + a.chunk - 1) / a.chunk : 0;
    int rank = 0, ebase = 0, entries = 0;
    for (int j = 0; j < 32; j++) {
        const unsigned kj = __shfl_sync(kFull, key, j);
        const int cj = __shfl_sync(kFull, nchunks, j);
        rank += kj < key;                                   // rows before this one
        ebase += (kj >> 5) < (key >> 5) ? cj : 0;          // entries of the slots before this one
        entries += cj;
    }
    const int rows = __popc(__ballot_sync(kFull, valid));
    if (lane < a.R) a.pos[lane] = valid ? rank : -1;
    if (valid) {
        a.row_pair[rank] = lane;
        a.row_slot[rank] = p;
    }
    if (lane == 0) {
        a.counts[0] = rows;
        a.counts[1] = 2 * entries;
        a.counts[2] = entries;
    }
    for (int c = 0; c < nchunks; c++) {
        const int r0 = rank + c * a.chunk;               // the leader's rank is its slot's first row
        const int nr = n - c * a.chunk < a.chunk ? n - c * a.chunk : a.chunk;
        const int idx = ebase + c;
        for (int j = 0; j < 2; j++) {
            GroupEntry ge = {};
            ge.code = a.bank.w13 + (j == 0 ? a.bank.off_w1[p] : a.bank.off_w3[p]);
            ge.post = a.bank.w13_svh + ((int64_t)p * 2 + j) * a.I;
            ge.post2 = nullptr;
            ge.K = a.bank.k_gu[p];
            ge.OC = a.I;
            ge.u_row0 = j * a.R + r0;
            ge.out_off = j * a.R + r0;
            ge.nrows = nr;
            ge.slot = p;
            a.ent1[2 * idx + j] = ge;
        }
        GroupEntry ge = {};
        ge.code = a.bank.w2 + a.bank.off_w2[p];
        ge.post = a.bank.w2_svh + (int64_t)p * a.H;
        ge.post2 = nullptr;
        ge.K = a.bank.k_d[p];
        ge.OC = a.H;
        ge.u_row0 = r0;
        ge.out_off = r0;
        ge.nrows = nr;
        a.ent2[idx] = ge;
    }
    if (a.y_zero) {
        // tokens whose routes are all invalid get y = 0 (no combine reaches them)
        const unsigned vb = __ballot_sync(kFull, valid);
        const unsigned mk = a.topk >= 32 ? 0xFFFFFFFFu : (1u << a.topk) - 1u;
        const int T = a.R / a.topk;
        for (int t = 0; t < T; t++) {
            if ((vb >> (t * a.topk)) & mk) continue;
            for (int c = 8 * lane; c < a.H; c += 8 * 32)
                *reinterpret_cast<uint4 *>(a.y_zero + (int64_t)t * a.H + c) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Input rotation per (token, route) pair, before the rows are known:
// u[j][i] = Had(x_t * w13_suh[p][j]) for pair i = t * topk + k routed to slot p
// (pairs whose expert id, slot or bitrate is invalid are skipped; the routing
// records them).
struct PairRotateArgs {
    const uint16_t *x;
    const int32_t *ids;
    int R, topk, E, H;
    exl3_moe_bank bank;
    uint16_t *u;         // fp16 [2][R][H]
    const float *logits; // non-null: the ids are this launch's own top-k of the logits [T][E]
};

__device__ __forceinline__ void rotate_pairs(const PairRotateArgs &a, int wid, int nwarps, int lane) {
    const int blocks = a.H / kHad;
    int t_have = -1, id_have = 0;   // the token whose top-k this warp holds, lane k's choice
    for (int task = wid; task < a.R * blocks; task += nwarps) {
        const int i = task / blocks, c = (task - i * blocks) * kHad + 4 * lane;
        int e;
        if (a.logits) {
            // the warp ranks the token's logits itself (the same result as the routing
            // CTA's, which writes ids and w) rather than wait for another CTA
            const int t = i / a.topk;
            if (t != t_have) {
                float unused;
                topk_warp(a.logits + (int64_t)t * a.E, a.E, a.topk, lane, &id_have, &unused);
                t_have = t;
            }
            e = __shfl_sync(kFull, id_have, i - t * a.topk);
        } else {
            e = a.ids[i];
        }
        if (e < 0 || e >= a.E) continue;
        const int p = a.bank.perm[e];
        if (p < 0 || p >= a.E) continue;
        const int kg = a.bank.k_gu[p], kd = a.bank.k_d[p];
        if (kg < 2 || kg > 4 || kd < 2 || kd > 4) continue;
        const int t = i / a.topk;
        const uint2 xv = *reinterpret_cast<const uint2 *>(a.x + (int64_t)t * a.H + c);
        uint2 sv[2];
#pragma unroll
        for (int j = 0; j < 2; j++) sv[j] = __ldg(reinterpret_cast<const uint2 *>(a.bank.w13_suh + ((int64_t)p * 2 + j) * a.H + c));
        const uint32_t xs[2] = {xv.x, xv.y};
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const uint32_t ss[2] = {sv[j].x, sv[j].y};
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; k++)
                v[k] = bf16_bits_to_f32((xs[k >> 1] >> (16 * (k & 1))) & 0xFFFFu) *
                       f16_bits_to_f32((uint16_t)(ss[k >> 1] >> (16 * (k & 1))));
            warp_fwht128(v, lane);
            uint2 o;
            o.x = (uint32_t)f32_to_f16_bits(v[0] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[1] * kHadNorm) << 16);
            o.y = (uint32_t)f32_to_f16_bits(v[2] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[3] * kHadNorm) << 16);
            *reinterpret_cast<uint2 *>(a.u + ((int64_t)j * a.R + i) * a.H + c) = o;
        }
    }
}

// The first kernel of the small-T chain: CTA 0 routes, the others rotate the
// pairs' inputs meanwhile (both need only the ids).  With router logits (r.logits
// non-null) CTA 0 first takes each token's top-k (one warp per token) and writes
// them to ids_out (the ids the routing reads) and w_out, and every rotating warp
// ranks its own token's logits.
__global__ void __launch_bounds__(1024) route_rotate_kernel(const RouteArgs a, const PairRotateArgs r,
                                                            int32_t *ids_out, float *w_out) {
    // launched as a dependent of the kernel that wrote the ids or the logits: wait
    // for it; let FC1 be scheduled
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (blockIdx.x == 0) {
        if (r.logits) {
            const int lane = threadIdx.x & 31, T = a.R / a.topk;
            for (int t = threadIdx.x >> 5; t < T; t += blockDim.x >> 5) {
                int id = 0;
                float wt = 0.f;
                topk_warp(r.logits + (int64_t)t * a.E, a.E, a.topk, lane, &id, &wt);
                if (lane < a.topk) {
                    ids_out[(int64_t)t * a.topk + lane] = id;
                    w_out[(int64_t)t * a.topk + lane] = wt;
                }
            }
            __syncthreads();   // the routing below reads the ids
        }
        if (a.R <= 32) {
            if (threadIdx.x < 32) route_small(a, threadIdx.x);
            return;
        }
        route_body(a);
        return;
    }
    rotate_pairs(r, (blockIdx.x - 1) * (blockDim.x >> 5) + (threadIdx.x >> 5), (gridDim.x - 1) * (blockDim.x >> 5),
                 threadIdx.x & 31);
}

// ------------------------------------------------------------------ rotate
// One warp per (row, projection j, 128-block): u[j*R + r] = Had(x_t * suh[p][j]).
__global__ void __launch_bounds__(256) rotate_kernel(const uint16_t *__restrict__ x, int H, int R, int topk,
                                                     const uint16_t *__restrict__ suh,
                                                     const int32_t *__restrict__ row_pair,
                                                     const int32_t *__restrict__ row_slot,
                                                     const int32_t *__restrict__ counts,
                                                     uint16_t *__restrict__ u, int parts) {
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    // `parts` warps per row (many when there are few rows), each a contiguous run of 128-blocks
    const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int r = wid / parts, part = wid - r * parts;
    if (r >= R || r >= counts[0]) return;
    const int span = H / parts;                                  // channels per warp, a multiple of 128
    const int c_begin = part * span, c_end = c_begin + span;
    const int t = row_pair[r] / topk;
    const int p = row_slot[r];
    const uint16_t *xr = x + (int64_t)t * H;
    const uint16_t *sj[2] = {suh + (int64_t)p * 2 * H, suh + ((int64_t)p * 2 + 1) * H};
    uint16_t *uj[2] = {u + (int64_t)r * H, u + ((int64_t)R + r) * H};
    // two 128-blocks per iteration, every load issued before the transforms; the
    // token's x block serves both projections
    for (int c0 = c_begin + 4 * lane; c0 < c_end; c0 += 2 * kHad) {
        const bool two = c0 + kHad < c_end;
        uint2 xv[2], sv[2][2];
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int c = c0 + h * kHad;
            if (h == 0 || two) {
                xv[h] = *reinterpret_cast<const uint2 *>(xr + c);
                sv[h][0] = __ldg(reinterpret_cast<const uint2 *>(sj[0] + c));
                sv[h][1] = __ldg(reinterpret_cast<const uint2 *>(sj[1] + c));
            }
        }
#pragma unroll
        for (int h = 0; h < 2; h++) {
            if (h == 1 && !two) break;
            const int c = c0 + h * kHad;
            const uint32_t xs[2] = {xv[h].x, xv[h].y};
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const uint32_t ss[2] = {sv[h][j].x, sv[h][j].y};
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    v[i] = bf16_bits_to_f32((xs[i >> 1] >> (16 * (i & 1))) & 0xFFFFu) *
                           f16_bits_to_f32((uint16_t)(ss[i >> 1] >> (16 * (i & 1))));
                warp_fwht128(v, lane);
                uint2 o;
                o.x = (uint32_t)f32_to_f16_bits(v[0] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[1] * kHadNorm) << 16);
                o.y = (uint32_t)f32_to_f16_bits(v[2] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[3] * kHadNorm) << 16);
                *reinterpret_cast<uint2 *>(uj[j] + c) = o;
            }
        }
    }
}

// ------------------------------------------------------------------ act
// One warp per (row, 128-block of I): h = silu(g) * u, then FC2's input
// transform h2 = Had(h * w2_suh[p]).  g and u already carry their output Had
// and svh scale (FC1 epilogue).
__global__ void __launch_bounds__(256) act_kernel(const float *__restrict__ st1, int I, int R,
                                                  const uint16_t *__restrict__ w2_suh,
                                                  const int32_t *__restrict__ row_slot,
                                                  const int32_t *__restrict__ counts,
                                                  uint16_t *__restrict__ h2) {
    asm volatile("griddepcontrol.launch_dependents;");
    // may be launched as a dependent of FC1: wait for its rows
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);   // R * I / 128 < 2^31
    const int blocks = I / kHad;
    const int rows = counts[0];
    const int r = wid / blocks;
    if (r >= rows || r >= R) return;
    const int c0 = (wid - r * blocks) * kHad + 4 * lane;
    const int p = row_slot[r];
    const float4 g = *reinterpret_cast<const float4 *>(st1 + (int64_t)r * I + c0);
    const float4 uu = *reinterpret_cast<const float4 *>(st1 + ((int64_t)R + r) * I + c0);
    const uint2 sv = __ldg(reinterpret_cast<const uint2 *>(w2_suh + (int64_t)p * I + c0));
    const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {uu.x, uu.y, uu.z, uu.w};
    const uint32_t ss[2] = {sv.x, sv.y};
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float silu = gv[i] / (1.0f + __expf(-gv[i]));
        v[i] = (silu * uv[i]) * f16_bits_to_f32((uint16_t)(ss[i >> 1] >> (16 * (i & 1))));
    }
    warp_fwht128(v, lane);
    uint2 o;
    o.x = (uint32_t)f32_to_f16_bits(v[0] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[1] * kHadNorm) << 16);
    o.y = (uint32_t)f32_to_f16_bits(v[2] * kHadNorm) | ((uint32_t)f32_to_f16_bits(v[3] * kHadNorm) << 16);
    *reinterpret_cast<uint2 *>(h2 + (int64_t)r * I + c0) = o;
}

// ------------------------------------------------------------------ combine
// One warp per (token, 128-block of H): y_t = sum_k w[t][k] * d[pos(t, k)],
// k in order; routes whose expert id was invalid contribute nothing.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ st2, int H, int T, int topk,
                                                      const float *__restrict__ w,
                                                      const int32_t *__restrict__ pos,
                                                      uint16_t *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);   // T * H / 128 < 2^31
    const int blocks = H / kHad;
    const int t = wid / blocks;
    if (t >= T) return;
    const int c0 = (wid - t * blocks) * kHad + 4 * lane;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < topk; k++) {
        const int r = pos[(int64_t)t * topk + k];
        if (r < 0) continue;
        const float wk = w[(int64_t)t * topk + k];
        const float4 d = *reinterpret_cast<const float4 *>(st2 + (int64_t)r * H + c0);
        acc[0] += wk * d.x;
        acc[1] += wk * d.y;
        acc[2] += wk * d.z;
        acc[3] += wk * d.w;
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(acc[0]) | ((uint32_t)f32_to_bf16_bits(acc[1]) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(acc[2]) | ((uint32_t)f32_to_bf16_bits(acc[3]) << 16);
    *reinterpret_cast<uint2 *>(y + (int64_t)t * H + c0) = o;
}

inline unsigned warp_grid(int64_t warps) { return (unsigned)((warps + 7) / 8); }

}  // namespace

extern "C" {

exl3_status exl3_moe_topk_softmax(const float *logits, int32_t T, int32_t E, int32_t topk, int32_t *ids, float *w,
                                  exl3_stream stream) {
    if (T < 0 || E < 1 || E > kMoeMaxE || topk < 1 || topk > kMoeMaxTopk || topk > E)
        return fail(EXL3_EINVAL, "moe_topk_softmax: T = %d, E = %d (1..%d), topk = %d (1..%d, <= E)", T, E,
                    kMoeMaxE, topk, kMoeMaxTopk);
    if (T == 0) return EXL3_OK;
    if (!logits || !ids || !w) return fail(EXL3_EINVAL, "moe_topk_softmax: null pointer");
    cudaError_t e = launch_topk(logits, T, E, topk, ids, w, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "moe_topk_softmax");
    return EXL3_OK;
}

size_t exl3_moe_workspace_bytes(int32_t T, int32_t H, int32_t I, int32_t E, int32_t topk) {
    if (T < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || E < 1 || E > kMoeMaxE || topk < 1 ||
        topk > kMoeMaxTopk)
        return 0;
    const int64_t P = moe_pass_tokens(H, I, E, topk);
    if (P < 1) return 0;
    if (T <= P) return moe_layout(T, H, I, E, topk).total;
    // several passes of P tokens and a shorter last one
    const size_t full = moe_layout((int)P, H, I, E, topk).total;
    const int rest = (int)(T % P);
    const size_t last = rest ? moe_layout(rest, H, I, E, topk).total : 0;
    return full > last ? full : last;
}

}  // extern "C"

namespace {

// The layer on T tokens.  logits null: ids and w are the caller's routing
// (inputs).  logits non-null: ids and w are outputs, this call's own top-k of the
// logits (the top-k kernel runs first).
exl3_status moe_layer(const char *fn, const uint16_t *x, const float *logits, int32_t T, int32_t H, int32_t I,
                      int32_t E, int32_t topk, int32_t *ids, float *w, const exl3_moe_bank *bank, uint16_t *y,
                      void *wsp, size_t ws_bytes, exl3_stream stream) {
    if (T < 0 || H <= 0 || I <= 0 || H % 128 || I % 128)
        return fail(EXL3_EINVAL, "%s: T = %d, H = %d, I = %d (H and I positive multiples of 128)", fn, T, H, I);
    if (E < 1 || E > kMoeMaxE || topk < 1 || topk > kMoeMaxTopk)
        return fail(EXL3_EINVAL, "%s: E = %d (1..%d), topk = %d (1..%d)", fn, E, kMoeMaxE, topk, kMoeMaxTopk);
    if ((int64_t)T * topk > (1 << 24)) return fail(EXL3_EINVAL, "%s: T * topk = %lld routes is too many", fn,
                                                   (long long)T * topk);
    const int64_t P = moe_pass_tokens(H, I, E, topk);
    if (P < 1)
        return fail(EXL3_EINVAL, "%s: H = %d, I = %d, E = %d: more column groups than the workspace's %zu counters",
                    fn, H, I, E, kWorkspaceCounters);
    if (T == 0) return EXL3_OK;
    if (T > P) {
        // passes of P tokens: each is the whole layer on its own rows of x, ids, w and y
        if (!x || !ids || !w || !y) return fail(EXL3_EINVAL, "%s: null pointer", fn);
        for (int64_t t0 = 0; t0 < T; t0 += P) {
            const int32_t n = (int32_t)(T - t0 < P ? T - t0 : P);
            const exl3_status st = moe_layer(fn, x + t0 * H, logits ? logits + t0 * E : nullptr, n, H, I, E, topk,
                                             ids + t0 * topk, w + t0 * topk, bank, y + t0 * H, wsp, ws_bytes, stream);
            if (st != EXL3_OK) return st;
        }
        return EXL3_OK;
    }
    if (!x || !ids || !w || !y || !bank) return fail(EXL3_EINVAL, "%s: null pointer", fn);
    const exl3_moe_bank &b = *bank;
    if (!b.w13 || !b.w2 || !b.off_w1 || !b.off_w3 || !b.off_w2 || !b.perm || !b.k_gu || !b.k_d || !b.w13_suh ||
        !b.w13_svh || !b.w2_suh || !b.w2_svh)
        return fail(EXL3_EINVAL, "%s: null pointer in the expert bank", fn);
    if ((((uintptr_t)x | (uintptr_t)y | (uintptr_t)b.w13 | (uintptr_t)b.w2) & 15u) ||
        (((uintptr_t)b.w13_suh | (uintptr_t)b.w13_svh | (uintptr_t)b.w2_suh | (uintptr_t)b.w2_svh) & 7u))
        return fail(EXL3_EINVAL, "%s: x, y and the code banks must be 16-byte aligned, scale vectors 8-byte", fn);
    const MoeLayout L = moe_layout(T, H, I, E, topk);
    if (!wsp || (reinterpret_cast<uintptr_t>(wsp) & 255u) || ws_bytes < L.total)
        return fail(EXL3_EWORKSPACE, "%s: workspace %p of %zu bytes; this call needs %zu bytes, 256-byte aligned",
                    fn, wsp, ws_bytes, L.total);
    char *base = static_cast<char *>(wsp);
    int32_t *err = workspace_err(wsp);
    int32_t *counters = workspace_counters(wsp);
    int32_t *pos = reinterpret_cast<int32_t *>(base + L.pos);
    int32_t *row_pair = reinterpret_cast<int32_t *>(base + L.row_pair);
    int32_t *row_slot = reinterpret_cast<int32_t *>(base + L.row_slot);
    int32_t *counts = reinterpret_cast<int32_t *>(base + L.counts);
    GroupEntry *ent1 = reinterpret_cast<GroupEntry *>(base + L.ent1);
    GroupEntry *ent2 = reinterpret_cast<GroupEntry *>(base + L.ent2);
    uint16_t *u13 = reinterpret_cast<uint16_t *>(base + L.u13);
    float *st1 = reinterpret_cast<float *>(base + L.st1);
    uint16_t *h2 = reinterpret_cast<uint16_t *>(base + L.h2);
    float *st2 = reinterpret_cast<float *>(base + L.st2);
    float *slab = reinterpret_cast<float *>(base + L.slab);
    cudaStream_t s = (cudaStream_t)stream;
    const int R = L.R;

    // One 8-row block per entry: the routing with the per-pair input rotation
    // alongside (and, up to kFoldTopkTokens tokens, the top-k), FC1 on the pairs'
    // rows with the activation in its epilogue, FC2 with the weighted combine in
    // its epilogue, chained as programmatic dependents.  Otherwise the separate
    // passes below.
    const int GH = H / kHad;
    const bool chain = !L.fused && L.nb == 1 &&
                       (int64_t)L.max_entries * (2 * (I / kHad) > GH ? 2 * (I / kHad) : GH) <= kCombCounterBase &&
                       (int64_t)T * GH <= (int64_t)kWorkspaceCounters - kCombCounterBase;
    RouteArgs ra = {ids, R, topk, E, H, I, L.chunk, b, pos, row_pair, row_slot, counts, ent1, ent2, err,
                    chain ? y : nullptr};
    cudaError_t e;
    cudaLaunchAttribute pdl_attr[1];
    pdl_attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl_attr[0].val.programmaticStreamSerializationAllowed = 1;
    // At a few tokens the chain's first launch takes the top-k itself (one launch
    // fewer; every rotating warp then ranks its own token's logits, which costs
    // more than the launch it saves once there are many routes: T = 64 measured
    // 198.7 -> 206.2 us, T = 1 36.9 -> 35.7 us).
    const bool fold_topk = logits && chain && T <= kFoldTopkTokens;
    if (logits && !fold_topk) {
        // the routing below reads ids and w: the top-k first (a programmatic
        // dependent of whatever precedes the layer, and the routing of it)
        if ((e = launch_topk(logits, T, E, topk, ids, w, s)) != cudaSuccess) return cuda_fail(e, "moe: top-k");
    }
    if (chain) {
        PairRotateArgs pr = {x, ids, R, topk, E, H, b, u13, fold_topk ? logits : nullptr};
        const int64_t tasks = (int64_t)R * (H / kHad);
        const int64_t rot_ctas = (tasks + 31) / 32 < 4 * (int64_t)device_info().sm_count ? (tasks + 31) / 32
                                                                                          : 4 * (int64_t)device_info().sm_count;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(1 + rot_ctas));
        cfg.blockDim = dim3(1024);
        cfg.stream = s;
        cfg.attrs = pdl_attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, route_rotate_kernel, ra, pr, ids, w)) != cudaSuccess)
            return cuda_fail(e, "moe_grouped: route");
        GroupGemmArgs g1 = {};
        g1.u = u13;
        g1.IC = H;
        g1.mode = kModeRows;
        g1.entries = ent1;
        g1.n_entries_dev = counts + 1;
        g1.n_groups_per_entry = I / kHad;
        g1.partials = slab;
        g1.counters = counters;
        g1.gather = 1;
        g1.R = R;
        g1.topk = topk;
        g1.row_pair = row_pair;
        // w1 and w3 of an expert row block in one column group: the epilogue applies
        // the activation and FC2's input transform (no fp32 FC1 rows, no act launch)
        g1.pair_act = 1;
        g1.act_suh = b.w2_suh;
        g1.act_out = h2;
        if ((e = launch_group_gemm(g1, 1, true, s)) != cudaSuccess) return cuda_fail(e, "moe_grouped: FC1");
        GroupGemmArgs g2 = {};
        g2.u = h2;
        g2.IC = I;
        g2.mode = kModeRows;
        g2.entries = ent2;
        g2.n_entries_dev = counts + 2;
        g2.n_groups_per_entry = GH;
        g2.out_rows = st2;
        g2.partials = slab;
        g2.counters = counters;
        g2.R = R;
        g2.topk = topk;
        g2.row_pair = row_pair;
        g2.comb = 1;
        g2.comb_w = w;
        g2.comb_pos = pos;
        g2.comb_y = y;
        g2.comb_counters = counters + kCombCounterBase;
        // the routing launch, two before, wrote the entry lists and tables; FC1 only h2
        g2.entries_ready = 1;
        // when every column group can have its own CTA (at most R entries of H/128
        // groups), whole groups per 16-warp CTA, three or so tile rows a warp
        g2.wide = (int64_t)R * (H / kHad) <= device_info().sm_count ? 1 : 0;
        if ((e = launch_group_gemm(g2, 1, true, s)) != cudaSuccess) return cuda_fail(e, "moe_grouped: FC2");
        trace("%s T=%d H=%d I=%d E=%d topk=%d rows<=%d gemm=decode (3 launches)", fn, T, H, I, E, topk, R);
        return EXL3_OK;
    }
    route_kernel<<<1, 1024, 0, s>>>(ra);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "moe_grouped: route");

    // warps per row: enough warps to fill the GPU when few rows are routed, whole rows otherwise
    int parts = 1;
    while (parts * 2 <= H / kHad && (H / kHad) % (parts * 2) == 0 && (int64_t)R * parts < 32768) parts *= 2;
    rotate_kernel<<<warp_grid((int64_t)R * parts), 256, 0, s>>>(x, H, R, topk, b.w13_suh, row_pair, row_slot, counts,
                                                               u13, parts);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "moe_grouped: rotate");

    if (L.fused) {
        FusedArgs f1 = {};
        f1.IC = H;
        f1.entries = ent1;
        f1.n_entries_dev = counts + 1;
        f1.groups_per_entry = I / kHad;
        f1.OC_rows = I;
        f1.out_rows = st1;
        f1.partials = slab;
        f1.counters = counters;
        f1.err = err;
        if ((e = launch_fused_rows(f1, u13, 2 * (int64_t)R, 2 * (int64_t)L.max_entries, s)) != cudaSuccess)
            return cuda_fail(e, "moe_grouped: FC1");
        act_kernel<<<warp_grid((int64_t)R * (I / kHad)), 256, 0, s>>>(st1, I, R, b.w2_suh, row_slot, counts, h2);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "moe_grouped: act");
        FusedArgs f2 = f1;
        f2.IC = I;
        f2.entries = ent2;
        f2.n_entries_dev = counts + 2;
        f2.groups_per_entry = H / kHad;
        f2.OC_rows = H;
        f2.out_rows = st2;
        if ((e = launch_fused_rows(f2, h2, (int64_t)R, (int64_t)L.max_entries, s)) != cudaSuccess)
            return cuda_fail(e, "moe_grouped: FC2");
    } else {
        GroupGemmArgs g1 = {};
        g1.u = u13;
        g1.IC = H;
        g1.mode = kModeRows;
        g1.entries = ent1;
        g1.n_entries_dev = counts + 1;
        g1.n_groups_per_entry = I / kHad;
        g1.out_rows = st1;
        g1.partials = slab;
        g1.counters = counters;
        // the entry lists come from route_kernel, the launch before the rotation
        g1.entries_ready = 1;
        if ((e = launch_group_gemm(g1, L.nb, true, s)) != cudaSuccess) return cuda_fail(e, "moe_grouped: FC1");

        act_kernel<<<warp_grid((int64_t)R * (I / kHad)), 256, 0, s>>>(st1, I, R, b.w2_suh, row_slot, counts, h2);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "moe_grouped: act");

        GroupGemmArgs g2 = g1;
        g2.u = h2;
        g2.IC = I;
        g2.entries = ent2;
        g2.n_entries_dev = counts + 2;
        g2.n_groups_per_entry = H / kHad;
        g2.out_rows = st2;
        if ((e = launch_group_gemm(g2, L.nb, true, s)) != cudaSuccess) return cuda_fail(e, "moe_grouped: FC2");
    }

    combine_kernel<<<warp_grid((int64_t)T * (H / kHad)), 256, 0, s>>>(st2, H, T, topk, w, pos, y);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "moe_grouped: combine");
    trace("%s T=%d H=%d I=%d E=%d topk=%d rows<=%d nb=%d gemm=%s", fn, T, H, I, E, topk, R, L.nb,
          L.fused ? "fused" : "decode");
    return EXL3_OK;
}

}  // namespace

extern "C" {

exl3_status exl3_moe_grouped(const uint16_t *x, int32_t T, int32_t H, int32_t I, int32_t E, int32_t topk,
                             const int32_t *ids, const float *w, const exl3_moe_bank *bank, uint16_t *y, void *wsp,
                             size_t ws_bytes, exl3_stream stream) {
    return moe_layer("moe_grouped", x, nullptr, T, H, I, E, topk, const_cast<int32_t *>(ids), const_cast<float *>(w),
                     bank, y, wsp, ws_bytes, stream);
}

exl3_status exl3_moe_forward(const uint16_t *x, const float *logits, int32_t T, int32_t H, int32_t I, int32_t E,
                             int32_t topk, const exl3_moe_bank *bank, int32_t *ids, float *w, uint16_t *y, void *wsp,
                             size_t ws_bytes, exl3_stream stream) {
    if (T > 0 && !logits) return fail(EXL3_EINVAL, "moe_forward: null logits");
    if (topk > E) return fail(EXL3_EINVAL, "moe_forward: topk = %d > E = %d", topk, E);
    return moe_layer("moe_forward", x, logits, T, H, I, E, topk, ids, w, bank, y, wsp, ws_bytes, stream);
}

}  // extern "C"
