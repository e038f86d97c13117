// fused_tc.cu -- EXL3 linear for 8 < M <= 128 rows on the tensor cores, with
// the trellis decoded straight into shared-memory operand tiles
// (radiance_escha.py, module docstring "THE FORWARD": the middle factor
// u @ decode(code), followed by the output Had128 and the rout, s_out scales).
//
// v^T = W^T u^T runs as tcgen05 MMAs with the output columns on the MMA's M
// (128 = one Had128 block) and the rows on its N (16..128).  Per 64-channel
// slice of the input ("stage"):
//   A (W^T, 128 columns x 64 channels, K-major, 128-byte swizzle) is written by
//     a group of four decoder warps: a thread decodes one quarter of a 16x16
//     trellis tile and stores the fp16 weights (lo + hi of the codebook, rounded
//     once, as the format defines them);
//   B (rows x 64 channels) is a TMA tile of the pre-transformed activations.
// One tcgen05.mma covers 128 x 16 weights and occupies the issuing thread for
// about 60 cycles whatever N is, so two threads on different SM sub-partitions
// issue the MMAs of alternate stages into two accumulators that the epilogue
// adds.  Code words and B tiles arrive through rings of their own, deep enough
// to cover HBM and TMA latency.
//
// Warp roles (640 threads, one CTA per SM):
//   warp 0        TMEM allocation; MMA issuer for even stages
//   warp 1        TMA producer of the B tiles (released in chunks of 2 stages)
//   warp 2        TMA producer of the code ring (one 3-D box per stage)
//   warp 3        MMA issuer for odd stages
//   warps 4..7    epilogue: TMEM -> registers -> split-K slab or shared
//                 transpose -> per-row Had128 -> rout, s_out -> bf16
//   warps 8..19   decoders: three groups of four warps; group p decodes the
//                 stages g with g % 3 == p (three warps per sub-partition, so
//                 one group's ring waits overlap the others' arithmetic)
// Work units (column group x stage) of all shards are split evenly over the
// persistent grid; the accumulators are double-buffered in TMEM so that the
// epilogue of one column group overlaps the MMAs of the next.  CTAs that share
// a column group reduce through the split-K slab; the last one to arrive
// applies the epilogue.  Every mbarrier wait is bounded (tc_ptx.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace exl3 {

namespace {

constexpr int FT_NGROUPS = 3;                      // decoder groups (4 warps each); group p decodes stages g % 3 == p
constexpr int FT_ASLOTS = 6;                       // A ring depth (two slots per decoder group)
constexpr int FT_MAX_CSTAGES = 12;                 // code ring depth (fewer at 128 rows)
constexpr int FT_CSLOT = 4096;                     // code bytes per stage: 4 trellis rows x 8 tiles x 32K, K <= 4
constexpr int FT_BM = 128;                         // output columns per tile (one Had128 block)
constexpr int FT_KC = 64;                          // input channels per stage
constexpr int FT_A_BYTES = FT_BM * FT_KC * 2;      // 16 KB
constexpr int FT_THREADS = 256 + FT_NGROUPS * 128;
constexpr int W_MMA0 = 0, W_BLOAD = 1, W_CODE = 2, W_MMA1 = 3, W_EPI = 4, W_DEC = 8;
constexpr int FT_TSTRIDE = 144;                    // transpose buffer: 4 parts x 36 floats per row
constexpr int FT_T_BYTES = 32 * FT_TSTRIDE * 4;
constexpr int FT_MAX_BCHUNKS = 12;                 // B ring: chunks of 2 stages
constexpr int FT_SMEM_LIMIT = 232448;              // opt-in shared memory per CTA
constexpr int kFtMaxEntries = 32;                  // rows mode: entries one CTA may touch (cached in shared memory)
// barriers
constexpr int B_FULL = 0, B_EMPTY = B_FULL + FT_ASLOTS, B_BFULL = B_EMPTY + FT_ASLOTS,
              B_BEMPTY = B_BFULL + FT_MAX_BCHUNKS, B_CFULL = B_BEMPTY + FT_MAX_BCHUNKS,
              B_CEMPTY = B_CFULL + FT_MAX_CSTAGES, B_ACCF = B_CEMPTY + FT_MAX_CSTAGES, B_ACCE = B_ACCF + 2,
              B_DONE = B_ACCE + 2, B_COUNT = B_DONE + 2;

template <int NT>
struct FtCfg {
    static constexpr int B_BYTES = NT * FT_KC * 2;                   // one stage of activations
    static constexpr int CHUNK_BYTES = 2 * B_BYTES;
    static constexpr int CSTAGES = NT >= 128 ? 9 : FT_MAX_CSTAGES;   // code ring depth (a multiple of the groups)
    static constexpr int FIXED = FT_ASLOTS * FT_A_BYTES + CSTAGES * FT_CSLOT + FT_T_BYTES + 4 * FT_BM +
                                 kFtMaxEntries * (int)sizeof(GroupEntry) + B_COUNT * 8 + 64 + 1024;
    static constexpr int FIT = (FT_SMEM_LIMIT - FIXED) / CHUNK_BYTES;
    static constexpr int BCHUNKS = FIT < FT_MAX_BCHUNKS ? FIT : FT_MAX_BCHUNKS;
    static constexpr int B_OFF = FT_ASLOTS * FT_A_BYTES;
    static constexpr int CODE_OFF = B_OFF + BCHUNKS * CHUNK_BYTES;
    static constexpr int T_OFF = CODE_OFF + CSTAGES * FT_CSLOT;
    static constexpr int SC_OFF = T_OFF + FT_T_BYTES;                 // the segment's rout, s_out (fp16)
    static constexpr int ENT_OFF = SC_OFF + 2 * FT_BM * 2;            // rows mode: cached entries
    static constexpr int BAR_OFF = ENT_OFF + kFtMaxEntries * (int)sizeof(GroupEntry);
    static constexpr int SMEM = BAR_OFF + B_COUNT * 8 + 64 + 1024;
    static constexpr int BUF = NT < 32 ? 32 : NT;                    // TMEM columns per accumulator
    static constexpr int TMEM_COLS = 4 * BUF;                        // 2 issuers x 2 buffers
    static constexpr uint32_t IDESC = make_idesc_f16(FT_BM, NT);
    static_assert(BCHUNKS >= 2 && SMEM <= FT_SMEM_LIMIT, "shared-memory plan does not fit");
    static_assert(TMEM_COLS <= 512, "tensor memory plan does not fit");
    static_assert(CSTAGES % FT_NGROUPS == 0 && FT_ASLOTS % FT_NGROUPS == 0, "rings must rotate with the groups");
};

// Stage g of a CTA is work unit f0 + g: column group gi = unit / ST, stage
// st = unit % ST.  A segment is the run of stages of one column group; its
// accumulator is buffer (gi - first group of the CTA) & 1.  What a role needs
// about a segment's column group:
struct SegDesc {
    const char *code;                // the code tensor (bytes)
    const uint16_t *post, *post2;    // dense: rout, s_out; rows mode: the post-scale, nullptr
    int K, TO, G;                    // bits per weight, tiles per trellis row, column group in the tensor
    int u_row;                       // first activation row
    int rows;                        // rows of the segment
    int64_t out0;                    // dense: first output column; rows mode: first output row
    int tm;                          // dense: code tensor map index; rows mode: -1 (bulk copies)
};


template <int K>
__device__ __forceinline__ void lds_quarter(uint32_t (&w)[2 * K], uint32_t addr) {
    if constexpr (K == 3) {
#pragma unroll
        for (int j = 0; j < 3; j++)
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w[2 * j]), "=r"(w[2 * j + 1]) : "r"(addr + 8 * j));
    } else {
#pragma unroll
        for (int j = 0; j < K / 2; j++)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * j]), "=r"(w[4 * j + 1]), "=r"(w[4 * j + 2]), "=r"(w[4 * j + 3])
                         : "r"(addr + 16 * j));
    }
}

// A decoder thread's share of a stage is quarter q (tile rows 4q..4q+3, all 16
// columns) of tile (kt, oc_tile).  Tile column c is operand row c*8 + oc_tile;
// its four weights are the 8 bytes at channel 16*kt + 4*q of that row, i.e.
// 16-byte chunk 2*kt + q/2, half q%2, 128-byte swizzled (chunk ^ row % 8).
// oc_tile is spread over the lanes so that each half-warp's 8-byte stores hit
// 16 distinct bank pairs.

// Wait for a stage's code and load this thread's quarter into registers.  The
// ring slot stays held until the quarter is decoded (ft_decode_quarter).
template <int K>
__device__ __forceinline__ bool ft_fetch(const FusedArgs &a, uint32_t (&w)[2 * K], uint32_t cfull, uint32_t cph,
                                         uint32_t code_slot, int kt, int oc_tile, int q, volatile int *abort) {
    if (!__all_sync(kFull, mbar_wait(cfull, cph, a.err, abort))) return false;
    lds_quarter<K>(w, code_slot + (uint32_t)(kt * 256 * K + oc_tile * 32 * K + q * 8 * K));
    return true;
}

// Decode a quarter held in registers into its A slot, publish it to the MMA
// issuer and release the code slot it came from.
template <int K>
__device__ __forceinline__ bool ft_decode_quarter(const FusedArgs &a, const uint32_t (&w)[2 * K], uint32_t empty,
                                                  uint32_t empty_parity, uint32_t full, uint32_t cempty,
                                                  uint32_t a_base, int kt, int oc_tile, int q, int lane,
                                                  volatile int *abort) {
    if (!__all_sync(kFull, mbar_wait(empty, empty_parity, a.err, abort))) return false;
    QuarterStream<K> st;
    st.build(w, quarter_prev_word(w[2 * K - 1], lane));
    const uint32_t hx = a.hash_xor;
    const uint32_t off = (uint32_t)((((2 * kt + (q >> 1)) ^ oc_tile) << 4) + ((q & 1) << 3));
#pragma unroll
    for (int c = 0; c < 16; c++) {
        const uint32_t z0 = trellis_hash_x(st.state(c, a.pow2), hx);
        const uint32_t z1 = trellis_hash_x(st.state(16 + c, a.pow2), hx);
        const uint32_t z2 = trellis_hash_x(st.state(32 + c, a.pow2), hx);
        const uint32_t z3 = trellis_hash_x(st.state(48 + c, a.pow2), hx);
        const uint32_t w01 = trellis_weight_pair(z0, z1), w23 = trellis_weight_pair(z2, z3);
        const uint32_t addr = a_base + (uint32_t)(c * 8 + oc_tile) * 128u + off;
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(w01), "r"(w23) : "memory");
    }
    // Every thread orders its generic-proxy accesses of shared memory before what
    // the async proxy does next: its stores to the A slot before the MMAs read
    // them, and its loads of the code slot before the next TMA copy into that
    // slot (a write-after-read across proxies, which the mbarrier alone does not
    // order: released without this fence, a slot was seen overwritten before the
    // last warp had read it).  Then one arrival per warp on each barrier.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        mbar_arrive(full);
        mbar_arrive(cempty);
    }
    return true;
}

// Ring positions of a decoder group: code slot / phase and A slot / the parity
// its "empty" wait takes, of the group's next stage.
struct DecState {
    int cs, cph, slot, eph;
};

// Decode this group's stages g, g + FT_NGROUPS, ... below end, all of one shard
// (one K).  g is left at the first stage not decoded.
template <int K, int CSTAGES>
__device__ __forceinline__ bool ft_decode_run(const FusedArgs &a, uint32_t code_base, uint32_t a_ring, uint32_t bar0,
                                              int &g, int end, DecState &ds, int kt, int oc_tile, int q, int lane,
                                              volatile int *abort) {
    for (; g < end; g += FT_NGROUPS) {
        uint32_t w[2 * K];
        const uint32_t cempty = bar0 + 8u * (B_CEMPTY + ds.cs);
        if (!ft_fetch<K>(a, w, bar0 + 8u * (B_CFULL + ds.cs), ds.cph, code_base + ds.cs * FT_CSLOT, kt, oc_tile, q,
                         abort))
            return false;
        ds.cs += FT_NGROUPS;
        if (ds.cs >= CSTAGES) { ds.cs -= CSTAGES; ds.cph ^= 1; }
        if (!ft_decode_quarter<K>(a, w, bar0 + 8u * (B_EMPTY + ds.slot), ds.eph, bar0 + 8u * (B_FULL + ds.slot),
                                  cempty, a_ring + ds.slot * FT_A_BYTES, kt, oc_tile, q, lane, abort))
            return false;
        ds.slot += FT_NGROUPS;
        if (ds.slot >= FT_ASLOTS) { ds.slot -= FT_ASLOTS; ds.eph ^= 1; }
    }
    return true;
}

template <int NT, bool ROWS>
__global__ void __launch_bounds__(FT_THREADS, 1) fused_tc_kernel(const __grid_constant__ FusedArgs a) {
    using C = FtCfg<NT>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *sbase = smem_raw + (base - raw);
    float *T = reinterpret_cast<float *>(sbase + C::T_OFF);
    uint16_t *s_scale = reinterpret_cast<uint16_t *>(sbase + C::SC_OFF);   // [0, 128) rout, [128, 256) s_out
    GroupEntry *s_ent = reinterpret_cast<GroupEntry *>(sbase + C::ENT_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + C::BAR_OFF);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + B_COUNT);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    volatile int *s_last = reinterpret_cast<volatile int *>(s_tmem + 2);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [bar0](int i) { return bar0 + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ST = a.IC / FT_KC, M = a.M;

    if (threadIdx.x == 0) {
        for (int i = 0; i < FT_ASLOTS; i++) {
            mbar_init(bar(B_FULL + i), 4);      // the four warps of a decoder group
            mbar_init(bar(B_EMPTY + i), 1);     // MMA commit
        }
        for (int i = 0; i < C::BCHUNKS; i++) {
            mbar_init(bar(B_BFULL + i), 1);     // B producer (arrive + transaction bytes)
            mbar_init(bar(B_BEMPTY + i), 2);    // one commit from each issuer
        }
        for (int i = 0; i < C::CSTAGES; i++) {
            mbar_init(bar(B_CFULL + i), 1);     // code producer (arrive + transaction bytes)
            mbar_init(bar(B_CEMPTY + i), 4);    // the four warps of a decoder group
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_ACCF + i), 2);      // one commit from each issuer
            mbar_init(bar(B_ACCE + i), 4);      // the four epilogue warps
            mbar_init(bar(B_DONE + i), 1);
        }
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == W_MMA0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                     "r"(C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // Rows mode reads the entry lists the preceding kernel (the routing) built, so
    // it waits for that kernel here.  Dense mode takes from the preceding kernel
    // (the pre-transform) only the activations and the row scales: the two roles
    // that read them, the B producer and the epilogue, wait before their first
    // access, and the code fetch and the decode start while that kernel still
    // runs.  Before its wait a role reads only the code (never written by a kernel)
    // and writes only shared and tensor memory.
    if constexpr (ROWS) asm volatile("griddepcontrol.wait;" ::: "memory");

    int n_groups = 0;
    if constexpr (ROWS) {
        n_groups = *a.n_entries_dev * a.groups_per_entry;
    } else {
        for (int i = 0; i < a.n_shards; i++) n_groups += a.sh[i].OC / kHad;
    }
    const int64_t total = (int64_t)n_groups * ST;
    const int nCTA = (int64_t)gridDim.x < total ? (int)gridDim.x : (int)total;
    const int c = blockIdx.x;
    const int64_t f0 = c < nCTA ? (int64_t)c * total / nCTA : 0;
    int n = c < nCTA ? (int)((int64_t)(c + 1) * total / nCTA - f0) : 0;   // stages of this CTA
    const int gi0 = (int)(f0 / ST), st0 = (int)(f0 - (int64_t)gi0 * ST);
    int issued = 0;   // copies issued by a producer thread (drained on abort)

    // rows mode: the entries this CTA's column groups belong to, cached in shared memory
    int e_first = 0;
    if constexpr (ROWS) {
        e_first = gi0 / a.groups_per_entry;
        int e_cnt = n > 0 ? (gi0 + (st0 + n - 1) / ST) / a.groups_per_entry - e_first + 1 : 0;
        if (e_cnt > kFtMaxEntries) {
            // the host sizes the grid so that this cannot happen; do no work rather than overrun
            if (threadIdx.x == 0) record_error(a.err, kErrRouteOverflow);
            n = 0;
            e_cnt = 0;
        }
        static_assert(sizeof(GroupEntry) % 8 == 0, "entries are copied in 8-byte words");
        for (int i = threadIdx.x; i < e_cnt * (int)(sizeof(GroupEntry) / 8); i += blockDim.x)
            reinterpret_cast<long long *>(s_ent)[i] = __ldg(reinterpret_cast<const long long *>(a.entries + e_first) + i);
        __syncthreads();
    }
    // Everything a role needs about column group gi (one segment).
    auto seg_desc = [&](int gi) -> SegDesc {
        SegDesc d;
        if constexpr (ROWS) {
            const int e = gi / a.groups_per_entry;
            const GroupEntry &ge = s_ent[e - e_first];
            d.code = reinterpret_cast<const char *>(ge.code);
            d.post = ge.post;
            d.post2 = nullptr;
            d.K = ge.K;
            d.TO = ge.OC / kTile;
            d.G = gi - e * a.groups_per_entry;
            d.u_row = ge.u_row0;
            d.rows = ge.nrows;
            d.out0 = ge.out_off;
            d.tm = -1;
        } else {
            int sidx = 0;
            while (sidx + 1 < a.n_shards && a.sh[sidx + 1].g0 <= gi) sidx++;
            const FusedShard &sh = a.sh[sidx];
            d.code = reinterpret_cast<const char *>(sh.code);
            d.post = sh.rout;
            d.post2 = sh.s_out;
            d.K = sh.K;
            d.TO = sh.OC / kTile;
            d.G = gi - sh.g0;
            d.u_row = sh.u_slot * M;
            d.rows = M;
            d.out0 = sh.col0;
            d.tm = sidx;
        }
        return d;
    };
    // Segment walk: segment j holds stages [lo, hi) of column group gi0 + j, starting at stage st_lo.
#define FT_FOR_SEGMENTS(...)                                                                  \
    for (int lo_ = 0, hi_ = (ST - st0 < n ? ST - st0 : n), j_ = 0; lo_ < n;                  \
         lo_ = hi_, hi_ = (hi_ + ST < n ? hi_ + ST : n), j_++) {                              \
        const int lo = lo_, hi = hi_, jseg = j_, gi = gi0 + j_, st_lo = j_ == 0 ? st0 : 0;    \
        (void)lo; (void)hi; (void)jseg; (void)gi; (void)st_lo;                                \
        __VA_ARGS__                                                                           \
    }

    if (warp == W_MMA0 || warp == W_MMA1) {
        // ---------------- MMA issuers: stages of parity p into accumulator p
        // (the loop touches only this issuer's stages and keeps every index
        // incremental: it shares its sub-partition with two busy decoder warps)
        if (lane == 0) {
            const int p = warp == W_MMA0 ? 0 : 1;
            const uint64_t da0 = smem_desc_sw128(base);
            const uint64_t db0 = smem_desc_sw128(base + C::B_OFF + p * C::B_BYTES);
            int slot = p, aph = 0;   // A slot of stage g and its phase
            int ch = 0, bph = 0;     // B chunk of stage g and its phase
            int j = 0;               // segment index; segment j ends before stage seg_end
            int seg_end = ST - st0 < n ? ST - st0 : n;
            uint32_t d = 0;
            bool fresh = true;
            auto open_seg = [&]() -> bool {
                // the epilogue must have drained this accumulator buffer
                if (!mbar_wait(bar(B_ACCE + (j & 1)), ((j >> 1) & 1) ^ 1, a.err, s_abort)) return false;
                tc_fence_after();
                d = tmem + (uint32_t)((2 * (j & 1) + p) * C::BUF);
                fresh = true;
                return true;
            };
            bool ok = n > 0 && open_seg();
            for (int g = p; ok; g += 2) {
                while (g >= seg_end) {
                    // no stage of this parity left in segment j: close it (an issuer
                    // without stages in it still arrives), open the next one
                    umma_commit(bar(B_ACCF + (j & 1)));
                    if (seg_end >= n) break;
                    j++;
                    seg_end = seg_end + ST < n ? seg_end + ST : n;
                    if (!(ok = open_seg())) break;
                }
                if (!ok || g >= n) break;
                if (!mbar_wait(bar(B_FULL + slot), aph, a.err, s_abort) ||
                    !mbar_wait(bar(B_BFULL + ch), bph, a.err, s_abort))
                    break;
                tc_fence_after();
                const uint64_t da = da0 + (uint64_t)(slot * (FT_A_BYTES >> 4));
                const uint64_t db = db0 + (uint64_t)(ch * (C::CHUNK_BYTES >> 4));
#pragma unroll
                for (int k = 0; k < FT_KC / 16; k++) umma_f16(d, da + 2 * k, db + 2 * k, C::IDESC, (!fresh) || k);
                fresh = false;
                umma_commit(bar(B_EMPTY + slot));
                umma_commit(bar(B_BEMPTY + ch));
                slot += 2;
                if (slot >= FT_ASLOTS) { slot -= FT_ASLOTS; aph ^= 1; }
                if (++ch == C::BCHUNKS) { ch = 0; bph ^= 1; }
            }
            // every MMA must be complete before the CTA releases TMEM and shared memory
            umma_commit(bar(B_DONE + p));
            mbar_drain(bar(B_DONE + p), 0);
        }
    } else if (warp == W_BLOAD) {
        // ---------------- TMA producer of the B tiles, two stages per chunk
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");   // the activations
            bool ok = true;
            FT_FOR_SEGMENTS({
                if (!ok) break;
                const SegDesc d = seg_desc(gi);
                for (int g = lo; g < hi; g++) {
                    const int jc = g >> 1, ch = jc % C::BCHUNKS;
                    if ((g & 1) == 0) {
                        if (!mbar_wait(bar(B_BEMPTY + ch), ((jc / C::BCHUNKS) & 1) ^ 1, a.err, s_abort)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(bar(B_BFULL + ch), (g + 1 < n ? 2 : 1) * C::B_BYTES);
                        issued++;
                    }
                    tma_load_2d(base + C::B_OFF + ch * C::CHUNK_BYTES + (g & 1) * C::B_BYTES, &a.tm_u,
                                (st_lo + g - lo) * FT_KC, d.u_row, bar(B_BFULL + ch));
                }
            })
        }
    } else if (warp == W_CODE) {
        // ---------------- producer of the code ring: per stage one 3-D TMA box (4 tile rows
        // x 8 tiles) when the code tensor has a tensor map, else four bulk copies
        if (lane == 0) {
            bool ok = true;
            FT_FOR_SEGMENTS({
                if (!ok) break;
                const SegDesc d = seg_desc(gi);
                const uint32_t bytes = 256u * (uint32_t)d.K;        // 8 tiles of one trellis row
                for (int g = lo; g < hi; g++) {
                    const int cs = g % C::CSTAGES, st = st_lo + g - lo;
                    if (!mbar_wait(bar(B_CEMPTY + cs), ((g / C::CSTAGES) & 1) ^ 1, a.err, s_abort)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar(B_CFULL + cs), 4 * bytes);
                    const uint32_t dst = base + C::CODE_OFF + cs * FT_CSLOT;
                    if (d.tm >= 0) {
                        tma_load_3d(dst, &a.tm_code[d.tm], 0, 8 * d.G, 4 * st, bar(B_CFULL + cs));
                    } else {
#pragma unroll
                        for (int kt = 0; kt < 4; kt++)
                            bulk_load(dst + kt * bytes, d.code + ((int64_t)(4 * st + kt) * d.TO + 8 * d.G) * 32 * d.K,
                                      bytes, bar(B_CFULL + cs));
                    }
                    issued++;
                }
            })
        }
    } else if (warp >= W_DEC) {
        // ---------------- decoders: group p decodes the stages g % FT_NGROUPS == p
        const int p = (warp - W_DEC) >> 2;
        const int kt = (warp - W_DEC) & 3;
        const int oc_tile = ((lane >> 2) & 3) * 2 + (lane >> 4);
        const int q = lane & 3;
        DecState ds;
        ds.cs = p;
        ds.cph = 0;
        ds.slot = p;
        ds.eph = 1;
        // decode this group's stages segment by segment with a loop specialised for the segment's K
        int g = p;
        FT_FOR_SEGMENTS({
            if (g >= hi) continue;
            const int K = seg_desc(gi).K;
            bool ok;
            if (K == 2)
                ok = ft_decode_run<2, C::CSTAGES>(a, base + C::CODE_OFF, base, bar0, g, hi, ds, kt, oc_tile, q, lane,
                                                  s_abort);
            else if (K == 3)
                ok = ft_decode_run<3, C::CSTAGES>(a, base + C::CODE_OFF, base, bar0, g, hi, ds, kt, oc_tile, q, lane,
                                                  s_abort);
            else
                ok = ft_decode_run<4, C::CSTAGES>(a, base + C::CODE_OFF, base, bar0, g, hi, ds, kt, oc_tile, q, lane,
                                                  s_abort);
            if (!ok) break;
        })
    } else {
        // ---------------- epilogue, warps 4..7 (128 threads, named barrier 1)
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the row scales; outputs after the preceding kernel
        const int r = (warp & 3) * 32 + lane;         // TMEM lane = operand row of this thread
        const int et = (warp - W_EPI) * 32 + lane;    // 0..127
        const int ti = et >> 2, part = et & 3;        // transpose phase: row in chunk, quarter of the block
        const int64_t frag = (int64_t)M * FT_BM;   // split-K slab slot: M (the row bound) x 128 columns
        FT_FOR_SEGMENTS({
            const int seg_len = hi - lo;
            // which issuers accumulated into this segment: parity lo always, the other one if it is longer than 1
            const bool has[2] = {(lo & 1) == 0 || seg_len > 1, (lo & 1) == 1 || seg_len > 1};
            const SegDesc d = seg_desc(gi);
            const int G = d.G;
            const int rows = d.rows < NT ? d.rows : NT;
            const int b = jseg & 1;
            // this column group's output scales, fetched while the MMAs finish
            s_scale[et] = __ldg(d.post + G * kHad + et);
            if constexpr (!ROWS) s_scale[FT_BM + et] = __ldg(d.post2 + G * kHad + et);
            const bool have = mbar_wait(bar(B_ACCF + b), (jseg >> 1) & 1, a.err, s_abort);
            tc_fence_after();
            if (!named_bar_and(1, 128, have)) break;
            const uint32_t tb = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(2 * b * C::BUF);
            // CTAs sharing this column group
            const int64_t x0 = (int64_t)gi * ST, x1 = x0 + ST - 1;
            const int c_first = (int)(((x0 + 1) * nCTA - 1) / total);
            const int c_last = (int)(((x1 + 1) * nCTA - 1) / total);
            const bool split = c_first != c_last;
            auto load_acc = [&](int c0, float (&v)[32]) {
#pragma unroll
                for (int i = 0; i < 32; i++) v[i] = 0.f;
#pragma unroll
                for (int pp = 0; pp < 2; pp++) {
                    if (!has[pp]) continue;
                    float t[32];
                    tmem_ld32(tb + (uint32_t)(pp * C::BUF) + c0, t);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i++) v[i] += t[i];
                }
            };
            // The first contributor of a split group (its range ends in this group, so
            // this is its last segment) usually arrives last, at the end of its work.
            // If every other contributor has arrived already, it keeps its own part in
            // TMEM and adds only theirs: the sum runs in the same CTA order (its own
            // part first), so the result is the same, bit for bit.
            // (dense launches only: in rows mode it measured slower)
            bool own_in_tmem = false;
            if (!ROWS && split && c == c_first) {
                if (et == 0)
                    *s_last = *reinterpret_cast<volatile int32_t *>(a.counters + gi) == c_last - c_first;
                named_bar(1, 128);
                own_in_tmem = *s_last != 0;
                named_bar(1, 128);   // s_last is written again below
                if (own_in_tmem) {
                    __threadfence();   // the others wrote their partials before arriving
                    if (et == 0) a.counters[gi] = 0;
                }
            }
            if (split && !own_in_tmem) {
                float *slot = a.partials + (int64_t)(c + gi) * frag;
                for (int c0 = 0; c0 < rows; c0 += 32) {
                    float v[32];
                    load_acc(c0, v);
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        if (c0 + i < rows) __stcg(slot + (int64_t)(c0 + i) * FT_BM + r, v[i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_ACCE + b));
                __threadfence();
                named_bar(1, 128);
                if (et == 0) *s_last = (atomicAdd(a.counters + gi, 1) == c_last - c_first);
                named_bar(1, 128);
                if (!*s_last) continue;
                __threadfence();
                if (et == 0) a.counters[gi] = 0;
            }
            for (int c0 = 0; c0 < rows; c0 += 32) {
                if (split && !own_in_tmem) {
                    // sum the contributors' slabs for rows c0 .. c0 + 31 (32 x 128
                    // floats): thread et takes float4 f = et + 128 k, coalesced; two
                    // contributors' loads in flight at a time, added in ascending
                    // CTA order (the same order whichever CTA finishes last)
                    const float4 *pbase = reinterpret_cast<const float4 *>(a.partials + (int64_t)c0 * FT_BM);
#pragma unroll
                    for (int kb = 0; kb < 8; kb += 4) {
                        float4 acc[4];
#pragma unroll
                        for (int k = 0; k < 4; k++) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int cc = c_first; cc <= c_last; cc += 2) {
                            const bool two = cc + 1 <= c_last;
                            const float4 *p0 = pbase + (int64_t)(cc + gi) * (frag / 4);
                            const float4 *p1 = p0 + frag / 4;
                            float4 t0[4], t1[4];
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                const int f = et + 128 * (kb + k);
                                const bool live = c0 + (f >> 5) < rows;
                                t0[k] = live ? __ldcg(p0 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
                                t1[k] = live && two ? __ldcg(p1 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                acc[k].x += t0[k].x; acc[k].y += t0[k].y; acc[k].z += t0[k].z; acc[k].w += t0[k].w;
                                if (two) {
                                    acc[k].x += t1[k].x; acc[k].y += t1[k].y; acc[k].z += t1[k].z; acc[k].w += t1[k].w;
                                }
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 4; k++) {
                            const int f = et + 128 * (kb + k), row = f >> 5, cq = f & 31;   // columns 4 cq .. 4 cq + 3
                            *reinterpret_cast<float4 *>(T + row * FT_TSTRIDE + (cq >> 3) * 36 + 4 * (cq & 7)) = acc[k];
                        }
                    }
                } else {
                    float v[32];
                    load_acc(c0, v);
#pragma unroll
                    for (int i = 0; i < 32; i++) T[i * FT_TSTRIDE + (r >> 5) * 36 + (r & 31)] = v[i];
                    if (own_in_tmem) {
                        // this CTA's part is in T: add the other contributors' slabs in CTA
                        // order, every load of a contributor issued at once (thread et: float4
                        // f = et + 128 k; a thread reads and rewrites only its own positions)
                        named_bar(1, 128);
                        const float4 *pbase = reinterpret_cast<const float4 *>(a.partials + (int64_t)c0 * FT_BM);
#pragma unroll
                        for (int kb = 0; kb < 8; kb += 4) {
                            float4 acc[4];
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                const int f = et + 128 * (kb + k), row = f >> 5, cq = f & 31;
                                acc[k] = *reinterpret_cast<const float4 *>(T + row * FT_TSTRIDE + (cq >> 3) * 36 + 4 * (cq & 7));
                            }
                            for (int cc = c_first + 1; cc <= c_last; cc++) {
                                const float4 *pc = pbase + (int64_t)(cc + gi) * (frag / 4);
                                float4 t[4];
#pragma unroll
                                for (int k = 0; k < 4; k++) {
                                    const int f = et + 128 * (kb + k);
                                    t[k] = c0 + (f >> 5) < rows ? __ldcg(pc + f) : make_float4(0.f, 0.f, 0.f, 0.f);
                                }
#pragma unroll
                                for (int k = 0; k < 4; k++) {
                                    acc[k].x += t[k].x; acc[k].y += t[k].y; acc[k].z += t[k].z; acc[k].w += t[k].w;
                                }
                            }
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                const int f = et + 128 * (kb + k), row = f >> 5, cq = f & 31;
                                *reinterpret_cast<float4 *>(T + row * FT_TSTRIDE + (cq >> 3) * 36 + 4 * (cq & 7)) = acc[k];
                            }
                        }
                    }
                }
                named_bar(1, 128);
                // row c0 + ti, values of operand rows 32*part .. 32*part + 31
                float x[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(T + ti * FT_TSTRIDE + part * 36 + i);
                    x[i] = t4.x; x[i + 1] = t4.y; x[i + 2] = t4.z; x[i + 3] = t4.w;
                }
                // Had128 over the block.  The operand-row order is a permutation of
                // the bits of the column index, under which the Sylvester matrix is
                // invariant, so the transform runs on operand rows directly.
#pragma unroll
                for (int hs = 1; hs < 32; hs <<= 1) {
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        if (i & hs) continue;
                        const float p0 = x[i], p1 = x[i + hs];
                        x[i] = p0 + p1;
                        x[i + hs] = p0 - p1;
                    }
                }
#pragma unroll
                for (int m = 1; m < 4; m <<= 1) {
                    const float sgn = (part & m) ? -1.f : 1.f;   // o - x or x + o as one exact-sign FMA
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const float o = __shfl_xor_sync(kFull, x[i], m);
                        x[i] = fmaf(sgn, x[i], o);
                    }
                }
                const int nrow = c0 + ti;
                if (nrow < rows) {
                    // operand row 32*part + k holds column 16*(k % 8) + 4*part + k / 8
                    const int colb = G * kHad + 4 * part;
                    if constexpr (ROWS) {
                        // fp32 rows: y = Had128(v) * post
                        float *dst = a.out_rows + (int64_t)(d.out0 + nrow) * a.OC_rows + colb;
#pragma unroll
                        for (int jj = 0; jj < 8; jj++) {
                            const uint2 rv = *reinterpret_cast<const uint2 *>(s_scale + 4 * part + 16 * jj);
                            float4 o;
                            o.x = (x[jj] * kHadNorm) * f16_bits_to_f32((uint16_t)(rv.x & 0xFFFFu));
                            o.y = (x[jj + 8] * kHadNorm) * f16_bits_to_f32((uint16_t)(rv.x >> 16));
                            o.z = (x[jj + 16] * kHadNorm) * f16_bits_to_f32((uint16_t)(rv.y & 0xFFFFu));
                            o.w = (x[jj + 24] * kHadNorm) * f16_bits_to_f32((uint16_t)(rv.y >> 16));
                            *reinterpret_cast<float4 *>(dst + 16 * jj) = o;
                        }
                    } else {
                        uint16_t *dst = a.out + (int64_t)nrow * a.ldo + d.out0 + colb;
                        // the Hadamard scale, times the row's activation scale when there is one
                        const float hn = a.row_scale ? kHadNorm * __ldg(a.row_scale + d.u_row + nrow) : kHadNorm;
#pragma unroll
                        for (int jj = 0; jj < 8; jj++) {
                            const int cl = 4 * part + 16 * jj;     // column within the block
                            const uint2 rv = *reinterpret_cast<const uint2 *>(s_scale + cl);
                            const uint2 sv = *reinterpret_cast<const uint2 *>(s_scale + FT_BM + cl);
                            const uint32_t rw[2] = {rv.x, rv.y}, sw[2] = {sv.x, sv.y};
                            uint32_t o2[2];
#pragma unroll
                            for (int h = 0; h < 2; h++) {
                                float y0 = (x[jj + 16 * h] * hn) * f16_bits_to_f32((uint16_t)(rw[h] & 0xFFFFu));
                                float y1 = (x[jj + 16 * h + 8] * hn) * f16_bits_to_f32((uint16_t)(rw[h] >> 16));
                                y0 *= f16_bits_to_f32((uint16_t)(sw[h] & 0xFFFFu));
                                y1 *= f16_bits_to_f32((uint16_t)(sw[h] >> 16));
                                o2[h] = (uint32_t)f32_to_bf16_bits(y0) | ((uint32_t)f32_to_bf16_bits(y1) << 16);
                            }
                            *reinterpret_cast<uint2 *>(dst + 16 * jj) = make_uint2(o2[0], o2[1]);
                        }
                    }
                }
                named_bar(1, 128);   // T is rewritten by the next chunk
            }
            if (!split || own_in_tmem) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_ACCE + b));
            }
        })
    }
#undef FT_FOR_SEGMENTS

    tc_fence_before();
    __syncthreads();
    if (*s_abort && lane == 0 && (warp == W_BLOAD || warp == W_CODE)) {
        // let this thread's copies in flight land before the CTA exits
        const int depth = warp == W_BLOAD ? C::BCHUNKS : C::CSTAGES;
        const int b0 = warp == W_BLOAD ? B_BFULL : B_CFULL;
        for (int g = issued - depth > 0 ? issued - depth : 0; g < issued; g++)
            mbar_drain(bar(b0 + g % depth), (g / depth) & 1);
    }
    __syncthreads();
    if (warp == W_MMA0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
    }
}

template <int NT, bool ROWS>
cudaError_t launch_fused_t(const FusedArgs &a, int64_t total_units, cudaStream_t s) {
    using C = FtCfg<NT>;
    const cudaError_t ea = kernel_smem_optin((const void *)fused_tc_kernel<NT, ROWS>, C::SMEM);
    if (ea != cudaSuccess) return ea;
    int64_t grid = device_info().sm_count;       // one CTA per SM (shared memory)
    if (grid > kFusedMaxCtas) grid = kFusedMaxCtas;
    if (grid > total_units) grid = total_units;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(FT_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_tc_kernel<NT, ROWS>, a);
}

}  // namespace

size_t fused_slab_floats(int max_groups, int64_t rows) {
    if (rows > kFusedMaxRows) rows = kFusedMaxRows;
    return (size_t)(kFusedMaxCtas + max_groups) * FT_BM * (size_t)rows;
}

bool fused_supported() { return tma_encode_available(); }

cudaError_t launch_fused(FusedArgs &a, const uint16_t *u, cudaStream_t s) {
    if (a.M <= 0 || a.M > kFusedMaxRows || a.IC <= 0 || a.IC % 128 || a.n_shards < 1 || a.n_shards > 4)
        return cudaErrorInvalidValue;
    const int nt = a.M <= 16 ? 16 : (a.M <= 32 ? 32 : (a.M <= 64 ? 64 : 128));
    int slots = 0;
    for (int i = 0; i < a.n_shards; i++)
        if (a.sh[i].u_slot < 0) return cudaErrorInvalidValue;
        else if (a.sh[i].u_slot + 1 > slots) slots = a.sh[i].u_slot + 1;
    if (!make_map_f16(&a.tm_u, u, (int64_t)slots * a.M, a.IC, nt)) return cudaErrorInvalidValue;
    for (int i = 0; i < a.n_shards; i++)
        if (!make_map_code(&a.tm_code[i], a.sh[i].code, a.IC, a.sh[i].OC, a.sh[i].K)) return cudaErrorInvalidValue;
    a.entries = nullptr;
    a.n_entries_dev = nullptr;
    a.hash_xor = kHashXor;
    for (int i = 0; i < 17; i++) a.pow2[i] = 1u << i;
    int64_t groups = 0;
    for (int i = 0; i < a.n_shards; i++) groups += a.sh[i].OC / kHad;
    const int64_t total = groups * (a.IC / FT_KC);
    switch (nt) {
        case 16: return launch_fused_t<16, false>(a, total, s);
        case 32: return launch_fused_t<32, false>(a, total, s);
        case 64: return launch_fused_t<64, false>(a, total, s);
        default: return launch_fused_t<128, false>(a, total, s);
    }
}

bool fused_rows_fits(int64_t max_entries, int groups_per_entry, int IC) {
    // every CTA's column groups must fall in at most kFtMaxEntries entries
    int64_t grid = device_info().sm_count;
    if (grid > kFusedMaxCtas) grid = kFusedMaxCtas;
    const int64_t units = max_entries * groups_per_entry * (int64_t)(IC / FT_KC);
    const int64_t per_cta = (units + grid - 1) / grid;
    const int64_t per_entry = (int64_t)groups_per_entry * (IC / FT_KC);
    return per_cta / per_entry + 2 <= kFtMaxEntries;
}

cudaError_t launch_fused_rows(FusedArgs &a, const uint16_t *u, int64_t u_rows, int64_t max_entries,
                              cudaStream_t s) {
    if (a.IC <= 0 || a.IC % 128 || a.groups_per_entry < 1 || !a.entries || !a.n_entries_dev || !a.out_rows)
        return cudaErrorInvalidValue;
    a.M = kFusedRowsNT;
    a.n_shards = 0;
    if (!make_map_f16(&a.tm_u, u, u_rows, a.IC, kFusedRowsNT)) return cudaErrorInvalidValue;
    a.hash_xor = kHashXor;
    for (int i = 0; i < 17; i++) a.pow2[i] = 1u << i;
    const int64_t total = max_entries * a.groups_per_entry * (int64_t)(a.IC / FT_KC);
    return launch_fused_t<kFusedRowsNT, true>(a, total, s);
}

}  // namespace exl3
