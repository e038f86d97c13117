// internal.h -- host-side launch interfaces between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace exl3 {

// Rows of the decode-mode GEMM per pass: tokens are processed in n-blocks of 8
// (the MMA's N), at most kDecodeMaxNB blocks held in registers at once.
constexpr int kDecodeMaxNB = 4;
constexpr int kDecodeMaxRows = 8 * kDecodeMaxNB;
// Upper bound on decode-GEMM CTAs (persistent grid); sizes the partial slab.
constexpr int kDecodeMaxCtas = 1024;
constexpr int kDecodeWarps = 8;
// Arrival counters in every workspace: one per output column group of a launch.
constexpr size_t kWorkspaceCounters = 65536;

struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
};
const DeviceInfo &device_info();
// Opt `kernel` in to `smem` bytes of dynamic shared memory on the current device
// (once per kernel and device), and its resident CTAs per SM with `threads`
// threads per CTA.
cudaError_t kernel_smem_optin(const void *kernel, size_t smem);
cudaError_t kernel_occupancy(const void *kernel, int threads, size_t smem, int *occ);

// Workspace carving shared by the linear entry points.
struct LinearWorkspace {
    int32_t *err = nullptr;        // error word
    int32_t *counters = nullptr;   // per output column group (128 columns)
    uint16_t *u = nullptr;         // pre-transformed activations fp16 [M][IC]
    float *partials = nullptr;     // split-K slab
    uint16_t *wt = nullptr;        // prefill: decoded W^T fp16 [OC][IC]
    size_t counters_n = 0, u_elems = 0, partial_elems = 0, wt_elems = 0;
};
size_t linear_workspace_layout(int64_t max_M, int32_t max_IC, int32_t max_OC,
                               LinearWorkspace *ws, void *base);

cudaError_t launch_pretransform(const uint16_t *x, int64_t M, int IC, const uint16_t *s_in,
                                const uint16_t *rin, uint16_t *u, cudaStream_t s);
// Pre-transform of x once per shard: u[shard][m][:] with shard s using (s_in[s], rin[s]).
struct PretransformShards {
    const uint16_t *s_in[4];
    const uint16_t *rin[4];
    int n;
};
cudaError_t launch_pretransform_shards(const uint16_t *x, int64_t M, int IC, const PretransformShards &p,
                                       uint16_t *u, cudaStream_t s);
// pdl: launch as a programmatic dependent of the preceding kernel, which must
// itself have waited for everything before it before triggering (the
// pre-transforms do): the reconstruct then overlaps that kernel and completes
// after it.
cudaError_t launch_reconstruct(const int16_t *code, int IC, int OC, int K, uint16_t *W,
                               bool transposed, cudaStream_t s, bool pdl = false);
cudaError_t launch_codebook_table(uint16_t *table, cudaStream_t s);

// One problem of the grouped decode-mode GEMM: a code tensor [IC/16][OC/16][16K]
// applied to rows [u_row0, u_row0 + nrows) of the activation matrix.
struct GroupEntry {
    const int16_t *code;
    const uint16_t *post;     // dense: rout [OC]; rows mode: post-scale [OC]
    const uint16_t *post2;    // dense: s_out [OC]; rows mode: unused
    int64_t out_off;          // dense: column of out where this entry starts; rows: first output row
    int32_t K;
    int32_t OC;
    int32_t u_row0;
    int32_t nrows;            // <= 8 * NB of the launch
    int32_t g0;               // first global column-group index of this entry
    int32_t slot;             // MoE: the expert's bank slot (the paired FC1 epilogue's w2_suh row)
};

enum GroupMode : int32_t {
    kModeDense = 0,   // y = (Had128(v) * post) * post2 -> bf16 out[row][out_off + col], row stride ldo
    kModeRows = 1,    // y = Had128(v) * post -> fp32 out_rows[(out_off + row) * OC + col]
};

struct GroupGemmArgs {
    const uint16_t *u;            // fp16 activations, row stride IC (or 8-bit codes, below)
    int IC;
    int mode;
    const GroupEntry *entries;    // device array (MoE) or nullptr (use inline)
    const int32_t *n_entries_dev; // device entry count (MoE) or nullptr
    int n_groups_per_entry;       // > 0: every entry has this many column groups (MoE)
    int n_inline;
    GroupEntry inline_e[4];       // dense: up to 4 shards passed by value
    uint16_t *out;                // dense output base (bf16), row stride ldo
    int64_t ldo;
    float *out_rows;              // rows-mode output (fp32)
    float *partials;
    int32_t *counters;
    uint32_t hash_xor;            // the codebook's xor constant, kept in a register
    uint32_t pow2[17];            // pow2[o] = 1 << o (multipliers of the state extraction)
    int32_t max_rows;             // rows per entry the launch was sized for
    int32_t parts;                // > 0: CTA c takes part c % parts of group c / parts (set by the launcher)
    // Rows mode with gathered activations (grouped MoE, one 8-row block per
    // entry): u holds two halves of R rows each, stored per (token, route) pair;
    // entry row g (routed row r = e.u_row0 - j R + g of half j) reads row
    // row_pair[r] of its half.
    int32_t gather;
    int32_t R, topk;
    const int32_t *row_pair;
    // Combine epilogue (FC2): after writing routed row r, the last of token t's
    // valid routes to arrive at column group G sums y[t] = sum_k comb_w[t][k] *
    // out_rows[comb_pos[t][k]] in k order into comb_y (bf16 [T][OC]).
    int32_t comb;
    const float *comb_w;
    const int32_t *comb_pos;
    uint16_t *comb_y;
    int32_t *comb_counters;       // [T][OC / 128], zero between calls
    // 8-bit activations: u holds uint8 codes q + 128 (row stride IC bytes); the
    // epilogue multiplies row r = e.u_row0 + n by row_scale[r] (non-null only
    // then; one 8-row block per entry)
    int32_t codes;
    const float *row_scale;
    // Paired FC1 (gathered rows, entries 2i / 2i + 1 = w1 / w3 of one expert row
    // block): the epilogue writes FC2's input act_out[row][col] (fp16, row stride
    // OC) = Had128((silu(g) * u) * act_suh[slot][col]) instead of fp32 rows.
    int32_t pair_act;
    const uint16_t *act_suh;
    uint16_t *act_out;
    // The device entry list (and the routed-row tables) were written by a kernel
    // that completed before the preceding kernel in the stream let this launch
    // start: read them, and request the first code words, before waiting for
    // the preceding kernel (whose output is only the activations).
    int32_t entries_ready;
    // Rows mode over device entry lists, one 8-row block of fp16 rows (MoE FC2
    // at few routed pairs): one 16-warp CTA per column group at a time, the
    // group's tile rows split over its warps (group_wide_kernel).
    int32_t wide;
};
constexpr int kMaxInlineEntries = 4;

// Launch the grouped decode-mode GEMM; `max_groups` bounds the total number of
// column groups (for the partial slab), rows per entry <= 8 * nb.  A launch with
// gathered activations (a.gather) needs nb == 1.
cudaError_t launch_group_gemm(const GroupGemmArgs &a, int nb, bool pdl, cudaStream_t s);
size_t group_slab_floats(int max_groups, int nb);

// Fused decode + tensor-core GEMM for 8 < M <= kFusedMaxRows rows: the trellis
// is decoded into shared-memory operand tiles that tcgen05 MMAs multiply by the
// pre-transformed activations u [shard][M][IC] (fp16).
constexpr int kFusedMaxRows = 128;
constexpr int kFusedMaxCtas = 256;
constexpr int kFusedRowsNT = 64;      // rows mode (grouped MoE entries): rows per entry
struct FusedShard {
    const int16_t *code;
    const uint16_t *rout, *s_out;
    int64_t col0;        // first output column of this shard
    int32_t K, OC;
    int32_t g0;          // first global column-group index
    int32_t u_slot;      // this shard's activations are rows [u_slot * M, (u_slot + 1) * M) of u
};
struct FusedArgs {
    CUtensorMap tm_u;        // u [n_shards * M][IC], box 64 channels x rows-per-tile
    CUtensorMap tm_code[4];  // per shard: the code as (tile words, tiles, tile rows)
    FusedShard sh[4];
    int32_t n_shards, M, IC, pad_;
    uint16_t *out;       // bf16, row stride ldo
    int64_t ldo;
    // rows mode (device-built entry lists, e.g. the grouped MoE): per entry a code
    // tensor applied to rows [u_row0, u_row0 + nrows) of u, written as fp32 rows
    // out_rows[(out_off + row) * OC_rows + col] = Had128(v) * post
    const GroupEntry *entries;
    const int32_t *n_entries_dev;
    int32_t groups_per_entry;   // OC_rows / 128
    int32_t OC_rows;
    float *out_rows;
    float *partials;     // split-K slab, fused_slab_floats() floats
    int32_t *counters;
    int32_t *err;
    uint32_t hash_xor;
    uint32_t pow2[17];
    // dense mode, 8-bit activations: output row r of shard s is scaled by
    // row_scale[u_slot * M + r] (u then holds the codes' exact fp16 values)
    const float *row_scale;
};
bool fused_supported();
size_t fused_slab_floats(int max_groups, int64_t rows);
cudaError_t launch_fused(FusedArgs &a, const uint16_t *u, cudaStream_t s);
// Rows mode over a device-built entry list of at most max_entries entries, each
// with at most kFusedRowsNT rows; u has u_rows rows.  fused_rows_fits() tells
// whether a launch of that size fits the kernel's per-CTA entry cache.
bool fused_rows_fits(int64_t max_entries, int groups_per_entry, int IC);
cudaError_t launch_fused_rows(FusedArgs &a, const uint16_t *u, int64_t u_rows, int64_t max_entries,
                              cudaStream_t s);

// The GEMM path pinned by exl3_set_gemm_path: 0 none (by rows), 1 decode, 2 fused, 3 prefill.
int forced_mode();

bool prefill_supported();
// epi 0: the EXL3 output transform (OC a multiple of 128); epi 1: a per-column
// scale rout, no transform (any OC).
// row_scale (epi 0 only, may be null): output row m is scaled by row_scale[m].
cudaError_t launch_prefill(const uint16_t *u, const uint16_t *wt, int64_t M, int IC, int OC,
                           const uint16_t *rout, const uint16_t *s_out, uint16_t *out,
                           int64_t ldo, int32_t *err, cudaStream_t s, bool *launched, int epi = 0,
                           const float *row_scale = nullptr);

// 8-bit activations.  Pre-transform (once per shard, as launch_pretransform_shards)
// plus per-row quantization of x [M][IC]: row r = shard * M + m of dst and As,
// As[r] = amax_r / 127, q = round-half-even(u / As) clamped to [-127, 127];
// f16_out = false: codes q + 128 into dst as uint8 [n * M][IC]; true: q as exact
// fp16 into dst as uint16 [n * M][IC].  IC * 4 bytes of shared memory per row.
cudaError_t launch_quantize_a8(const uint16_t *x, int64_t M, int IC, const PretransformShards &p, void *dst,
                               bool f16_out, float *As, cudaStream_t s);
size_t quantize_a8_smem_bytes(int IC);
// uint8 codes [n] -> q = code - 128 as exact fp16 (n a multiple of 8, both 16-byte aligned).
cudaError_t launch_codes_to_f16(const uint8_t *A, int64_t n, uint16_t *dst, cudaStream_t s);

// int8 output head, few rows (M <= 32), x16 the fp16 activations: ctr = two
// zeroed workspace counters.
cudaError_t launch_lm_head_decode(const uint16_t *x16, int M, int H, const int8_t *q, const uint16_t *scale, int64_t V,
                                  uint16_t *out, int64_t ldo, int32_t *ctr, cudaStream_t s);
// Conversions for the tensor-core head: int8 rows -> fp16, bf16 rows -> fp16 (exact).
cudaError_t launch_i8_to_f16(const int8_t *q, int64_t n, uint16_t *dst, cudaStream_t s);
cudaError_t launch_bf16_to_f16(const uint16_t *x, int64_t n, uint16_t *dst, cudaStream_t s);

cudaError_t launch_gather(const int8_t *q, const uint16_t *scale, int64_t V, int H,
                          const int32_t *ids, int64_t N, uint16_t *out, int32_t *n_bad,
                          cudaStream_t s);

}  // namespace exl3
