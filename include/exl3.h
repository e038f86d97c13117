/*
 * exl3.h -- C ABI of the GB300 (sm_103a) EXL3 trellis library.
 *
 * The library computes the EXL3 (exllamav3 trellis) quantized linear layer
 *
 *     y = s_out * rout * Had128( Had128((x * s_in) * rin) @ decode(code) )
 *
 * (radiance_escha.py, module docstring "THE FORWARD": rin is a pre-scale
 * applied before its Hadamard, rout a post-scale applied after its own, rin
 * already carries the weight scale and is applied exactly once, and no bias is
 * applied), its merged-shard column-slice form (radiance_escha.py,
 * escha_linear_into and EschaLinearMethod.apply: one call per source tensor,
 * each writing its own columns of one output buffer), the grouped MoE form
 * over a flat expert bank (bank.py: w13 = [w1 | w3] per slot, w2, K-sorted
 * slots) and the int8 embedding gather (vllm-quantpack exl3/embedding.py,
 * embedding()).
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller, unless a comment
 *     says otherwise.  The library never allocates or frees device memory and
 *     never synchronizes the stream; every call is asynchronous on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream).
 *   - bf16 and fp16 values are passed as uint16_t bit patterns.
 *   - Code tensors are int16 [IC/16][OC/16][16*K], one block of 16*K words per
 *     16x16 weight tile, the first index along the input channels
 *     (radiance_escha.py: the module's 16-wide tile constant and the code
 *     tensor shape it documents; K is the last dimension divided by 16).  K must
 *     be 2, 3 or 4.
 *   - IC and OC must be multiples of 128: the incoherence transform is blocked
 *     at 128 channels and a boundary inside a block would change the transform
 *     (radiance_escha.py, create_weights / process_weights_after_loading).
 *   - Arguments are validated on the host before any launch.  A bad argument
 *     returns EXL3_EINVAL (nothing is launched) and exl3_last_error() names the
 *     sizes involved.  No entry point aborts the process.
 *   - M == 0 (no rows) is a no-op returning EXL3_OK (radiance_escha.py,
 *     escha_linear_into returns at once when there are no rows).
 *
 * Trellis decode reading (the pages give only the tensor shapes): a tile's
 * 16K words are a stream read most-significant bit first; weight t (0..255,
 * at tile row t/16 along IC and column t%16 along OC) decodes the 16-bit state
 * formed by stream bits [(t+1)K-16, (t+1)K), taken modulo the tile's 256K bits
 * (tail-biting), through the QTIP 3INST hash
 *     z = 89226354*s + 64248484 (mod 2^32); z' = (z & 0x8FFF8FFF) ^ 0x3B603B60;
 *     w = fp16(half(z' & 0xFFFF) + half(z' >> 16)).
 */
#ifndef EXL3_GB300_H
#define EXL3_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EXL3_OK = 0,
    EXL3_EINVAL = 1,        /* bad size, alignment, K or pointer; nothing launched */
    EXL3_EWORKSPACE = 2,    /* workspace missing or smaller than the query says */
    EXL3_ECUDA = 3,         /* a CUDA runtime call or launch failed */
    EXL3_EUNSUPPORTED = 4,  /* valid request this build does not implement */
    EXL3_EDEVICE = 5        /* a kernel recorded an error (see exl3_workspace_error) */
} exl3_status;

/* A cudaStream_t, passed opaquely so that this header needs no CUDA headers. */
typedef void *exl3_stream;

/* Message of the last failing call on this host thread ("" if none). */
const char *exl3_last_error(void);

/* Library version string. */
const char *exl3_version(void);

/* ---------------------------------------------------------------- workspace */

/*
 * Bytes of workspace exl3_linear / exl3_linear_into need for any call with
 * M <= max_M, IC <= max_IC and OC <= max_OC.  It holds the pre-transformed
 * activations, the split-K partial slab with its per-column-group arrival
 * counters (radiance_escha.py, _ensure_scratch: an fp32 partial slab plus an
 * int32 block counter, allocated once per device outside graph capture), an
 * error word, and for large M the decoded weight staging of the prefill path.
 * Returns 0 for invalid sizes.
 */
size_t exl3_linear_workspace_bytes(int64_t max_M, int32_t max_IC, int32_t max_OC);

/*
 * Prepare a freshly allocated workspace (zeroes counters and the error word).
 * Must run once before the workspace's first use; the kernels leave the
 * counters at zero again after every call.  ws must be 256-byte aligned.
 * Two calls that share one workspace must not run concurrently.
 */
exl3_status exl3_workspace_init(void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * Copy the workspace's device error word to *flag_host (host pointer) and
 * synchronize `stream`.  0 = no kernel recorded an error.  A nonzero value
 * names the first failure a kernel recorded (for example a bounded wait that
 * gave up); the word stays set until exl3_workspace_init runs again.
 */
exl3_status exl3_workspace_error(const void *ws, size_t ws_bytes, int32_t *flag_host,
                                 exl3_stream stream);

/* ------------------------------------------------------------------ linear */

/*
 * Test and measurement hook: pin the GEMM path every linear call takes,
 * process-wide, instead of choosing it by the number of rows.  Workspace
 * queries made while a path is pinned size for that path, so query after
 * pinning.  EXL3_PATH_BY_ROWS (the default) restores the normal choice.  The
 * decode path serves any M (in passes of 32 rows); the fused path applies to
 * M <= 128 and otherwise falls back to the choice by rows.  Returns
 * EXL3_EINVAL for any other value.  Not for concurrent use with running calls.
 */
enum {
    EXL3_PATH_BY_ROWS = 0,
    EXL3_PATH_DECODE = 1,
    EXL3_PATH_FUSED = 2,
    EXL3_PATH_PREFILL = 3
};
exl3_status exl3_set_gemm_path(int32_t path);

/*
 * One EXL3 projection into a column slice of a caller-owned output
 * (radiance_escha.py, escha_linear_into):
 *   x      bf16 [M][IC], row-major, contiguous
 *   code   int16 [IC/16][OC/16][16*K]
 *   s_in, rin    fp16 [IC]      pre-scales, applied before the input Had128
 *   rout, s_out  fp16 [OC]      post-scales, applied after the output Had128
 *   out    bf16 [M][ldo]; only columns [col0, col0 + OC) are written, every
 *          other column is left untouched (a merged layer calls this once per
 *          shard, advancing col0 by that shard's OC)
 *   ws     workspace of at least exl3_linear_workspace_bytes(M, IC, OC) bytes
 * Requires ldo >= OC, 0 <= col0, col0 + OC <= ldo, and 16-byte aligned x,
 * code, and out + col0 rows (ldo and col0 multiples of 8).
 * The GEMM path is chosen by M inside this call (radiance_escha.py,
 * escha_linear_into: the small-M / large-M switch lives in the op): a
 * register-resident trellis decode for M <= 16, the trellis decoded into
 * tensor-core operand tiles for M <= 128, reconstruct + tensor-core GEMM above
 * (exl3_set_gemm_path pins one path for tests and measurements).
 */
exl3_status exl3_linear_into(const uint16_t *x, int64_t M, int32_t IC,
                             const int16_t *code, int32_t OC, int32_t K,
                             const uint16_t *s_in, const uint16_t *rin,
                             const uint16_t *rout, const uint16_t *s_out,
                             uint16_t *out, int64_t ldo, int64_t col0,
                             void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * Steps 2 and 3 of THE FORWARD on activations that are already transformed:
 *   out[:, col0:col0+OC] = bf16( (Had128(u @ decode(code)) * rout) * s_out )
 *   u  fp16 [M][IC] = Had128((x * s_in) * rin), as exl3_pretransform writes it.
 * For callers whose shards share one input transform (the radiance_escha.py
 * docstring says rin and s_in are shared across merged shards, while its
 * loader measured them differing per shard): transform once, then call this
 * per shard.  Same requirements as exl3_linear_into, with u in place of x.
 */
exl3_status exl3_gemm_into(const uint16_t *u, int64_t M, int32_t IC,
                           const int16_t *code, int32_t OC, int32_t K,
                           const uint16_t *rout, const uint16_t *s_out,
                           uint16_t *out, int64_t ldo, int64_t col0,
                           void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * exl3_linear_into without a workspace, for callers that cannot allocate
 * device memory: code running where cudaMalloc is not allowed or not wanted
 * (inside a host callback, under an allocator-owning framework or plugin host
 * that hands out no spare buffer, or on a path that must never trigger an
 * allocation or its implicit synchronization).  No page the library follows
 * has a counterpart of this call.
 *
 * Same arguments and result as exl3_linear_into, minus the workspace; the
 * caller still owns x, code, the scale vectors and out.  Scratch comes from one
 * fixed array of about 6.8 MB that the library declares in device memory:
 * every GPU that loads the library holds it until the process exits.  Limits:
 * M <= 8, IC <= 32768, OC <= 65536; larger requests return EXL3_EINVAL and
 * launch nothing.  The call allocates and frees nothing.
 *
 * Every call looks up the array's device address on the current device; the
 * first call on a device may load the library's device code there, so make
 * that first call before any stream capture.  Every call on a device shares
 * the one array and clears its counters on entry, so calls that overlap on
 * the GPU (different streams, or other threads) race and give wrong results:
 * serialize them.
 */
exl3_status exl3_linear_into_noalloc(const uint16_t *x, int64_t M, int32_t IC,
                                     const int16_t *code, int32_t OC, int32_t K,
                                     const uint16_t *s_in, const uint16_t *rin,
                                     const uint16_t *rout, const uint16_t *s_out,
                                     uint16_t *out, int64_t ldo, int64_t col0,
                                     exl3_stream stream);

/*
 * One merged layer (radiance_escha.py, EschaLinearMethod.apply: gate_up_proj
 * = gate_proj + up_proj, qkv_proj = q/k/v, each source tensor its own EXL3
 * tensor with its own K and scale vectors) in one call: the result equals
 * calling exl3_linear_into once per shard, in order, on the same x and out.
 * All shards share IC; each has its own code, K, OC, four scale vectors and
 * column offset col0 (the caller advances col0 by each shard's OC, as
 * EschaLinearMethod.apply does).  The shards run in one pre-transform launch
 * and one grouped GEMM launch (for M <= 32 rows per pass), so the merged
 * layer has one tail instead of one per shard.
 *   shards   HOST array of n_shards descriptors, 1 <= n_shards <= 4
 *   ws       exl3_linear_shards_workspace_bytes(M, IC, shards, n_shards) bytes
 */
/*
 * Codebook of a tensor.  EXL3 checkpoints mark a tensor's codebook with
 * per-tensor marker entries (vllm-quantpack linear.py, LINEAR_SUFFIXES lists
 * mcg and mul1 beside trellis, read as present / absent per shard; in the vLLM
 * PR #190 thread a commit treats the two markers as sentinels and sends
 * MCG-marked modules to one kernel, legacy and MUL1 shards to another).  The pages give neither
 * variant's constants, so this build decodes the default (3INST) codebook only:
 * a shard marked MCG or MUL1 returns EXL3_EUNSUPPORTED before any launch.
 */
enum {
    EXL3_CODEBOOK_3INST = 0,   /* no marker: the default codebook */
    EXL3_CODEBOOK_MCG = 1,     /* "mcg" marker present */
    EXL3_CODEBOOK_MUL1 = 2     /* "mul1" marker present */
};

typedef struct exl3_shard {
    const int16_t *code;      /* [IC/16][OC/16][16*K] */
    const uint16_t *s_in;     /* fp16 [IC] */
    const uint16_t *rin;      /* fp16 [IC] */
    const uint16_t *rout;     /* fp16 [OC] */
    const uint16_t *s_out;    /* fp16 [OC] */
    int32_t OC;
    int32_t K;
    int64_t col0;
    int32_t codebook;         /* EXL3_CODEBOOK_*; 0 (zero-initialised) is the default */
    int32_t reserved;         /* 0 */
} exl3_shard;

size_t exl3_linear_shards_workspace_bytes(int64_t max_M, int32_t IC, const exl3_shard *shards,
                                          int32_t n_shards);

exl3_status exl3_linear_into_shards(const uint16_t *x, int64_t M, int32_t IC,
                                    const exl3_shard *shards, int32_t n_shards,
                                    uint16_t *out, int64_t ldo,
                                    void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * exl3_linear_into_shards with x and out in host memory.  x_host and out_host
 * are pinned host buffers mapped into the device's address space
 * (cudaMallocHost / cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped; with unified addressing all pinned memory is
 * mapped).  The pre-transform reads x, and the GEMM's epilogue writes out,
 * through those mappings (over the host link: NVLink-C2C on Grace parts):
 * there are no staging copies and no device copies of x or out.  For
 * decode-sized M, where x and out are small, this is the cheapest way to run
 * the layer on host-resident activations.
 *   x_host    HOST pinned bf16 [M][IC] (8-byte aligned)
 *   out_host  HOST pinned bf16 [M][ldo]; only the shards' column slices are written
 *   shards, ws, stream: as for exl3_linear_into_shards (device memory)
 * Returns EXL3_EINVAL before any launch if x_host or out_host is not mapped
 * pinned host memory (pageable host memory and device memory included).
 * Asynchronous like every call: synchronize the stream before reading out_host.
 */
exl3_status exl3_linear_into_shards_host(const uint16_t *x_host, int64_t M, int32_t IC,
                                         const exl3_shard *shards, int32_t n_shards,
                                         uint16_t *out_host, int64_t ldo,
                                         void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * exl3_linear_into_shards on activations already transformed per shard:
 * u fp16 [n_shards][M][IC], u[i] = Had128((x * s_in_i) * rin_i) (as
 * exl3_pretransform writes it); the shards' s_in / rin pointers are ignored.
 * One grouped GEMM launch per 32 rows.
 */
exl3_status exl3_gemm_into_shards(const uint16_t *u, int64_t M, int32_t IC,
                                  const exl3_shard *shards, int32_t n_shards,
                                  uint16_t *out, int64_t ldo,
                                  void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * Several projections of one layer (for a decoder layer: qkv, o, gate_up, down)
 * in one call on one workspace, in order: projection i is exl3_linear_into_shards
 * on its own x_i, IC_i, shards and out_i.  Inputs that several projections read
 * are transformed once: projections with the same x pointer share the
 * pre-transformed rows of every distinct (s_in, rin) pointer pair among their
 * shards (equal values under different pointers are not detected).  All
 * projections have M rows.  The call only enqueues work (graph-capturable);
 * a projection's x may be the output of an earlier one in the same call.
 *   projs     HOST array of n descriptors, 1 <= n <= 16; shards HOST arrays
 *   ws        exl3_projections_workspace_bytes(M, projs, n) bytes, prepared by
 *             exl3_workspace_init
 */
typedef struct exl3_projection {
    const uint16_t *x;          /* bf16 [M][IC] */
    int32_t IC;
    int32_t n_shards;           /* 1..4 */
    const exl3_shard *shards;   /* HOST array of n_shards descriptors */
    uint16_t *out;              /* bf16 [M][ldo] */
    int64_t ldo;
} exl3_projection;

size_t exl3_projections_workspace_bytes(int64_t max_M, const exl3_projection *projs, int32_t n);

exl3_status exl3_linear_projections(const exl3_projection *projs, int32_t n, int64_t M,
                                    void *ws, size_t ws_bytes, exl3_stream stream);

/* exl3_linear_into with out = y [M][OC] contiguous (ldo = OC, col0 = 0). */
exl3_status exl3_linear(const uint16_t *x, int64_t M, int32_t IC,
                        const int16_t *code, int32_t OC, int32_t K,
                        const uint16_t *s_in, const uint16_t *rin,
                        const uint16_t *rout, const uint16_t *s_out,
                        uint16_t *y, void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * The activation pre-transform on its own (step 1 of THE FORWARD):
 *   u[m][:] = Had128((x[m][:] * s_in) * rin) per 128-channel block, fp16 out.
 * x bf16 [M][IC], u fp16 [M][IC].
 */
exl3_status exl3_pretransform(const uint16_t *x, int64_t M, int32_t IC,
                              const uint16_t *s_in, const uint16_t *rin,
                              uint16_t *u, exl3_stream stream);

/*
 * Decode a whole code tensor to dense fp16 weights W [IC][OC] (row-major):
 * W[16a + t/16][16b + t%16] = weight t of tile code[a][b].  The exllamav3
 * reconstruct kernel plays this role on the pages (vllm-quantpack linear.py,
 * _cut_tp: "the reconstruct kernel rejects an output width that is not a
 * multiple of 128"); here it is the decoded-weight parity hook.
 */
exl3_status exl3_reconstruct(const int16_t *code, int32_t IC, int32_t OC, int32_t K,
                             uint16_t *W, exl3_stream stream);

/* Decode every 16-bit trellis state: table[s] = fp16 weight of state s,
 * table has 65536 entries. */
exl3_status exl3_codebook_table(uint16_t *table, exl3_stream stream);

/* ------------------------------------------------------- 8-bit activations */

/*
 * The 8-bit activation variant (radiance_escha.py, escha_linear_into: the
 * projection fills a uint8 activation buffer A [M][IC] and a float32 scale
 * As [M] from a per-row amax before its GEMM; the page gives the buffers, not
 * the encoding).  The encoding read here, per row of the pre-transformed
 * activations u = Had128((x * s_in) * rin):
 *   As = amax / 127 (amax = max_c |u[c]|),
 *   q[c] = u[c] / As rounded half to even, clamped to [-127, 127] (0 if amax = 0),
 *   A[c] = q[c] + 128,
 * and the projection multiplies q * As in place of u:
 *   out[:, col0:col0+OC] = bf16( (Had128((q * As) @ decode(code)) * rout) * s_out ).
 * u, amax, As and q / As are computed in fp32 on the device.
 */

/* Bytes of workspace for exl3_linear_into_a8 / exl3_gemm_a8_into with up to
 * max_M rows (0 on invalid sizes); never decreases as max_M grows. */
size_t exl3_linear_a8_workspace_bytes(int64_t max_M, int32_t max_IC, int32_t max_OC);

/*
 * The quantizer on its own: x bf16 [M][IC] -> A uint8 [M][IC], As fp32 [M]
 * (device pointers; x, s_in, rin 8-byte aligned, A and As 4-byte aligned).
 * IC * 4 bytes of shared memory serve one row: EXL3_EUNSUPPORTED past the
 * device's limit (IC above about 56000 on this GPU).
 */
exl3_status exl3_quantize_a8(const uint16_t *x, int64_t M, int32_t IC,
                             const uint16_t *s_in, const uint16_t *rin,
                             uint8_t *A, float *As, exl3_stream stream);

/*
 * exl3_linear_into with 8-bit activations: same arguments, requirements and
 * GEMM paths; ws of at least exl3_linear_a8_workspace_bytes(M, IC, OC) bytes.
 * M <= 8 rows on the decode path multiply the codes straight from the
 * workspace; other paths expand them to exact fp16 values first.
 */
exl3_status exl3_linear_into_a8(const uint16_t *x, int64_t M, int32_t IC,
                                const int16_t *code, int32_t OC, int32_t K,
                                const uint16_t *s_in, const uint16_t *rin,
                                const uint16_t *rout, const uint16_t *s_out,
                                uint16_t *out, int64_t ldo, int64_t col0,
                                void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * The GEMM and output transform on activations already quantized (A, As as
 * exl3_quantize_a8 writes them; A 16-byte aligned): exl3_gemm_into with
 * q * As in place of u.  ws of at least exl3_linear_a8_workspace_bytes(M, IC,
 * OC) bytes.
 */
exl3_status exl3_gemm_a8_into(const uint8_t *A, const float *As, int64_t M, int32_t IC,
                              const int16_t *code, int32_t OC, int32_t K,
                              const uint16_t *rout, const uint16_t *s_out,
                              uint16_t *out, int64_t ldo, int64_t col0,
                              void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * exl3_linear_into_shards with 8-bit activations: every shard's activations
 * are quantized with its own (s_in, rin), then one grouped GEMM launch serves
 * all shards.  ws of at least exl3_linear_shards_a8_workspace_bytes(M, IC,
 * shards, n_shards) bytes.
 */
size_t exl3_linear_shards_a8_workspace_bytes(int64_t max_M, int32_t IC, const exl3_shard *shards,
                                             int32_t n_shards);
exl3_status exl3_linear_into_shards_a8(const uint16_t *x, int64_t M, int32_t IC,
                                       const exl3_shard *shards, int32_t n_shards,
                                       uint16_t *out, int64_t ldo,
                                       void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * exl3_gemm_into_shards on 8-bit activations: A uint8 [n_shards][M][IC] (16-byte
 * aligned) and As fp32 [n_shards][M], shard i's rows quantized with its own
 * (s_in, rin) as exl3_quantize_a8 writes them; the shards' s_in / rin pointers
 * are ignored.  ws as for exl3_linear_into_shards_a8.
 */
exl3_status exl3_gemm_a8_into_shards(const uint8_t *A, const float *As, int64_t M, int32_t IC,
                                     const exl3_shard *shards, int32_t n_shards,
                                     uint16_t *out, int64_t ldo,
                                     void *ws, size_t ws_bytes, exl3_stream stream);

/* -------------------------------------------------------------------- MoE */

/*
 * One layer's EXL3 expert bank (bank.py, Exl3Bank: allocate / views / tables).
 * All pointers are device pointers; "per slot" arrays are indexed by physical
 * slot p, and perm maps logical expert e to its slot p = perm[e].
 *   w13      int16, flat: slot p's w1 code tensor [H/16][I/16][16*k_gu[p]]
 *            starts at word off_w1[p], its w3 tensor (same shape) at off_w3[p]
 *   w2       int16, flat: slot p's w2 code tensor [I/16][H/16][16*k_d[p]]
 *            starts at word off_w2[p]
 *   off_w1, off_w3, off_w2   int64 [E]  word offsets (multiples of 8)
 *   perm     int32 [E]  logical expert -> slot
 *   k_gu, k_d   int32 [E]  per slot: K of w1/w3 and of w2, each 2, 3 or 4
 *   w13_suh  fp16 [E][2][H]   input pre-scales of w1 (index 0) and w3 (1)
 *   w13_svh  fp16 [E][2][I]   output post-scales of w1 and w3
 *   w2_suh   fp16 [E][I]      input pre-scale of w2
 *   w2_svh   fp16 [E][H]      output post-scale of w2
 */
typedef struct exl3_moe_bank {
    const int16_t *w13;
    const int16_t *w2;
    const int64_t *off_w1;
    const int64_t *off_w3;
    const int64_t *off_w2;
    const int32_t *perm;
    const int32_t *k_gu;
    const int32_t *k_d;
    const uint16_t *w13_suh;
    const uint16_t *w13_svh;
    const uint16_t *w2_suh;
    const uint16_t *w2_svh;
} exl3_moe_bank;

/*
 * Router helper: per token, the topk largest logits (equal logits: lower
 * expert id first) and their softmax weights over the selected topk.
 *   logits fp32 [T][E]; ids int32 [T][topk]; w fp32 [T][topk].
 * Requires 1 <= topk <= 32 and E <= 1024.
 */
exl3_status exl3_moe_topk_softmax(const float *logits, int32_t T, int32_t E, int32_t topk,
                                  int32_t *ids, float *w, exl3_stream stream);

/* Workspace bytes exl3_moe_grouped and exl3_moe_forward need for T tokens of this geometry. */
size_t exl3_moe_workspace_bytes(int32_t T, int32_t H, int32_t I, int32_t E, int32_t topk);

/*
 * Grouped SiLU-gated MoE layer over an EXL3 expert bank.  For token t and its
 * routes k = 0..topk-1 (expert e = ids[t][k], slot p = bank->perm[e]):
 *   g = Had(Had(x_t * w13_suh[p][0]) @ W1_p) * w13_svh[p][0]
 *   u = Had(Had(x_t * w13_suh[p][1]) @ W3_p) * w13_svh[p][1]
 *   d = Had(Had((silu(g) * u) * w2_suh[p]) @ W2_p) * w2_svh[p]
 *   y_t = sum over k = 0..topk-1, in that order, of w[t][k] * d
 *   x bf16 [T][H]; ids int32 [T][topk]; w fp32 [T][topk]; y bf16 [T][H].
 * Ids outside [0, E) are an error the kernels record in the workspace error
 * word (their rows contribute nothing).  Requires H, I multiples of 128,
 * topk <= 32.  ws: exl3_moe_workspace_bytes(T, H, I, E, topk) bytes,
 * prepared by exl3_workspace_init.
 */
exl3_status exl3_moe_grouped(const uint16_t *x, int32_t T, int32_t H, int32_t I,
                             int32_t E, int32_t topk, const int32_t *ids, const float *w,
                             const exl3_moe_bank *bank, uint16_t *y,
                             void *ws, size_t ws_bytes, exl3_stream stream);

/*
 * The whole MoE layer from the router logits: exl3_moe_topk_softmax followed by
 * exl3_moe_grouped, with ids [T][topk] and w [T][topk] as outputs (the routing
 * the layer used), in one call on the caller's stream.  logits fp32 [T][E];
 * requires topk <= E; other arguments and the workspace as for
 * exl3_moe_grouped.
 */
exl3_status exl3_moe_forward(const uint16_t *x, const float *logits, int32_t T, int32_t H,
                             int32_t I, int32_t E, int32_t topk, const exl3_moe_bank *bank,
                             int32_t *ids, float *w, uint16_t *y,
                             void *ws, size_t ws_bytes, exl3_stream stream);

/* ------------------------------------------------------------- embedding */

/*
 * int8 embedding gather with per-row scale (vllm-quantpack exl3/embedding.py,
 * embedding(): only the gathered rows are converted, so the table stays int8
 * in memory):  out[i][:] = bf16(q[ids[i]][:] * scale[ids[i]]), one rounding.
 *   q int8 [V][H] (row-major), scale fp16 [V], ids int32 [N], out bf16 [N][H].
 * An id outside [0, V) writes a row of zeros (the masking vLLM's vocab-parallel
 * embedding applies, same file's module docstring) and, if n_bad (device
 * int32, may be NULL) is given, is added to *n_bad.  Requires H % 16 == 0 and
 * 16-byte aligned q and out.
 */
exl3_status exl3_embed_int8_gather(const int8_t *q, const uint16_t *scale, int64_t V,
                                   int32_t H, const int32_t *ids, int64_t N,
                                   uint16_t *out, int32_t *n_bad, exl3_stream stream);

/* ------------------------------------------------------------ output head */

/*
 * The int8 table as the output projection (vllm-quantpack exl3/embedding.py,
 * Exl3EmbeddingMethod.apply: the weight is the int8 table times its per-row
 * scale, and the head computes x @ weight^T):
 *     out[m][v] = bf16( scale[v] * sum_h x[m][h] * q[v][h] )
 * with the row scale taken out of the sum and one rounding of the result.
 *   x      bf16 [M][H], 16-byte aligned; its values are multiplied as fp16 (exact
 *          for magnitudes in fp16's normal range, 2^-14 .. 65504)
 *   q      int8 [V][H] row-major (the embedding table's layout), 16-byte aligned
 *   scale  fp16 [V]
 *   out    bf16 [M][ldo], columns [0, V) written, ldo >= V
 *   ws     exl3_lm_head_workspace_bytes(M, H, V) bytes, prepared by
 *          exl3_workspace_init (counters that return to zero after each call)
 * Requires H a multiple of 256.  Up to 32 rows stream the table once through
 * registers (HBM-bound); more rows run on the tensor cores over table chunks
 * converted to fp16 in the workspace.
 */
size_t exl3_lm_head_workspace_bytes(int64_t max_M, int32_t H, int64_t V);

exl3_status exl3_lm_head_int8(const uint16_t *x, int64_t M, int32_t H,
                              const int8_t *q, const uint16_t *scale, int64_t V,
                              uint16_t *out, int64_t ldo,
                              void *ws, size_t ws_bytes, exl3_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_GB300_H */
