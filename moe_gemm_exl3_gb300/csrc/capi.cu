// capi.cu -- the extern "C" boundary: argument validation, workspace carving,
// the decode/prefill choice by M, and error reporting.  No entry point
// allocates device memory or synchronizes the caller's stream (except
// exl3_workspace_error, which is documented to).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/exl3.h"
#include "internal.h"

namespace exl3 {

static thread_local char g_err[512] = "";

// EXL3_TRACE in the environment (read once) prints every call's path and every
// error message to stderr.
static bool trace_on() {
    static const bool on = std::getenv("EXL3_TRACE") != nullptr;
    return on;
}

exl3_status fail(exl3_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    if (trace_on()) std::fprintf(stderr, "[exl3] error: %s\n", g_err);
    return st;
}

exl3_status cuda_fail(cudaError_t e, const char *where) {
    return fail(EXL3_ECUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

void trace(const char *fmt, ...) {
    if (!trace_on()) return;
    va_list ap;
    va_start(ap, fmt);
    std::fprintf(stderr, "[exl3] ");
    std::vfprintf(stderr, fmt, ap);
    std::fprintf(stderr, "\n");
    va_end(ap);
}

const DeviceInfo &device_info() {
    static DeviceInfo info[64];
    static bool done[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        cudaDeviceGetAttribute(&info[dev].sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&info[dev].max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (info[dev].sm_count <= 0) info[dev].sm_count = 1;
        done[dev] = true;
    }
    return info[dev];
}

// Per (kernel, device): the dynamic shared-memory opt-in and the resident CTAs
// per SM.  Both are properties of the current device, so they are cached per
// device, under a lock (calls may come from several host threads).
struct KernelSetup {
    const void *kernel;
    int dev;
    size_t smem;
    cudaError_t err;
    int occ;
};

static KernelSetup kernel_setup(const void *kernel, int threads, size_t smem) {
    static std::mutex mu;
    static KernelSetup done[256];
    static int n_done = 0;
    // per (kernel, device): the largest dynamic shared memory opted in so far; the
    // opt-in only ever grows, so a launch sized earlier keeps fitting
    static struct { const void *kernel; int dev; size_t smem; } optin[128];
    static int n_optin = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; i++)
        if (done[i].kernel == kernel && done[i].dev == dev && done[i].smem == smem) return done[i];
    KernelSetup k = {kernel, dev, smem, cudaSuccess, 1};
    if (smem > 48 * 1024) {
        int o = 0;
        while (o < n_optin && !(optin[o].kernel == kernel && optin[o].dev == dev)) o++;
        if (o == n_optin || optin[o].smem < smem) {
            k.err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (k.err == cudaSuccess) {
                if (o == n_optin && n_optin < 128) n_optin++;
                if (o < 128) optin[o] = {kernel, dev, smem};
            }
        }
    }
    if (k.err == cudaSuccess && threads > 0) {
        k.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.occ, kernel, threads, smem);
        if (k.occ < 1) k.occ = 1;
    }
    if (n_done < 256) done[n_done++] = k;
    return k;
}

cudaError_t kernel_smem_optin(const void *kernel, size_t smem) { return kernel_setup(kernel, 0, smem).err; }

cudaError_t kernel_occupancy(const void *kernel, int threads, size_t smem, int *occ) {
    const KernelSetup k = kernel_setup(kernel, threads, smem);
    *occ = k.occ;
    return k.err;
}

static inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
size_t linear_workspace_layout_n(int64_t max_M, int32_t IC, int n_shards, int total_groups, int32_t max_OC,
                                 LinearWorkspace *ws, void *base);

// Fixed part of every workspace: error word, then the arrival counters.
constexpr size_t kHeaderBytes = 256;
constexpr size_t kCounterCount = kWorkspaceCounters;
constexpr size_t kFixedBytes = kHeaderBytes + kCounterCount * sizeof(int32_t);

size_t fixed_workspace_bytes() { return kFixedBytes; }
int32_t *workspace_err(void *base) { return reinterpret_cast<int32_t *>(base); }
int32_t *workspace_counters(void *base) {
    return reinterpret_cast<int32_t *>(static_cast<char *>(base) + kHeaderBytes);
}

// Which GEMM path serves M rows:
//   decode   M <= kDecodeModeMaxRows: register-resident decode + mma.sync, rows on the MMA's N
//   fused    M <= kFusedMaxRows: decode into shared memory + tcgen05 MMAs
//   prefill  larger M: reconstruct W^T once, then the persistent tcgen05 GEMM
// The boundaries are where the measured times of neighbouring paths cross on
// the 5120 -> 2 x 17408 projection.  exl3_set_gemm_path() pins one path for
// tests and A/B measurements; workspace queries made while it is pinned size
// for that path too.
constexpr int64_t kDecodeModeMaxRows = 16;
enum class GemmMode { kDecode, kFused, kPrefill };

static std::atomic<int> g_gemm_path{0};

int forced_mode() { return g_gemm_path.load(std::memory_order_relaxed); }

GemmMode gemm_mode(int64_t M) {
    const int force = forced_mode();
    if (force == 1) return GemmMode::kDecode;
    if (force == 2 && M <= kFusedMaxRows && fused_supported()) return GemmMode::kFused;
    if (force == 3 && prefill_supported()) return GemmMode::kPrefill;
    if (M <= kDecodeModeMaxRows) return GemmMode::kDecode;
    if (M <= kFusedMaxRows && fused_supported()) return GemmMode::kFused;
    if (prefill_supported()) return GemmMode::kPrefill;
    return GemmMode::kDecode;
}

size_t linear_workspace_layout(int64_t max_M, int32_t max_IC, int32_t max_OC, LinearWorkspace *ws,
                               void *base) {
    return linear_workspace_layout_n(max_M, max_IC, 1, max_OC / 128, max_OC, ws, base);
}

// Sized for every path that some M <= max_M can take, so the byte count never
// decreases as max_M grows.
size_t linear_workspace_layout_n(int64_t max_M, int32_t IC, int n_shards, int total_groups, int32_t max_OC,
                                 LinearWorkspace *ws, void *base) {
    if (max_M < 0 || IC <= 0 || max_OC <= 0 || n_shards <= 0) return 0;
    const int64_t dec_rows = max_M < kDecodeMaxRows ? max_M : kDecodeMaxRows;
    const int nb = (int)((dec_rows + 7) / 8 > 0 ? (dec_rows + 7) / 8 : 1);
    size_t off = kFixedBytes;
    const size_t u_elems = (size_t)n_shards * max_M * IC;
    const size_t u_off = off;
    off = align256(off + u_elems * sizeof(uint16_t));
    size_t part_elems = group_slab_floats(total_groups, nb);
    if (fused_supported() && max_M > 0) {
        const size_t f = fused_slab_floats(total_groups, max_M);
        if (f > part_elems) part_elems = f;
    }
    const size_t part_off = off;
    off = align256(off + part_elems * sizeof(float));
    size_t wt_elems = 0, wt_off = off;
    if ((max_M > kFusedMaxRows || (max_M > 0 && forced_mode() == 3)) && prefill_supported()) {
        wt_elems = (size_t)max_OC * IC;
        off = align256(off + wt_elems * sizeof(uint16_t));
    }
    if (ws) {
        char *b = static_cast<char *>(base);
        ws->err = workspace_err(base);
        ws->counters = workspace_counters(base);
        ws->counters_n = kCounterCount;
        ws->u = reinterpret_cast<uint16_t *>(b + u_off);
        ws->u_elems = u_elems;
        ws->partials = reinterpret_cast<float *>(b + part_off);
        ws->partial_elems = part_elems;
        ws->wt = wt_elems ? reinterpret_cast<uint16_t *>(b + wt_off) : nullptr;
        ws->wt_elems = wt_elems;
    }
    return off;
}

}  // namespace exl3

using namespace exl3;

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" {

const char *exl3_last_error(void) { return g_err; }

const char *exl3_version(void) { return "exl3-gb300 0.2.0 (sm_103a)"; }

exl3_status exl3_set_gemm_path(int32_t path) {
    if (path < EXL3_PATH_BY_ROWS || path > EXL3_PATH_PREFILL)
        return fail(EXL3_EINVAL, "set_gemm_path: path = %d (0 by rows, 1 decode, 2 fused, 3 prefill)", path);
    g_gemm_path.store(path, std::memory_order_relaxed);
    return EXL3_OK;
}

size_t exl3_linear_workspace_bytes(int64_t max_M, int32_t max_IC, int32_t max_OC) {
    if (max_M < 0 || max_IC <= 0 || max_OC <= 0 || max_IC % 128 || max_OC % 128 ||
        (int64_t)max_OC / 128 > (int64_t)kCounterCount)
        return 0;
    return linear_workspace_layout(max_M, max_IC, max_OC, nullptr, nullptr);
}

exl3_status exl3_workspace_init(void *ws, size_t ws_bytes, exl3_stream stream) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return fail(EXL3_EINVAL, "workspace_init: workspace pointer %p is null or not 256-byte aligned", ws);
    if (ws_bytes < kFixedBytes)
        return fail(EXL3_EWORKSPACE, "workspace_init: %zu bytes < the %zu-byte minimum", ws_bytes, kFixedBytes);
    cudaError_t e = cudaMemsetAsync(ws, 0, kFixedBytes, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "workspace_init");
    return EXL3_OK;
}

exl3_status exl3_workspace_error(const void *ws, size_t ws_bytes, int32_t *flag_host, exl3_stream stream) {
    if (!ws || !flag_host || ws_bytes < kFixedBytes)
        return fail(EXL3_EINVAL, "workspace_error: null pointer or workspace of %zu bytes", ws_bytes);
    cudaError_t e = cudaMemcpyAsync(flag_host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "workspace_error");
    return EXL3_OK;
}

static exl3_status check_linear_args(const char *fn, const uint16_t *x, int64_t M, int32_t IC,
                                     const int16_t *code, int32_t OC, int32_t K,
                                     const uint16_t *s_in, const uint16_t *rin,
                                     const uint16_t *rout, const uint16_t *s_out) {
    if (M < 0) return fail(EXL3_EINVAL, "%s: M = %lld is negative", fn, (long long)M);
    if (K < 2 || K > 4)
        return fail(EXL3_EUNSUPPORTED, "%s: K = %d bits per weight; this build decodes K in {2, 3, 4}", fn, K);
    if (IC <= 0 || OC <= 0 || IC % 128 || OC % 128)
        return fail(EXL3_EINVAL, "%s: IC = %d and OC = %d must be positive multiples of 128 "
                    "(the Hadamard transform is blocked at 128)", fn, IC, OC);
    if ((int64_t)OC / 128 > (int64_t)kCounterCount)
        return fail(EXL3_EINVAL, "%s: OC = %d exceeds %lld column groups", fn, OC, (long long)kCounterCount);
    if (!code || !s_in || !rin || !rout || !s_out || (M > 0 && !x))
        return fail(EXL3_EINVAL, "%s: null input pointer", fn);
    if (!aligned16(code) || (M > 0 && !aligned16(x)))
        return fail(EXL3_EINVAL, "%s: x (%p) and code (%p) must be 16-byte aligned", fn, x, code);
    if (((uintptr_t)s_in | (uintptr_t)rin | (uintptr_t)rout | (uintptr_t)s_out) & 7u)
        return fail(EXL3_EINVAL, "%s: scale vectors must be 8-byte aligned", fn);
    return EXL3_OK;
}

exl3_status exl3_pretransform(const uint16_t *x, int64_t M, int32_t IC, const uint16_t *s_in,
                              const uint16_t *rin, uint16_t *u, exl3_stream stream) {
    if (M < 0 || IC <= 0 || IC % 128)
        return fail(EXL3_EINVAL, "pretransform: M = %lld, IC = %d (IC must be a positive multiple of 128)",
                    (long long)M, IC);
    if (M == 0) return EXL3_OK;
    if (!x || !s_in || !rin || !u) return fail(EXL3_EINVAL, "pretransform: null pointer");
    if (((uintptr_t)x | (uintptr_t)u | (uintptr_t)s_in | (uintptr_t)rin) & 7u)
        return fail(EXL3_EINVAL, "pretransform: pointers must be 8-byte aligned");
    cudaError_t e = launch_pretransform(x, M, IC, s_in, rin, u, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "pretransform");
    return EXL3_OK;
}

struct ShardDesc {
    const int16_t *code;
    const uint16_t *s_in, *rin, *rout, *s_out;
    int32_t OC, K;
    int64_t col0;
};

// Trellis GEMM + epilogue for n shards whose pre-transformed activations sit
// in u as [slot][M][IC] (fp16); shard i uses slot slots[i] (i if slots is null).
// 8-bit activations: row_scale [slots][M] multiplies each output row; with
// codes, u holds uint8 codes (q + 128, M <= 8 rows per decode pass) instead of
// fp16 values.
static exl3_status run_gemm(const char *fn, const uint16_t *u, int64_t M, int32_t IC, const ShardDesc *sh, int n,
                            uint16_t *out, int64_t ldo, const LinearWorkspace &ws, bool pdl, cudaStream_t s,
                            const int *slots = nullptr, const float *row_scale = nullptr, bool codes = false) {
    cudaError_t e;
    auto slot = [&](int i) { return slots ? slots[i] : i; };
    const GemmMode mode = gemm_mode(M);
    if (codes && mode != GemmMode::kDecode) return fail(EXL3_EINVAL, "%s: 8-bit codes need the decode path", fn);
    if (mode == GemmMode::kFused) {
        FusedArgs a = {};
        a.row_scale = row_scale;
        a.n_shards = n;
        a.M = (int32_t)M;
        a.IC = IC;
        int g0 = 0;
        for (int i = 0; i < n; i++) {
            FusedShard &f = a.sh[i];
            f.code = sh[i].code;
            f.rout = sh[i].rout;
            f.s_out = sh[i].s_out;
            f.col0 = sh[i].col0;
            f.K = sh[i].K;
            f.OC = sh[i].OC;
            f.g0 = g0;
            f.u_slot = slot(i);
            g0 += sh[i].OC / 128;
        }
        a.out = out;
        a.ldo = ldo;
        a.partials = ws.partials;
        a.counters = ws.counters;
        a.err = ws.err;
        e = launch_fused(a, u, s);
        if (e != cudaSuccess) return cuda_fail(e, fn);
        trace("%s M=%lld IC=%d shards=%d mode=fused", fn, (long long)M, IC, n);
        return EXL3_OK;
    }
    if (mode == GemmMode::kPrefill) {
        for (int i = 0; i < n; i++) {
            bool launched = false;
            // a programmatic dependent of the kernel before it only when that kernel is
            // this call's pre-transform (pdl) or the previous shard's GEMM (which triggers
            // only by completing): both have waited for all earlier work, so the staging
            // buffer is free and the reconstruct may overlap the pre-transform
            e = launch_reconstruct(sh[i].code, IC, sh[i].OC, sh[i].K, ws.wt, /*transposed=*/true, s, pdl || i > 0);
            if (e != cudaSuccess) return cuda_fail(e, fn);
            e = launch_prefill(u + (int64_t)slot(i) * M * IC, ws.wt, M, IC, sh[i].OC, sh[i].rout, sh[i].s_out,
                               out + sh[i].col0, ldo, ws.err, s, &launched, 0,
                               row_scale ? row_scale + (int64_t)slot(i) * M : nullptr);
            if (e != cudaSuccess) return cuda_fail(e, fn);
            if (!launched) return fail(EXL3_EUNSUPPORTED, "%s: prefill path unavailable", fn);
        }
        trace("%s M=%lld IC=%d shards=%d mode=prefill", fn, (long long)M, IC, n);
        return EXL3_OK;
    }
    // decode mode: passes of up to kDecodeMaxRows rows (8 with codes), all shards in
    // one launch per pass
    const int64_t pass_rows = codes ? 8 : kDecodeMaxRows;
    for (int64_t r0 = 0; r0 < M; r0 += pass_rows) {
        const int rows = (int)((M - r0) < pass_rows ? (M - r0) : pass_rows);
        GroupGemmArgs a = {};
        a.u = u;
        a.IC = IC;
        a.mode = kModeDense;
        a.codes = codes ? 1 : 0;
        a.row_scale = row_scale;
        a.n_inline = n;
        int g0 = 0;
        for (int i = 0; i < n; i++) {
            GroupEntry &ge = a.inline_e[i];
            ge.code = sh[i].code;
            ge.post = sh[i].rout;
            ge.post2 = sh[i].s_out;
            ge.out_off = sh[i].col0;
            ge.K = sh[i].K;
            ge.OC = sh[i].OC;
            ge.u_row0 = (int32_t)((int64_t)slot(i) * M + r0);
            ge.nrows = rows;
            ge.g0 = g0;
            g0 += sh[i].OC / 128;
        }
        a.out = out + r0 * ldo;
        a.ldo = ldo;
        a.partials = ws.partials;
        a.counters = ws.counters;
        e = launch_group_gemm(a, (rows + 7) / 8, pdl, s);
        if (e != cudaSuccess) return cuda_fail(e, fn);
    }
    trace("%s M=%lld IC=%d shards=%d mode=decode", fn, (long long)M, IC, n);
    return EXL3_OK;
}

static exl3_status check_out_ws(const char *fn, int64_t M, int32_t OC, const uint16_t *out, int64_t ldo,
                                int64_t col0, void *wsp, size_t ws_bytes, size_t need) {
    if (ldo < OC || col0 < 0 || col0 + OC > ldo)
        return fail(EXL3_EINVAL, "%s: column slice [%lld, %lld) does not fit ldo = %lld", fn,
                    (long long)col0, (long long)col0 + OC, (long long)ldo);
    if (M == 0) return EXL3_OK;
    if (!out) return fail(EXL3_EINVAL, "%s: null output", fn);
    if ((ldo % 8) || (col0 % 8) || !aligned16(out))
        return fail(EXL3_EINVAL, "%s: out (%p), ldo = %lld and col0 = %lld must give 16-byte "
                    "aligned rows (ldo, col0 multiples of 8)", fn, out, (long long)ldo, (long long)col0);
    if (!wsp || (reinterpret_cast<uintptr_t>(wsp) & 255u) || ws_bytes < need)
        return fail(EXL3_EWORKSPACE, "%s: workspace %p of %zu bytes; this call needs %zu bytes, "
                    "256-byte aligned", fn, wsp, ws_bytes, need);
    return EXL3_OK;
}

exl3_status exl3_linear_into(const uint16_t *x, int64_t M, int32_t IC, const int16_t *code, int32_t OC,
                             int32_t K, const uint16_t *s_in, const uint16_t *rin, const uint16_t *rout,
                             const uint16_t *s_out, uint16_t *out, int64_t ldo, int64_t col0, void *wsp,
                             size_t ws_bytes, exl3_stream stream) {
    exl3_status st = check_linear_args("linear_into", x, M, IC, code, OC, K, s_in, rin, rout, s_out);
    if (st == EXL3_OK)
        st = check_out_ws("linear_into", M, OC, out, ldo, col0, wsp, ws_bytes, exl3_linear_workspace_bytes(M, IC, OC));
    if (st != EXL3_OK || M == 0) return st;
    LinearWorkspace ws;
    linear_workspace_layout(M, IC, OC, &ws, wsp);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_pretransform(x, M, IC, s_in, rin, ws.u, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into: pretransform");
    ShardDesc d = {code, s_in, rin, rout, s_out, OC, K, col0};
    return run_gemm("linear_into", ws.u, M, IC, &d, 1, out, ldo, ws, true, s);
}

exl3_status exl3_gemm_into(const uint16_t *u, int64_t M, int32_t IC, const int16_t *code, int32_t OC, int32_t K,
                           const uint16_t *rout, const uint16_t *s_out, uint16_t *out, int64_t ldo, int64_t col0,
                           void *wsp, size_t ws_bytes, exl3_stream stream) {
    exl3_status st = check_linear_args("gemm_into", u, M, IC, code, OC, K, rout, rout, rout, s_out);
    if (st == EXL3_OK)
        st = check_out_ws("gemm_into", M, OC, out, ldo, col0, wsp, ws_bytes, exl3_linear_workspace_bytes(M, IC, OC));
    if (st != EXL3_OK || M == 0) return st;
    LinearWorkspace ws;
    linear_workspace_layout(M, IC, OC, &ws, wsp);
    ShardDesc d = {code, nullptr, nullptr, rout, s_out, OC, K, col0};
    return run_gemm("gemm_into", u, M, IC, &d, 1, out, ldo, ws, false, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- 8-bit activations
// Workspace: the linear layout, then As [max_M] (fp32).  M <= 8 rows on the
// decode path keep the uint8 codes in the activation region; other paths keep
// the codes' exact fp16 values there.
static size_t a8_layout(int64_t max_M, int32_t IC, int32_t OC, LinearWorkspace *ws, void *base, float **As) {
    const size_t off = linear_workspace_layout(max_M, IC, OC, ws, base);
    if (!off) return 0;
    if (As) *As = reinterpret_cast<float *>(static_cast<char *>(base) + off);
    return off + align256((size_t)max_M * sizeof(float));
}

size_t exl3_linear_a8_workspace_bytes(int64_t max_M, int32_t max_IC, int32_t max_OC) {
    if (!exl3_linear_workspace_bytes(max_M, max_IC, max_OC)) return 0;
    return a8_layout(max_M, max_IC, max_OC, nullptr, nullptr, nullptr);
}

static exl3_status check_a8_ic(const char *fn, int32_t IC) {
    const size_t smem = quantize_a8_smem_bytes(IC);
    if (smem + 1024 > (size_t)device_info().max_smem_optin)
        return fail(EXL3_EUNSUPPORTED, "%s: IC = %d needs %zu bytes of shared memory per row (%d available)", fn, IC,
                    smem, device_info().max_smem_optin);
    return EXL3_OK;
}

exl3_status exl3_quantize_a8(const uint16_t *x, int64_t M, int32_t IC, const uint16_t *s_in, const uint16_t *rin,
                             uint8_t *A, float *As, exl3_stream stream) {
    if (M < 0 || IC <= 0 || IC % 128)
        return fail(EXL3_EINVAL, "quantize_a8: M = %lld, IC = %d (IC must be a positive multiple of 128)",
                    (long long)M, IC);
    if (M == 0) return EXL3_OK;
    if (!x || !s_in || !rin || !A || !As) return fail(EXL3_EINVAL, "quantize_a8: null pointer");
    if (((uintptr_t)x | (uintptr_t)s_in | (uintptr_t)rin) & 7u || ((uintptr_t)A | (uintptr_t)As) & 3u)
        return fail(EXL3_EINVAL, "quantize_a8: x, s_in, rin must be 8-byte aligned and A, As 4-byte aligned");
    exl3_status st = check_a8_ic("quantize_a8", IC);
    if (st != EXL3_OK) return st;
    PretransformShards p = {};
    p.s_in[0] = s_in;
    p.rin[0] = rin;
    p.n = 1;
    cudaError_t e = launch_quantize_a8(x, M, IC, p, A, false, As, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "quantize_a8");
    return EXL3_OK;
}

exl3_status exl3_linear_into_a8(const uint16_t *x, int64_t M, int32_t IC, const int16_t *code, int32_t OC,
                                int32_t K, const uint16_t *s_in, const uint16_t *rin, const uint16_t *rout,
                                const uint16_t *s_out, uint16_t *out, int64_t ldo, int64_t col0, void *wsp,
                                size_t ws_bytes, exl3_stream stream) {
    exl3_status st = check_linear_args("linear_into_a8", x, M, IC, code, OC, K, s_in, rin, rout, s_out);
    if (st == EXL3_OK)
        st = check_out_ws("linear_into_a8", M, OC, out, ldo, col0, wsp, ws_bytes,
                          exl3_linear_a8_workspace_bytes(M, IC, OC));
    if (st == EXL3_OK && M > 0) st = check_a8_ic("linear_into_a8", IC);
    if (st != EXL3_OK || M == 0) return st;
    LinearWorkspace ws;
    float *As = nullptr;
    a8_layout(M, IC, OC, &ws, wsp, &As);
    cudaStream_t s = (cudaStream_t)stream;
    const bool codes = gemm_mode(M) == GemmMode::kDecode && M <= 8;
    PretransformShards p = {};
    p.s_in[0] = s_in;
    p.rin[0] = rin;
    p.n = 1;
    cudaError_t e = launch_quantize_a8(x, M, IC, p, ws.u, !codes, As, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_a8: quantize");
    ShardDesc d = {code, s_in, rin, rout, s_out, OC, K, col0};
    return run_gemm("linear_into_a8", ws.u, M, IC, &d, 1, out, ldo, ws, true, s, nullptr, As, codes);
}

exl3_status exl3_gemm_a8_into(const uint8_t *A, const float *As, int64_t M, int32_t IC, const int16_t *code,
                              int32_t OC, int32_t K, const uint16_t *rout, const uint16_t *s_out, uint16_t *out,
                              int64_t ldo, int64_t col0, void *wsp, size_t ws_bytes, exl3_stream stream) {
    exl3_status st = check_linear_args("gemm_a8_into", reinterpret_cast<const uint16_t *>(A), M, IC, code, OC, K,
                                       rout, rout, rout, s_out);
    if (st == EXL3_OK && M > 0 && (!As || ((uintptr_t)As & 3u)))
        return fail(EXL3_EINVAL, "gemm_a8_into: As (%p) must be a non-null 4-byte aligned pointer", (const void *)As);
    if (st == EXL3_OK)
        st = check_out_ws("gemm_a8_into", M, OC, out, ldo, col0, wsp, ws_bytes,
                          exl3_linear_a8_workspace_bytes(M, IC, OC));
    if (st != EXL3_OK || M == 0) return st;
    LinearWorkspace ws;
    a8_layout(M, IC, OC, &ws, wsp, nullptr);
    cudaStream_t s = (cudaStream_t)stream;
    ShardDesc d = {code, nullptr, nullptr, rout, s_out, OC, K, col0};
    if (gemm_mode(M) == GemmMode::kDecode && M <= 8)
        return run_gemm("gemm_a8_into", reinterpret_cast<const uint16_t *>(A), M, IC, &d, 1, out, ldo, ws, false, s,
                        nullptr, As, true);
    cudaError_t e = launch_codes_to_f16(A, M * IC, ws.u, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_a8_into: codes");
    return run_gemm("gemm_a8_into", ws.u, M, IC, &d, 1, out, ldo, ws, true, s, nullptr, As, false);
}

// A shard's codebook marker: only the default codebook is decoded (its constants
// are the only ones the method's description fixes).
static exl3_status check_codebook(const char *fn, const exl3_shard &h, int i) {
    if (h.codebook == EXL3_CODEBOOK_3INST) return EXL3_OK;
    if (h.codebook == EXL3_CODEBOOK_MCG || h.codebook == EXL3_CODEBOOK_MUL1)
        return fail(EXL3_EUNSUPPORTED, "%s: shard %d is marked with the %s codebook; this build decodes the default "
                    "(3INST) codebook only", fn, i, h.codebook == EXL3_CODEBOOK_MCG ? "MCG" : "MUL1");
    return fail(EXL3_EINVAL, "%s: shard %d: codebook = %d (0 default, 1 MCG, 2 MUL1)", fn, i, h.codebook);
}

static bool shards_shape(const exl3_shard *shards, int32_t n, int *groups, int32_t *max_oc) {
    if (!shards || n < 1 || n > kMaxInlineEntries) return false;
    *groups = 0;
    *max_oc = 0;
    for (int i = 0; i < n; i++) {
        if (shards[i].OC <= 0 || shards[i].OC % 128) return false;
        *groups += shards[i].OC / 128;
        if (shards[i].OC > *max_oc) *max_oc = shards[i].OC;
    }
    return *groups <= (int)kCounterCount;
}

size_t exl3_linear_shards_workspace_bytes(int64_t max_M, int32_t IC, const exl3_shard *shards, int32_t n) {
    int groups;
    int32_t max_oc;
    if (max_M < 0 || IC <= 0 || IC % 128 || !shards_shape(shards, n, &groups, &max_oc)) return 0;
    return linear_workspace_layout_n(max_M, IC, n, groups, max_oc, nullptr, nullptr);
}

static exl3_status shards_prepare(const char *fn, const uint16_t *x, int64_t M, int32_t IC, const exl3_shard *shards,
                                  int32_t n, uint16_t *out, int64_t ldo, void *wsp, size_t ws_bytes, bool need_in,
                                  ShardDesc *d, LinearWorkspace *ws) {
    int groups;
    int32_t max_oc;
    if (!shards_shape(shards, n, &groups, &max_oc))
        return fail(EXL3_EINVAL, "%s: need 1..%d shard descriptors with OC a positive multiple of 128", fn,
                    kMaxInlineEntries);
    for (int i = 0; i < n; i++) {
        const exl3_shard &h = shards[i];
        const uint16_t *si = need_in ? h.s_in : h.rout, *ri = need_in ? h.rin : h.rout;
        exl3_status st = check_codebook(fn, h, i);
        if (st != EXL3_OK) return st;
        st = check_linear_args(fn, x, M, IC, h.code, h.OC, h.K, si, ri, h.rout, h.s_out);
        if (st == EXL3_OK)
            st = check_out_ws(fn, M, h.OC, out, ldo, h.col0, wsp, ws_bytes,
                              exl3_linear_shards_workspace_bytes(M, IC, shards, n));
        if (st != EXL3_OK) return st;
        d[i] = {h.code, h.s_in, h.rin, h.rout, h.s_out, h.OC, h.K, h.col0};
    }
    if (M > 0) linear_workspace_layout_n(M, IC, n, groups, max_oc, ws, wsp);
    return EXL3_OK;
}

exl3_status exl3_linear_into_shards(const uint16_t *x, int64_t M, int32_t IC, const exl3_shard *shards,
                                    int32_t n, uint16_t *out, int64_t ldo, void *wsp, size_t ws_bytes,
                                    exl3_stream stream) {
    ShardDesc d[kMaxInlineEntries];
    LinearWorkspace ws;
    exl3_status st = shards_prepare("linear_into_shards", x, M, IC, shards, n, out, ldo, wsp, ws_bytes, true, d, &ws);
    if (st != EXL3_OK || M == 0) return st;
    cudaStream_t s = (cudaStream_t)stream;
    PretransformShards p = {};
    p.n = n;
    for (int i = 0; i < n; i++) {
        p.s_in[i] = d[i].s_in;
        p.rin[i] = d[i].rin;
    }
    cudaError_t e = launch_pretransform_shards(x, M, IC, p, ws.u, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_shards: pretransform");
    return run_gemm("linear_into_shards", ws.u, M, IC, d, n, out, ldo, ws, true, s);
}

// The device address of mapped pinned host memory p; nullptr if p is anything
// else (pageable host memory, device memory, an unknown pointer).
static void *mapped_host(const void *p) {
    cudaPointerAttributes attr;
    if (!p || cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

exl3_status exl3_linear_into_shards_host(const uint16_t *x_host, int64_t M, int32_t IC, const exl3_shard *shards,
                                         int32_t n, uint16_t *out_host, int64_t ldo, void *wsp, size_t ws_bytes,
                                         exl3_stream stream) {
    const uint16_t *x = x_host;
    uint16_t *out = out_host;
    if (M > 0) {
        x = static_cast<const uint16_t *>(mapped_host(x_host));
        out = static_cast<uint16_t *>(mapped_host(out_host));
        if (!x) return fail(EXL3_EINVAL, "linear_into_shards_host: x_host (%p) is not mapped pinned host memory", x_host);
        if (!out)
            return fail(EXL3_EINVAL, "linear_into_shards_host: out_host (%p) is not mapped pinned host memory", out_host);
    }
    return exl3_linear_into_shards(x, M, IC, shards, n, out, ldo, wsp, ws_bytes, stream);
}

exl3_status exl3_gemm_into_shards(const uint16_t *u, int64_t M, int32_t IC, const exl3_shard *shards, int32_t n,
                                  uint16_t *out, int64_t ldo, void *wsp, size_t ws_bytes, exl3_stream stream) {
    ShardDesc d[kMaxInlineEntries];
    LinearWorkspace ws;
    exl3_status st = shards_prepare("gemm_into_shards", u, M, IC, shards, n, out, ldo, wsp, ws_bytes, false, d, &ws);
    if (st != EXL3_OK || M == 0) return st;
    return run_gemm("gemm_into_shards", u, M, IC, d, n, out, ldo, ws, false, (cudaStream_t)stream);
}

size_t exl3_linear_shards_a8_workspace_bytes(int64_t max_M, int32_t IC, const exl3_shard *shards, int32_t n) {
    const size_t b = exl3_linear_shards_workspace_bytes(max_M, IC, shards, n);
    return b ? b + align256((size_t)n * max_M * sizeof(float)) : 0;
}

exl3_status exl3_linear_into_shards_a8(const uint16_t *x, int64_t M, int32_t IC, const exl3_shard *shards,
                                       int32_t n, uint16_t *out, int64_t ldo, void *wsp, size_t ws_bytes,
                                       exl3_stream stream) {
    ShardDesc d[kMaxInlineEntries];
    LinearWorkspace ws;
    exl3_status st = shards_prepare("linear_into_shards_a8", x, M, IC, shards, n, out, ldo, wsp, ws_bytes, true, d,
                                    &ws);
    if (st == EXL3_OK && M > 0 && ws_bytes < exl3_linear_shards_a8_workspace_bytes(M, IC, shards, n))
        st = fail(EXL3_EWORKSPACE, "linear_into_shards_a8: workspace of %zu bytes; this call needs %zu bytes",
                  ws_bytes, exl3_linear_shards_a8_workspace_bytes(M, IC, shards, n));
    if (st == EXL3_OK && M > 0) st = check_a8_ic("linear_into_shards_a8", IC);
    if (st != EXL3_OK || M == 0) return st;
    float *As = reinterpret_cast<float *>(static_cast<char *>(wsp) + exl3_linear_shards_workspace_bytes(M, IC, shards, n));
    cudaStream_t s = (cudaStream_t)stream;
    const bool codes = gemm_mode(M) == GemmMode::kDecode && M <= 8;
    PretransformShards p = {};
    p.n = n;
    for (int i = 0; i < n; i++) {
        p.s_in[i] = d[i].s_in;
        p.rin[i] = d[i].rin;
    }
    cudaError_t e = launch_quantize_a8(x, M, IC, p, ws.u, !codes, As, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_shards_a8: quantize");
    return run_gemm("linear_into_shards_a8", ws.u, M, IC, d, n, out, ldo, ws, true, s, nullptr, As, codes);
}

exl3_status exl3_gemm_a8_into_shards(const uint8_t *A, const float *As, int64_t M, int32_t IC,
                                     const exl3_shard *shards, int32_t n, uint16_t *out, int64_t ldo, void *wsp,
                                     size_t ws_bytes, exl3_stream stream) {
    ShardDesc d[kMaxInlineEntries];
    LinearWorkspace ws;
    exl3_status st = shards_prepare("gemm_a8_into_shards", reinterpret_cast<const uint16_t *>(A), M, IC, shards, n,
                                    out, ldo, wsp, ws_bytes, false, d, &ws);
    if (st == EXL3_OK && M > 0 && (!As || ((uintptr_t)As & 3u)))
        st = fail(EXL3_EINVAL, "gemm_a8_into_shards: As (%p) must be a non-null 4-byte aligned pointer",
                  (const void *)As);
    if (st == EXL3_OK && M > 0 && ws_bytes < exl3_linear_shards_a8_workspace_bytes(M, IC, shards, n))
        st = fail(EXL3_EWORKSPACE, "gemm_a8_into_shards: workspace of %zu bytes; this call needs %zu bytes",
                  ws_bytes, exl3_linear_shards_a8_workspace_bytes(M, IC, shards, n));
    if (st != EXL3_OK || M == 0) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (gemm_mode(M) == GemmMode::kDecode && M <= 8)
        return run_gemm("gemm_a8_into_shards", reinterpret_cast<const uint16_t *>(A), M, IC, d, n, out, ldo, ws, false,
                        s, nullptr, As, true);
    cudaError_t e = launch_codes_to_f16(A, (int64_t)n * M * IC, ws.u, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_a8_into_shards: codes");
    return run_gemm("gemm_a8_into_shards", ws.u, M, IC, d, n, out, ldo, ws, true, s, nullptr, As, false);
}

exl3_status exl3_linear(const uint16_t *x, int64_t M, int32_t IC, const int16_t *code, int32_t OC, int32_t K,
                        const uint16_t *s_in, const uint16_t *rin, const uint16_t *rout, const uint16_t *s_out,
                        uint16_t *y, void *ws, size_t ws_bytes, exl3_stream stream) {
    return exl3_linear_into(x, M, IC, code, OC, K, s_in, rin, rout, s_out, y, OC, 0, ws, ws_bytes, stream);
}

exl3_status exl3_reconstruct(const int16_t *code, int32_t IC, int32_t OC, int32_t K, uint16_t *W,
                             exl3_stream stream) {
    if (K < 2 || K > 4) return fail(EXL3_EUNSUPPORTED, "reconstruct: K = %d; this build decodes K in {2, 3, 4}", K);
    if (IC <= 0 || OC <= 0 || IC % 16 || OC % 16)
        return fail(EXL3_EINVAL, "reconstruct: IC = %d, OC = %d must be positive multiples of 16", IC, OC);
    if (!code || !W || !aligned16(code) || !aligned16(W) || (OC % 128 && OC % 8))
        return fail(EXL3_EINVAL, "reconstruct: code and W must be non-null and 16-byte aligned");
    cudaError_t e = launch_reconstruct(code, IC, OC, K, W, false, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "reconstruct");
    return EXL3_OK;
}

exl3_status exl3_codebook_table(uint16_t *table, exl3_stream stream) {
    if (!table) return fail(EXL3_EINVAL, "codebook_table: null table");
    cudaError_t e = launch_codebook_table(table, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "codebook_table");
    return EXL3_OK;
}

exl3_status exl3_embed_int8_gather(const int8_t *q, const uint16_t *scale, int64_t V, int32_t H,
                                   const int32_t *ids, int64_t N, uint16_t *out, int32_t *n_bad,
                                   exl3_stream stream) {
    if (V <= 0 || H <= 0 || H % 16 || N < 0)
        return fail(EXL3_EINVAL, "embed_int8_gather: V = %lld, H = %d (multiple of 16), N = %lld",
                    (long long)V, H, (long long)N);
    if (N == 0) return EXL3_OK;
    if (!q || !scale || !ids || !out) return fail(EXL3_EINVAL, "embed_int8_gather: null pointer");
    if (N * (int64_t)(H / 16) >= 0x7FFFFF00LL)
        return fail(EXL3_EINVAL, "embed_int8_gather: N * H / 16 = %lld chunks; one call handles fewer than 2^31",
                    (long long)(N * (int64_t)(H / 16)));
    if (!aligned16(q) || !aligned16(out))
        return fail(EXL3_EINVAL, "embed_int8_gather: q (%p) and out (%p) must be 16-byte aligned", q, out);
    cudaError_t e = launch_gather(q, scale, V, H, ids, N, out, n_bad, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "embed_int8_gather");
    return EXL3_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ projections
namespace {

constexpr int kMaxProjections = 16;
constexpr int kMaxSlots = 16;   // distinct (s_in, rin) pre-transforms of one input

// A call's plan: projections that read the same x share one group of
// pre-transformed rows, one slot per distinct (s_in, rin) pair (pointer equality).
struct ProjPlan {
    struct Group {
        const uint16_t *x;
        int32_t IC;
        int nslots;
        const uint16_t *s_in[kMaxSlots], *rin[kMaxSlots];
        size_t off;          // byte offset of its rows [slot][M][IC] in the u region
        int first_proj;      // the projection that transforms it
    } g[kMaxProjections];
    int ng = 0;
    int group_of[kMaxProjections];
    int slot_of[kMaxProjections][kMaxInlineEntries];
    size_t u_bytes = 0, part_elems = 0, wt_elems = 0;
};

const char *plan_projections(const exl3_projection *p, int32_t n, int64_t M, ProjPlan *pl) {
    if (!p || n < 1 || n > kMaxProjections) return "need 1..16 projections";
    for (int i = 0; i < n; i++) {
        const exl3_projection &pr = p[i];
        int groups;
        int32_t max_oc;
        if (pr.IC <= 0 || pr.IC % 128 || !shards_shape(pr.shards, pr.n_shards, &groups, &max_oc))
            return "a projection needs IC a positive multiple of 128 and 1..4 shards of OC a multiple of 128";
        int gi = 0;
        while (gi < pl->ng && !(pl->g[gi].x == pr.x && pl->g[gi].IC == pr.IC)) gi++;
        if (gi == pl->ng) {
            ProjPlan::Group &g = pl->g[pl->ng++];
            g.x = pr.x;
            g.IC = pr.IC;
            g.nslots = 0;
            g.first_proj = i;
        }
        ProjPlan::Group &g = pl->g[gi];
        pl->group_of[i] = gi;
        for (int k = 0; k < pr.n_shards; k++) {
            int sl = 0;
            while (sl < g.nslots && !(g.s_in[sl] == pr.shards[k].s_in && g.rin[sl] == pr.shards[k].rin)) sl++;
            if (sl == g.nslots) {
                if (g.nslots == kMaxSlots) return "more than 16 distinct (s_in, rin) pairs on one input";
                g.s_in[sl] = pr.shards[k].s_in;
                g.rin[sl] = pr.shards[k].rin;
                g.nslots++;
            }
            pl->slot_of[i][k] = sl;
        }
        // split-K slab and prefill staging of this projection's GEMM (shared, used in turn)
        const int64_t dec_rows = M < kDecodeMaxRows ? M : kDecodeMaxRows;
        const int nb = (int)((dec_rows + 7) / 8 > 0 ? (dec_rows + 7) / 8 : 1);
        size_t part = group_slab_floats(groups, nb);
        if (fused_supported() && M > 0) {
            const size_t f = fused_slab_floats(groups, M);
            if (f > part) part = f;
        }
        if (part > pl->part_elems) pl->part_elems = part;
        if ((M > kFusedMaxRows || (M > 0 && forced_mode() == 3)) && prefill_supported()) {
            const size_t wt = (size_t)max_oc * pr.IC;
            if (wt > pl->wt_elems) pl->wt_elems = wt;
        }
    }
    size_t off = 0;
    for (int gi = 0; gi < pl->ng; gi++) {
        pl->g[gi].off = off;
        off = align256(off + sizeof(uint16_t) * (size_t)pl->g[gi].nslots * M * pl->g[gi].IC);
    }
    pl->u_bytes = off;
    return nullptr;
}

// Workspace: fixed header | u region | split-K slab | prefill staging.
size_t projections_layout(const ProjPlan &pl, size_t *u_off, size_t *part_off, size_t *wt_off) {
    size_t off = kFixedBytes;
    *u_off = off;
    off = align256(off + pl.u_bytes);
    *part_off = off;
    off = align256(off + sizeof(float) * pl.part_elems);
    *wt_off = off;
    off = align256(off + sizeof(uint16_t) * pl.wt_elems);
    return off;
}

}  // namespace

extern "C" {

size_t exl3_projections_workspace_bytes(int64_t max_M, const exl3_projection *p, int32_t n) {
    if (max_M < 0) return 0;
    ProjPlan pl;
    if (plan_projections(p, n, max_M, &pl)) return 0;
    size_t a, b, c;
    return projections_layout(pl, &a, &b, &c);
}

exl3_status exl3_linear_projections(const exl3_projection *p, int32_t n, int64_t M, void *wsp, size_t ws_bytes,
                                    exl3_stream stream) {
    const char *fn = "linear_projections";
    if (M < 0) return fail(EXL3_EINVAL, "%s: M = %lld is negative", fn, (long long)M);
    ProjPlan pl;
    if (const char *why = plan_projections(p, n, M, &pl)) return fail(EXL3_EINVAL, "%s: %s", fn, why);
    size_t u_off, part_off, wt_off;
    const size_t need = projections_layout(pl, &u_off, &part_off, &wt_off);
    for (int i = 0; i < n; i++) {
        const exl3_projection &pr = p[i];
        for (int k = 0; k < pr.n_shards; k++) {
            const exl3_shard &h = pr.shards[k];
            exl3_status st = check_codebook(fn, h, k);
            if (st == EXL3_OK)
                st = check_linear_args(fn, pr.x, M, pr.IC, h.code, h.OC, h.K, h.s_in, h.rin, h.rout, h.s_out);
            if (st == EXL3_OK) st = check_out_ws(fn, M, h.OC, pr.out, pr.ldo, h.col0, wsp, ws_bytes, need);
            if (st != EXL3_OK) return st;
        }
    }
    if (M == 0) return EXL3_OK;
    char *b = static_cast<char *>(wsp);
    LinearWorkspace ws;
    ws.err = workspace_err(wsp);
    ws.counters = workspace_counters(wsp);
    ws.counters_n = kCounterCount;
    ws.partials = reinterpret_cast<float *>(b + part_off);
    ws.partial_elems = pl.part_elems;
    ws.wt = pl.wt_elems ? reinterpret_cast<uint16_t *>(b + wt_off) : nullptr;
    ws.wt_elems = pl.wt_elems;
    cudaStream_t s = (cudaStream_t)stream;
    for (int i = 0; i < n; i++) {
        const exl3_projection &pr = p[i];
        const ProjPlan::Group &g = pl.g[pl.group_of[i]];
        uint16_t *u = reinterpret_cast<uint16_t *>(b + u_off + g.off);
        if (g.first_proj == i) {
            // every pre-transform of this input, once (up to four per launch)
            for (int s0 = 0; s0 < g.nslots; s0 += 4) {
                PretransformShards pt = {};
                pt.n = g.nslots - s0 < 4 ? g.nslots - s0 : 4;
                for (int k = 0; k < pt.n; k++) {
                    pt.s_in[k] = g.s_in[s0 + k];
                    pt.rin[k] = g.rin[s0 + k];
                }
                cudaError_t e = launch_pretransform_shards(pr.x, M, pr.IC, pt, u + (int64_t)s0 * M * pr.IC, s);
                if (e != cudaSuccess) return cuda_fail(e, "linear_projections: pretransform");
            }
        }
        ShardDesc d[kMaxInlineEntries];
        for (int k = 0; k < pr.n_shards; k++) {
            const exl3_shard &h = pr.shards[k];
            d[k] = {h.code, h.s_in, h.rin, h.rout, h.s_out, h.OC, h.K, h.col0};
        }
        exl3_status st = run_gemm(fn, u, M, pr.IC, d, pr.n_shards, pr.out, pr.ldo, ws, true, s, pl.slot_of[i]);
        if (st != EXL3_OK) return st;
    }
    return EXL3_OK;
}

}  // extern "C"
