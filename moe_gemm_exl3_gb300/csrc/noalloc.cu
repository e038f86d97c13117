// noalloc.cu -- exl3_linear_into_noalloc: the small-M EXL3 projection with
// its scratch in a fixed, library-owned device array, for callers that cannot
// allocate device memory or hand the library a workspace.
//
// The scratch array is a file-scope __device__ variable: it exists on every
// GPU that loads this library, from module load until process exit, and every
// call on that GPU shares it.  Host code cannot use the array's name as a
// device address (on the host it names a host-side shadow), so every call
// looks the real address up with cudaGetSymbolAddress while the caller's
// device is current, and every launch is given that address.  The look-up is
// not cached: after a device reset the module is loaded again at a new address.
#include <cuda_runtime.h>

#include "../../include/exl3.h"
#include "internal.h"

namespace exl3 {
exl3_status fail(exl3_status st, const char *fmt, ...);
exl3_status cuda_fail(cudaError_t e, const char *where);
}  // namespace exl3

using namespace exl3;

namespace {

// Limits of the allocation-free variant (also stated in include/exl3.h).
constexpr int64_t kNaMaxM = 8;          // one decode pass of one 8-row block
constexpr int32_t kNaMaxIC = 32768;
constexpr int32_t kNaMaxOC = 65536;
constexpr int32_t kNaMaxGroups = kNaMaxOC / 128;

// Scratch layout: [error word + pad | counters | activations | split-K slab].
constexpr size_t kNaHeader = 256;
constexpr size_t kNaCounters = (size_t)kNaMaxGroups * sizeof(int32_t);
constexpr size_t kNaU = (size_t)kNaMaxM * kNaMaxIC * sizeof(uint16_t);
constexpr size_t kNaSlab = (size_t)(kDecodeMaxCtas + kNaMaxGroups) * (8 * 1 * 4 * 32) * sizeof(float);  // NB = 1
constexpr size_t kNaBytes = kNaHeader + kNaCounters + kNaU + kNaSlab;   // 6.8 MB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

// The scratch array's device address on the current device.
exl3_status scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_noalloc: cudaGetSymbolAddress");
    *out = p;
    return EXL3_OK;
}

}  // namespace

extern "C" exl3_status exl3_linear_into_noalloc(const uint16_t *x, int64_t M, int32_t IC, const int16_t *code,
                                                int32_t OC, int32_t K, const uint16_t *s_in, const uint16_t *rin,
                                                const uint16_t *rout, const uint16_t *s_out, uint16_t *out,
                                                int64_t ldo, int64_t col0, exl3_stream stream) {
    const char *fn = "linear_into_noalloc";
    if (M < 0 || M > kNaMaxM || IC <= 0 || IC > kNaMaxIC || OC <= 0 || OC > kNaMaxOC)
        return fail(EXL3_EINVAL, "%s: M = %lld, IC = %d, OC = %d exceed this entry point's fixed scratch "
                    "(M <= %lld, IC <= %d, OC <= %d); use exl3_linear_into with a workspace",
                    fn, (long long)M, IC, OC, (long long)kNaMaxM, kNaMaxIC, kNaMaxOC);
    if (K < 2 || K > 4) return fail(EXL3_EUNSUPPORTED, "%s: K = %d; this build decodes K in {2, 3, 4}", fn, K);
    if (IC % 128 || OC % 128)
        return fail(EXL3_EINVAL, "%s: IC = %d and OC = %d must be multiples of 128", fn, IC, OC);
    if (ldo < OC || col0 < 0 || col0 + OC > ldo)
        return fail(EXL3_EINVAL, "%s: column slice [%lld, %lld) does not fit ldo = %lld", fn, (long long)col0,
                    (long long)col0 + OC, (long long)ldo);
    if (M == 0) return EXL3_OK;
    if (!x || !code || !s_in || !rin || !rout || !s_out || !out)
        return fail(EXL3_EINVAL, "%s: null pointer", fn);
    if (((uintptr_t)x | (uintptr_t)code | (uintptr_t)out) & 15u || (ldo % 8) || (col0 % 8) ||
        (((uintptr_t)s_in | (uintptr_t)rin | (uintptr_t)rout | (uintptr_t)s_out) & 7u))
        return fail(EXL3_EINVAL, "%s: x, code and out rows must be 16-byte aligned (ldo, col0 multiples of 8), "
                    "scale vectors 8-byte aligned", fn);

    void *base = nullptr;
    exl3_status st = scratch_address(&base);
    if (st != EXL3_OK) return st;
    char *b = static_cast<char *>(base);
    int32_t *counters = reinterpret_cast<int32_t *>(b + kNaHeader);
    uint16_t *u = reinterpret_cast<uint16_t *>(b + kNaHeader + kNaCounters);
    float *slab = reinterpret_cast<float *>(b + kNaHeader + kNaCounters + kNaU);
    cudaStream_t s = (cudaStream_t)stream;

    // The array keeps whatever the previous call left; the arrival counters
    // (and the error word) must start at zero.
    cudaError_t e = cudaMemsetAsync(b, 0, kNaHeader + kNaCounters, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_noalloc: clear counters");
    e = launch_pretransform(x, M, IC, s_in, rin, u, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_noalloc: pretransform");
    GroupGemmArgs a = {};
    a.u = u;
    a.IC = IC;
    a.mode = kModeDense;
    a.n_inline = 1;
    GroupEntry &ge = a.inline_e[0];
    ge.code = code;
    ge.post = rout;
    ge.post2 = s_out;
    ge.out_off = col0;
    ge.K = K;
    ge.OC = OC;
    ge.u_row0 = 0;
    ge.nrows = (int32_t)M;
    ge.g0 = 0;
    a.out = out;
    a.ldo = ldo;
    a.partials = slab;
    a.counters = counters;
    e = launch_group_gemm(a, 1, false, s);
    if (e != cudaSuccess) return cuda_fail(e, "linear_into_noalloc: decode gemm");
    return EXL3_OK;
}
