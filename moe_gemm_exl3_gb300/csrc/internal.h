// internal.h -- host-side launch interfaces between the C ABI layer and the kernels.
#pragma once

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

struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
};
const DeviceInfo &device_info();

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
cudaError_t launch_reconstruct(const int16_t *code, int IC, int OC, int K, uint16_t *W,
                               bool transposed, cudaStream_t s);
cudaError_t launch_codebook_table(uint16_t *table, cudaStream_t s);

struct DecodeGemmArgs {
    const uint16_t *u;        // fp16 [M][IC]
    const int16_t *code;
    int IC, OC, K;
    int M;                    // rows in this pass (<= kDecodeMaxRows)
    const uint16_t *rout, *s_out;
    uint16_t *out;            // bf16, row stride ldo, already offset by col0
    int64_t ldo;
    float *partials;
    int32_t *counters;
};
cudaError_t launch_decode_gemm(const DecodeGemmArgs &a, cudaStream_t s);

bool prefill_supported();
cudaError_t launch_prefill(const uint16_t *u, const uint16_t *wt, int64_t M, int IC, int OC,
                           const uint16_t *rout, const uint16_t *s_out, uint16_t *out,
                           int64_t ldo, int32_t *err, cudaStream_t s, bool *launched);

cudaError_t launch_gather(const int8_t *q, const uint16_t *scale, int64_t V, int H,
                          const int32_t *ids, int64_t N, uint16_t *out, int32_t *n_bad,
                          cudaStream_t s);

}  // namespace exl3
