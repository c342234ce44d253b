// gemm_tc.cuh - host-side interface of gemm_tc.cu (the prefill product):
// the x conversion, the two tcgen05 GEMMs and their launch plans.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace qg {

// Token-tile width (128 or 256) and k-split parts of a GEMM launch.
struct GemmPlan {
    int bn, ks;
};

// f32 -> f16 (round to nearest even) of n values (n a multiple of 8).
cudaError_t launch_f32_to_f16(const float *x, __half *out, int64_t n, int sms, cudaStream_t s);

// Y[n_tok][n_out] = A[n_out][K] . B[n_tok][K]^T for f16 A, B (16-byte aligned,
// K a multiple of 8), tiles as gemm_f16_plan chooses them.
cudaError_t launch_gemm_f16_tc(const __half *A, const __half *B, float *y, int64_t n_out, int64_t n_tok, int64_t K,
                               int32_t *err, int sms, int device, cudaStream_t s);

// The same for Q4_K W, dequantized into tensor memory inside the GEMM, with
// the tiles and k split of `plan`; a split's partial products go to `part`
// ((plan.ks - 1) n_tok n_out f32) and one more launch adds them to y.
cudaError_t launch_gemm_q4k_tmem(const uint8_t *W, const __half *B, float *y, int64_t n_out, int64_t n_tok,
                                 int64_t K, GemmPlan plan, float *part, int32_t *err, int sms, int device,
                                 cudaStream_t s);

GemmPlan gemm_q4k_tmem_plan(int64_t n_out, int64_t n_tok, int64_t K, int sms, int max_parts, size_t scratch_bytes);
GemmPlan gemm_f16_plan(int64_t n_out, int64_t n_tok, int64_t K, int sms);

}  // namespace qg
