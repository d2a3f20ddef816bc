// gemm.cuh -- launch interface of the library's matrix products.
#pragma once

#include "common.cuh"

namespace lstm {

// C(m, n) = sum_k A(m, k) * B(k, n) (+ bias[n]), fp32 accumulate and output.
//   A(m, k) = A[m*sam + k*sak]   (one of sam, sak is 1)
//   B(k, n) = B[row(k)*sbk + n*sbn], row(k) = b_rows ? b_rows[k] : k; a
//             negative b_rows entry makes that B row zero (one of sbk, sbn is 1)
//   C(m, n) = C[m*ldc + n]
// With k_splits > 1 the K range is cut into k_splits pieces whose partial
// products go to `partial` ([k_splits][M][N]) and are then added in split
// order (deterministic), plus bias, into C.
struct GemmDesc {
    int M = 0, N = 0, K = 0;
    const void* A = nullptr; int64_t sam = 0, sak = 0; int a_bf16 = 0;
    const void* B = nullptr; int64_t sbk = 0, sbn = 0; int b_bf16 = 0;
    const int32_t* b_rows = nullptr;
    float* C = nullptr; int64_t ldc = 0;
    const float* bias = nullptr;
    int round_bf16 = 0;       // round fp32 operands to bf16 before multiplying
    int k_splits = 1;
    float* partial = nullptr;
};

// Number of K splits the launcher will use, and the partial-sum floats needed.
int gemm_choose_splits(const GemmDesc& d, int num_sms);
size_t gemm_partial_floats(const GemmDesc& d, int num_sms);

lstm_status gemm_simt_run(const GemmDesc& d, int num_sms, cudaStream_t s);
// Same, traced under `kind` in the plan's tracer.
lstm_status gemm_simt(const GemmDesc& d, const Plan& p, int kind, cudaStream_t s);

// bf16 A[M][K] x B[N][K]^T (+ bias) on tcgen05 tensor cores, fp32 out.
bool gemm_tc_supported(int M, int N, int K, const void* A, const void* B);
lstm_status gemm_tc_bf16_nt(const Plan& p, int kind, const void* A, const void* B, float* C, int64_t ldc,
                            const float* bias, int M, int N, int K, cudaStream_t s);

}  // namespace lstm
