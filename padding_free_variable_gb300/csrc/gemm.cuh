// gemm.cuh -- launch interface of the library's matrix products.
#pragma once

#include <cuda.h>

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
    int accumulate = 0;       // C += result instead of C = result (taken unsplit)
    float* partial = nullptr;
};

// Number of K splits the launcher will use, and the partial-sum floats needed.
int gemm_choose_splits(const GemmDesc& d, int num_sms);
size_t gemm_partial_floats(const GemmDesc& d, int num_sms);

lstm_status gemm_simt_run(const GemmDesc& d, int num_sms, cudaStream_t s);
// Same, traced under `kind` in the plan's tracer.
lstm_status gemm_simt(const GemmDesc& d, const Plan& p, int kind, cudaStream_t s);

// bf16 A[M][K] x B[N][K]^T (+ bias) on tcgen05 tensor cores, fp32 out.
// Row pitches lda, ldb in elements (multiples of 8); K may be any positive
// size (the tail reads zeros).  splits > 1 cuts K into that many ranges whose
// partial products go to `partial` ([splits][M][N]) and are then added in
// split order, plus bias, into C.
bool gemm_tc_supported(int M, int N, int K, const void* A, const void* B);
int gemm_tc_splits(int M, int N, int K, int num_sms, int max_splits);
lstm_status gemm_tc_bf16(const Plan& p, int kind, const void* A, int64_t lda, const void* B, int64_t ldb, int M,
                         int N, int K, float* C, int64_t ldc, const float* bias, int splits, float* partial,
                         cudaStream_t s);

// dstT[c][r] = bf16(src[row(r)][col0 + c]) (row(r) = map ? map[r] : r, negative
// map entries read 0), optionally also dst_rm[r][c]; src fp32 or bf16.
lstm_status transpose_to_bf16(const Plan& p, const void* src, bool src_bf16, int64_t lds, int col0,
                              const int32_t* map, int rows, int cols, void* dstT, int64_t ldt, void* dst_rm,
                              int64_t ldm, cudaStream_t s);

// One product C[M][N] = A[M][K] B[N][K]^T (bf16, K-major, fp32 out, no bias)
// with its tensor maps encoded once, for launches that repeat with varying M
// (M <= rows_max; rows past M are computed from whatever A holds there and
// not stored).
// With splits > 1 the K range is cut into that many pieces and piece z writes its partial
// product into slice z of C (slices rows_max * ldc floats apart); the reader adds the
// slices in order.
struct TcOperands {
    CUtensorMap A, B;
    int N = 0, K = 0;
    float* C = nullptr;
    int64_t ldc = 0;
    int splits = 1;
    int64_t split_stride = 0;
};
bool gemm_tc_prepare(TcOperands* o, const void* A, int64_t lda, int rows_max, const void* B, int64_t ldb, int N,
                     int K, float* C, int64_t ldc, int splits);
// K splits that fill the GPU with `products` products of up to rows_max x N.
int gemm_tc_pair_splits(int rows_max, int N, int K, int products, int num_sms);
// Two prepared products (o1 may be null; equal splits) in one launch, with M0 and M1 rows.
lstm_status gemm_tc_pair(const Plan& p, int kind, const TcOperands& o0, int M0, const TcOperands* o1, int M1,
                         cudaStream_t s);

// TMA map of a row-major fp32 matrix [rows][cols] (row pitch ld elements) in
// boxes of box_cols x box_rows without swizzle; out-of-range elements read 0.
// False when the driver entry point is missing or the layout is not
// TMA-addressable (16-byte aligned base, pitch and box row).
bool make_map_f32(CUtensorMap* map, const float* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                  int box_rows);

// TMA map of a row-major bf16 matrix [rows][cols] (row pitch ld elements) in boxes of 64
// columns x box_rows rows with the 128-byte swizzle (the K-major operand layout of
// tc::sdesc_sw128); out-of-range elements read 0.
bool make_map_bf16_sw128(CUtensorMap* map, const void* ptr, int rows, int cols, int64_t ld, int box_rows);

// The same with a padded row range (rows in [rows, rows_pad) written as 0)
// and an fp32 split into three bf16 pieces v0 + v1 + v2 written as six K
// segments (kSplitSegments, kseg_t / kseg_m elements apart in the transposed /
// row-major output): pattern 1 = pieces [1, 2, 0, 1, 0, 0], pattern 2 =
// [1, 0, 2, 0, 1, 0], so that a pattern-1 operand times a pattern-2 operand is
// the sum of the six piece products above 2^-24 of the leading one; pattern 0
// = v0 only.  dstT may be null.
constexpr int kSplitSegments = 6;
lstm_status transpose_to_bf16_split(const Plan& p, const void* src, bool src_bf16, int64_t lds, int col0,
                                    const int32_t* map, int rows, int rows_pad, int cols, int pattern, void* dstT,
                                    int64_t ldt, int64_t kseg_t, void* dst_rm, int64_t ldm, int64_t kseg_m,
                                    cudaStream_t s);

// C = sum over splits (in split order) of partial, + bias.
cudaError_t splitk_reduce(const float* partial, int splits, int M, int N, float* C, int64_t ldc,
                          const float* bias, int num_sms, cudaStream_t s);
lstm_status gemm_tc_bf16_nt(const Plan& p, int kind, const void* A, const void* B, float* C, int64_t ldc,
                            const float* bias, int M, int N, int K, cudaStream_t s);

}  // namespace lstm
