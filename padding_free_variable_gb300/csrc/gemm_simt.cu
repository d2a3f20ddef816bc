// gemm_simt.cu -- CUDA-core matrix products (fp32 path, and any shape the
// tensor-core kernel does not take).
//
// RETURNN paper, Sec. 4.2: the non-recurrent part of the LSTM forward pass is
// one matrix product over the whole batch of sequences, and so are the
// gradients with respect to the weights and the inputs after the recurrent
// part has been back-propagated.  The fp32 path keeps full fp32 products
// (CUDA-core FFMA): tf32 tensor cores would not hold a 1e-4 relative error.
#include <algorithm>

#include "gemm.cuh"

namespace lstm {

namespace {

constexpr int BM = 128, BN = 128, BK = 16, TM = 8, TN = 8, THREADS = 256;

template <typename T> __device__ __forceinline__ float ldf(const T* p, int64_t i);
template <> __device__ __forceinline__ float ldf<float>(const float* p, int64_t i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}

// Tile loaders: element e of the thread's share walks the contiguous
// dimension across consecutive threads so each warp reads contiguous runs.
template <typename TA, bool A_KC>
__device__ __forceinline__ void load_a(const GemmDesc& d, const TA* A, int m0, int k0, int kend,
                                       float (&As)[BK][BM + 4])
{
#pragma unroll
    for (int i = 0; i < (BM * BK) / THREADS; ++i) {
        const int e = i * THREADS + threadIdx.x;
        int m, k;
        if (A_KC) { k = e % BK; m = e / BK; }
        else { m = e % BM; k = e / BM; }
        const int gm = m0 + m, gk = k0 + k;
        float v = 0.f;
        if (gm < d.M && gk < kend) {
            v = ldf<TA>(A, (int64_t)gm * d.sam + (int64_t)gk * d.sak);
            if (d.round_bf16) v = bf16_round(v);
        }
        As[k][m] = v;
    }
}

template <typename TB, bool B_KC>
__device__ __forceinline__ void load_b(const GemmDesc& d, const TB* B, int n0, int k0, int kend,
                                       float (&Bs)[BK][BN + 4])
{
#pragma unroll
    for (int i = 0; i < (BN * BK) / THREADS; ++i) {
        const int e = i * THREADS + threadIdx.x;
        int n, k;
        if (B_KC) { k = e % BK; n = e / BK; }
        else { n = e % BN; k = e / BN; }
        const int gn = n0 + n, gk = k0 + k;
        float v = 0.f;
        if (gn < d.N && gk < kend) {
            int64_t row = gk;
            if (d.b_rows) row = __ldg(d.b_rows + gk);
            if (row >= 0) {
                v = ldf<TB>(B, row * d.sbk + (int64_t)gn * d.sbn);
                if (d.round_bf16) v = bf16_round(v);
            }
        }
        Bs[k][n] = v;
    }
}

template <typename TA, typename TB, bool A_KC, bool B_KC>
__global__ void __launch_bounds__(THREADS) gemm_simt_kernel(GemmDesc d, int k_chunk)
{
    __shared__ __align__(16) float As[2][BK][BM + 4];
    __shared__ __align__(16) float Bs[2][BK][BN + 4];
    const TA* A = reinterpret_cast<const TA*>(d.A);
    const TB* B = reinterpret_cast<const TB*>(d.B);
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int kbeg = blockIdx.z * k_chunk;
    const int kend = min(d.K, kbeg + k_chunk);
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    int buf = 0;
    if (kbeg < kend) {
        load_a<TA, A_KC>(d, A, m0, kbeg, kend, As[0]);
        load_b<TB, B_KC>(d, B, n0, kbeg, kend, Bs[0]);
    }
    __syncthreads();
    for (int k0 = kbeg; k0 < kend; k0 += BK) {
        if (k0 + BK < kend) {
            load_a<TA, A_KC>(d, A, m0, k0 + BK, kend, As[buf ^ 1]);
            load_b<TB, B_KC>(d, B, n0, k0 + BK, kend, Bs[buf ^ 1]);
        }
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
            // rows ty*4 + {0..3} and 64 + ty*4 + {0..3}: conflict-free float4 reads
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w; a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w; b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
        buf ^= 1;
    }
    float* out = d.C;
    int64_t ldo = d.ldc;
    const bool split = d.k_splits > 1;
    if (split) { out = d.partial + (int64_t)blockIdx.z * d.M * d.N; ldo = d.N; }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (gm >= d.M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (gn >= d.N) continue;
            float v = acc[i][j];
            if (!split && d.bias) v += __ldg(d.bias + gn);
            if (!split && d.accumulate) v += out[(int64_t)gm * ldo + gn];
            out[(int64_t)gm * ldo + gn] = v;
        }
    }
}

// C = sum over splits (in split order) + bias
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, int M, int N,
                                     float* __restrict__ C, int64_t ldc, const float* __restrict__ bias)
{
    const int64_t total = (int64_t)M * N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int z = 0; z < splits; ++z) s += partial[(int64_t)z * total + i];
        const int64_t m = i / N, n = i - m * N;
        if (bias) s += bias[n];
        C[m * ldc + n] = s;
    }
}

template <typename TA, typename TB>
lstm_status launch_typed(const GemmDesc& desc, int splits, int k_chunk, int num_sms, cudaStream_t s)
{
    GemmDesc d = desc;
    d.k_splits = splits;          // the kernel writes partial sums only when really split
    const dim3 grid((d.N + BN - 1) / BN, (d.M + BM - 1) / BM, splits);
    const bool akc = d.sak == 1, bkc = d.sbk == 1 && d.b_rows == nullptr;
    if (akc && bkc) gemm_simt_kernel<TA, TB, true, true><<<grid, THREADS, 0, s>>>(d, k_chunk);
    else if (akc && !bkc) gemm_simt_kernel<TA, TB, true, false><<<grid, THREADS, 0, s>>>(d, k_chunk);
    else if (!akc && bkc) gemm_simt_kernel<TA, TB, false, true><<<grid, THREADS, 0, s>>>(d, k_chunk);
    else gemm_simt_kernel<TA, TB, false, false><<<grid, THREADS, 0, s>>>(d, k_chunk);
    if (cudaGetLastError() != cudaSuccess) return LSTM_ERR_CUDA;
    if (splits > 1 && splitk_reduce(d.partial, splits, d.M, d.N, d.C, d.ldc, d.bias, num_sms, s) != cudaSuccess)
        return LSTM_ERR_CUDA;
    return LSTM_OK;
}

}  // namespace

cudaError_t splitk_reduce(const float* partial, int splits, int M, int N, float* C, int64_t ldc,
                          const float* bias, int num_sms, cudaStream_t s)
{
    const int64_t total = (int64_t)M * N;
    if (total == 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 8);
    splitk_reduce_kernel<<<blocks, 256, 0, s>>>(partial, splits, M, N, C, ldc, bias);
    return cudaGetLastError();
}

int gemm_choose_splits(const GemmDesc& d, int num_sms)
{
    if (d.k_splits <= 1 || d.accumulate) return 1;
    const int tiles = ((d.N + BN - 1) / BN) * ((d.M + BM - 1) / BM);
    int splits = (2 * num_sms + tiles - 1) / tiles;
    const int max_by_k = (d.K + 255) / 256;
    splits = std::min(splits, std::min(max_by_k, d.k_splits));
    return std::max(1, splits);
}

size_t gemm_partial_floats(const GemmDesc& d, int num_sms)
{
    const int s = gemm_choose_splits(d, num_sms);
    return s > 1 ? (size_t)s * d.M * d.N : 0;
}

lstm_status gemm_simt(const GemmDesc& d, const Plan& p, int kind, cudaStream_t s)
{
    if (d.M <= 0 || d.N <= 0) return LSTM_OK;
    const int num_sms = p.num_sms;
    trace_begin(p, kind, s);
    lstm_status st = gemm_simt_run(d, num_sms, s);
    const int splits = d.K > 0 ? gemm_choose_splits(d, num_sms) : 1;
    trace_end(p, kind, s, splits > 1 ? 2 : 1);
    return st;
}

lstm_status gemm_simt_run(const GemmDesc& d, int num_sms, cudaStream_t s)
{
    const int splits = gemm_choose_splits(d, num_sms);
    if (d.K <= 0) {
        if (d.accumulate) return LSTM_OK;             // C += 0
        // empty reduction: C = bias (or 0)
        GemmDesc z = d;
        z.k_splits = 1;
        return launch_typed<float, float>(z, 1, 0, num_sms, s);
    }
    const int k_chunk = ((d.K + splits - 1) / splits + BK - 1) / BK * BK;
    if (splits > 1 && !d.partial) return LSTM_ERR_INVALID_ARG;
    if (d.a_bf16 && d.b_bf16) return launch_typed<__nv_bfloat16, __nv_bfloat16>(d, splits, k_chunk, num_sms, s);
    if (d.a_bf16) return launch_typed<__nv_bfloat16, float>(d, splits, k_chunk, num_sms, s);
    if (d.b_bf16) return launch_typed<float, __nv_bfloat16>(d, splits, k_chunk, num_sms, s);
    return launch_typed<float, float>(d, splits, k_chunk, num_sms, s);
}

}  // namespace lstm
