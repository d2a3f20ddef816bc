// convert.cu -- bf16 operand preparation for the tensor-core gradient products.
//
// RETURNN paper, Sec. 4.2: the weight and input gradients are each one
// product over all frames once the recurrent part has been back-propagated.
// On the bf16 path those products run on tcgen05 with both operands K-major,
// so the frame dimension (K of dW and dR) has to be innermost: this kernel
// writes bf16 transposes (and, optionally, a row-major bf16 copy) of a column
// block of a row-major matrix, reading its rows through an optional row map.
#include "common.cuh"
#include "gemm.cuh"

namespace lstm {

namespace {

template <typename Tin>
__device__ __forceinline__ float load_f(const Tin* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// dstT[c][r] = bf16(src[row(r)][col0 + c]) and, if dst_rm, dst_rm[r][c] = the same value,
// for r < rows, c < cols; row(r) = map ? map[r] : r, and a negative map entry reads 0.
template <typename Tin>
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const Tin* __restrict__ src, int64_t lds, int col0,
                                                             const int32_t* __restrict__ map, int rows, int cols,
                                                             __nv_bfloat16* __restrict__ dstT, int64_t ldt,
                                                             __nv_bfloat16* __restrict__ dst_rm, int64_t ldm)
{
    __shared__ __nv_bfloat16 tile[32][34];
    const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        __nv_bfloat16 v = __float2bfloat16_rn(0.f);
        if (r < rows && c < cols) {
            const int64_t sr = map ? (int64_t)__ldg(map + r) : (int64_t)r;
            if (sr >= 0) v = __float2bfloat16_rn(load_f<Tin>(src + sr * lds + col0 + c));
            if (dst_rm) dst_rm[(int64_t)r * ldm + c] = v;
        }
        tile[i][tx] = v;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (c < cols && r < rows) dstT[(int64_t)c * ldt + r] = tile[tx][i];
    }
}

}  // namespace

lstm_status transpose_to_bf16(const Plan& p, const void* src, bool src_bf16, int64_t lds, int col0,
                              const int32_t* map, int rows, int cols, void* dstT, int64_t ldt, void* dst_rm,
                              int64_t ldm, cudaStream_t s)
{
    if (rows <= 0 || cols <= 0) return LSTM_OK;
    const dim3 grid((rows + 31) / 32, (cols + 31) / 32);
    trace_begin(p, K_CONVERT, s);
    if (src_bf16)
        transpose_bf16_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16*)src, lds, col0, map, rows, cols, (__nv_bfloat16*)dstT, ldt,
            (__nv_bfloat16*)dst_rm, ldm);
    else
        transpose_bf16_kernel<float><<<grid, 256, 0, s>>>((const float*)src, lds, col0, map, rows, cols,
                                                          (__nv_bfloat16*)dstT, ldt, (__nv_bfloat16*)dst_rm, ldm);
    const cudaError_t e = cudaGetLastError();
    trace_end(p, K_CONVERT, s, e == cudaSuccess ? 1 : 0);
    return e == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

}  // namespace lstm
