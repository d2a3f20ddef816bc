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

constexpr int kSplitSegs = 6;

// piece of segment sg under `pattern` (0 = the leading piece only)
__device__ __forceinline__ int seg_piece(int pattern, int sg)
{
    if (pattern == 1) return (0x001021 >> (4 * sg)) & 15;    // [1, 2, 0, 1, 0, 0]
    if (pattern == 2) return (0x010201 >> (4 * sg)) & 15;    // [1, 0, 2, 0, 1, 0]
    return 0;
}

__device__ __forceinline__ void split3(float v, __nv_bfloat16 (&p)[3])
{
    p[0] = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(p[0]);
    p[1] = __float2bfloat16_rn(r1);
    p[2] = __float2bfloat16_rn(r1 - __bfloat162float(p[1]));
}

template <typename Tin>
__device__ __forceinline__ float load_f(const Tin* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// dstT[c][r] = bf16(src[row(r)][col0 + c]) and, if dst_rm, dst_rm[r][c] = the same value,
// for r < rows, c < cols; row(r) = map ? map[r] : r, and a negative map entry reads 0.
// Rows in [rows, rows_pad) are written as zeros into dstT only (the padded tail of a K
// range); dst_rm has rows rows.
// Split patterns, for fp32 products on bf16 tensor cores as six products
// concatenated along K: each value v becomes three bf16 pieces v0 = bf16(v),
// v1 = bf16(v - v0), v2 = bf16(v - v0 - v1) (the two differences are exact in
// fp32, and v0 + v1 + v2 is v to within 2^-24 of |v|), written into six K
// segments (kseg_t apart in dstT rows, kseg_m apart in dst_rm rows).  Pattern 1
// (the A side, x) writes pieces [1, 2, 0, 1, 0, 0] and pattern 2 (the B side,
// y) pieces [1, 0, 2, 0, 1, 0], so that the product of a pattern-1 and a
// pattern-2 operand is x1 y1 + x2 y0 + x0 y2 + x1 y0 + x0 y1 + x0 y0: every
// piece product above 2^-24 of x0 y0 (the other three are below 2^-26).
// Pattern 0 writes v0 only.
template <typename Tin>
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const Tin* __restrict__ src, int64_t lds, int col0,
                                                             const int32_t* __restrict__ map, int rows,
                                                             int rows_pad, int cols, int pattern,
                                                             __nv_bfloat16* __restrict__ dstT, int64_t ldt,
                                                             int64_t kseg_t, __nv_bfloat16* __restrict__ dst_rm,
                                                             int64_t ldm, int64_t kseg_m)
{
    __shared__ __nv_bfloat16 tp[3][32][34];
    const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int nseg = pattern == 0 ? 1 : kSplitSegs;
    const int npc = pattern == 0 ? 1 : 3;
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        float f = 0.f;
        if (r < rows && c < cols) {
            const int64_t sr = map ? (int64_t)__ldg(map + r) : (int64_t)r;
            if (sr >= 0) f = load_f<Tin>(src + sr * lds + col0 + c);
        }
        __nv_bfloat16 pc[3];
        split3(f, pc);
        if (dst_rm && r < rows && c < cols)           // the row-major copy has no padded rows
            for (int sg = 0; sg < nseg; ++sg) dst_rm[(int64_t)r * ldm + sg * kseg_m + c] = pc[seg_piece(pattern, sg)];
        for (int q = 0; q < npc; ++q) tp[q][i][tx] = pc[q];
    }
    __syncthreads();
    if (!dstT) return;
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (c < cols && r < rows_pad)
            for (int sg = 0; sg < nseg; ++sg) dstT[(int64_t)c * ldt + sg * kseg_t + r] = tp[seg_piece(pattern, sg)][tx][i];
    }
}

template <typename Tin>
__device__ __forceinline__ void load4(const Tin* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4])
{
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4])
{
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(x.x << 16); v[1] = __uint_as_float(x.x & 0xffff0000u);
    v[2] = __uint_as_float(x.y << 16); v[3] = __uint_as_float(x.y & 0xffff0000u);
}

// The same conversion in 64 x 64 tiles with 4-element loads, 8-byte row-major stores and
// 16-byte transposed stores, for layouts where every piece is aligned (cols, col0, lds,
// ldm and kseg_m multiples of 4; ldt and kseg_t multiples of 8; 16-byte aligned bases).
template <typename Tin>
__global__ void __launch_bounds__(256) transpose_bf16_v4_kernel(const Tin* __restrict__ src, int64_t lds, int col0,
                                                                const int32_t* __restrict__ map, int rows,
                                                                int rows_pad, int cols, int pattern,
                                                                __nv_bfloat16* __restrict__ dstT, int64_t ldt,
                                                                int64_t kseg_t, __nv_bfloat16* __restrict__ dst_rm,
                                                                int64_t ldm, int64_t kseg_m)
{
    __shared__ __align__(16) __nv_bfloat16 tp[3][64][72];     // [piece][column][row]
    const int r0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
    const int tid = threadIdx.x;
    const int nseg = pattern == 0 ? 1 : kSplitSegs;
    const int npc = pattern == 0 ? 1 : 3;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int rr = (tid >> 4) + 16 * it, q = tid & 15;
        const int r = r0 + rr, c = c0 + 4 * q;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < rows && c < cols) {
            const int64_t sr = map ? (int64_t)__ldg(map + r) : (int64_t)r;
            if (sr >= 0) load4<Tin>(src + sr * lds + col0 + c, v);
        }
        __nv_bfloat16 pc[4][3];
#pragma unroll
        for (int e = 0; e < 4; ++e) split3(v[e], pc[e]);
        if (dst_rm && r < rows && c < cols) {
            uint2 pw[3];
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                pw[k].x = (uint32_t)__bfloat16_as_ushort(pc[0][k]) | ((uint32_t)__bfloat16_as_ushort(pc[1][k]) << 16);
                pw[k].y = (uint32_t)__bfloat16_as_ushort(pc[2][k]) | ((uint32_t)__bfloat16_as_ushort(pc[3][k]) << 16);
            }
            for (int sg = 0; sg < nseg; ++sg)
                *reinterpret_cast<uint2*>(dst_rm + (int64_t)r * ldm + sg * kseg_m + c) = pw[seg_piece(pattern, sg)];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int k = 0; k < 3; ++k)
                if (k < npc) tp[k][4 * q + e][rr] = pc[e][k];
    }
    __syncthreads();
    if (!dstT) return;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int cc = (tid >> 3) + 32 * it, o = tid & 7;
        const int c = c0 + cc, r = r0 + 8 * o;
        if (c >= cols || r >= rows_pad) continue;
        for (int sg = 0; sg < nseg; ++sg) {
            const __nv_bfloat16* t = &tp[seg_piece(pattern, sg)][cc][8 * o];
            __nv_bfloat16* d = dstT + (int64_t)c * ldt + sg * kseg_t + r;
            if (r + 8 <= rows_pad) {
                *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(t);
            } else {
                for (int e = 0; e < 8 && r + e < rows_pad; ++e) d[e] = t[e];
            }
        }
    }
}

}  // namespace

lstm_status transpose_to_bf16_split(const Plan& p, const void* src, bool src_bf16, int64_t lds, int col0,
                                    const int32_t* map, int rows, int rows_pad, int cols, int pattern, void* dstT,
                                    int64_t ldt, int64_t kseg_t, void* dst_rm, int64_t ldm, int64_t kseg_m,
                                    cudaStream_t s)
{
    rows_pad = rows_pad < rows ? rows : rows_pad;
    if (rows_pad <= 0 || cols <= 0) return LSTM_OK;
    const bool v4 = cols % 4 == 0 && col0 % 4 == 0 && lds % 4 == 0 && ((uintptr_t)src & 15u) == 0 &&
                    (!dst_rm || (ldm % 4 == 0 && kseg_m % 4 == 0 && ((uintptr_t)dst_rm & 15u) == 0)) &&
                    (!dstT || (ldt % 8 == 0 && kseg_t % 8 == 0 && ((uintptr_t)dstT & 15u) == 0));
    if (v4) {
        const dim3 grid4((rows_pad + 63) / 64, (cols + 63) / 64);
        trace_begin(p, K_CONVERT, s);
        if (src_bf16)
            transpose_bf16_v4_kernel<__nv_bfloat16><<<grid4, 256, 0, s>>>(
                (const __nv_bfloat16*)src, lds, col0, map, rows, rows_pad, cols, pattern, (__nv_bfloat16*)dstT, ldt,
                kseg_t, (__nv_bfloat16*)dst_rm, ldm, kseg_m);
        else
            transpose_bf16_v4_kernel<float><<<grid4, 256, 0, s>>>((const float*)src, lds, col0, map, rows, rows_pad,
                                                                  cols, pattern, (__nv_bfloat16*)dstT, ldt, kseg_t,
                                                                  (__nv_bfloat16*)dst_rm, ldm, kseg_m);
        const cudaError_t e = cudaGetLastError();
        trace_end(p, K_CONVERT, s, e == cudaSuccess ? 1 : 0);
        return e == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
    }
    const dim3 grid((rows_pad + 31) / 32, (cols + 31) / 32);
    trace_begin(p, K_CONVERT, s);
    if (src_bf16)
        transpose_bf16_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16*)src, lds, col0, map, rows, rows_pad, cols, pattern, (__nv_bfloat16*)dstT, ldt,
            kseg_t, (__nv_bfloat16*)dst_rm, ldm, kseg_m);
    else
        transpose_bf16_kernel<float><<<grid, 256, 0, s>>>((const float*)src, lds, col0, map, rows, rows_pad, cols,
                                                          pattern, (__nv_bfloat16*)dstT, ldt, kseg_t,
                                                          (__nv_bfloat16*)dst_rm, ldm, kseg_m);
    const cudaError_t e = cudaGetLastError();
    trace_end(p, K_CONVERT, s, e == cudaSuccess ? 1 : 0);
    return e == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

lstm_status transpose_to_bf16(const Plan& p, const void* src, bool src_bf16, int64_t lds, int col0,
                              const int32_t* map, int rows, int cols, void* dstT, int64_t ldt, void* dst_rm,
                              int64_t ldm, cudaStream_t s)
{
    return transpose_to_bf16_split(p, src, src_bf16, lds, col0, map, rows, rows, cols, 0, dstT, ldt, 0, dst_rm, ldm,
                                   0, s);
}

}  // namespace lstm
