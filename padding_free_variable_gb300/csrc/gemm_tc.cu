// gemm_tc.cu -- bf16 products on the 5th-generation tensor cores.
//
// RETURNN paper, Sec. 4.2: the non-recurrent part of the forward pass is one
// matrix product over all frames of the batch.  On GB300 that product runs as
// C[M][N] = A[M][K] B[N][K]^T + bias[N] with A, B bf16 (both K-major, i.e.
// row-major with K innermost) and fp32 accumulation in tensor memory:
//
//   warp 0      TMA producer: 128x64 tiles of A and 256x64 tiles of B into a
//               4-stage ring of 128-byte-swizzled shared-memory slots
//   warp 1      owns the 256 TMEM columns; one thread issues tcgen05.mma
//               (M=128, N=256, K=16) and commits each stage back to the ring
//   warps 2..5  epilogue: tcgen05.ld of their TMEM lane quarter, + bias, store (the
//               persistent kernel stages 32 x 32 pieces in shared memory and writes them
//               with TMA stores: whole 128-byte rows instead of 16-byte pieces of 32 rows)
//
// Every mbarrier wait is bounded; a timeout is recorded in the plan's status
// word and the CTA still frees its tensor memory before returning.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "gemm.cuh"
#include "tc_ptx.cuh"

namespace lstm {

namespace {

constexpr int TBM = 128, TBN = 256, TBK = 64, TSTAGES = 4;
constexpr int TC_THREADS = 192;
constexpr uint32_t A_BYTES = TBM * TBK * 2;
constexpr uint32_t B_BYTES = TBN * TBK * 2;
constexpr uint32_t TMEM_COLS = 256;
constexpr size_t TC_SMEM = 1024 + (size_t)TSTAGES * (A_BYTES + B_BYTES) + 256;
// persistent kernel: the epilogue warps' output staging, two 32 x 32 fp32 boxes per warp
constexpr int EPI_COLS = 32;
constexpr uint32_t EPI_BOX_BYTES = 32 * EPI_COLS * 4;
constexpr uint32_t EPI_BYTES = 4 * 2 * EPI_BOX_BYTES;
constexpr size_t TC_SMEM_P = TC_SMEM + EPI_BYTES;
static_assert(TC_SMEM_P <= 227 * 1024, "shared memory of the persistent kernel");

struct TcArgs {
    int M, N, K;
    int k_chunk;          // k range of split z: [z*k_chunk, min(K, (z+1)*k_chunk)), multiple of 64
    float* C;
    int64_t ldc;
    const float* bias;    // added only without split
    float* partial;       // split > 1: [z][M][N], or [z] slices split_stride apart with row pitch ldc
    int64_t split_stride; // 0: slices of M x N
    DeviceStatus* status;
    unsigned long long limit_ns;
};

__device__ __forceinline__ void fail(const TcArgs& a, int* s_abort, unsigned where)
{
    record_failure(a.status, LSTM_ERR_TIMEOUT, 0x80000u | where);
    *(volatile int*)s_abort = 1;
}

// One 128 x 256 output tile (blockIdx.x, blockIdx.y) of split zs of nzs.
__device__ __forceinline__ void tc_gemm_tile(const CUtensorMap* mapA, const CUtensorMap* mapB, const TcArgs& a,
                                             int zs, int nzs)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = base;
    uint8_t* sB = base + TSTAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + TSTAGES * (A_BYTES + B_BYTES));
    uint64_t* empty = full + TSTAGES;
    uint64_t* accf = empty + TSTAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * TBM, n0 = blockIdx.x * TBN;
    const int kbeg = zs * a.k_chunk;
    const int kend = min(a.K, kbeg + a.k_chunk);
    const int nk = kend > kbeg ? (kend - kbeg + TBK - 1) / TBK : 0;
    const bool split = nzs > 1;
    float* const Cout = split ? a.partial + (int64_t)zs * (a.split_stride ? a.split_stride : (int64_t)a.M * a.N) : a.C;
    const int64_t ldo = split ? (a.split_stride ? a.ldc : (int64_t)a.N) : a.ldc;
    const float* const bias = split ? nullptr : a.bias;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(accf, 1);
        *s_abort = 0;
        tc::fence_mbar_init();
        tc::prefetch_tensormap(mapA);
        tc::prefetch_tensormap(mapB);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- producer
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % TSTAGES;
            if (kb >= TSTAGES && !tc::mbar_wait(&empty[s], ((kb / TSTAGES) - 1) & 1, a.limit_ns)) {
                fail(a, s_abort, 1);
                break;
            }
            if (*(volatile int*)s_abort) break;
            tc::mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
            tc::tma_load_2d(sA + s * A_BYTES, mapA, &full[s], kbeg + kb * TBK, m0);
            tc::tma_load_2d(sB + s * B_BYTES, mapB, &full[s], kbeg + kb * TBK, n0);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16_f32(TBM, TBN);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % TSTAGES;
            if (*(volatile int*)s_abort) break;
            if (!tc::mbar_wait(&full[s], (kb / TSTAGES) & 1, a.limit_ns)) {
                fail(a, s_abort, 2);
                break;
            }
            tc::tc_fence_after_sync();
            const uint32_t a0 = tc::smem_u32(sA + s * A_BYTES), b0 = tc::smem_u32(sB + s * B_BYTES);
#pragma unroll
            for (int kk = 0; kk < TBK / 16; ++kk)
                tc::mma_bf16_ss(tmem, tc::sdesc_sw128(a0 + kk * 32), tc::sdesc_sw128(b0 + kk * 32), idesc,
                                (kb | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(accf);      // arrives once every MMA issued above has completed
    } else if (warp >= 2) {
        // ---- epilogue: this warp may read TMEM lanes 32*(warp%4) .. +31
        const int q = warp & 3;
        const int row = m0 + q * 32 + lane;
        const bool ok = tc::mbar_wait(accf, 0, a.limit_ns);
        if (!ok && lane == 0) fail(a, s_abort, 3);
        tc::tc_fence_after_sync();
        if (__all_sync(0xffffffffu, ok) && !*(volatile int*)s_abort) {
            const bool vec = (ldo % 4) == 0 && (((uintptr_t)Cout) & 15u) == 0;
            for (int c = 0; c < TBN; c += 16) {
                if (n0 + c >= a.N) break;                      // uniform across the warp
                uint32_t r[16];
                if (nk > 0) {
                    tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, r);
                    tc::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = 0u;   // empty k range: a zero product
                }
                if (row < a.M) {
                    const int n = n0 + c;
                    float* out = Cout + (int64_t)row * ldo + n;
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
                    if (n + 16 <= a.N && vec) {
                        if (bias) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] += __ldg(bias + n + e);
                        }
#pragma unroll
                        for (int e = 0; e < 16; e += 4)
                            *reinterpret_cast<float4*>(out + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (n + e < a.N) out[e] = v[e] + (bias ? __ldg(bias + n + e) : 0.f);
                    }
                }
            }
        }
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Persistent form: one CTA per SM walks the (split, m, n) tiles of the product with stride
// gridDim.x (n fastest, so the CTAs in flight share A tiles and all of B through L2).  The
// shared-memory ring continues across tiles, and the accumulator is double-buffered in
// tensor memory (2 x 256 columns): the epilogue warps drain tile i from one buffer while the
// MMA warp accumulates tile i + 1 into the other.  Barriers: full / empty per ring stage,
// accf per buffer (MMA -> epilogue) and acce per buffer (the 4 epilogue warps -> MMA).
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_bf16_persistent_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                               const __grid_constant__ CUtensorMap mapC, TcArgs a, int nM, int nN, int splits,
                               int tma_c)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = base;
    uint8_t* sB = base + TSTAGES * A_BYTES;
    uint8_t* stg = base + TSTAGES * (A_BYTES + B_BYTES);      // 1024-aligned output staging
    uint64_t* full = reinterpret_cast<uint64_t*>(stg + EPI_BYTES);
    uint64_t* empty = full + TSTAGES;
    uint64_t* accf = empty + TSTAGES;        // [2]
    uint64_t* acce = accf + 2;               // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
    int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = nM * nN * splits;
    const bool split = splits > 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TSTAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&accf[b], 1);
            tc::mbar_init(&acce[b], 4);
        }
        *s_abort = 0;
        tc::fence_mbar_init();
        tc::prefetch_tensormap(&mapA);
        tc::prefetch_tensormap(&mapB);
        if (tma_c) tc::prefetch_tensormap(&mapC);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 2 * TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    auto decode = [&](int tile, int& z, int& m0, int& n0, int& kbeg, int& nk) {
        z = tile / (nM * nN);
        const int rem = tile - z * nM * nN;
        m0 = (rem / nN) * TBM;
        n0 = (rem % nN) * TBN;
        kbeg = z * a.k_chunk;
        const int kend = min(a.K, kbeg + a.k_chunk);
        nk = kend > kbeg ? (kend - kbeg + TBK - 1) / TBK : 0;
    };

    if (warp == 0 && lane == 0) {
        // ---- producer: the ring's k-blocks of every tile of this CTA, in order
        int g = 0;
        for (int tile = blockIdx.x; tile < ntiles && !*(volatile int*)s_abort; tile += gridDim.x) {
            int z, m0, n0, kbeg, nk;
            decode(tile, z, m0, n0, kbeg, nk);
            for (int kb = 0; kb < nk; ++kb, ++g) {
                const int s = g % TSTAGES;
                if (g >= TSTAGES && !tc::mbar_wait(&empty[s], ((g / TSTAGES) - 1) & 1, a.limit_ns)) {
                    fail(a, s_abort, 11);
                    break;
                }
                if (*(volatile int*)s_abort) break;
                tc::mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
                tc::tma_load_2d(sA + s * A_BYTES, &mapA, &full[s], kbeg + kb * TBK, m0);
                tc::tma_load_2d(sB + s * B_BYTES, &mapB, &full[s], kbeg + kb * TBK, n0);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: tile i into accumulator buffer i & 1
        constexpr uint32_t idesc = tc::idesc_bf16_f32(TBM, TBN);
        int g = 0, i = 0;
        for (int tile = blockIdx.x; tile < ntiles && !*(volatile int*)s_abort; tile += gridDim.x, ++i) {
            int z, m0, n0, kbeg, nk;
            decode(tile, z, m0, n0, kbeg, nk);
            const int b = i & 1;
            if (i >= 2 && !tc::mbar_wait(&acce[b], ((i >> 1) - 1) & 1, a.limit_ns)) {
                fail(a, s_abort, 12);
                break;
            }
            tc::tc_fence_after_sync();
            const uint32_t d = tmem + (uint32_t)(b * TMEM_COLS);
            bool ok = true;
            for (int kb = 0; kb < nk; ++kb, ++g) {
                const int s = g % TSTAGES;
                if (*(volatile int*)s_abort || !tc::mbar_wait(&full[s], (g / TSTAGES) & 1, a.limit_ns)) {
                    if (!*(volatile int*)s_abort) fail(a, s_abort, 13);
                    ok = false;
                    break;
                }
                tc::tc_fence_after_sync();
                const uint32_t a0 = tc::smem_u32(sA + s * A_BYTES), b0 = tc::smem_u32(sB + s * B_BYTES);
#pragma unroll
                for (int kk = 0; kk < TBK / 16; ++kk)
                    tc::mma_bf16_ss(d, tc::sdesc_sw128(a0 + kk * 32), tc::sdesc_sw128(b0 + kk * 32), idesc,
                                    (kb | kk) != 0 ? 1u : 0u);
                tc::mma_commit(&empty[s]);
            }
            if (!ok) break;
            tc::mma_commit(&accf[b]);    // arrives once every MMA of this tile has completed
        }
    } else if (warp >= 2) {
        // ---- epilogue: this warp reads TMEM lanes 32*(warp%4) .. +31 of the tile's buffer
        const int q = warp & 3;
        // tma_c: 32-column pieces go through this warp's two staging boxes (128-byte swizzle:
        // 16-byte chunk j of row r at chunk j ^ (r & 7), so each 8-lane phase of the v4 stores
        // covers all banks) and leave as one TMA store each: whole 128-byte rows, clipped to C
        float* const box0 = reinterpret_cast<float*>(stg + (size_t)q * 2 * EPI_BOX_BYTES);
        int pieces = 0;                       // this warp's staged pieces so far (box = pieces & 1)
        int i = 0;
        for (int tile = blockIdx.x; tile < ntiles && !*(volatile int*)s_abort; tile += gridDim.x, ++i) {
            int z, m0, n0, kbeg, nk;
            decode(tile, z, m0, n0, kbeg, nk);
            const int b = i & 1;
            const bool ok = tc::mbar_wait(&accf[b], (i >> 1) & 1, a.limit_ns);
            if (!ok && lane == 0) fail(a, s_abort, 14);
            tc::tc_fence_after_sync();
            if (!__all_sync(0xffffffffu, ok) || *(volatile int*)s_abort) break;
            float* const Cout = split ? a.partial + (int64_t)z * a.M * a.N : a.C;
            const int64_t ldo = split ? (int64_t)a.N : a.ldc;
            const float* const bias = split ? nullptr : a.bias;
            const bool vec = (ldo % 4) == 0 && (((uintptr_t)Cout) & 15u) == 0;
            const int row = m0 + q * 32 + lane;
            if (tma_c && !split) {
                // a warp whose 32 rows all lie past M (last row block) has nothing to store
                const int cend = m0 + q * 32 < a.M ? TBN : 0;
                const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * TMEM_COLS);
                for (int c = 0; c < cend; c += EPI_COLS) {
                    if (n0 + c >= a.N) break;                  // uniform across the warp
                    uint32_t r0[16], r1[16];
                    if (nk > 0) {
                        tc::tmem_ld_32x32b_x16(tq + (uint32_t)c, r0);
                        tc::tmem_ld_32x32b_x16(tq + (uint32_t)(c + 16), r1);
                        tc::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) r0[e] = r1[e] = 0u;   // empty k range: a zero product
                    }
                    // bias of the piece's 32 columns: one coalesced load, then broadcast by shuffle
                    const int nb = n0 + c + lane;
                    const float bl = (bias && nb < a.N) ? __ldg(bias + nb) : 0.f;
                    float* const box = box0 + (pieces & 1) * (EPI_BOX_BYTES / 4);
                    if (lane == 0) tc::bulk_wait_group_read<1>();   // this box's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = 4 * j + e;
                            const uint32_t raw = col < 16 ? r0[col] : r1[col - 16];
                            v[e] = __uint_as_float(raw) + __shfl_sync(0xffffffffu, bl, col);
                        }
                        *reinterpret_cast<float4*>(box + lane * EPI_COLS + ((j ^ (lane & 7)) * 4)) =
                            make_float4(v[0], v[1], v[2], v[3]);
                    }
                    tc::fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc::tma_store_2d(&mapC, box, n0 + c, m0 + q * 32);
                        tc::bulk_commit_group();
                    }
                    ++pieces;
                }
            } else {
                for (int c = 0; c < TBN; c += 16) {
                    if (n0 + c >= a.N) break;                      // uniform across the warp
                    uint32_t r[16];
                    if (nk > 0) {
                        tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * TMEM_COLS + c), r);
                        tc::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = 0u;   // empty k range: a zero product
                    }
                    if (row < a.M) {
                        const int n = n0 + c;
                        float* out = Cout + (int64_t)row * ldo + n;
                        float v[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
                        if (n + 16 <= a.N && vec) {
                            if (bias) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) v[e] += __ldg(bias + n + e);
                            }
#pragma unroll
                            for (int e = 0; e < 16; e += 4)
                                *reinterpret_cast<float4*>(out + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                if (n + e < a.N) out[e] = v[e] + (bias ? __ldg(bias + n + e) : 0.f);
                        }
                    }
                }
            }
            // this warp has read the buffer: one arrival per warp frees it for tile i + 2
            tc::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acce[b]);
        }
        // the stores must be complete before the kernel ends
        if (tma_c && lane == 0) tc::bulk_wait_group_all();
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * TMEM_COLS);
    }
}

// Two independent products in one launch (blockIdx.z = product * splits + split): the grid
// covers the larger of the two, and a CTA past its own product's extent returns before it
// touches any barrier or tensor memory.  With splits > 1 each split writes its own slice.
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_bf16_pair_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapB0,
                         const __grid_constant__ CUtensorMap mapA1, const __grid_constant__ CUtensorMap mapB1,
                         TcArgs a0, TcArgs a1, int splits)
{
    const bool second = (int)blockIdx.z >= splits;
    const int zs = (int)blockIdx.z - (second ? splits : 0);
    const TcArgs& a = second ? a1 : a0;
    if ((int)blockIdx.y * TBM >= a.M || (int)blockIdx.x * TBN >= a.N) return;
    tc_gemm_tile(second ? &mapA1 : &mapA0, second ? &mapB1 : &mapB0, a, zs, splits);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Row-major bf16 [rows][cols] with row pitch ld elements (cols = K innermost)
// as 128-byte-swizzled boxes of 64 x box_rows; out-of-range elements read 0.
bool make_map(CUtensorMap* map, const void* ptr, int rows, int cols, int64_t ld, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)TBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_map_bf16_sw128(CUtensorMap* map, const void* ptr, int rows, int cols, int64_t ld, int box_rows)
{
    return ((uintptr_t)ptr & 15u) == 0 && (ld * 2) % 16 == 0 && make_map(map, ptr, rows, cols, ld, box_rows);
}

bool make_map_f32(CUtensorMap* map, const float* ptr, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                  int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc || ((uintptr_t)ptr & 15u) || (ld * 4) % 16 != 0 || (box_cols * 4) % 16 != 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The kernel's dynamic shared-memory limit, raised once per device (the attribute belongs
// to the device's context, so a process driving several GPUs sets it on each).
static bool smem_attr_ready(const void* fn, int bytes)
{
    constexpr int kMaxDevices = 64;
    static std::atomic<uint64_t> done_persistent{0}, done_pair{0};
    std::atomic<uint64_t>& done =
        fn == (const void*)gemm_tc_bf16_persistent_kernel ? done_persistent : done_pair;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
    const uint64_t bit = dev < kMaxDevices ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    if (bit) done.fetch_or(bit, std::memory_order_release);
    return true;
}

// C[M][N] fp32 with row pitch ldc as the epilogue's store target: 32 x 32 boxes, 128-byte
// swizzle (the staging layout of the persistent kernel's epilogue warps).
static bool make_map_c(CUtensorMap* map, float* C, int M, int N, int64_t ldc)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc || ((uintptr_t)C & 15u) || (ldc * 4) % 16 != 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)ldc * 4};
    cuuint32_t box[2] = {(cuuint32_t)EPI_COLS, 32u};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_tc_supported(int M, int N, int K, const void* A, const void* B)
{
    // TMA: 16-byte aligned bases and row pitches; x coordinates are multiples of 64 elements.
    return M > 0 && N > 0 && K > 0 && K % 8 == 0 && ((uintptr_t)A & 15u) == 0 && ((uintptr_t)B & 15u) == 0 &&
           encode_fn() != nullptr;
}

int gemm_tc_splits(int M, int N, int K, int num_sms, int max_splits)
{
    const int tiles = ((N + TBN - 1) / TBN) * ((M + TBM - 1) / TBM);
    const int kblocks = (K + TBK - 1) / TBK;
    int splits = std::max(1, num_sms / std::max(1, tiles));
    splits = std::min(splits, std::min(max_splits, std::max(1, kblocks / 4)));
    return std::max(1, splits);
}

lstm_status gemm_tc_bf16(const Plan& p, int kind, const void* A, int64_t lda, const void* B, int64_t ldb, int M,
                         int N, int K, float* C, int64_t ldc, const float* bias, int splits, float* partial,
                         cudaStream_t s)
{
    if (M <= 0 || N <= 0) return LSTM_OK;
    if (K <= 0 || lda % 8 != 0 || ldb % 8 != 0 || ((uintptr_t)A & 15u) || ((uintptr_t)B & 15u) || !encode_fn())
        return LSTM_ERR_UNSUPPORTED;
    if (splits > 1 && !partial) return LSTM_ERR_INVALID_ARG;
    CUtensorMap mapA, mapB;
    if (!make_map(&mapA, A, M, K, lda, TBM) || !make_map(&mapB, B, N, K, ldb, TBN)) return LSTM_ERR_UNSUPPORTED;
    if (!smem_attr_ready((const void*)gemm_tc_bf16_persistent_kernel, (int)TC_SMEM_P)) return LSTM_ERR_CUDA;
    const int kblocks = (K + TBK - 1) / TBK;
    if (splits < 1) splits = 1;
    const int kb_per = (kblocks + splits - 1) / splits;
    splits = (kblocks + kb_per - 1) / kb_per;          // every split gets at least one k-block
    TcArgs a;
    a.M = M; a.N = N; a.K = K; a.k_chunk = kb_per * TBK;
    a.C = C; a.ldc = ldc; a.bias = bias; a.partial = partial; a.split_stride = 0;
    a.status = p.d_status; a.limit_ns = p.wait_limit_ns;
    const int nM = (M + TBM - 1) / TBM, nN = (N + TBN - 1) / TBN;
    const int ntiles = nM * nN * splits;
    const dim3 grid((unsigned)std::min(ntiles, std::max(1, p.num_sms)));
    // unsplit products store their tiles by TMA when C allows a tensor map
    CUtensorMap mapC;
    memset(&mapC, 0, sizeof(mapC));
    const int tma_c = splits == 1 && make_map_c(&mapC, C, M, N, ldc) ? 1 : 0;
    trace_begin(p, kind, s);
    gemm_tc_bf16_persistent_kernel<<<grid, TC_THREADS, TC_SMEM_P, s>>>(mapA, mapB, mapC, a, nM, nN, splits, tma_c);
    cudaError_t e = cudaGetLastError();
    int launched = e == cudaSuccess ? 1 : 0;
    if (e == cudaSuccess && splits > 1) {
        e = splitk_reduce(partial, splits, M, N, C, ldc, bias, p.num_sms, s);
        launched += e == cudaSuccess ? 1 : 0;
    }
    trace_end(p, kind, s, launched);
    return e == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

bool gemm_tc_prepare(TcOperands* o, const void* A, int64_t lda, int rows_max, const void* B, int64_t ldb, int N,
                     int K, float* C, int64_t ldc, int splits)
{
    if (rows_max <= 0 || N <= 0 || K <= 0 || splits < 1 || lda % 8 != 0 || ldb % 8 != 0 || ((uintptr_t)A & 15u) ||
        ((uintptr_t)B & 15u) || !encode_fn())
        return false;
    if (!make_map(&o->A, A, rows_max, K, lda, TBM) || !make_map(&o->B, B, N, K, ldb, TBN)) return false;
    o->N = N; o->K = K; o->C = C; o->ldc = ldc;
    o->splits = splits; o->split_stride = (int64_t)rows_max * ldc;
    return true;
}

int gemm_tc_pair_splits(int rows_max, int N, int K, int products, int num_sms)
{
    const int tiles = products * ((rows_max + TBM - 1) / TBM) * ((N + TBN - 1) / TBN);
    const int kblocks = (K + TBK - 1) / TBK;
    // splitting pays only when the tiles alone leave most of the GPU idle: each split adds a
    // slice of partial sums to write and read back (measured: 64 tiles of 256 x 4096 x 1024
    // products are faster unsplit)
    if (4 * tiles >= num_sms) return 1;
    int splits = std::max(1, num_sms / std::max(1, tiles));
    return std::max(1, std::min(splits, kblocks / 4));
}

lstm_status gemm_tc_pair(const Plan& p, int kind, const TcOperands& o0, int M0, const TcOperands* o1, int M1,
                         cudaStream_t s)
{
    if (!smem_attr_ready((const void*)gemm_tc_bf16_pair_kernel, (int)TC_SMEM)) return LSTM_ERR_CUDA;
    if (!o1) { o1 = &o0; M1 = 0; }
    const int Mmax = std::max(M0, M1), Nmax = std::max(o0.N, o1->N);
    if (Mmax <= 0) return LSTM_OK;
    if (o1->splits != o0.splits) return LSTM_ERR_INVALID_ARG;
    const int splits = o0.splits;
    auto args = [&](const TcOperands& o, int M) {
        TcArgs a;
        const int kblocks = (o.K + TBK - 1) / TBK;
        a.M = M; a.N = o.N; a.K = o.K; a.k_chunk = (kblocks + splits - 1) / splits * TBK;
        a.C = o.C; a.ldc = o.ldc; a.bias = nullptr;
        a.partial = splits > 1 ? o.C : nullptr;           // split z writes slice z of C
        a.split_stride = o.split_stride;
        a.status = p.d_status; a.limit_ns = p.wait_limit_ns;
        return a;
    };
    const TcArgs a0 = args(o0, M0), a1 = args(*o1, M1);
    const dim3 grid((Nmax + TBN - 1) / TBN, (Mmax + TBM - 1) / TBM, 2 * splits);
    trace_begin(p, kind, s);
    gemm_tc_bf16_pair_kernel<<<grid, TC_THREADS, TC_SMEM, s>>>(o0.A, o0.B, o1->A, o1->B, a0, a1, splits);
    const cudaError_t e = cudaGetLastError();
    trace_end(p, kind, s, e == cudaSuccess ? 1 : 0);
    return e == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

lstm_status gemm_tc_bf16_nt(const Plan& p, int kind, const void* A, const void* B, float* C, int64_t ldc,
                            const float* bias, int M, int N, int K, cudaStream_t s)
{
    if (!gemm_tc_supported(M, N, K, A, B)) return LSTM_ERR_UNSUPPORTED;
    return gemm_tc_bf16(p, kind, A, K, B, K, M, N, K, C, ldc, bias, 1, nullptr, s);
}

}  // namespace lstm
