// recurrent_cluster.cuh -- internals shared by the cluster recurrent kernels'
// translation units (forward: recurrent_cluster.cu; backward and the db / dpeep sums:
// recurrent_cluster_bwd.cu): constants, PTX helpers, the cell's vector helpers, and the
// launch configuration helpers.  Everything here has internal linkage.
#pragma once
#include <cooperative_groups.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "gemm.cuh"
#include "recurrent.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace lstm {

namespace {

constexpr int kCU = 32;        // units per CTA
constexpr int kCM = 128;       // gate rows per CTA (MMA M)
constexpr int kCT = 256;       // threads
constexpr int kSumChunks = 128; // row chunks of the db / dpeep sums
// bound on the teardown wait for a product still in flight after a timeout
// (an MMA takes microseconds; TMEM is freed only after it has completed)
constexpr unsigned long long kTeardownWaitNs = 1000000000ull;
// the thread that issues the TMA operand tiles: lane 0 of the last warp, which never issues
// MMAs (at most 4 issuing warps), so the tile loads do not delay the next product
constexpr int kTileIssuer = kCT - 32;
// forward: steps between the L2 prefetch of a step's gate tiles and their load into shared
// memory (the load itself is issued one step ahead; the rows mostly come from HBM).  The
// backward issues its tiles two microseconds before their use and takes no prefetch
// (measured slower with one)
constexpr int kTileAhead = 3;

__device__ __forceinline__ float sigm_c(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float tanh_c(float x)
{
    const float e = __expf(2.0f * fminf(fmaxf(x, -40.0f), 40.0f));
    return 1.0f - __fdividef(2.0f, e + 1.0f);
}

// byte offset of the 8-element chunk holding column k of row `row` in a
// K-major operand of `rows` rows: 64-column blocks, 128-byte rows, 16-byte
// chunks swizzled by (row mod 8)
__device__ __forceinline__ uint32_t sw_off(int row, int k, int rows)
{
    const int kb = k >> 6, ch = (k & 63) >> 3;
    return (uint32_t)kb * (uint32_t)rows * 128u + (uint32_t)row * 128u + (uint32_t)((ch ^ (row & 7)) << 4);
}

// same for a 4-element (8-byte) piece starting at column k (k a multiple of 4)
__device__ __forceinline__ uint32_t sw_off4(int row, int k, int rows)
{
    return sw_off(row, k, rows) + (uint32_t)((k & 7) << 1);
}

__device__ __forceinline__ uint32_t bf16x2(float lo_k, float hi_k)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_k), "f"(lo_k));
    return r;
}

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Bring rows [row0, row0 + n) of a row-major fp32 matrix (columns [col0,
// col0 + 32) only) into L2 ahead of use: one 128-byte line per row.
__device__ __forceinline__ void prefetch_rows(const float* m, int64_t ld, int row0, int n, int col0)
{
    for (int j = threadIdx.x; j < n; j += kCT) prefetch_l2(m + (int64_t)(row0 + j) * ld + col0);
}

// 4 fp32 values -> NP bf16 pieces, 2 per word: piece 0 = bf16(v), piece k = bf16 of what
// pieces 0..k-1 leave of v (each difference is exact in fp32)
template <int NP>
__device__ __forceinline__ void split4(const float (&v)[4], uint2 (&pc)[NP])
{
    float r[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        const uint32_t w0 = bf16x2(r[0], r[1]), w1 = bf16x2(r[2], r[3]);
        pc[k] = make_uint2(w0, w1);
        r[0] -= __uint_as_float(w0 << 16);
        r[1] -= __uint_as_float(w0 & 0xffff0000u);
        r[2] -= __uint_as_float(w1 << 16);
        r[3] -= __uint_as_float(w1 & 0xffff0000u);
    }
}


// U (2 or 4) consecutive fp32 values moved as one vector, and their NP bf16 pieces packed
// two per word (the cell's per-thread unit chunk)
template <int U> struct VecF;
template <> struct VecF<4> { using T = float4; };
template <> struct VecF<2> { using T = float2; };
template <int U> struct PkU;
template <> struct PkU<4> { using T = uint2; };
template <> struct PkU<2> { using T = uint32_t; };

template <int U>
__device__ __forceinline__ void ld_u(const float* p, float (&v)[U])
{
    if constexpr (U == 4) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
        const float2 x = *reinterpret_cast<const float2*>(p);
        v[0] = x.x; v[1] = x.y;
    }
}
template <int U>
__device__ __forceinline__ void ldg_u(const float* p, float (&v)[U])
{
    if constexpr (U == 4) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
        const float2 x = __ldg(reinterpret_cast<const float2*>(p));
        v[0] = x.x; v[1] = x.y;
    }
}
template <int U>
__device__ __forceinline__ void st_u(float* p, const float (&v)[U])
{
    if constexpr (U == 4) *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    else *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}
template <int U, int NP>
__device__ __forceinline__ void split_u(const float (&v)[U], typename PkU<U>::T (&pc)[NP])
{
    if constexpr (U == 4) {
        split4<NP>(v, pc);
    } else {
        float r0 = v[0], r1 = v[1];
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const uint32_t w0 = bf16x2(r0, r1);
            pc[k] = w0;
            r0 -= __uint_as_float(w0 << 16);
            r1 -= __uint_as_float(w0 & 0xffff0000u);
        }
    }
}
// byte offset of units [U q, U q + U) of row j in one 32-unit block of the 64-byte swizzled
// layout (16-byte chunks swizzled by (j >> 1) & 3)
template <int U>
__device__ __forceinline__ uint32_t sw64_off_u(int j, int q)
{
    const int start = U * q;
    return (uint32_t)j * 64u + (uint32_t)((((start >> 3) ^ ((j >> 1) & 3))) << 4) + (uint32_t)(start & 7) * 2u;
}

__device__ __forceinline__ void fence_proxy_async_cta()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_cluster()
{
    asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}

// Phase stamps of CTA 0 of each direction, in the grid kernels' slots:
// 0 = 1 = step start (this design waits at the end of a step), 2 = 5 = after
// the product reached shared memory, 3 = after the cell and the exchange,
// 4 = after the cluster barrier.
__device__ __forceinline__ void cstamp(const RecArgs& a, bool bwd, int dir, int rank, int s, int k0, int k1)
{
    if (threadIdx.x == 0 && a.trace && rank == 0 && s < a.trace_steps) {
        const long long now = clock64();
        long long* d = a.trace + (((size_t)(bwd ? 1 : 0) * a.ndir + dir) * a.trace_steps + s) * 8;
        d[k0] = now;
        d[k1] = now;
    }
}

// Split cluster barrier: arrive (release) now, wait (acquire) later; every
// thread of every CTA runs both, in the same order, once per phase.
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrival without memory ordering: for "this CTA has finished reading"
// signals whose reads are already complete (an MMA observed through its
// mbarrier, shared-memory loads whose values have been consumed); it does
// not wait for this thread's outstanding global loads and stores.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32 consecutive fp32 (or bf16) weights -> NP pieces of 16 bf16x2 words (as split4)
template <int NP>
__device__ __forceinline__ void split32(const float (&v)[32], uint32_t (&pc)[NP][16])
{
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        float r0 = v[2 * e], r1 = v[2 * e + 1];
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const uint32_t w = bf16x2(r0, r1);
            pc[k][e] = w;
            r0 -= __uint_as_float(w << 16);
            r1 -= __uint_as_float(w & 0xffff0000u);
        }
    }
}

// One K = 16 step of D += A B^T with both operands in NP bf16 pieces: A piece k at TMEM
// column a + k * ap, B piece k at descriptor b + k * bp.  NP = 3: the six piece products
// x_i y_j with i + j <= 2 (each of the others is below 2^-26 of x0 y0), smallest first.
template <int NP>
__device__ __forceinline__ void mma_k16(uint32_t d, uint32_t a, uint32_t ap, uint64_t b, uint64_t bp, uint32_t idesc,
                                        uint32_t acc)
{
    if (NP == 1) {
        tc::mma_bf16_ts(d, a, b, idesc, acc);
    } else {
        tc::mma_bf16_ts(d, a + ap, b + bp, idesc, acc);          // x1 y1
        tc::mma_bf16_ts(d, a + 2u * ap, b, idesc, 1u);            // x2 y0
        tc::mma_bf16_ts(d, a, b + 2u * bp, idesc, 1u);            // x0 y2
        tc::mma_bf16_ts(d, a + ap, b, idesc, 1u);                 // x1 y0
        tc::mma_bf16_ts(d, a, b + bp, idesc, 1u);                 // x0 y1
        tc::mma_bf16_ts(d, a, b, idesc, 1u);                      // x0 y0
    }
}

// One chain of the forward product: k-steps i = 4J + ch + v*NCH (v < 4/NCH)
// over the 64-column blocks J of the B operand.  A (R slice) in TMEM from
// column a0 (pieces ap apart), B in shared memory from descriptor b0 (pieces
// bp apart), `bstep` = descriptor units between B blocks.
template <int NCH, int NP>
__device__ __forceinline__ void issue_chain(uint32_t d, uint32_t a0, uint32_t ap, uint64_t b0, uint64_t bp,
                                            uint32_t bstep, int nks, int ch, uint32_t idesc)
{
    uint32_t acc = 0u;
    for (int J = 0; 4 * J < nks; ++J) {
#pragma unroll
        for (int v = 0; v < 4 / NCH; ++v) {
            const int w = ch + v * NCH;
            const int i = 4 * J + w;
            if (i < nks) {
                const uint64_t bo = (uint64_t)(J * bstep + 2 * w);      // 32 bytes per k-step of 16
                const uint32_t ac = (uint32_t)(i * 8);                  // 8 columns per k-step of 16
                mma_k16<NP>(d, a0 + ac, ap, b0 + bo, bp, idesc, acc);
                acc = 1u;
            }
        }
    }
}

// The same chain over a B operand in 32-column blocks (64-byte swizzle, two
// k-steps of 16 per block).
template <int NCH, int NP>
__device__ __forceinline__ void issue_chain32(uint32_t d, uint32_t a0, uint32_t ap, uint64_t b0, uint64_t bp,
                                              uint32_t bstep, int nks, int ch, uint32_t idesc)
{
    uint32_t acc = 0u;
#pragma unroll 2
    for (int i = ch; i < nks; i += NCH) {
        const uint64_t bo = (uint64_t)((uint32_t)(i >> 1) * bstep + (uint32_t)(i & 1) * 2u);
        const uint32_t ac = (uint32_t)(i * 8);
        mma_k16<NP>(d, a0 + ac, ap, b0 + bo, bp, idesc, acc);
        acc = 1u;
    }
}

// The same with a compile-time k-step count, fully unrolled (the issuing
// thread's own instruction stream bounds the issue rate of small MMAs).
template <int NCH, int NKS, int KPB, int NP>
__device__ __forceinline__ void issue_chain_fixed(uint32_t d, uint32_t a0, uint32_t ap, uint64_t b0, uint64_t bp,
                                                  uint32_t bstep, int ch, uint32_t idesc)
{
#pragma unroll
    for (int jj = 0; jj < NKS / NCH; ++jj) {
        const int i = ch + jj * NCH;
        const uint64_t bo = (uint64_t)((uint32_t)(i / KPB) * bstep + (uint32_t)(i % KPB) * 2u);
        const uint32_t ac = (uint32_t)(i * 8);
        mma_k16<NP>(d, a0 + ac, ap, b0 + bo, bp, idesc, jj == 0 ? 0u : 1u);
    }
}

template <int NP>
__device__ __forceinline__ void issue_chains32(int nch, uint32_t d, uint32_t a0, uint32_t ap, uint64_t b0,
                                               uint64_t bp, uint32_t bstep, int nks, int ch, uint32_t idesc)
{
    if (nch == 4 && nks == 16) issue_chain_fixed<4, 16, 2, NP>(d, a0, ap, b0, bp, bstep, ch, idesc);
    else if (nch == 4 && nks == 32) issue_chain_fixed<4, 32, 2, NP>(d, a0, ap, b0, bp, bstep, ch, idesc);
    else if (nch == 4 && nks == 8) issue_chain_fixed<4, 8, 2, NP>(d, a0, ap, b0, bp, bstep, ch, idesc);
    else if (nch == 2 && nks == 16) issue_chain_fixed<2, 16, 2, NP>(d, a0, ap, b0, bp, bstep, ch, idesc);
    else if (nch == 4) issue_chain32<4, NP>(d, a0, ap, b0, bp, bstep, nks, ch, idesc);
    else if (nch == 2) issue_chain32<2, NP>(d, a0, ap, b0, bp, bstep, nks, ch, idesc);
    else issue_chain32<1, NP>(d, a0, ap, b0, bp, bstep, nks, ch, idesc);
}

// Shared-memory descriptor of a K-major operand in the 64-byte swizzled
// layout: rows of 64 bytes (32 bf16), groups of 8 rows 512 bytes apart, the
// 16-byte chunk c of row r stored at chunk c ^ ((r >> 1) & 3).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1 << 16;                           // leading byte offset (unused for this layout)
    d |= (uint64_t)(512u >> 4) << 32;                 // stride byte offset: 8 rows x 64 B
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)4 << 61;                           // 64-byte swizzle
    return d;
}

// byte offset of units [4q, 4q + 4) (q < 8) of row j in one 32-unit block of
// the 64-byte swizzled layout
__device__ __forceinline__ uint32_t sw64_off4(int j, int q)
{
    return (uint32_t)j * 64u + (uint32_t)((((q >> 1) ^ ((j >> 1) & 3))) << 4) + (uint32_t)(q & 1) * 8u;
}

__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Bulk copy of `bytes` from this CTA's shared memory into a peer's
// (shared::cluster address), completing on the peer's mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                             uint32_t mbar_cluster)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst_cluster), "r"(tc::smem_u32(src)), "r"(bytes), "r"(mbar_cluster)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk copies except the newest group have finished reading their source
__device__ __forceinline__ void bulk_wait_read_all_but_one()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// this thread's bulk copies have all finished reading their source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk copies have completed (destination written)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Sum of the accumulator chains at columns col0 + ch * stride (ch < nch <= 4)
// for 16 consecutive columns of this warp's 32 lanes: the loads are issued
// together and waited for once.
__device__ __forceinline__ void tmem_sum_chains(uint32_t taddr0, uint32_t stride, int nch, float (&v)[16])
{
    uint32_t r[4][16];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        if (ch < nch) tc::tmem_ld_32x32b_x16(taddr0 + (uint32_t)ch * stride, r[ch]);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[0][e]);
#pragma unroll
    for (int ch = 1; ch < 4; ++ch)
        if (ch < nch) {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] += __uint_as_float(r[ch][e]);
        }
}

template <int NP>
__device__ __forceinline__ void issue_chains(int nch, uint32_t d, uint32_t a0, uint32_t ap, uint64_t b0,
                                             uint64_t bp, uint32_t bstep, int nks, int ch, uint32_t idesc)
{
    if (nch == 4) issue_chain<4, NP>(d, a0, ap, b0, bp, bstep, nks, ch, idesc);
    else if (nch == 2) issue_chain<2, NP>(d, a0, ap, b0, bp, bstep, nks, ch, idesc);
    else issue_chain<1, NP>(d, a0, ap, b0, bp, bstep, nks, ch, idesc);
}


static inline size_t al(size_t v, size_t a) { return (v + a - 1) / a * a; }

static inline uint32_t pow2_cols(int need)
{
    uint32_t cols = 32;
    while (cols < (uint32_t)need) cols <<= 1;
    return cols;
}

// Dynamic shared memory for a cluster kernel that allocates `tcols` TMEM
// columns per CTA: at least enough that no more CTAs fit on one SM than
// their columns fit in its 512 (a CTA whose allocation waited for another
// CTA of the same cluster would never see it leave).
static inline size_t tmem_safe_smem(const Plan& p, size_t smem, uint32_t tcols)
{
    int per_sm = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p.device) != cudaSuccess)
        return 0;
    const int fit = 512 / (int)tcols;                 // CTAs whose columns fit together
    if (fit >= 2048 / kCT) return smem;               // the thread limit already caps residency
    const size_t reserved = 1024;                     // per-CTA shared memory reserved by the system
    const size_t need = (size_t)per_sm / (size_t)(fit + 1) - reserved + 64;
    return std::max(smem, need);
}

// True when at least one cluster of `G` CTAs with `smem` bytes can be resident.
static inline bool cluster_schedulable(const Plan& p, const void* fn, int G, size_t smem)
{
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device) != cudaSuccess) return false;
    if (smem > (size_t)optin) return false;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (G > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return clusters >= 1;
}

static inline int max_active_rows(const Plan& p)
{
    int bmax = 0;
    for (int t = 0; t < p.T; ++t) bmax = std::max(bmax, p.h_bs[t]);
    return bmax;
}

// Sequence groups: the sorted slots are cut into ng contiguous groups of S slots, one cluster
// per (direction, group).  S is the smallest multiple of 8 (at least 8) for which every
// cluster has an SM of its own, or the plan's forced size; one group when S covers the batch.
// False when a group would need more than 128 rows (the cell's row items).
static inline bool choose_groups(const Plan& p, int G, int ndir, int* S_out, int* ng_out)
{
    int S;
    if (p.forced_group_rows > 0) {
        S = p.forced_group_rows;
    } else {
        const int maxg = std::max(1, p.num_sms / (G * ndir));
        S = std::max(8, (ceil_div(p.B, maxg) + 7) / 8 * 8);
    }
    if (S >= p.B) S = p.B;
    if (S > 128) return false;
    *S_out = S;
    *ng_out = ceil_div(p.B, S);
    return true;
}

// Units a thread takes in the cell: 2 (twice the threads busy) or 4.  Measured: the backward
// cell gains from 2 up to 16 rows a group (3.68 -> 3.47 us a step at 16 rows, 3.42 -> 3.08 at
// 8); the forward gains at 8 rows (3.03 -> 2.95) and loses at 16 (2.45 -> 2.52).
static inline int cell_units(int group_rows, bool backward) { return group_rows <= (backward ? 16 : 8) ? 2 : 4; }

// One cluster of c.G CTAs per (direction, sequence group).
static inline lstm_status cluster_launch(const RecConfig& c, const void* fn, void** args, int ndir, cudaStream_t s)
{
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem) != cudaSuccess)
        return LSTM_ERR_CUDA;
    if (c.G > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return LSTM_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(c.G * ndir * c.ngroups);
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c.G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) { cudaGetLastError(); return LSTM_ERR_UNSUPPORTED; }
    return LSTM_OK;
}

}  // namespace
}  // namespace lstm
