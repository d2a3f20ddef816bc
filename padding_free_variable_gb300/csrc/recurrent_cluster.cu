// recurrent_cluster.cu -- cluster-resident recurrent kernels (forward and BPTT).
//
// The same recurrence as lstm_rec_fwd_kernel ("Single Stream Parallelization
// of Generalized LSTM-Like RNNs on a GPU", Sec. 3: one sequential step per
// frame, the delayed connection R h_{t-1} then the cell), laid out for
// thread-block clusters when one direction's R fits in a cluster:
//
//  * sequence groups: the sorted slots are cut into contiguous groups of S
//    slots, and every (direction, group) pair is one cluster of G = H/32
//    CTAs.  Sequences are independent, so the clusters never communicate;
//    a group runs only as many steps as its longest sequence, and each
//    cluster moves only its own rows between its CTAs every step;
//  * CTA c of a cluster owns units [32c, 32c+32) and their 128 gate rows of
//    R, resident in TENSOR MEMORY as the MMA's A operand.  bf16 weights are
//    one bf16 piece; fp32 weights (and the fp32 B operands h_{t-1} or the
//    gate errors) are three bf16 pieces v0 + v1 + v2 (v0 = bf16(v), each
//    further piece the bf16 rounding of what the earlier ones leave), and
//    each K = 16 step issues the six piece products above 2^-24 of the
//    leading one, so the product keeps fp32 accuracy.  With A in tensor
//    memory an M=128, N<=32, K=16 MMA reads only its B tile from shared
//    memory (measured on GB300: ~19 cycles per MMA with 4 issuing warps,
//    against ~43 with A in shared memory);
//  * per step up to 4 warps each issue one chain of tcgen05.mma into their
//    own accumulator columns (chains summed at read-out); N is the group's
//    active rows rounded up to 16;
//  * the cell runs on the summed chains, and each CTA sends its h_t (bf16
//    pieces, swizzled) to every peer of its cluster.  Two exchanges:
//    BULK -- the operand is double-buffered per step parity; each CTA stages
//    its h_t and pushes it with one cp.async.bulk per peer and piece into the
//    peer's buffer of the other parity, completing on the peer's mbarrier of
//    that parity.  The data's arrival is the step's synchronisation: no
//    cluster barrier runs in the step loop.  Otherwise (the double buffers do
//    not fit): one operand buffer written with DSMEM stores between the two
//    halves of a split cluster barrier.
// Every wait but the hardware cluster barrier (which every CTA of a cluster
// reaches by construction) is bounded, and a timeout is recorded in the
// plan's status word.
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

}  // namespace

// Shared memory (RecArgs offsets): off_acc = accs, off_state = cell states,
// off_contrib = B operand (h_{t-1}, its NP pieces), off_sums = mbarriers, TMEM
// slot, failure flag and the group's step count, off_tab = tables, off_peep =
// peepholes.  Tensor memory: accumulator chains in columns [0, chains * NBM),
// the R slice (NP pieces of H/2 columns each) from column tm_acol.
//
// The cluster serves sorted slots [j0, j0 + S) of direction `dir`: its step t
// has rows off[t] + j0 .. + n - 1, n = min(max(bs[t] - j0, 0), S), and it runs
// the Tg steps with n > 0 (Tg = the group's longest length).
//
// Two exchanges of h_t between the CTAs of a cluster:
//  * BULK: the operand is double-buffered per step parity, in 32-unit blocks
//    of the 64-byte swizzled layout, so that one CTA's units of all rows are
//    one contiguous block.  Each CTA stages its h_t there in its own shared
//    memory and copies it with one cp.async.bulk per peer and piece, which
//    completes on the peer's mbarrier of that parity: the arrival of the
//    data is the step's synchronisation, and no cluster barrier runs inside
//    the step loop.  A peer can only send h_{t+1} into buffer (s & 1) after
//    it received this CTA's h_t, which is sent after this CTA's product of
//    step s has read that buffer; each mbarrier is re-armed for its next use
//    before this CTA's copies of the step go out, so no byte can arrive at an
//    unarmed barrier.
//  * otherwise (the double buffer does not fit): one operand buffer, written
//    by the peers with plain DSMEM stores between two halves of a split
//    cluster barrier.
//
// With a.tma_pre the gate pre-activations of a step (4 gates x NBM rows x this
// CTA's 32 units, fp32) arrive in shared memory by four TMA tile loads, issued
// by one thread right after the previous step's cell has read the tile: the
// product's window stays free of the 256 threads' global loads (measured to
// delay the MMAs' completion by ~0.8 us).
template <int NP, bool BULK>
__global__ void __launch_bounds__(kCT, 1) lstm_rec_fwd_cluster_kernel(RecArgs a, const __grid_constant__ CUtensorMap pre_map)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cl = cg::this_cluster();
    const int G = a.G;
    const int rank = (int)cl.block_rank();
    const int ng = a.ngroups;
    const int dir = (int)(blockIdx.x / G) / ng, grp = (int)(blockIdx.x / G) % ng;
    const int S = a.grp_rows, j0 = grp * S;           // this cluster's sorted slots [j0, j0 + S)
    const int srank = grp == 0 ? rank : -1;           // the phase stamps come from group 0
    const int H = a.H, T = a.T, NBM = a.JC;          // JC carries the operand buffer rows (multiple of 16)
    const int KB = (H + 63) / 64;
    const int u0 = rank * kCU;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const int nch = a.tm_chains;
    float* accs = reinterpret_cast<float*>(base + a.off_acc);        // [NBM][128]
    float* cst = reinterpret_cast<float*>(base + a.off_state);       // [S][32]
    // B operand: BULK [2 parity][NP][G][NBM][64 B], else [NP][KB][NBM][128 B]
    uint8_t* Bb = base + a.off_contrib;
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(base + a.off_sums);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
    int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
    uint64_t* full_bar = mma_bar + 2;                                // BULK: [2] operand arrival per parity
    uint64_t* pre_bar = mma_bar + 4;                                 // tma_pre: arrival of a step's tile
    int* s_tg = reinterpret_cast<int*>(mma_bar + 6);                 // the group's step count
    float* pre_tile = reinterpret_cast<float*>(base + a.off_red);    // tma_pre: [4 gates][NBM][32]
    const bool tma_pre = a.tma_pre != 0;
    float* peep_s = reinterpret_cast<float*>(base + a.off_peep);     // [3][32]
    int* s_bs = reinterpret_cast<int*>(base + a.off_tab);            // [T] the group's active rows
    int* s_off = s_bs + T;                                           // [T+1] the group's first row
    int* s_len = s_off + T + 1;                                      // [S] lengths of the group's slots
    uint8_t* stage = base + a.off_h;                                 // BULK: [2 parity][NP][NBM][64 B]
    const size_t bsz = BULK ? (size_t)G * NBM * 64 : (size_t)KB * NBM * 128;   // bytes of one B piece
    const size_t ssz = (size_t)NBM * 64;                             // bytes of one staged h piece
    auto Bop = [&](int parity, int piece) -> uint8_t* {
        return Bb + (BULK ? (size_t)parity * NP * bsz : 0) + (size_t)piece * bsz;
    };
    auto Stg = [&](int parity, int piece) -> uint8_t* { return stage + (size_t)(parity * NP + piece) * ssz; };
    int Tg = 0;
    // rows of h of step s2 - 1 that step s2 reads: the rows continuing into step s2.  Rows past
    // them are never read going forward (finished sequences) and were never written going
    // backward (sequences not yet started: still zero from the set-up)
    auto step_rows = [&](int s2) -> int {
        const int tp = dir == 0 ? s2 - 1 : Tg - s2, tn = dir == 0 ? s2 : Tg - 1 - s2;
        return min(s_bs[tp], s_bs[tn]);
    };
    // bytes a CTA receives for step s2: those rows from every other CTA (its own it writes itself)
    auto step_bytes = [&](int s2) -> uint32_t {
        return (uint32_t)(G - 1) * (uint32_t)NP * (uint32_t)step_rows(s2) * 64u;
    };
    const uint32_t tcols = (uint32_t)a.Umax;                         // Umax carries the TMEM columns
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up: operand zeroed, the group's tables, barriers, tensor memory
    for (size_t i = threadIdx.x; i < (BULK ? 2 : 1) * NP * bsz / 16; i += kCT)
        reinterpret_cast<uint4*>(Bb)[i] = make_uint4(0, 0, 0, 0);
    if (BULK)
        for (size_t i = threadIdx.x; i < 2 * NP * ssz / 16; i += kCT) reinterpret_cast<uint4*>(stage)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) *s_tg = 0;
    __syncthreads();
    // bs is non-increasing in t, so the group's steps are t < Tg, Tg = the one t whose
    // successor has no row of the group
    for (int i = threadIdx.x; i < T; i += kCT) {
        const int n = min(max(a.bs[i] - j0, 0), S);
        s_bs[i] = n;
        if (n > 0 && (i + 1 == T || a.bs[i + 1] <= j0)) *s_tg = i + 1;
    }
    for (int i = threadIdx.x; i <= T; i += kCT) s_off[i] = a.off[i] + j0;
    for (int i = threadIdx.x; i < S; i += kCT) s_len[i] = j0 + i < a.B ? a.slot_len[j0 + i] : 0;
    for (int i = threadIdx.x; i < 3 * kCU; i += kCT) {
        const int q = i / kCU, uu = i - q * kCU;
        peep_s[i] = a.peep[(size_t)dir * 3 * H + q * H + u0 + uu];
    }
    __syncthreads();
    Tg = *s_tg;
    if (threadIdx.x == 0) {
        tc::mbar_init(mma_bar, (uint32_t)nch);
        *s_fail = 0;
        if (BULK) {
            tc::mbar_init(&full_bar[0], 1);
            tc::mbar_init(&full_bar[1], 1);
        }
        if (tma_pre) tc::mbar_init(pre_bar, 1);
        tc::fence_mbar_init();
        // the operand of step 1 (parity 1) is armed before the cluster barrier below,
        // i.e. before any peer can send
        if (BULK && Tg > 1) tc::mbar_arrive_expect_tx(&full_bar[1], step_bytes(1));
    }
    if (threadIdx.x < 32) {
        tc::tmem_alloc(tmem_slot, tcols);
        tc::tmem_relinquish();
    }
    fence_proxy_async_cta();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a0 = tmem + (uint32_t)a.tm_acol, ap = (uint32_t)(H / 2);
    // R slice -> tensor memory: lane 32g + uu holds gate row g of unit u0 + uu (the MMA's row
    // order), column c of the slice holds k = 2c and 2c + 1; warps g and g + 4 share the lanes
    // of gate g and take alternate 32-wide k chunks
    {
        const int g = warp & 3;
        const size_t grow = (size_t)dir * 4 * H * H + (size_t)(g * H + u0 + lane) * H;
        const uint32_t lanes = (uint32_t)(32 * g) << 16;
        for (int cc = warp >> 2; cc < H / 32; cc += 2) {
            float v[32];
            if (NP > 1) {
                const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.R) + grow + 32 * cc);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 x = __ldg(src + e);
                    v[4 * e] = x.x; v[4 * e + 1] = x.y; v[4 * e + 2] = x.z; v[4 * e + 3] = x.w;
                }
            } else {
                const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(a.R) + grow + 32 * cc;
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __bfloat162float(src[e]);
            }
            uint32_t pc[NP][16];
            split32<NP>(v, pc);
#pragma unroll
            for (int k = 0; k < NP; ++k) tc::tmem_st_32x32b_x16(a0 + (uint32_t)k * ap + lanes + (uint32_t)(16 * cc), pc[k]);
        }
        tc::tmem_wait_st();
    }
    if (a.h_n) {
        for (int idx = threadIdx.x; idx < S * kCU; idx += kCT) {
            const int j = idx / kCU, uu = idx - j * kCU;
            if (j0 + j < a.B && s_len[j] == 0) {        // an empty sequence ends in its initial state
                const size_t o = ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uu;
                a.h_n[o] = a.h0 ? a.h0[o] : 0.f;
                if (a.c_n) a.c_n[o] = a.c0 ? a.c0[o] : 0.f;
            }
        }
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    // tma_pre: the four gate tiles of step s2 (rows from off[t2], NBM of them; rows past the
    // packed rows read 0), one thread, completing on pre_bar
    auto issue_pre = [&](int s2, bool fence) {
        const int t2 = dir == 0 ? s2 : Tg - 1 - s2;
        if (fence) fence_proxy_async_cta();
        tc::mbar_arrive_expect_tx(pre_bar, (uint32_t)(4 * NBM * kCU * 4));
#pragma unroll
        for (int g = 0; g < 4; ++g)
            tc::tma_load_2d(pre_tile + (size_t)g * NBM * kCU, &pre_map, pre_bar, dir * 4 * H + g * H + u0, s_off[t2]);
    };
    int last_tile = -1;                   // tile issuer: the last step whose tile was issued
    if (tma_pre && threadIdx.x == kTileIssuer && Tg > 0) { issue_pre(0, true); last_tile = 0; }
    cl.sync();     // every CTA of the cluster is resident before any remote write

    const int jq = threadIdx.x >> 3, q8 = threadIdx.x & 7;          // cell item: row jq (+32k), units q8*4..+4
    const int nks = (H + 15) / 16;                                   // MMA k-steps
    float pk[3][4];                                                  // peepholes i, f, o of units q8*4..+4
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[q][e] = peep_s[q * kCU + q8 * 4 + e];
    const uint32_t bstep = (uint32_t)(NBM * (BULK ? 64 : 128)) >> 4;  // descriptor units between B blocks
    bool failed = false;                  // CTA-uniform: an MMA completion wait timed out
    bool pre_ok_prev = true;              // this thread's wait for the previous step's tile
    for (int s = 0; s < Tg; ++s) {
        const int t = dir == 0 ? s : Tg - 1 - s;
        const int n = s_bs[t];
        const int rowbase = s_off[t];
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < Tg ? s_bs[t + 1] : 0);
        const int NBs = (n + 15) & ~15;
        const int par = BULK ? (s & 1) : 0;
        bool arrived = true;          // this step's operand (and the previous step's tile) arrived
        if (BULK) {
            cstamp(a, false, dir, srank, s, 0, 0);
            // h_{t-1} of every peer has arrived in this step's operand
            if (s > 0 && !failed)
                arrived = tc::mbar_wait(&full_bar[par], (uint32_t)(((s - 1) >> 1) & 1), a.wait_limit_ns);
        } else {
            if (s > 0) {
                cluster_wait();    // h_{t-1} of every peer is in this CTA's operand
                // every thread of this CTA arrived after its cell: the tile is free
                if (tma_pre && threadIdx.x == kTileIssuer && !failed) { issue_pre(s, true); last_tile = s; }
                cstamp(a, false, dir, srank, s - 1, 4, 4);
            }
            cstamp(a, false, dir, srank, s, 0, 0);
        }
        // D[gate rows][rows] = R_slice x h_{t-1}^T: chain ch is issued by warp ch into its own
        // accumulator, so the chains overlap
        if (lane == 0 && warp < nch && !failed) {
            fence_proxy_async_cta();
            tc::tc_fence_after_sync();
            cstamp(a, false, dir, srank, s, 1, 1);
            const uint32_t idesc = tc::idesc_bf16_f32(kCM, NBs);
            const uint64_t bp = (uint64_t)(bsz >> 4);                  // descriptor units between B pieces
            if (BULK) {
                const uint64_t db0 = sdesc_sw64(tc::smem_u32(Bop(par, 0)));
                issue_chains32<NP>(nch, tmem + (uint32_t)(warp * NBM), a0, ap, db0, bp, bstep, nks, warp, idesc);
            } else {
                const uint64_t db0 = tc::sdesc_sw128(tc::smem_u32(Bop(0, 0)));
                issue_chains<NP>(nch, tmem + (uint32_t)(warp * NBM), a0, ap, db0, bp, bstep, nks, warp, idesc);
            }
            if (!(s == 0 && dir == 0 && grp == 0 && rank == a.debug_skip_cta)) tc::mma_commit(mma_bar);   // test hook
        }
        if (warp < nch) __syncwarp();     // the issuing lane's warp does not poll while it issues
        cstamp(a, false, dir, srank, s, 6, 6);
        // meanwhile (without tma_pre): the cell items' own operands (gate pre-activations),
        // rows jq and jq + 32
        float pre[2][4][4];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int j = jq + it * 32;
            if (!tma_pre && j < n) {
                const float* gr = a.ga + (size_t)(rowbase + j) * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H);
                    pre[it][g][0] = x.x; pre[it][g][1] = x.y; pre[it][g][2] = x.z; pre[it][g][3] = x.w;
                }
            }
        }
        if (!tma_pre && s + 1 < Tg) {   // next step's own rows into L2 (4 gate blocks of this CTA's units)
            const int t2 = dir == 0 ? s + 1 : Tg - 2 - s;
            for (int g = 0; g < 4; ++g)
                prefetch_rows(a.ga, nd4H, s_off[t2], s_bs[t2], dir * 4 * H + g * H + u0);
        }
        // A timeout (of the product, or of the operand's arrival) becomes a CTA-uniform decision
        // at the barrier after the read-out: from then on the CTA issues no product, waits for
        // no operand, re-arms nothing and sends nothing (so no barrier is armed twice and
        // unmatched bytes stay within two steps), and the teardown waits for the product in
        // flight before freeing tensor memory.  The read-out of the failing step itself may see
        // partial sums; the status word marks the results as invalid.
        const bool ok = failed ? true : tc::mbar_wait(mma_bar, (uint32_t)(s & 1), a.wait_limit_ns);
        arrived = arrived && pre_ok_prev;
        if ((!ok || !arrived) && !failed) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, (ok ? 0x60000u : 0x40000u) | (unsigned)s);
            *s_fail = 1 + s;
        }
        cstamp(a, false, dir, srank, s, 7, 7);
        tc::tc_fence_after_sync();
        if (!BULK) cluster_arrive_relaxed();   // this CTA's product has read its operand: peers may overwrite it
        // accumulators -> shared: warp (quarter q = gate, half) reads lanes 32q.. in 16-column blocks
        if (!failed) {
            const int q = warp & 3, half = warp >> 2;
            for (int c0 = half * 16; c0 < NBs; c0 += 32) {
                float v[16];
                tmem_sum_chains(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, (uint32_t)NBM, nch, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) accs[(size_t)(c0 + e) * kCM + q * 32 + lane] = v[e];
            }
        }
        tc::tc_fence_before_sync();
        if (__syncthreads_or(!ok || !arrived)) failed = true;
        // BULK: re-arm this parity for step s + 2 before this CTA's h_t goes out (a peer
        // needs h_t before it can send h_{t+1})
        if (BULK && threadIdx.x == 0 && !failed && s + 2 < Tg)
            tc::mbar_arrive_expect_tx(&full_bar[par], step_bytes(s + 2));
        cstamp(a, false, dir, srank, s, 2, 2);
        // cell: row j, units u0 + q8*4 .. +4; h_t kept (split) for the exchange.  Without the bulk
        // exchange the global outputs of rows jq and jq + 32 are written after the exchange's
        // barrier arrival, so that the arrival (a release) does not wait for them
        bool pre_ok = true;
        if (tma_pre && !failed) pre_ok = tc::mbar_wait(pre_bar, (uint32_t)(s & 1), a.wait_limit_ns);
        if (!pre_ok && !failed) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, 0x70000u | (unsigned)s);
            *s_fail = 1 + s;
        }
        uint2 xp[4][NP];
        float og_[2][4][4], oc_[2][4], oh_[2][4];
        auto store_outputs = [&](int j, const float (&gg)[4][4], const float (&cv)[4], const float (&hv)[4],
                                 uint2 hi) {
            const int row = rowbase + j;
            const int len = s_len[j];
            float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<float4*>(gr + g * H) = make_float4(gg[g][0], gg[g][1], gg[g][2], gg[g][3]);
            const size_t yo = (size_t)row * ndH + dir * H + u0 + q8 * 4;
            *reinterpret_cast<float4*>(a.cbuf + yo) = make_float4(cv[0], cv[1], cv[2], cv[3]);
            *reinterpret_cast<float4*>(a.y + yo) = make_float4(hv[0], hv[1], hv[2], hv[3]);
            if (a.y_lo) *reinterpret_cast<uint2*>(a.y_lo + yo) = hi;
            if (a.h_n && ((dir == 0 && t == len - 1) || (dir == 1 && t == 0 && len > 0))) {
                const size_t o = ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + q8 * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a.h_n[o + e] = hv[e];
                    if (a.c_n) a.c_n[o + e] = cv[e];
                }
            }
        };
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int j = jq + it * 32;
            if (j >= n) continue;
            const int len = s_len[j];
            float pv[4][4];
            if (tma_pre) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(pre_tile + ((size_t)g * NBM + j) * kCU + q8 * 4);
                    pv[g][0] = x.x; pv[g][1] = x.y; pv[g][2] = x.z; pv[g][3] = x.w;
                }
            } else if (it < 2) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < 4; ++e) pv[g][e] = it == 0 ? pre[0][g][e] : pre[1][g][e];
            } else {
                const float* gr = a.ga + (size_t)(rowbase + j) * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H);
                    pv[g][0] = x.x; pv[g][1] = x.y; pv[g][2] = x.z; pv[g][3] = x.w;
                }
            }
            float hv[4], cv[4], gg[4][4];
            // the row's products of the 4 gates and its previous cell states, 4 units at a time
            float acv[4][4], cpv[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 x = *reinterpret_cast<const float4*>(accs + (size_t)j * kCM + g * kCU + q8 * 4);
                acv[g][0] = x.x; acv[g][1] = x.y; acv[g][2] = x.z; acv[g][3] = x.w;
            }
            {
                const float4 x = j < n_prev ? *reinterpret_cast<const float4*>(cst + j * kCU + q8 * 4)
                                 : a.c0 ? __ldg(reinterpret_cast<const float4*>(
                                              a.c0 + ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + q8 * 4))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                cpv[0] = x.x; cpv[1] = x.y; cpv[2] = x.z; cpv[3] = x.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float cp = cpv[e];
                const float ig = sigm_c(pv[0][e] + acv[0][e] + pk[0][e] * cp);
                const float fg = sigm_c(pv[1][e] + acv[1][e] + pk[1][e] * cp);
                const float zg = tanh_c(pv[2][e] + acv[2][e]);
                float c = fg * cp + ig * zg;
                const float og = sigm_c(pv[3][e] + acv[3][e] + pk[2][e] * c);
                float h = og * tanh_c(c);
                if (a.padded && t >= len) { c = 0.f; h = 0.f; }
                gg[0][e] = ig; gg[1][e] = fg; gg[2][e] = zg; gg[3][e] = og; cv[e] = c; hv[e] = h;
            }
            *reinterpret_cast<float4*>(cst + j * kCU + q8 * 4) = make_float4(cv[0], cv[1], cv[2], cv[3]);
            split4<NP>(hv, xp[it]);
            if (!BULK && it < 2) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) og_[it][g][e] = gg[g][e];
                    oc_[it][e] = cv[e];
                    oh_[it][e] = hv[e];
                }
            } else {
                store_outputs(j, gg, cv, hv, xp[it][0]);
            }
        }
        cstamp(a, false, dir, srank, s, 5, 5);
        if (BULK) {
            // h_t (rows [0, NBs)) staged in this CTA's 32-unit block, then one bulk copy per peer
            // and half into that peer's operand of step s + 1
            if (s + 1 < Tg) {
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int j = jq + it * 32;
                    if (j >= n) continue;
                    const uint32_t o = sw64_off4(j, q8);
                    // this CTA's own block of the next step's operand is written in place
                    const size_t ob = (size_t)rank * NBM * 64 + o;
#pragma unroll
                    for (int k = 0; k < NP; ++k) {
                        *reinterpret_cast<uint2*>(Stg(par, k) + o) = xp[it][k];
                        *reinterpret_cast<uint2*>(Bop(par ^ 1, k) + ob) = xp[it][k];
                    }
                }
            }
            fence_proxy_async_cta();
            __syncthreads();
            // lane 0 of warp w sends to peers w, w + 8 (copies issued by one warp's lanes serialise)
            const bool sender = lane == 0 && warp < G;
            if (s + 1 < Tg && sender && !failed) {
                const uint32_t nxt = (uint32_t)(par ^ 1);
                const uint32_t bytes = (uint32_t)step_rows(s + 1) * 64u;
                for (int p2 = warp; p2 < G; p2 += kCT / 32) {
                    if (p2 == (int)rank || bytes == 0) continue;
                    const uint32_t bar = mapa_u32(tc::smem_u32(&full_bar[nxt]), (uint32_t)p2);
#pragma unroll
                    for (int k = 0; k < NP; ++k)
                        bulk_to_peer(mapa_u32(tc::smem_u32(Bop(nxt, k) + (size_t)rank * NBM * 64), (uint32_t)p2),
                                     Stg(par, k), bytes, bar);
                }
                bulk_commit();
            }
            cstamp(a, false, dir, srank, s, 4, 4);
            if (tma_pre && threadIdx.x == kTileIssuer && s + 1 < Tg && !failed) {   // the tile has been read
                issue_pre(s + 1, false);
                last_tile = s + 1;
            }
            if (s + 1 < Tg && sender && !failed) bulk_wait_read_all_but_one();   // step s - 1's staging
        } else {
            cluster_wait();        // every peer's product of this step is done with its operand
            // h_t into every peer's operand of the next step (row j, columns u0 + q8*4 ..)
            if (s + 1 < Tg) {
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int j = jq + it * 32;
                    if (j >= n) continue;
                    const uint32_t o = sw_off4(j, u0 + q8 * 4, NBM);
                    for (int p2 = 0; p2 < G; ++p2)
#pragma unroll
                        for (int k = 0; k < NP; ++k)
                            *reinterpret_cast<uint2*>(cl.map_shared_rank(Bop(0, k) + o, p2)) = xp[it][k];
                }
            }
            fence_proxy_async_cluster();
            cluster_arrive();      // release: this CTA's h_t is in every peer's operand
        }
        if (!BULK) {
#pragma unroll
            for (int it = 0; it < 2; ++it)
                if (jq + it * 32 < n) store_outputs(jq + it * 32, og_[it], oc_[it], oh_[it], xp[it][0]);
        }
        pre_ok_prev = pre_ok;
        cstamp(a, false, dir, srank, s, 3, 3);
    }
    // after a timeout the last tile issued may not have been waited for: no load may still be
    // writing this CTA's shared memory when it exits (bounded wait)
    if (tma_pre && threadIdx.x == kTileIssuer && last_tile >= 0)
        tc::mbar_wait(pre_bar, (uint32_t)(last_tile & 1), kTeardownWaitNs);
    if (BULK) {
        if (lane == 0 && warp < G) bulk_wait_all();   // no copy of this CTA is still in flight
        cl.sync();                              // nor one into it: every CTA has passed its last wait
    } else if (Tg > 0) {
        cluster_wait();            // the last step's arrival
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        __syncwarp();
        tc::tc_fence_after_sync();
        if (failed) tc::mbar_wait(mma_bar, (uint32_t)((*s_fail - 1) & 1), kTeardownWaitNs);
        tc::tmem_dealloc(tmem, tcols);
    }
}

// ------------------------------------------------------------------------- backward
//
// BPTT of the same recurrence ("Single Stream Parallelization...", Sec. 2) in
// the same cluster layout.  The error reaching h_t through R is
// R^T da_{t+1}; CTA c holds its 128 gate rows of R (as R^T, in tensor memory)
// and the gate errors it computes for them, so it forms the partial product
// P_c = R_c^T da_c for every unit on the tensor cores, and sends the part of
// P_c that belongs to CTA c' (its 32 units) into c''s inbox.  At the next step
// each CTA adds the G partials of its units in CTA order.  db and dpeep are
// summed afterwards by lstm_param_sums_kernel.
// Shared memory (RecArgs offsets): off_contrib = B (gate errors, NP pieces),
// off_acc = inbox, off_state = dc carry, off_sums = mbarriers, TMEM slot,
// failure flag, the group's step count, off_peep = peepholes, off_tab =
// tables; BULK also off_h = staging of the outgoing partials [G][NBM][32];
// with a.tma_pre off_red = operand tiles [7][NBM][32] (gates i f z o, c_t,
// c_{t-1}, dy).  Tensor memory: accumulators (tile m, chain ch) at columns
// (m * chains + ch) * NBM; piece k of R^T tile m from column
// tm_acol + 64 MT k + 64 m.  Sequence groups as in the forward kernel.
//
// Exchanges of the partials:
//  * BULK: the inbox is double-buffered per step parity ([2][G][NBM][32]);
//    the TMEM read-out lands in a staging buffer laid out per owner, and one
//    cp.async.bulk per owner copies it into the owner's inbox, completing on
//    the owner's mbarrier of that parity (re-armed before the CTA's own copies
//    go out, as in the forward kernel).  A source can only write parity
//    (s & 1) again for step s + 2 after it received this CTA's partials of
//    step s + 1, which are formed after this CTA's cell of step s has read the
//    inbox.
// The cell's own operands arrive as TMA tiles when they fit (a.tma_pre),
// issued after the barrier that follows the cell (every thread has read them).
//  * otherwise: one inbox written with plain DSMEM stores between the two
//    halves of a split cluster barrier.
template <int NP, bool BULK>
__global__ void __launch_bounds__(kCT, 1) lstm_rec_bwd_cluster_kernel(RecArgs a,
                                                                     const __grid_constant__ CUtensorMap map_ga,
                                                                     const __grid_constant__ CUtensorMap map_c,
                                                                     const __grid_constant__ CUtensorMap map_dy)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cl = cg::this_cluster();
    const int G = a.G;
    const int rank = (int)cl.block_rank();
    const int ng = a.ngroups;
    const int dir = (int)(blockIdx.x / G) / ng, grp = (int)(blockIdx.x / G) % ng;
    const int S = a.grp_rows, j0 = grp * S;           // this cluster's sorted slots [j0, j0 + S)
    const int srank = grp == 0 ? rank : -1;           // the phase stamps come from group 0
    const int H = a.H, T = a.T, NBM = a.JC;
    const int MT = (H + kCM - 1) / kCM;              // 128-unit tiles of the partial product
    const int u0 = rank * kCU;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const int nch = a.tm_chains;                     // chains per tile; issuers = MT * nch
    uint8_t* Bb = base + a.off_contrib;              // [NP][2 k-blocks][NBM][128 B]
    const size_t bsz = (size_t)2 * NBM * 128;        // bytes of one B piece
    float* inbox = reinterpret_cast<float*>(base + a.off_acc);       // [BULK ? 2 : 1][G][NBM][32]
    float* stage = reinterpret_cast<float*>(base + a.off_h);         // BULK: [G][NBM][32]
    float* tiles = reinterpret_cast<float*>(base + a.off_red);       // BULK + tma_pre: [7][NBM][32]
    float* dcc = reinterpret_cast<float*>(base + a.off_state);       // [S][32]
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(base + a.off_sums);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
    int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
    uint64_t* full_bar = mma_bar + 2;                                // BULK: [2] inbox arrival per parity
    uint64_t* opnd_bar = mma_bar + 4;                                // operand tiles' arrival
    int* s_tg = reinterpret_cast<int*>(mma_bar + 6);                 // the group's step count
    float* peep_s = reinterpret_cast<float*>(base + a.off_peep);
    int* s_bs = reinterpret_cast<int*>(base + a.off_tab);            // [T] the group's active rows
    int* s_off = s_bs + T;                                           // [T+1] the group's first row
    int* s_len = s_off + T + 1;                                      // [S] lengths of the group's slots
    const uint32_t tcols = (uint32_t)a.Umax;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool tma_opnd = a.tma_pre != 0;
    auto inbox_at = [&](int parity, int src, int j) -> float* {
        return inbox + (((size_t)(BULK ? parity : 0) * G + src) * NBM + j) * kCU;
    };
    auto tile = [&](int k, int j) -> float* { return tiles + ((size_t)k * NBM + j) * kCU; };
    int Tg = 0;
    // rows of the partials of step s2 - 1 that step s2 reads: its rows with a step after them
    // (in recurrence order); the cell reads no others
    auto step_rows = [&](int s2) -> int {
        const int tp = dir == 0 ? Tg - s2 : s2 - 1, tn = dir == 0 ? Tg - 1 - s2 : s2;
        return min(s_bs[tp], s_bs[tn]);
    };
    // bytes a CTA receives for step s2: those rows from every other CTA (its own it writes itself)
    auto step_bytes = [&](int s2) -> uint32_t {
        return (uint32_t)(G - 1) * (uint32_t)step_rows(s2) * (uint32_t)(kCU * 4);
    };

    for (int i = threadIdx.x; i < NP * bsz / 16; i += kCT) reinterpret_cast<uint4*>(Bb)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < (BULK ? 2 : 1) * G * NBM * kCU; i += kCT) inbox[i] = 0.f;
    if (threadIdx.x == 0) *s_tg = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < T; i += kCT) {
        const int n = min(max(a.bs[i] - j0, 0), S);
        s_bs[i] = n;
        if (n > 0 && (i + 1 == T || a.bs[i + 1] <= j0)) *s_tg = i + 1;
    }
    for (int i = threadIdx.x; i <= T; i += kCT) s_off[i] = a.off[i] + j0;
    for (int i = threadIdx.x; i < S; i += kCT) s_len[i] = j0 + i < a.B ? a.slot_len[j0 + i] : 0;
    for (int i = threadIdx.x; i < 3 * kCU; i += kCT) {
        const int q = i / kCU, uu = i - q * kCU;
        peep_s[i] = a.peep[(size_t)dir * 3 * H + q * H + u0 + uu];
    }
    __syncthreads();
    Tg = *s_tg;
    if (threadIdx.x == 0) {
        tc::mbar_init(mma_bar, (uint32_t)(MT * nch));
        *s_fail = 0;
        if (BULK) {
            tc::mbar_init(&full_bar[0], 1);
            tc::mbar_init(&full_bar[1], 1);
        }
        if (tma_opnd) tc::mbar_init(opnd_bar, 1);
        tc::fence_mbar_init();
        // the inbox of step 1 (parity 1) is armed before the cluster barrier below
        if (BULK && Tg > 1) tc::mbar_arrive_expect_tx(&full_bar[1], step_bytes(1));
    }
    if (threadIdx.x < 32) {
        tc::tmem_alloc(tmem_slot, tcols);
        tc::tmem_relinquish();
    }
    fence_proxy_async_cta();
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a0 = tmem + (uint32_t)a.tm_acol, ap = (uint32_t)(64 * MT);
    // R^T slice -> tensor memory: tile m, lane l = unit 128m + l (zero past H); column 64m + c
    // holds this CTA's gate rows r = 2c, 2c + 1 (r = 32g + uu); warps q and q + 4 share the
    // lanes 32q.. and take alternate gates
    {
        const int q = warp & 3;
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        for (int m = 0; m < MT; ++m) {
            const int up = 128 * m + 32 * q + lane;
            for (int g = warp >> 2; g < 4; g += 2) {
                float v[32];
#pragma unroll
                for (int uu = 0; uu < 32; ++uu) {
                    const size_t src = (size_t)dir * 4 * H * H + (size_t)(g * H + u0 + uu) * H + up;
                    v[uu] = up < H ? (NP > 1 ? __ldg(reinterpret_cast<const float*>(a.R) + src)
                                             : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.R)[src]))
                                   : 0.f;
                }
                uint32_t pc[NP][16];
                split32<NP>(v, pc);
#pragma unroll
                for (int k = 0; k < NP; ++k)
                    tc::tmem_st_32x32b_x16(a0 + (uint32_t)k * ap + lanes + (uint32_t)(64 * m + 16 * g), pc[k]);
            }
        }
        tc::tmem_wait_st();
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    // tma_opnd: the seven operand tiles of step s2 (NBM rows each; rows past the packed rows read
    // 0), one thread, completing on opnd_bar
    auto issue_opnd = [&](int s2) {
        const int t2 = dir == 0 ? Tg - 1 - s2 : s2;
        const int y0 = s_off[t2];
        const int yp = dir == 0 ? (t2 >= 1 ? s_off[t2 - 1] : 0) : (t2 + 1 < Tg ? s_off[t2 + 1] : 0);
        tc::mbar_arrive_expect_tx(opnd_bar, (uint32_t)(7 * NBM * kCU * 4));
#pragma unroll
        for (int g = 0; g < 4; ++g) tc::tma_load_2d(tile(g, 0), &map_ga, opnd_bar, dir * 4 * H + g * H + u0, y0);
        tc::tma_load_2d(tile(4, 0), &map_c, opnd_bar, dir * H + u0, y0);
        tc::tma_load_2d(tile(5, 0), &map_c, opnd_bar, dir * H + u0, yp);
        tc::tma_load_2d(tile(6, 0), &map_dy, opnd_bar, dir * H + u0, y0);
    };
    int last_tile = -1;                   // tile issuer: the last step whose tiles were issued
    if (tma_opnd && threadIdx.x == kTileIssuer && Tg > 0) { issue_opnd(0); last_tile = 0; }
    cl.sync();

    const int jq = threadIdx.x >> 3, q8 = threadIdx.x & 7;          // cell item: row jq (+32k), units q8*4..+4
    const uint32_t bstep = (uint32_t)(NBM * 128) >> 4;
    float pk[3][4];                                                  // peepholes i, f, o of units q8*4..+4
#pragma unroll
    for (int q = 0; q < 3; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[q][e] = peep_s[q * kCU + q8 * 4 + e];
    // c0 of slot j's units u0 + q8*4 .. +4 (the state before its first step; zero without one)
    auto init_c = [&](int j) -> float4 {
        return a.c0 ? __ldg(reinterpret_cast<const float4*>(a.c0 + ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 +
                                                            q8 * 4))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    // own operands (gates, c_t, c_{t-1}, dy) of row jq of a step, loaded one step ahead
    // (without operand tiles)
    float nx[7][4];
    auto load_own = [&](int s2) {
        const int t2 = dir == 0 ? Tg - 1 - s2 : s2;
        const int n2 = s_bs[t2];
        if (jq >= n2) return;
        const int row = s_off[t2] + jq;
        const float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 x = *reinterpret_cast<const float4*>(gr + g * H);
            nx[g][0] = x.x; nx[g][1] = x.y; nx[g][2] = x.z; nx[g][3] = x.w;
        }
        const size_t yo = (size_t)row * ndH + dir * H + u0 + q8 * 4;
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(a.cbuf + yo));
        const float4 d0 = __ldg(reinterpret_cast<const float4*>(a.dy + yo));
        nx[4][0] = c0.x; nx[4][1] = c0.y; nx[4][2] = c0.z; nx[4][3] = c0.w;
        nx[6][0] = d0.x; nx[6][1] = d0.y; nx[6][2] = d0.z; nx[6][3] = d0.w;
        const int np2 = dir == 0 ? (t2 >= 1 ? n2 : 0) : (t2 + 1 < Tg ? s_bs[t2 + 1] : 0);
        if (jq < np2) {
            const int pb2 = dir == 0 ? s_off[t2 - 1] : s_off[t2 + 1];
            const float4 p0 = __ldg(reinterpret_cast<const float4*>(a.cbuf + (size_t)(pb2 + jq) * ndH + dir * H + u0 + q8 * 4));
            nx[5][0] = p0.x; nx[5][1] = p0.y; nx[5][2] = p0.z; nx[5][3] = p0.w;
        } else {
            const float4 p0 = init_c(jq);
            nx[5][0] = p0.x; nx[5][1] = p0.y; nx[5][2] = p0.z; nx[5][3] = p0.w;
        }
    };
    if (!tma_opnd && Tg > 0) load_own(0);
    bool failed = false;                  // CTA-uniform: a bounded wait ran out
    bool step_ok = true;                  // this thread's wait of the last product
    for (int s = 0; s < Tg; ++s) {
        const int t = dir == 0 ? Tg - 1 - s : s;
        const int n = s_bs[t];
        const int rowbase = s_off[t];
        const int n_next = dir == 0 ? (t + 1 < Tg ? s_bs[t + 1] : 0) : (t >= 1 ? n : 0);
        const int prev_base = dir == 0 ? (t >= 1 ? s_off[t - 1] : 0) : (t + 1 < Tg ? s_off[t + 1] : 0);
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < Tg ? s_bs[t + 1] : 0);
        const int NBs = (n + 15) & ~15;
        const int par = BULK ? (s & 1) : 0;
        cstamp(a, true, dir, srank, s, 0, 0);
        bool arrived = true;              // this step's inbox and operand tiles arrived
        if (BULK && s > 0 && !failed)
            arrived = tc::mbar_wait(&full_bar[par], (uint32_t)(((s - 1) >> 1) & 1), a.wait_limit_ns);
        if (tma_opnd && !failed && !tc::mbar_wait(opnd_bar, (uint32_t)(s & 1), a.wait_limit_ns)) arrived = false;
        if (!arrived && !failed) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, 0x60000u | (unsigned)s);
            *s_fail = 1 + s;
        }
        cstamp(a, true, dir, srank, s, 1, 1);
        for (int it = 0; it * 32 < n; ++it) {
            const int j = jq + it * 32;
            if (j >= n) continue;
            const int row = rowbase + j;
            const int uub = q8 * 4;
            float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + uub;
            float gv[4][4], cv[4], cpv[4], dyv[4];
            if (tma_opnd) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(tile(g, j) + uub);
                    gv[g][0] = x.x; gv[g][1] = x.y; gv[g][2] = x.z; gv[g][3] = x.w;
                }
                const float4 c0 = *reinterpret_cast<const float4*>(tile(4, j) + uub);
                const float4 p0 = *reinterpret_cast<const float4*>(tile(5, j) + uub);
                const float4 d0 = *reinterpret_cast<const float4*>(tile(6, j) + uub);
                cv[0] = c0.x; cv[1] = c0.y; cv[2] = c0.z; cv[3] = c0.w;
                dyv[0] = d0.x; dyv[1] = d0.y; dyv[2] = d0.z; dyv[3] = d0.w;
                const float4 pc = j < n_prev ? p0 : init_c(j);
                cpv[0] = pc.x; cpv[1] = pc.y; cpv[2] = pc.z; cpv[3] = pc.w;
            } else if (it == 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    gv[0][e] = nx[0][e]; gv[1][e] = nx[1][e]; gv[2][e] = nx[2][e]; gv[3][e] = nx[3][e];
                    cv[e] = nx[4][e]; cpv[e] = nx[5][e]; dyv[e] = nx[6][e];
                }
            } else {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H);
                    gv[g][0] = x.x; gv[g][1] = x.y; gv[g][2] = x.z; gv[g][3] = x.w;
                }
                const size_t yo = (size_t)row * ndH + dir * H + u0 + uub;
                const float4 c0 = __ldg(reinterpret_cast<const float4*>(a.cbuf + yo));
                cv[0] = c0.x; cv[1] = c0.y; cv[2] = c0.z; cv[3] = c0.w;
                const float4 d0 = __ldg(reinterpret_cast<const float4*>(a.dy + yo));
                dyv[0] = d0.x; dyv[1] = d0.y; dyv[2] = d0.z; dyv[3] = d0.w;
                const float4 p0 = j < n_prev ? __ldg(reinterpret_cast<const float4*>(
                                                   a.cbuf + (size_t)(prev_base + j) * ndH + dir * H + u0 + uub))
                                             : init_c(j);
                cpv[0] = p0.x; cpv[1] = p0.y; cpv[2] = p0.z; cpv[3] = p0.w;
            }
            const bool has_next = j < n_next;
            const bool real = !a.padded || t < s_len[j];
            // the G partial sums of R^T da of the step after, added in CTA order, and the carry
            float dhr[4] = {0.f, 0.f, 0.f, 0.f}, car[4] = {0.f, 0.f, 0.f, 0.f};
            const size_t so = ((size_t)dir * a.B + a.perm[j0 + j]) * H + u0 + uub;   // caller-order state
            if (has_next) {
                for (int c2 = 0; c2 < G; ++c2) {
                    const float4 x = *reinterpret_cast<const float4*>(inbox_at(par, c2, j) + uub);
                    dhr[0] += x.x; dhr[1] += x.y; dhr[2] += x.z; dhr[3] += x.w;
                }
                const float4 x = *reinterpret_cast<const float4*>(dcc + j * kCU + uub);
                car[0] = x.x; car[1] = x.y; car[2] = x.z; car[3] = x.w;
            } else {
                // the sequence's last step: the final state's own errors from outside
                if (a.dh_n) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(a.dh_n + so));
                    dhr[0] = x.x; dhr[1] = x.y; dhr[2] = x.z; dhr[3] = x.w;
                }
                if (a.dc_n) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(a.dc_n + so));
                    car[0] = x.x; car[1] = x.y; car[2] = x.z; car[3] = x.w;
                }
            }
            float da[4][4], cout[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float dai = 0.f, daf = 0.f, daz = 0.f, dao = 0.f, carry_out = 0.f;
                if (real) {
                    const float ig = gv[0][e], fg = gv[1][e], zg = gv[2][e], og = gv[3][e];
                    const float c = cv[e], cp = cpv[e];
                    const float dh = dyv[e] + dhr[e];
                    const float tc = tanh_c(c);
                    dao = dh * tc * og * (1.f - og);
                    const float dc = dh * og * (1.f - tc * tc) + dao * pk[2][e] + car[e];
                    dai = dc * zg * ig * (1.f - ig);
                    daf = dc * cp * fg * (1.f - fg);
                    daz = dc * ig * (1.f - zg * zg);
                    carry_out = dc * fg + dai * pk[0][e] + daf * pk[1][e];
                }
                da[0][e] = dai; da[1][e] = daf; da[2][e] = daz; da[3][e] = dao;
                cout[e] = carry_out;
            }
            *reinterpret_cast<float4*>(dcc + j * kCU + uub) = make_float4(cout[0], cout[1], cout[2], cout[3]);
            if (j >= n_prev && a.dc0)                    // the sequence's first step: dL/dc0
                *reinterpret_cast<float4*>(a.dc0 + so) = make_float4(cout[0], cout[1], cout[2], cout[3]);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                *reinterpret_cast<float4*>(gr + g * H) = make_float4(da[g][0], da[g][1], da[g][2], da[g][3]);
                uint2 pc[NP];
                split4<NP>(da[g], pc);
                const uint32_t o = sw_off4(j, g * kCU + uub, NBM);
#pragma unroll
                for (int k = 0; k < NP; ++k) *reinterpret_cast<uint2*>(Bb + (size_t)k * bsz + o) = pc[k];
            }
        }
        if (BULK) cstamp(a, true, dir, srank, s, 4, 4);   // (BULK: stamp 4 = cell done)
        if (!BULK) cluster_arrive_relaxed();   // this CTA has read its inbox: peers may overwrite it
        // the previous step's staging must have been read by its copies before this step's read-out
        if (BULK && lane == 0 && warp < G) bulk_wait_read_all();
        fence_proxy_async_cta();
        // a timeout (of the previous step's product, or of this step's arrivals) becomes a
        // CTA-uniform decision here, before the next issue: from then on the CTA issues, waits
        // for, re-arms and sends nothing (that step's read-out may have seen partial sums; the
        // status word marks the results as invalid)
        if (__syncthreads_or(!step_ok || !arrived)) failed = true;
        // the operand tiles and this parity's inbox have been read
        if (tma_opnd && threadIdx.x == kTileIssuer && s + 1 < Tg && !failed) {
            issue_opnd(s + 1);
            last_tile = s + 1;
        }
        // BULK: re-arm this parity for step s + 2 before this CTA's partials of step s go out
        if (BULK && threadIdx.x == 0 && !failed && s + 2 < Tg)
            tc::mbar_arrive_expect_tx(&full_bar[par], step_bytes(s + 2));
        cstamp(a, true, dir, srank, s, 2, 2);
        if (s + 1 < Tg) {
            // P[u'][j] = sum over this CTA's gate rows r of R[r][u'] da[j][r]: warp w issues tile
            // m = w / chains, chain ch = w % chains (k-steps ch, ch + chains, ... of the 8)
            if (lane == 0 && warp < MT * nch && !failed) {
                tc::tc_fence_after_sync();
                const int m = warp / nch, ch = warp - m * nch;
                const uint32_t idesc = tc::idesc_bf16_f32(kCM, NBs);
                const uint64_t db0 = tc::sdesc_sw128(tc::smem_u32(Bb)), bp = (uint64_t)(bsz >> 4);
                const uint32_t dm = tmem + (uint32_t)(warp * NBM), am = a0 + (uint32_t)(64 * m);
                if (nch == 4) issue_chain_fixed<4, 8, 4, NP>(dm, am, ap, db0, bp, bstep, ch, idesc);
                else if (nch == 2) issue_chain_fixed<2, 8, 4, NP>(dm, am, ap, db0, bp, bstep, ch, idesc);
                else issue_chain_fixed<1, 8, 4, NP>(dm, am, ap, db0, bp, bstep, ch, idesc);
                if (!(s == 0 && dir == 0 && grp == 0 && rank == a.debug_skip_cta)) tc::mma_commit(mma_bar);   // test hook
            }
            if (warp < MT * nch) __syncwarp();
            cstamp(a, true, dir, srank, s, 6, 6);
            step_ok = failed ? true : tc::mbar_wait(mma_bar, (uint32_t)(s & 1), a.wait_limit_ns);
            if (!step_ok) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, 0x50000u | (unsigned)s);
                *s_fail = 1 + s;
            }
            tc::tc_fence_after_sync();
            cstamp(a, true, dir, srank, s, 5, 7);
        }
        if (BULK) {
            if (s + 1 < Tg && !failed) {
                // read-out into the staging, per owner: tile m, lane quarter q -> owner 4m + q,
                // units 32q + lane of the tile, rows [0, NBs)
                for (int pq = warp; pq < MT * 4; pq += kCT / 32) {
                    const int m = pq >> 2, q = pq & 3;
                    const int owner = 4 * m + q;
                    if (owner >= G) continue;
                    // this CTA's own units go straight into its next inbox
                    float* dst = owner == (int)rank ? inbox_at(par ^ 1, rank, 0) : stage + (size_t)owner * NBM * kCU;
                    for (int c0 = 0; c0 < NBs; c0 += 16) {
                        float v[16];
                        tmem_sum_chains(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * nch * NBM + c0),
                                        (uint32_t)NBM, nch, v);
#pragma unroll
                        for (int e = 0; e < 16; ++e) dst[(size_t)(c0 + e) * kCU + lane] = v[e];
                    }
                }
            }
            tc::tc_fence_before_sync();
            fence_proxy_async_cta();
            __syncthreads();
            // lane 0 of warp w sends to owners w, w + 8 (copies issued by one warp's lanes serialise)
            if (s + 1 < Tg && !failed && lane == 0 && warp < G) {
                const uint32_t nxt = (uint32_t)(par ^ 1);
                const uint32_t bytes = (uint32_t)step_rows(s + 1) * (uint32_t)(kCU * 4);
                for (int o = warp; o < G; o += kCT / 32) {
                    if (o == (int)rank || bytes == 0) continue;
                    const uint32_t bar = mapa_u32(tc::smem_u32(&full_bar[nxt]), (uint32_t)o);
                    bulk_to_peer(mapa_u32(tc::smem_u32(inbox_at(nxt, rank, 0)), (uint32_t)o),
                                 stage + (size_t)o * NBM * kCU, bytes, bar);
                }
                bulk_commit();
            }
            if (!tma_opnd && s + 1 < Tg) load_own(s + 1);   // the next step's own operands
            cstamp(a, true, dir, srank, s, 3, 3);
        } else {
            cluster_wait();        // every peer has read its inbox of this step
            if (s + 1 < Tg && !failed) {
                // tile m, lane quarter q: units u' = 128m + 32q + lane, owned by CTA 4m + q
                for (int pq = warp; pq < MT * 4; pq += kCT / 32) {
                    const int m = pq >> 2, q = pq & 3;
                    const int owner = 4 * m + q;
                    if (owner >= G) continue;
                    float* dst_base = cl.map_shared_rank(inbox_at(0, rank, 0), owner);
                    for (int c0 = 0; c0 < NBs; c0 += 16) {
                        float v[16];
                        tmem_sum_chains(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * nch * NBM + c0),
                                        (uint32_t)NBM, nch, v);
                        // lanes are consecutive units: each store is one coalesced 128-byte row
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < n) dst_base[(size_t)(c0 + e) * kCU + lane] = v[e];
                    }
                }
                tc::tc_fence_before_sync();
            }
            cstamp(a, true, dir, srank, s, 3, 3);
            fence_proxy_async_cluster();
            cluster_arrive();      // release: this CTA's partial sums are in their owners' inboxes
            if (!tma_opnd && s + 1 < Tg) load_own(s + 1);   // the next step's own operands, in flight across the barrier
            cluster_wait();
            cstamp(a, true, dir, srank, s, 4, 4);
        }
    }
    // after a timeout the last tiles issued may not have been waited for (bounded wait)
    if (tma_opnd && threadIdx.x == kTileIssuer && last_tile >= 0)
        tc::mbar_wait(opnd_bar, (uint32_t)(last_tile & 1), kTeardownWaitNs);
    if (BULK) {
        if (lane == 0 && warp < G) bulk_wait_all();   // no copy of this CTA is still in flight
        cl.sync();                                    // nor one into it
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        __syncwarp();
        tc::tc_fence_after_sync();
        if (failed) tc::mbar_wait(mma_bar, (uint32_t)((*s_fail - 1) & 1), kTeardownWaitNs);
        tc::tmem_dealloc(tmem, tcols);
    }
}

// db and dpeep from the gate errors: column (direction, quantity q, unit u),
// q = 0..3 -> sum of da_q, 4 -> da_i c_{t-1}, 5 -> da_f c_{t-1}, 6 -> da_o c_t.
// Thread (direction, unit) takes all seven columns of its unit over one chunk of
// rows, in row order, so each row's gate errors and states are read once; the
// chunks are then added in chunk order (bitwise repeatable).  c_{t-1} of a
// sequence's first step is its initial state c0 (zero when c0 is null).
__global__ void lstm_param_sums_kernel(const float* __restrict__ ga, const float* __restrict__ cbuf,
                                       const int32_t* __restrict__ prev_fwd, const int32_t* __restrict__ prev_rev,
                                       const float* __restrict__ c0, const int32_t* __restrict__ row_slot,
                                       const int32_t* __restrict__ perm, int B,
                                       int rows, int H, int ndir, int chunk, float* __restrict__ partial)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= ndir * H) return;
    const int d = t / H, u = t - d * H;
    const int r0 = blockIdx.y * chunk, r1 = min(rows, r0 + chunk);
    const int nd4H = ndir * 4 * H, ndH = ndir * H;
    const int32_t* prev = d == 0 ? prev_fwd : prev_rev;
    float s[7] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int r = r0; r < r1; ++r) {
        const float* g = ga + (size_t)r * nd4H + (size_t)d * 4 * H + u;
        const float ai = __ldg(g), af = __ldg(g + H), az = __ldg(g + 2 * H), ao = __ldg(g + 3 * H);
        const int pr = __ldg(prev + r);
        const float cp = pr >= 0 ? __ldg(cbuf + (size_t)pr * ndH + d * H + u)
                       : c0 ? __ldg(c0 + ((size_t)d * B + __ldg(perm + __ldg(row_slot + r))) * H + u) : 0.f;
        const float ct = __ldg(cbuf + (size_t)r * ndH + d * H + u);
        s[0] += ai; s[1] += af; s[2] += az; s[3] += ao;
        s[4] += ai * cp; s[5] += af * cp; s[6] += ao * ct;
    }
    float* out = partial + (size_t)blockIdx.y * ndir * 7 * H + (size_t)d * 7 * H + u;
#pragma unroll
    for (int q = 0; q < 7; ++q) out[(size_t)q * H] = s[q];
}

__global__ void lstm_param_sums_combine(const float* __restrict__ partial, int chunks, int H, int ndir,
                                        float* __restrict__ db, float* __restrict__ dpeep)
{
    const int ncols = ndir * 7 * H;
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= ncols) return;
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) s += partial[(size_t)c * ncols + col];
    const int d = col / (7 * H), rem = col - d * 7 * H, q = rem / H, u = rem - q * H;
    if (q < 4) db[(size_t)d * 4 * H + q * H + u] = s;
    else dpeep[(size_t)d * 3 * H + (q - 4) * H + u] = s;
}

// ------------------------------------------------------------------------- configuration

static size_t al(size_t v, size_t a) { return (v + a - 1) / a * a; }

static uint32_t pow2_cols(int need)
{
    uint32_t cols = 32;
    while (cols < (uint32_t)need) cols <<= 1;
    return cols;
}

// Dynamic shared memory for a cluster kernel that allocates `tcols` TMEM
// columns per CTA: at least enough that no more CTAs fit on one SM than
// their columns fit in its 512 (a CTA whose allocation waited for another
// CTA of the same cluster would never see it leave).
static size_t tmem_safe_smem(const Plan& p, size_t smem, uint32_t tcols)
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
static bool cluster_schedulable(const Plan& p, const void* fn, int G, size_t smem)
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

static int max_active_rows(const Plan& p)
{
    int bmax = 0;
    for (int t = 0; t < p.T; ++t) bmax = std::max(bmax, p.h_bs[t]);
    return bmax;
}

// Sequence groups: the sorted slots are cut into ng contiguous groups of S slots, one cluster
// per (direction, group).  S is the smallest multiple of 8 (at least 8) for which every
// cluster has an SM of its own, or the plan's forced size; one group when S covers the batch.
// False when a group would need more than 128 rows (the cell's row items).
static bool choose_groups(const Plan& p, int G, int ndir, int* S_out, int* ng_out)
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

static const void* fwd_kernel(bool bf16, bool bulk)
{
    if (bulk) return bf16 ? (const void*)lstm_rec_fwd_cluster_kernel<1, true> : (const void*)lstm_rec_fwd_cluster_kernel<3, true>;
    return bf16 ? (const void*)lstm_rec_fwd_cluster_kernel<1, false> : (const void*)lstm_rec_fwd_cluster_kernel<3, false>;
}

bool rec_cluster_fwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* lay)
{
    if (p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % kCU != 0) return false;
    const int G = H / kCU;
    if (G > 16 || G * ndir > p.num_sms) return false;
    int S = 0, ng = 1;
    if (!choose_groups(p, G, ndir, &S, &ng)) return false;
    const int NBM = std::max(16, (std::min(S, max_active_rows(p)) + 15) & ~15);
    const int np = bf16 ? 1 : 3;                   // bf16 pieces of each operand
    const int KB = (H + 63) / 64;
    const int nks = (H + 15) / 16;
    const int acols = (H / 2) * np;                // R slice in TMEM, two bf16 per column and piece
    int nch = 4;
    while (nch > 1 && (nch > nks || nch * NBM + acols > 512)) nch >>= 1;
    if (nch * NBM + acols > 512) return false;
    const uint32_t cols = pow2_cols(nch * NBM + acols);
    // preference: TMA pre-activation tiles, then the bulk exchange (double-buffered operand +
    // staging); the single-buffered exchange without tiles needs the least shared memory
    const int order[4][2] = {{1, 1}, {0, 1}, {1, 0}, {0, 0}};
    for (int oi = 0; oi < 4; ++oi) {
        const int bulk = order[oi][0], pre = order[oi][1];
        if (p.forced_variant >= 0 && p.forced_variant != (bulk | pre << 1)) continue;
        const size_t bbytes = bulk ? 2 * (size_t)np * G * NBM * 64 : (size_t)np * KB * NBM * 128;
        size_t off = 0;
        const size_t o_b = off; off = al(off + bbytes, 1024);
        const size_t o_stage = off; if (bulk) off = al(off + 2 * (size_t)np * NBM * 64, 1024);
        const size_t o_pre = off; if (pre) off = al(off + 4 * (size_t)NBM * kCU * 4, 1024);
        const size_t o_acc = off; off = al(off + (size_t)NBM * kCM * 4, 16);
        const size_t o_cst = off; off = al(off + (size_t)S * kCU * 4, 16);
        const size_t o_bar = off; off = al(off + 64, 16);
        const size_t o_peep = off; off = al(off + 3 * kCU * 4, 16);
        const size_t o_tab = off; off = al(off + (size_t)(2 * p.T + 1 + S) * 4, 16);
        size_t smem = off + 1024 + 64;            // 1024 for the base alignment, 64 static
        smem = tmem_safe_smem(p, smem, cols);
        if (smem == 0) return false;
        if (!cluster_schedulable(p, fwd_kernel(bf16, bulk != 0), G, smem)) continue;
        RecConfig c;
        c.G = G; c.Umax = (int)cols; c.JC = NBM; c.smem = smem; c.cluster = 1;
        c.chains = nch; c.acol = (int)cols - acols; c.bulk = bulk; c.tma_pre = pre;
        c.grp_rows = S; c.ngroups = ng;
        *out = c;
        lay->off_contrib = (int)o_b; lay->off_h = (int)o_stage; lay->off_red = (int)o_pre; lay->off_acc = (int)o_acc;
        lay->off_state = (int)o_cst; lay->off_sums = (int)o_bar; lay->off_peep = (int)o_peep;
        lay->off_tab = (int)o_tab;
        return true;
    }
    return false;
}

// One cluster of c.G CTAs per (direction, sequence group).
static lstm_status cluster_launch(const RecConfig& c, const void* fn, void** args, int ndir, cudaStream_t s)
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

lstm_status rec_cluster_fwd_launch(const Plan& p, const RecConfig& c, RecArgs a, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC; a.tm_chains = c.chains; a.tm_acol = c.acol;
    a.grp_rows = c.grp_rows; a.ngroups = c.ngroups;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    const void* fn = fwd_kernel(a.bf16 != 0, c.bulk != 0);
    // the pre-activation tiles' map: ga as [rows][ndir*4H] fp32, boxes of 32 units x NBM rows
    CUtensorMap pre_map;
    memset(&pre_map, 0, sizeof(pre_map));
    const int nd4H = a.ndir * 4 * a.H;
    a.tma_pre = c.tma_pre && make_map_f32(&pre_map, a.ga, p.rows, nd4H, nd4H, kCU, c.JC) ? 1 : 0;
    void* args[] = {&a, &pre_map};
    trace_begin(p, K_REC_FWD, s);
    const lstm_status st = cluster_launch(c, fn, args, a.ndir, s);
    trace_end(p, K_REC_FWD, s, st == LSTM_OK ? 1 : 0);
    return st;
}

static const void* bwd_kernel(bool bf16, bool bulk)
{
    if (bulk) return bf16 ? (const void*)lstm_rec_bwd_cluster_kernel<1, true> : (const void*)lstm_rec_bwd_cluster_kernel<3, true>;
    return bf16 ? (const void*)lstm_rec_bwd_cluster_kernel<1, false> : (const void*)lstm_rec_bwd_cluster_kernel<3, false>;
}

bool rec_cluster_bwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* lay)
{
    if (p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % kCU != 0) return false;
    const int G = H / kCU;
    if (G > 16 || G * ndir > p.num_sms) return false;
    int S = 0, ng = 1;
    if (!choose_groups(p, G, ndir, &S, &ng)) return false;
    const int NBM = std::max(16, (std::min(S, max_active_rows(p)) + 15) & ~15);
    const int MT = (H + kCM - 1) / kCM;
    const int np = bf16 ? 1 : 3;                   // bf16 pieces of each operand
    const int acols = MT * 64 * np;                // R^T tiles in TMEM: 128 gate rows = 64 columns per piece
    int nch = 4;
    while (nch > 1 && (MT * nch > 4 || MT * nch * NBM + acols > 512)) nch >>= 1;
    if (MT * nch * NBM + acols > 512 || MT * nch > kCT / 32) return false;
    const uint32_t cols = pow2_cols(MT * nch * NBM + acols);
    // bulk exchange with operand tiles first, then the single-buffered barrier exchange with
    // and without tiles (the last needs the least shared memory)
    const int order[4][2] = {{1, 1}, {0, 1}, {0, 0}, {1, 0}};
    for (int oi = 0; oi < 4; ++oi) {
        const int bulk = order[oi][0], tiles = order[oi][1];
        if (oi == 3 && p.forced_variant < 0) break;   // the bulk exchange without tiles only on request
        if (p.forced_variant >= 0 && p.forced_variant != (bulk | tiles << 1)) continue;
        size_t off = 0;
        const size_t o_b = off; off = al(off + (size_t)np * 2 * NBM * 128, 1024);
        const size_t o_in = off; off = al(off + (bulk ? 2 : 1) * (size_t)G * NBM * kCU * 4, 1024);
        const size_t o_stage = off; if (bulk) off = al(off + (size_t)G * NBM * kCU * 4, 1024);
        const size_t o_tiles = off; if (tiles) off = al(off + 7 * (size_t)NBM * kCU * 4, 1024);
        const size_t o_dcc = off; off = al(off + (size_t)S * kCU * 4, 16);
        const size_t o_bar = off; off = al(off + 64, 16);
        const size_t o_peep = off; off = al(off + 3 * kCU * 4, 16);
        const size_t o_tab = off; off = al(off + (size_t)(2 * p.T + 1 + S) * 4, 16);
        size_t smem = off + 1024 + 64;
        smem = tmem_safe_smem(p, smem, cols);
        if (smem == 0) return false;
        if (!cluster_schedulable(p, bwd_kernel(bf16, bulk != 0), G, smem)) continue;
        RecConfig c;
        c.G = G; c.Umax = (int)cols; c.JC = NBM; c.smem = smem; c.cluster = 1;
        c.chains = nch; c.acol = (int)cols - acols; c.bulk = bulk; c.tma_pre = tiles;
        c.grp_rows = S; c.ngroups = ng;
        *out = c;
        lay->off_contrib = (int)o_b; lay->off_acc = (int)o_in; lay->off_h = (int)o_stage; lay->off_red = (int)o_tiles;
        lay->off_state = (int)o_dcc; lay->off_sums = (int)o_bar; lay->off_peep = (int)o_peep; lay->off_tab = (int)o_tab;
        return true;
    }
    return false;
}

size_t rec_cluster_bwd_sum_floats(int H, int ndir) { return (size_t)kSumChunks * ndir * 7 * H; }

lstm_status rec_cluster_bwd_launch(const Plan& p, const RecConfig& c, RecArgs a, float* sum_scratch, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC; a.tm_chains = c.chains; a.tm_acol = c.acol;
    a.grp_rows = c.grp_rows; a.ngroups = c.ngroups;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    const void* fn = bwd_kernel(a.bf16 != 0, c.bulk != 0);
    // operand tiles: ga as [rows][ndir*4H], c and dy as [rows][ndir*H] fp32, boxes of 32 x NBM
    CUtensorMap map_ga, map_c, map_dy;
    memset(&map_ga, 0, sizeof(map_ga));
    memset(&map_c, 0, sizeof(map_c));
    memset(&map_dy, 0, sizeof(map_dy));
    const int nd4H = a.ndir * 4 * a.H, ndH = a.ndir * a.H;
    a.tma_pre = c.tma_pre && make_map_f32(&map_ga, a.ga, p.rows, nd4H, nd4H, kCU, c.JC) &&
                make_map_f32(&map_c, a.cbuf, p.rows, ndH, ndH, kCU, c.JC) &&
                make_map_f32(&map_dy, a.dy, p.rows, ndH, ndH, kCU, c.JC) ? 1 : 0;
    void* args[] = {&a, &map_ga, &map_c, &map_dy};
    trace_begin(p, K_REC_BWD, s);
    lstm_status st = cluster_launch(c, fn, args, a.ndir, s);
    int launched = st == LSTM_OK ? 1 : 0;
    if (st == LSTM_OK) {
        st = param_sums_launch(p, a.ga, a.cbuf, a.H, a.ndir, a.db, a.dpeep, sum_scratch, s, a.c0);
        if (st == LSTM_OK) launched += 2;
    }
    trace_end(p, K_REC_BWD, s, launched);
    return st;
}

lstm_status param_sums_launch(const Plan& p, const float* ga, const float* cbuf, int H, int ndir, float* db,
                              float* dpeep, float* sum_scratch, cudaStream_t s, const float* c0)
{
    const int ncols = ndir * 7 * H;
    const int rows = (int)p.rows;
    const int chunk = (rows + kSumChunks - 1) / kSumChunks;
    lstm_param_sums_kernel<<<dim3((ndir * H + 127) / 128, kSumChunks), 128, 0, s>>>(
        ga, cbuf, p.d_prev_fwd, p.d_prev_rev, c0, p.d_row_slot, p.d_perm, p.B, rows, H, ndir, chunk, sum_scratch);
    lstm_param_sums_combine<<<(ncols + 255) / 256, 256, 0, s>>>(sum_scratch, kSumChunks, H, ndir, db, dpeep);
    return cudaGetLastError() == cudaSuccess ? LSTM_OK : LSTM_ERR_UNSUPPORTED;
}

}  // namespace lstm
