// recurrent_wide.cu -- persistent recurrent kernels for bf16 layers wider than a
// thread-block cluster (512 < H <= 1024).
//
// "Single Stream Parallelization of Generalized LSTM-Like RNNs on a GPU",
// Sec. 3: once the non-recurrent part is done for all frames, only the
// recurrent node remains sequential.  For H = 1024 one direction's R is 8 MB
// of bf16, more than one cluster holds, so one launch spreads it over H/16
// CTAs per direction (64 for H = 1024, both directions on 128 SMs):
//
//  * CTA c owns units [16c, 16c + 16).  Forward: its 64 gate rows of R (64 x H)
//    are loaded once by TMA into shared memory (128 KB) and stay there as the
//    MMA's B operand (N = 64) for every step.
//  * Every step the whole previous operand -- h_{t-1} forward, the previous
//    step's gate errors backward, bf16, one row per active sequence -- sits in
//    a double-buffered global array that L2 holds; a CTA streams the part it
//    needs in 128-row x 64-column TMA tiles through a ring of up to 4 stages
//    into tcgen05.mma (M = 128 rows of the batch per tile, fp32 accumulator in
//    tensor memory).  Forward, every CTA needs all of h_{t-1}: CTAs are grouped
//    in clusters of CS (4 when the device co-schedules them), each tile is read
//    from L2 once per cluster and multicast into all CS CTAs, and each CTA's
//    MMA completion frees the ring stage in all of them (multicast commit).
//  * Backward, R^T da needs all 4H gate errors for every unit.  In clusters of
//    four CTAs, CTA r takes only gate r's H errors against R^T rows of the
//    cluster's 64 units (64 x H resident, N = 64), so it streams a quarter of
//    the operand; the 16-column pieces of the partial products are exchanged
//    through distributed shared memory and added by the units' owners in a
//    fixed order.  Without clusters each CTA takes all 4H errors against its
//    own 16 units' R^T rows (16 x 4H, N = 16).
//  * The cell runs on the accumulator rows: thread r of a 128-thread half
//    reads row r of its tile from tensor memory (all four gates of the CTA's
//    16 units) and runs the forward cell (or its BPTT) after adding the step's
//    input projection; it keeps its row's cell state (forward) or cell-state
//    error (backward) in registers from step to step, and writes its 16 new
//    values of the operand for the next step.
//  * Steps of a direction are separated by a grid barrier: each CTA adds 1 to
//    the direction's counter (release) after its operand writes; a CTA starts
//    step s once the counter reaches s times the CTAs per direction (acquire;
//    the wait is bounded and a timeout is recorded in the plan's status word).
// One cooperative launch runs every step of both directions.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "gemm.cuh"
#include "recurrent.cuh"
#include "tc_ptx.cuh"

namespace lstm {

namespace {

constexpr int kWU = 16;                          // units per CTA
constexpr int kWT = 256;                         // threads: rows 0..127 and 128..255 of the batch
constexpr int kWMaxStages = 4;                   // operand ring stages at most (measured: 6 stages ran
                                                 // ~5% slower than 4 on H = 1024)
constexpr uint32_t kWTile = 128 * 64 * 2;        // one operand tile: 128 rows x 64 bf16
constexpr unsigned long long kWTeardownNs = 1000000000ull;

__device__ __forceinline__ float sigm_w(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float tanh_w(float x)
{
    const float e = __expf(2.0f * fminf(fmaxf(x, -40.0f), 40.0f));
    return 1.0f - __fdividef(2.0f, e + 1.0f);
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Distributed shared memory: a peer's address, a store into it, a release arrival on a peer's
// mbarrier, and the acquiring wait that pairs with it.
__device__ __forceinline__ uint32_t mapa_w(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float x, float y, float z, float w)
{
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}
__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(tc::smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Every CTA of the direction has published step `target` (bounded wait by thread 0; the
// outcome is the same for every thread of the CTA).
__device__ __forceinline__ bool grid_wait(const unsigned* ctr, unsigned target, const WideArgs& a, unsigned where)
{
    int fail = 0;
    if (threadIdx.x == 0) {
        const unsigned long long t0 = global_timer_ns();
        unsigned spins = 0;
        while ((int)(ld_acquire_gpu(ctr) - target) < 0) {
            if ((++spins & 63u) == 0) {
                if (failure_recorded(a.status)) { fail = 1; break; }
                if (global_timer_ns() - t0 > a.wait_limit_ns) {
                    record_failure(a.status, LSTM_ERR_TIMEOUT, where);
                    fail = 1;
                    break;
                }
            }
        }
    }
    return __syncthreads_or(fail) == 0;
}

// Phase stamps of CTA 0 of each direction, in the recurrent kernels' slots [kernel][dir][step][8]:
// 0 step start, 1 after the grid barrier, 5 product in tensor memory, 3 cell done, 4 published.
__device__ __forceinline__ void wstamp(const WideArgs& a, bool bwd, int dir, int cta, int s, int k)
{
    if (threadIdx.x == 0 && a.trace && cta == 0 && s < a.trace_steps)
        a.trace[(((size_t)(bwd ? 1 : 0) * a.ndir + dir) * a.trace_steps + s) * 8 + k] = clock64();
}

// Shared memory of both kernels: the resident weight slice (KBW blocks of rowsW x 128 B),
// the operand ring (`stages` tiles), the partial-product inbox of the split backward, barriers.
struct WideSmem {
    uint8_t* w;
    uint8_t* ring;
    float* inbox;           // split backward: [3 senders][B rows][16] fp32 (16-byte chunks swizzled)
    uint64_t* full;
    uint64_t* empty;
    uint64_t* mma_bar;
    uint64_t* w_bar;
    uint64_t* inbox_bar;    // split backward: one arrival from each of the three peers per step
    uint32_t* tmem_slot;
    int* counters;          // [0] loads issued, [1] tiles consumed (teardown after a timeout)
    float* peep;            // [3][16]
    int stages;
};

__device__ __forceinline__ WideSmem wide_smem(int KBW, int rowsW, int stages, size_t inbox_bytes)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    WideSmem m;
    m.stages = stages;
    m.w = base;
    m.ring = base + (size_t)KBW * rowsW * 128;
    m.inbox = reinterpret_cast<float*>(m.ring + (size_t)stages * kWTile);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(m.inbox) + inbox_bytes);
    m.full = bars;
    m.empty = bars + stages;
    m.mma_bar = bars + 2 * stages;
    m.w_bar = m.mma_bar + 1;
    m.inbox_bar = m.mma_bar + 2;
    m.tmem_slot = reinterpret_cast<uint32_t*>(m.mma_bar + 3);
    m.counters = reinterpret_cast<int*>(m.tmem_slot + 2);
    m.peep = reinterpret_cast<float*>(m.counters + 2);
    return m;
}

size_t wide_smem_bytes(int KBW, int rowsW, int stages, size_t inbox_bytes)
{
    return 1024 + (size_t)KBW * rowsW * 128 + (size_t)stages * kWTile + inbox_bytes + (2 * stages + 3) * 8 + 16 +
           3 * kWU * 4;
}

// Position in the operand ring: tiles issued (or consumed) so far, and the stage and lap
// parity of the next one, advanced without division.
struct RingPos {
    uint32_t it = 0;
    int st = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void advance(int stages)
    {
        ++it;
        if (++st == stages) { st = 0; ph ^= 1u; }
    }
};

// One step's product: D[tile m][rows][N] = sum over the KB blocks of A (the operand tiles of
// columns x0 + 64 kb, streamed from rows ybase + 128 m) times the resident weight slice (B, N
// rows per block).
// Thread 0 arms the ring and issues its share of the TMA tiles (with CS > 1: tile i by
// cluster rank i mod CS, multicast to the whole cluster), thread 32 issues the MMAs and frees
// each stage in every CTA of the cluster; prod / cons carry the ring position across
// steps (each only in its own thread).
template <int CS>
__device__ __forceinline__ bool wide_product(const WideSmem& m, const CUtensorMap* mapA, int x0, int ybase, int MT,
                                             int KB, int N, uint32_t tmem, const WideArgs& a, RingPos& prod,
                                             RingPos& cons, bool& w_ready, unsigned where, int crank)
{
    bool ok = true;
    constexpr uint16_t kMask = (uint16_t)((1u << CS) - 1u);
    if (threadIdx.x == 0) {
        fence_async_global();
        for (int t = 0; t < MT && ok; ++t)
            for (int kb = 0; kb < KB; ++kb, prod.advance(m.stages)) {
                const int st = prod.st;
                // the stage's previous tile has been consumed by every CTA of the cluster
                if (prod.it >= (uint32_t)m.stages && !tc::mbar_wait(&m.empty[st], prod.ph ^ 1u, a.wait_limit_ns)) {
                    record_failure(a.status, LSTM_ERR_TIMEOUT, where | 0x1000u);
                    ok = false;
                    break;
                }
                tc::mbar_arrive_expect_tx(&m.full[st], kWTile);
                if (CS == 1)
                    tc::tma_load_2d(m.ring + (size_t)st * kWTile, mapA, &m.full[st], x0 + kb * 64, ybase + t * 128);
                else if ((t * KB + kb) % CS == crank)
                    tc::tma_load_2d_multicast(m.ring + (size_t)st * kWTile, mapA, &m.full[st], x0 + kb * 64,
                                              ybase + t * 128, kMask);
                m.counters[0] = (int)prod.it + 1;
            }
    } else if (threadIdx.x == 32) {
        if (!w_ready) {
            if (!tc::mbar_wait(m.w_bar, 0, a.wait_limit_ns)) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, where | 0x2000u);
                ok = false;
            }
            w_ready = true;
        }
        const uint32_t idesc = tc::idesc_bf16_f32(128, N);
        const uint32_t wbytes = (uint32_t)N * 128;               // one block of the weight slice
        for (int t = 0; t < MT && ok; ++t)
            for (int kb = 0; kb < KB; ++kb, cons.advance(m.stages)) {
                const int st = cons.st;
                if (!tc::mbar_wait(&m.full[st], cons.ph, a.wait_limit_ns)) {
                    record_failure(a.status, LSTM_ERR_TIMEOUT, where | 0x3000u);
                    ok = false;
                    break;
                }
                tc::tc_fence_after_sync();
                const uint32_t a0 = tc::smem_u32(m.ring + (size_t)st * kWTile);
                const uint32_t b0 = tc::smem_u32(m.w + (size_t)kb * wbytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16_ss(tmem + (uint32_t)(t * N), tc::sdesc_sw128(a0 + kk * 32), tc::sdesc_sw128(b0 + kk * 32),
                                    idesc, (kb | kk) != 0 ? 1u : 0u);
                if (CS == 1) tc::mma_commit(&m.empty[st]);
                else tc::mma_commit_multicast(&m.empty[st], kMask);
                m.counters[1] = (int)cons.it + 1;
            }
        tc::mma_commit(m.mma_bar);
    }
    // the other lanes of the issuing warps wait here instead of polling while lane 0 works
    // (measured: polling lanes of the same warp slowed the issue loops ~3x)
    if (threadIdx.x < 64) __syncwarp();
    return ok;
}

// Before a CTA leaves: no TMA tile may still be landing in its shared memory, no MMA may
// still use its tensor memory, and (clusters) no peer's stage-release or partial product may
// still be on its way to it -- every wait bounded.  A clean run waits only for the peers'
// releases of the ring's last uses; after a timeout the CTA also waits for the tiles it armed
// and then gives any multicast tile already issued by a peer a millisecond to land.
// MC: CTAs sharing each operand tile (multicast); CL: the launch has clusters.
template <int MC, bool CL>
__device__ __forceinline__ void wide_finish(const WideSmem& m, uint32_t it_prod, uint32_t mma_phase, bool failed)
{
    if (threadIdx.x == 0) {
        const uint32_t ns = (uint32_t)m.stages;
        if (failed) {
            for (uint32_t it = (uint32_t)max(0, m.counters[1]); it < it_prod; ++it)
                tc::mbar_wait(&m.full[it % ns], (it / ns) & 1, kWTeardownNs);
            tc::mbar_wait(m.mma_bar, (mma_phase - 1) & 1, kWTeardownNs);
        }
        tc::mbar_wait(m.w_bar, 0, kWTeardownNs);
        if (MC > 1) {
            // each stage's last use released by every CTA of the cluster
            for (uint32_t it = it_prod > ns ? it_prod - ns : 0u; it < it_prod; ++it)
                tc::mbar_wait(&m.empty[it % ns], (it / ns) & 1, failed ? 1000000ull : kWTeardownNs);
            if (failed) {
                const unsigned long long t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 1000000ull) {
                }
            }
        }
    }
    if (CL) {
        __syncthreads();
        cooperative_groups::this_cluster().sync();      // no peer still sends into this CTA
    }
}

}  // namespace

// Forward.  Operand array a.xbuf: [ndir][2][B][H] bf16, step s reads parity s & 1 and
// writes parity (s + 1) & 1.  Tensor maps: mapW = R as [ndir*4H][H] (boxes 16 rows x 64),
// mapA = a.xbuf as [ndir*2*B][H] (boxes 128 rows x 64).
template <int CS>
__global__ void __launch_bounds__(kWT, 1) lstm_rec_fwd_wide_kernel(WideArgs a, const __grid_constant__ CUtensorMap mapW,
                                                                  const __grid_constant__ CUtensorMap mapA)
{
    const int H = a.H, T = a.T, B = a.B, NC = a.NC;
    const int KB = H / 64;
    const int dir = blockIdx.x / NC, cta = blockIdx.x - dir * NC, u0 = cta * kWU;
    const int nd4H = a.ndir * 4 * H, ndH = a.ndir * H;
    const WideSmem m = wide_smem(KB, 64, a.stages, 0);
    const int warp = threadIdx.x >> 5;
    const int crank = CS > 1 ? (int)cooperative_groups::this_cluster().block_rank() : 0;
    const int tile = threadIdx.x >> 7, j = threadIdx.x;      // this thread's row of the batch
    unsigned* ctr = a.ctr + dir;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            tc::mbar_init(&m.full[s], 1);
            tc::mbar_init(&m.empty[s], CS);          // one release from each CTA of the cluster
        }
        tc::mbar_init(m.mma_bar, 1);
        tc::mbar_init(m.w_bar, 1);
        m.counters[0] = m.counters[1] = 0;
        tc::fence_mbar_init();
        // the CTA's 64 gate rows of R (gate g, units u0..u0+15 -> slice rows 16 g ..), K-blocks of 64
        tc::mbar_arrive_expect_tx(m.w_bar, (uint32_t)KB * 64 * 128);
        for (int kb = 0; kb < KB; ++kb)
            for (int g = 0; g < 4; ++g)
                tc::tma_load_2d(m.w + (size_t)kb * 8192 + g * 2048, &mapW, m.w_bar, kb * 64, dir * 4 * H + g * H + u0);
    }
    if (warp == 0) {
        tc::tmem_alloc(m.tmem_slot, 128);
        tc::tmem_relinquish();
    }
    for (int i = threadIdx.x; i < 3 * kWU; i += kWT) m.peep[i] = a.peep[(size_t)dir * 3 * H + (i / kWU) * H + u0 + i % kWU];
    // empty sequences end in their initial state
    if (a.h_n && j < B && a.len[j] == 0)
        for (int k = 0; k < kWU; ++k) {
            const size_t o = ((size_t)dir * B + a.perm[j]) * H + u0 + k;
            a.h_n[o] = a.h0 ? a.h0[o] : 0.f;
            if (a.c_n) a.c_n[o] = a.c0 ? a.c0[o] : 0.f;
        }
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    if (CS > 1) cooperative_groups::this_cluster().sync();   // every peer's barriers exist before any multicast
    const uint32_t tmem = *m.tmem_slot;

    float creg[kWU];                                  // c of this thread's row, step to step
#pragma unroll
    for (int k = 0; k < kWU; ++k) creg[k] = 0.f;
    RingPos prod, cons;
    uint32_t mma_phase = 0;
    bool w_ready = false, failed = false;
    for (int s = 0; s < T && !failed; ++s) {
        const int t = dir == 0 ? s : T - 1 - s;
        const int n = a.bs[t];
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < T ? a.bs[t + 1] : 0);
        const int row = a.off[t] + j;
        wstamp(a, false, dir, cta, s, 0);
        // this row's input projection (own data: loaded before the wait)
        float pre[4][kWU];
        if (j < n) {
            const float* gr = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u0;
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int q = 0; q < kWU / 4; ++q) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H + 4 * q);
                    pre[g][4 * q] = x.x; pre[g][4 * q + 1] = x.y; pre[g][4 * q + 2] = x.z; pre[g][4 * q + 3] = x.w;
                }
        }
        if (s + 1 < T) {           // the next step's pre-activations of this row into L2
            const int t2 = dir == 0 ? s + 1 : T - 2 - s;
            if (j < a.bs[t2]) {
                const float* g2 = a.ga + (size_t)(a.off[t2] + j) * nd4H + (size_t)dir * 4 * H + u0;
#pragma unroll
                for (int g = 0; g < 4; ++g) asm volatile("prefetch.global.L2 [%0];" ::"l"(g2 + g * H));
            }
        }
        if (s > 0 && !grid_wait(ctr, (unsigned)(NC * s), a, 0x90000u | (unsigned)s)) { failed = true; break; }
        wstamp(a, false, dir, cta, s, 1);
        const int MT = (n_prev + 127) / 128;
        if (MT > 0) {
            bool ok = wide_product<CS>(m, &mapA, 0, (dir * 2 + (s & 1)) * B, MT, KB, 64, tmem, a, prod, cons,
                                       w_ready, 0xA0000u | (unsigned)(s & 0xfff), crank);
            ++mma_phase;
            // one thread polls the product's completion; the others wait at the barrier below
            if (threadIdx.x == 0) ok = tc::mbar_wait(m.mma_bar, (mma_phase - 1) & 1, a.wait_limit_ns) && ok;
            if (__syncthreads_or(!ok)) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, 0xB0000u | (unsigned)s);
                failed = true;
                break;
            }
            tc::tc_fence_after_sync();
        }
        wstamp(a, false, dir, cta, s, 5);
        // R h_{t-1} of this row (tensor-memory lane = row within the tile, warp-uniform loads),
        // added into the pre-activations one gate at a time
        if (tile < MT) {                  // (warp-uniform: the loads are warp-collective)
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                uint32_t r[16];
                tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(tile * 64 + g * 16), r);
                tc::tmem_wait_ld();
                if (j < n_prev)
#pragma unroll
                    for (int k = 0; k < kWU; ++k) pre[g][k] += __uint_as_float(r[k]);
            }
        }
        // the cell; h_t goes to the exchange buffer first and is published at once, the layer's
        // own outputs (gates, c, y) are stored after the publish, off the peers' critical path
        float hv[kWU], cv[kWU], gv[4][kWU];
        const int len = j < B ? a.len[j] : 0;
        const size_t so = j < B ? ((size_t)dir * B + a.perm[j]) * H + u0 : 0;          // caller-order state
        if (j < n) {
#pragma unroll
            for (int k = 0; k < kWU; ++k) {
                const float cp = j < n_prev ? creg[k] : (a.c0 ? __ldg(a.c0 + so + k) : 0.f);
                const float ig = sigm_w(pre[0][k] + m.peep[k] * cp);
                const float fg = sigm_w(pre[1][k] + m.peep[kWU + k] * cp);
                const float zg = tanh_w(pre[2][k]);
                float c = fg * cp + ig * zg;
                const float og = sigm_w(pre[3][k] + m.peep[2 * kWU + k] * c);
                float h = og * tanh_w(c);
                if (a.padded && t >= len) { c = 0.f; h = 0.f; }
                gv[0][k] = ig; gv[1][k] = fg; gv[2][k] = zg; gv[3][k] = og;
                cv[k] = c; hv[k] = h; creg[k] = c;
            }
        }
        uint32_t hb[kWU / 2];
#pragma unroll
        for (int e = 0; e < kWU / 2; ++e) {
            const __nv_bfloat162 p2 = __floats2bfloat162_rn(j < n ? hv[2 * e] : 0.f, j < n ? hv[2 * e + 1] : 0.f);
            hb[e] = *reinterpret_cast<const uint32_t*>(&p2);
        }
        if (j < n && s + 1 < T) {    // h_t for the next step's product
            uint4* xb = reinterpret_cast<uint4*>(a.xbuf + (((size_t)dir * 2 + ((s + 1) & 1)) * B + j) * H + u0);
            xb[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
            xb[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
        }
        fence_async_global();       // this thread's h_t is read by the peers' TMA tiles
        tc::tc_fence_before_sync();
        __syncthreads();
        wstamp(a, false, dir, cta, s, 3);
        // the release add is cumulative over the CTA's writes ordered before it by the barrier
        if (threadIdx.x == 0 && !(s == 0 && dir == 0 && cta == a.debug_skip_cta))   // (test hook)
            red_release_add(ctr, 1u);
        wstamp(a, false, dir, cta, s, 4);
        if (j < n) {
            float* gw = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u0;
            const size_t yo = (size_t)row * ndH + (size_t)dir * H + u0;
#pragma unroll
            for (int q = 0; q < kWU / 4; ++q) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    *reinterpret_cast<float4*>(gw + g * H + 4 * q) =
                        make_float4(gv[g][4 * q], gv[g][4 * q + 1], gv[g][4 * q + 2], gv[g][4 * q + 3]);
                *reinterpret_cast<float4*>(a.cbuf + yo + 4 * q) = make_float4(cv[4 * q], cv[4 * q + 1], cv[4 * q + 2], cv[4 * q + 3]);
                *reinterpret_cast<float4*>(a.y + yo + 4 * q) = make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
            }
            if (a.y_lo) {
                uint4* yl = reinterpret_cast<uint4*>(a.y_lo + yo);
                yl[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
                yl[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
            }
            if (a.h_n && ((dir == 0 && t == len - 1) || (dir == 1 && t == 0 && len > 0)))
#pragma unroll
                for (int k = 0; k < kWU; ++k) {
                    a.h_n[so + k] = hv[k];
                    if (a.c_n) a.c_n[so + k] = cv[k];
                }
        }
    }
    wide_finish<CS, (CS > 1)>(m, prod.it, mma_phase, failed);
    tc::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem, 128);
    }
}

// BPTT.  Operand array a.xbuf: [ndir][2][B][4H] bf16 gate errors (step s reads parity s & 1,
// the errors of the previous BPTT step; writes parity (s + 1) & 1).  mapW = R^T as
// [ndir*H][4H] (boxes 16 rows x 64), mapA = a.xbuf as [ndir*2*B][4H] (boxes 128 rows x 64).
//  KS = false: CTA c multiplies all 4H gate errors of each row by the R^T rows of its own 16
//    units (N = 16, K = 4H): every CTA streams the whole operand.
//  KS = true (clusters of four consecutive CTAs): CTA r of a cluster takes only gate r's H
//    errors (K = H) against the R^T rows of the cluster's 64 units (N = 64), a quarter of the
//    operand.  Of its partial product it keeps the 16 columns of its own units and stores the
//    other three 16-column pieces into their owners' inboxes (distributed shared memory); each
//    owner adds to its own partial those of ranks r+1, r+2, r+3 (mod 4), in that order, so the
//    sum does not depend on timing.  A peer writes into an inbox only after the grid barrier that follows the owner's
//    reading of it, so one inbox per CTA suffices.
template <bool KS>
__global__ void __launch_bounds__(kWT, 1) lstm_rec_bwd_wide_kernel(WideArgs a, const __grid_constant__ CUtensorMap mapW,
                                                                  const __grid_constant__ CUtensorMap mapA)
{
    constexpr int NU = KS ? 4 * kWU : kWU;            // product columns (units)
    constexpr uint32_t kTmemCols = 2 * NU < 32 ? 32 : 2 * NU;
    const int H = a.H, T = a.T, B = a.B, NC = a.NC;
    const int KB = (KS ? H : 4 * H) / 64;
    const int dir = blockIdx.x / NC, cta = blockIdx.x - dir * NC, u0 = cta * kWU;
    const int nd4H = a.ndir * 4 * H, ndH = a.ndir * H;
    const int crank = KS ? (int)cooperative_groups::this_cluster().block_rank() : 0;
    const int U0 = u0 - crank * kWU;                  // first unit of the product's columns
    const int x0 = crank * H;                         // first gate-error column of its K range
    const WideSmem m = wide_smem(KB, NU, a.stages, KS ? (size_t)3 * B * kWU * 4 : 0);
    const int warp = threadIdx.x >> 5;
    const int tile = threadIdx.x >> 7, j = threadIdx.x;
    unsigned* ctr = a.ctr + dir;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            tc::mbar_init(&m.full[s], 1);
            tc::mbar_init(&m.empty[s], 1);
        }
        tc::mbar_init(m.mma_bar, 1);
        tc::mbar_init(m.w_bar, 1);
        tc::mbar_init(m.inbox_bar, 3);
        m.counters[0] = m.counters[1] = 0;
        tc::fence_mbar_init();
        // R^T rows of the product's units over its K range, K-blocks of 64 (NU x 128 B each)
        tc::mbar_arrive_expect_tx(m.w_bar, (uint32_t)KB * NU * 128);
        for (int kb = 0; kb < KB; ++kb)
            for (int i = 0; i < NU / kWU; ++i)
                tc::tma_load_2d(m.w + (size_t)kb * NU * 128 + i * kWU * 128, &mapW, m.w_bar, x0 + kb * 64,
                                dir * H + U0 + i * kWU);
    }
    if (warp == 0) {
        tc::tmem_alloc(m.tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    for (int i = threadIdx.x; i < 3 * kWU; i += kWT) m.peep[i] = a.peep[(size_t)dir * 3 * H + (i / kWU) * H + u0 + i % kWU];
    tc::tc_fence_before_sync();
    __syncthreads();
    tc::tc_fence_after_sync();
    if (KS) cooperative_groups::this_cluster().sync();   // every peer's inbox barrier exists before any arrival
    const uint32_t tmem = *m.tmem_slot;
    // this thread's row in each peer's inbox (the slot a peer keeps for this CTA), 16-byte
    // chunks swizzled by row so that a warp's accesses spread over all banks
    uint32_t inbox_peer[4] = {0u, 0u, 0u, 0u};
    if (KS)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (c != crank) {
                const int slot = ((crank - c + 4) & 3) - 1;
                inbox_peer[c] = mapa_w(tc::smem_u32(m.inbox + ((size_t)slot * B + (j < B ? j : 0)) * kWU), (uint32_t)c);
            }
    const int swz = (j >> 1) & 3;

    float dcc[kWU];                                   // the cell-state error carried to the step before
#pragma unroll
    for (int k = 0; k < kWU; ++k) dcc[k] = 0.f;
    RingPos prod, cons;
    uint32_t mma_phase = 0, inbox_phase = 0;
    bool w_ready = false, failed = false;
    for (int s = 0; s < T && !failed; ++s) {
        const int t = dir == 0 ? T - 1 - s : s;
        const int n = a.bs[t];
        const int n_next = dir == 0 ? (t + 1 < T ? a.bs[t + 1] : 0) : (t >= 1 ? n : 0);
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < T ? a.bs[t + 1] : 0);
        const int prev_base = dir == 0 ? (t >= 1 ? a.off[t - 1] : 0) : (t + 1 < T ? a.off[t + 1] : 0);
        const int row = a.off[t] + j;
        wstamp(a, true, dir, cta, s, 0);
        // own operands of the row (before the wait): gates, c_t, c_{t-1}, dy
        float gv[4][kWU], cv[kWU], cp[kWU], dyv[kWU];
        const size_t so = j < B ? ((size_t)dir * B + a.perm[j]) * H + u0 : 0;   // caller-order state
        if (j < n) {
            const float* gr = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u0;
            const size_t yo = (size_t)row * ndH + (size_t)dir * H + u0;
            const size_t po = (size_t)(prev_base + j) * ndH + (size_t)dir * H + u0;
#pragma unroll
            for (int q = 0; q < kWU / 4; ++q) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H + 4 * q);
                    gv[g][4 * q] = x.x; gv[g][4 * q + 1] = x.y; gv[g][4 * q + 2] = x.z; gv[g][4 * q + 3] = x.w;
                }
                const float4 c4 = __ldg(reinterpret_cast<const float4*>(a.cbuf + yo + 4 * q));
                const float4 d4 = __ldg(reinterpret_cast<const float4*>(a.dy + yo + 4 * q));
                const float4 p4 = j < n_prev ? __ldg(reinterpret_cast<const float4*>(a.cbuf + po + 4 * q))
                                  : a.c0 ? __ldg(reinterpret_cast<const float4*>(a.c0 + so + 4 * q))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                cv[4 * q] = c4.x; cv[4 * q + 1] = c4.y; cv[4 * q + 2] = c4.z; cv[4 * q + 3] = c4.w;
                dyv[4 * q] = d4.x; dyv[4 * q + 1] = d4.y; dyv[4 * q + 2] = d4.z; dyv[4 * q + 3] = d4.w;
                cp[4 * q] = p4.x; cp[4 * q + 1] = p4.y; cp[4 * q + 2] = p4.z; cp[4 * q + 3] = p4.w;
            }
        }
        if (s + 1 < T) {           // the next step's gates, c and dy of this row into L2
            const int t2 = dir == 0 ? T - 2 - s : s + 1;
            if (j < a.bs[t2]) {
                const int r2 = a.off[t2] + j;
                const float* g2 = a.ga + (size_t)r2 * nd4H + (size_t)dir * 4 * H + u0;
#pragma unroll
                for (int g = 0; g < 4; ++g) asm volatile("prefetch.global.L2 [%0];" ::"l"(g2 + g * H));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.cbuf + (size_t)r2 * ndH + (size_t)dir * H + u0));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.dy + (size_t)r2 * ndH + (size_t)dir * H + u0));
            }
        }
        if (s > 0 && !grid_wait(ctr, (unsigned)(NC * s), a, 0xC0000u | (unsigned)s)) { failed = true; break; }
        wstamp(a, true, dir, cta, s, 1);
        // R^T da of the step after this one (recurrence order), for the rows that have one
        const int MT = (n_next + 127) / 128;
        if (MT > 0) {
            bool ok = wide_product<1>(m, &mapA, x0, (dir * 2 + (s & 1)) * B, MT, KB, NU, tmem, a, prod, cons,
                                      w_ready, 0xD0000u | (unsigned)(s & 0xfff), 0);
            ++mma_phase;
            if (threadIdx.x == 0) ok = tc::mbar_wait(m.mma_bar, (mma_phase - 1) & 1, a.wait_limit_ns) && ok;
            if (__syncthreads_or(!ok)) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, 0xE0000u | (unsigned)s);
                failed = true;
                break;
            }
            tc::tc_fence_after_sync();
        }
        wstamp(a, true, dir, cta, s, 5);
        float dhr[kWU];
#pragma unroll
        for (int k = 0; k < kWU; ++k) dhr[k] = 0.f;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        if (!KS) {
            if (tile < MT) {
                uint32_t r[16];
                tc::tmem_ld_32x32b_x16(tmem + lane_base + (uint32_t)(tile * kWU), r);
                tc::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < kWU; ++k) dhr[k] = j < n_next ? __uint_as_float(r[k]) : 0.f;
            }
        } else if (MT > 0) {
            // keep the own 16 columns, send the other three pieces to their owners
            if (tile < MT) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[16];
                    tc::tmem_ld_32x32b_x16(tmem + lane_base + (uint32_t)(tile * NU + c * kWU), r);
                    tc::tmem_wait_ld();
                    if (c == crank) {
#pragma unroll
                        for (int k = 0; k < kWU; ++k) dhr[k] = __uint_as_float(r[k]);
                    } else if (j < n_next) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            st_cluster_f4(inbox_peer[c] + (uint32_t)((q ^ swz) * 16), __uint_as_float(r[4 * q]),
                                          __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                                          __uint_as_float(r[4 * q + 3]));
                    }
                }
            }
            fence_acq_rel_cluster();
            __syncthreads();
            if (threadIdx.x == 0)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c != crank) mbar_arrive_remote(mapa_w(tc::smem_u32(m.inbox_bar), (uint32_t)c));
            // the three peers' pieces of this CTA's columns (every thread waits, bounded)
            int fail = 0;
            {
                const uint32_t par = inbox_phase & 1;
                if (!mbar_try_wait_cluster(m.inbox_bar, par)) {
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait_cluster(m.inbox_bar, par))
                        if (global_timer_ns() - t0 > a.wait_limit_ns || failure_recorded(a.status)) { fail = 1; break; }
                }
            }
            ++inbox_phase;
            if (__syncthreads_or(fail)) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, 0xF0000u | (unsigned)s);
                failed = true;
                break;
            }
            // own partial first, then the peers' in rank order after this CTA's (a fixed order
            // per unit: bitwise repeatable)
            if (j < n_next) {
#pragma unroll
                for (int slot = 0; slot < 3; ++slot) {
                    const float4* src = reinterpret_cast<const float4*>(m.inbox + ((size_t)slot * B + j) * kWU);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 v = src[q ^ swz];
                        dhr[4 * q] += v.x; dhr[4 * q + 1] += v.y; dhr[4 * q + 2] += v.z; dhr[4 * q + 3] += v.w;
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < kWU; ++k) dhr[k] = 0.f;
            }
        }
        wstamp(a, true, dir, cta, s, 2);
        // the cell; the bf16 gate errors go to the exchange buffer and are published first, the
        // fp32 gate errors (for the weight gradients) are stored after the publish
        float da[4][kWU];
        if (j < n) {
            const bool has_next = j < n_next;
            const bool real = !a.padded || t < a.len[j];
#pragma unroll
            for (int k = 0; k < kWU; ++k) {
                float dai = 0.f, daf = 0.f, daz = 0.f, dao = 0.f, carry_out = 0.f;
                if (real) {
                    // the sequence's last step: the final state's own errors from outside
                    const float dh = dyv[k] + (has_next ? dhr[k] : (a.dh_n ? __ldg(a.dh_n + so + k) : 0.f));
                    const float carry = has_next ? dcc[k] : (a.dc_n ? __ldg(a.dc_n + so + k) : 0.f);
                    const float ig = gv[0][k], fg = gv[1][k], zg = gv[2][k], og = gv[3][k];
                    const float tcv = tanh_w(cv[k]);
                    dao = dh * tcv * og * (1.f - og);
                    const float dc = dh * og * (1.f - tcv * tcv) + dao * m.peep[2 * kWU + k] + carry;
                    dai = dc * zg * ig * (1.f - ig);
                    daf = dc * cp[k] * fg * (1.f - fg);
                    daz = dc * ig * (1.f - zg * zg);
                    carry_out = dc * fg + dai * m.peep[k] + daf * m.peep[kWU + k];
                }
                da[0][k] = dai; da[1][k] = daf; da[2][k] = daz; da[3][k] = dao;
                dcc[k] = carry_out;
            }
            if (s + 1 < T) {         // bf16 gate errors for the next step's product
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t w8[kWU / 2];
#pragma unroll
                    for (int e = 0; e < kWU / 2; ++e) {
                        const __nv_bfloat162 p2 = __floats2bfloat162_rn(da[g][2 * e], da[g][2 * e + 1]);
                        w8[e] = *reinterpret_cast<const uint32_t*>(&p2);
                    }
                    uint4* xb = reinterpret_cast<uint4*>(
                        a.xbuf + (((size_t)dir * 2 + ((s + 1) & 1)) * B + j) * 4 * H + (size_t)g * H + u0);
                    xb[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
                    xb[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
                }
            }
        }
        fence_async_global();
        tc::tc_fence_before_sync();
        __syncthreads();
        wstamp(a, true, dir, cta, s, 3);
        if (threadIdx.x == 0 && !(s == 0 && dir == 0 && cta == a.debug_skip_cta))   // (test hook)
            red_release_add(ctr, 1u);
        wstamp(a, true, dir, cta, s, 4);
        if (j < n) {
            float* gw = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u0;
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int q = 0; q < kWU / 4; ++q)
                    *reinterpret_cast<float4*>(gw + g * H + 4 * q) =
                        make_float4(da[g][4 * q], da[g][4 * q + 1], da[g][4 * q + 2], da[g][4 * q + 3]);
            if (j >= n_prev && a.dc0 && (!a.padded || t < a.len[j]))     // the sequence's first step: dL/dc0
#pragma unroll
                for (int k = 0; k < kWU; ++k) a.dc0[so + k] = dcc[k];
        }
    }
    wide_finish<1, KS>(m, prod.it, mma_phase, failed);
    tc::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------- configuration

constexpr int kWCluster = 4;     // forward: CTAs sharing each operand tile; backward: the K split

static int optin_smem(const Plan& p)
{
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device) != cudaSuccess) return 0;
    return optin;
}

// Ring stages that fit beside a weight slice of KBW x rowsW x 128 B and an inbox: as many as
// fit, at most kWMaxStages and at most the plan's cap; 0 when fewer than two fit.
static int wide_stages(const Plan& p, int KBW, int rowsW, size_t inbox)
{
    const size_t optin = (size_t)optin_smem(p);
    int st = 0;
    for (int n = 2; n <= kWMaxStages; ++n)
        if (wide_smem_bytes(KBW, rowsW, n, inbox) <= optin) st = n;
    if (p.wide_stages > 0 && p.wide_stages < st) st = p.wide_stages;
    return st;
}

static size_t bwd_inbox_bytes(const Plan& p) { return (size_t)3 * p.B * kWU * 4; }

bool rec_wide_supported(const Plan& p, int H, int ndir, bool bf16)
{
    if (!bf16 || p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % 64 != 0 || H > 1024 || p.B > 256 || p.B < 1) return false;
    const int grid = ndir * H / kWU;
    if (grid > p.num_sms) return false;
    return wide_stages(p, H / 64, 64, 0) > 0 && wide_stages(p, 4 * H / 64, kWU, 0) > 0;
}

size_t rec_wide_xbuf_bytes(const Plan& p, int H, int ndir, bool bwd)
{
    return (size_t)ndir * 2 * p.B * (bwd ? 4 * H : H) * 2;
}

// One kernel form: its entry, shared memory and ring depth.
struct WideForm {
    const void* fn;
    size_t smem;
    int stages;
};

// One cooperative launch: the clustered form `f4` (clusters of kWCluster) when the plan allows
// it, it fits and the device co-schedules all of its clusters, else the plain form `f1` (when
// `plain` allows it; LSTM_ERR_UNSUPPORTED otherwise).  *cs receives the cluster size used.
static lstm_status wide_launch(const Plan& p, const WideForm& f1, const WideForm& f4, bool plain, WideArgs& a,
                               const CUtensorMap& mapW, const CUtensorMap& mapA, cudaStream_t s, int* cs)
{
    const int grid = a.ndir * a.NC;
    CUtensorMap mw = mapW, ma = mapA;
    void* args[] = {&a, &mw, &ma};
    if (cudaMemsetAsync(a.ctr, 0, sizeof(unsigned) * 2, s) != cudaSuccess) return LSTM_ERR_CUDA;
    if (p.wide_mode != 2 && a.NC % kWCluster == 0 && f4.stages > 0 &&
        cudaFuncSetAttribute(f4.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f4.smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kWT);
        cfg.dynamicSmemBytes = f4.smem;
        cfg.stream = s;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kWCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;                       // the occupancy query takes the cluster shape only
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, f4.fn, &cfg) == cudaSuccess && clusters * kWCluster >= grid) {
            cfg.numAttrs = 2;
            a.stages = f4.stages;
            if (cudaLaunchKernelExC(&cfg, f4.fn, args) == cudaSuccess) {
                *cs = kWCluster;
                return LSTM_OK;
            }
        }
        cudaGetLastError();                      // fall back to the plain launch below
    }
    if (!plain || f1.stages <= 0 ||
        cudaFuncSetAttribute(f1.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f1.smem) != cudaSuccess) {
        cudaGetLastError();
        return LSTM_ERR_UNSUPPORTED;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f1.fn, kWT, f1.smem) != cudaSuccess || per_sm < 1 ||
        per_sm * p.num_sms < grid) {
        cudaGetLastError();
        return LSTM_ERR_UNSUPPORTED;
    }
    a.stages = f1.stages;
    const cudaError_t e = cudaLaunchCooperativeKernel(f1.fn, dim3(grid), dim3(kWT), args, f1.smem, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorCooperativeLaunchTooLarge ? LSTM_ERR_UNSUPPORTED : LSTM_ERR_CUDA;
    }
    *cs = 1;
    return LSTM_OK;
}

lstm_status rec_wide_fwd_launch(const Plan& p, WideArgs a, const void* R, cudaStream_t s)
{
    a.NC = a.H / kWU;
    a.ctr = p.d_flags;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    CUtensorMap mapW, mapA;
    memset(&mapW, 0, sizeof(mapW));
    memset(&mapA, 0, sizeof(mapA));
    if (!make_map_bf16_sw128(&mapW, R, a.ndir * 4 * a.H, a.H, a.H, kWU) ||
        !make_map_bf16_sw128(&mapA, a.xbuf, a.ndir * 2 * a.B, a.H, a.H, 128))
        return LSTM_ERR_UNSUPPORTED;
    const int KB = a.H / 64, ns = wide_stages(p, KB, 64, 0);
    const WideForm f1 = {(const void*)lstm_rec_fwd_wide_kernel<1>, wide_smem_bytes(KB, 64, ns, 0), ns};
    const WideForm f4 = {(const void*)lstm_rec_fwd_wide_kernel<kWCluster>, f1.smem, ns};
    trace_begin(p, K_REC_FWD, s);
    int cs = 0;
    const lstm_status st = wide_launch(p, f1, f4, true, a, mapW, mapA, s, &cs);
    trace_end(p, K_REC_FWD, s, st == LSTM_OK ? 1 : 0);
    p.last_rec_variant[0] = cs;
    p.last_rec_stages[0] = st == LSTM_OK ? a.stages : 0;
    return st;
}

lstm_status rec_wide_bwd_launch(const Plan& p, WideArgs a, const void* RT, float* sum_scratch, float* db,
                                float* dpeep, cudaStream_t s)
{
    a.NC = a.H / kWU;
    a.ctr = p.d_flags;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    CUtensorMap mapW, mapA;
    memset(&mapW, 0, sizeof(mapW));
    memset(&mapA, 0, sizeof(mapA));
    if (!make_map_bf16_sw128(&mapW, RT, a.ndir * a.H, 4 * a.H, 4 * a.H, kWU) ||
        !make_map_bf16_sw128(&mapA, a.xbuf, a.ndir * 2 * a.B, 4 * a.H, 4 * a.H, 128))
        return LSTM_ERR_UNSUPPORTED;
    const int KB1 = 4 * a.H / 64, KB4 = a.H / 64;
    const size_t inbox = bwd_inbox_bytes(p);
    const int ns1 = wide_stages(p, KB1, kWU, 0), ns4 = wide_stages(p, KB4, 4 * kWU, inbox);
    const WideForm f1 = {(const void*)lstm_rec_bwd_wide_kernel<false>, wide_smem_bytes(KB1, kWU, ns1, 0), ns1};
    const WideForm f4 = {(const void*)lstm_rec_bwd_wide_kernel<true>, wide_smem_bytes(KB4, 4 * kWU, ns4, inbox), ns4};
    trace_begin(p, K_REC_BWD, s);
    int cs = 0;
    // automatic choice: only the split form (the plain one is slower than per-step launches)
    lstm_status st = wide_launch(p, f1, f4, p.wide_mode >= 1, a, mapW, mapA, s, &cs);
    p.last_rec_variant[1] = cs;
    p.last_rec_stages[1] = st == LSTM_OK ? a.stages : 0;
    int launched = st == LSTM_OK ? 1 : 0;
    if (st == LSTM_OK) {
        st = param_sums_launch(p, a.ga, a.cbuf, a.H, a.ndir, db, dpeep, sum_scratch, s, a.c0);
        if (st == LSTM_OK) launched += 2;
    }
    trace_end(p, K_REC_BWD, s, launched);
    return st;
}

}  // namespace lstm
