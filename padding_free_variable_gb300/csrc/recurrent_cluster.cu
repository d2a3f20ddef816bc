// recurrent_cluster.cu -- cluster-resident recurrent forward kernel.
//
// The same recurrence as lstm_rec_fwd_kernel ("Single Stream Parallelization
// of Generalized LSTM-Like RNNs on a GPU", Sec. 3: one sequential step per
// frame, the delayed connection R h_{t-1} then the cell), laid out for a
// thread-block cluster when one direction's R fits in the cluster:
//
//  * one cluster of G = H/32 CTAs per direction; CTA c owns units
//    [32c, 32c+32) and their 128 gate rows of R, resident in shared memory
//    in the tcgen05 128-byte-swizzled K-major layout (bf16; fp32 operands
//    are stored as bf16 hi + lo and multiplied as lo*hi + hi*lo + hi*hi);
//  * per step one thread issues tcgen05.mma: D[128 gate rows][n rows] in
//    tensor memory = R_slice x h_{t-1}^T, h taken from a shared-memory
//    operand buffer that the peers filled;
//  * the cell runs on the accumulator, and each CTA writes its new h (split
//    and swizzled) straight into every peer's next operand buffer through
//    distributed shared memory;
//  * one hardware cluster barrier per step replaces the grid-wide flag
//    barrier (measured on GB300: ~0.22 us for 16 CTAs against ~1.8 us for a
//    64-CTA flag barrier).
// Every CTA of a cluster runs exactly the same sequence of cluster barriers,
// so none can leave early; the only other wait (MMA completion) is bounded
// and a timeout is recorded in the plan's status word.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "recurrent.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace lstm {

namespace {

constexpr int kCU = 32;        // units per CTA
constexpr int kCM = 128;       // gate rows per CTA (MMA M)
constexpr int kCT = 256;       // threads
constexpr int kSumChunks = 64; // row chunks of the db / dpeep sums
constexpr int kChains = 4;     // independent TMEM accumulators per product (summed at read-out)

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

// 8 fp32 values -> bf16 hi (rounded) and lo (rounded remainder), packed 2 per word
__device__ __forceinline__ void split8(const float (&v)[8], uint4& hi, uint4& lo, bool want_lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = bf16x2(v[2 * i], v[2 * i + 1]);
        if (want_lo) {
            const float a = v[2 * i] - __uint_as_float(h[i] << 16);
            const float b = v[2 * i + 1] - __uint_as_float(h[i] & 0xffff0000u);
            l[i] = bf16x2(a, b);
        } else {
            l[i] = 0u;
        }
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
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

// 4 fp32 values -> bf16 hi and lo remainder, 2 per word
__device__ __forceinline__ void split4(const float (&v)[4], uint2& hi, uint2& lo, bool want_lo)
{
    const uint32_t h0 = bf16x2(v[0], v[1]), h1 = bf16x2(v[2], v[3]);
    hi = make_uint2(h0, h1);
    if (want_lo) {
        lo = make_uint2(bf16x2(v[0] - __uint_as_float(h0 << 16), v[1] - __uint_as_float(h0 & 0xffff0000u)),
                        bf16x2(v[2] - __uint_as_float(h1 << 16), v[3] - __uint_as_float(h1 & 0xffff0000u)));
    } else {
        lo = make_uint2(0u, 0u);
    }
}

__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

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

}  // namespace

// RecArgs offsets reused: off_h = A_hi, off_red = A_lo, off_acc = accs,
// off_state = cell states, off_contrib = B buffers, off_sums = mbarrier and
// TMEM slot, off_tab = tables, off_peep = peepholes.
template <bool SPLIT>
__global__ void __launch_bounds__(kCT, 1) lstm_rec_fwd_cluster_kernel(RecArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cl = cg::this_cluster();
    const int G = a.G;
    const int rank = (int)cl.block_rank();
    const int dir = blockIdx.x / G;
    const int H = a.H, T = a.T, NBM = a.JC;          // JC carries the operand buffer rows (multiple of 16)
    const int KB = (H + 63) / 64;
    const int u0 = rank * kCU;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    uint8_t* Ahi = base + a.off_h;
    uint8_t* Alo = base + a.off_red;
    float* accs = reinterpret_cast<float*>(base + a.off_acc);        // [NBM][128]
    float* cst = reinterpret_cast<float*>(base + a.off_state);       // [B][32]
    uint8_t* Bb = base + a.off_contrib;                              // [2 parity][2 hi/lo][KB][NBM][128 B]
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(base + a.off_sums);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
    int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
    float* peep_s = reinterpret_cast<float*>(base + a.off_peep);     // [3][32]
    int* s_bs = reinterpret_cast<int*>(base + a.off_tab);
    int* s_off = s_bs + T;
    int* s_len = s_off + T + 1;
    const size_t bsz = (size_t)KB * NBM * 128;                       // bytes of one B operand
    auto Bop = [&](int parity, int lo) -> uint8_t* { return Bb + (size_t)(parity * 2 + lo) * bsz; };
    const uint32_t tcols = (uint32_t)a.Umax;                         // Umax carries the TMEM columns

    // ---- set-up: R slice, operands zeroed, tables, barrier, tensor memory
    const __nv_bfloat16* Rb = reinterpret_cast<const __nv_bfloat16*>(a.R);
    const float* Rf = reinterpret_cast<const float*>(a.R);
    for (int idx = threadIdx.x; idx < kCM * KB * 8; idx += kCT) {
        const int r = idx / (KB * 8), rem = idx - r * (KB * 8);
        const int k0 = rem * 8;
        const int g = r / kCU, uu = r - g * kCU;
        const size_t grow = (size_t)dir * 4 * H * H + (size_t)(g * H + u0 + uu) * H;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int k = k0 + e;
            v[e] = k < H ? (SPLIT ? Rf[grow + k] : __bfloat162float(Rb[grow + k])) : 0.f;
        }
        uint4 hi, lo;
        split8(v, hi, lo, SPLIT);
        const uint32_t o = sw_off(r, k0, kCM);
        *reinterpret_cast<uint4*>(Ahi + o) = hi;
        if (SPLIT) *reinterpret_cast<uint4*>(Alo + o) = lo;
    }
    for (size_t i = threadIdx.x; i < 4 * bsz / 16; i += kCT) reinterpret_cast<uint4*>(Bb)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < T; i += kCT) s_bs[i] = a.bs[i];
    for (int i = threadIdx.x; i <= T; i += kCT) s_off[i] = a.off[i];
    for (int i = threadIdx.x; i < a.B; i += kCT) s_len[i] = a.slot_len[i];
    for (int i = threadIdx.x; i < 3 * kCU; i += kCT) {
        const int q = i / kCU, uu = i - q * kCU;
        peep_s[i] = a.peep[(size_t)dir * 3 * H + q * H + u0 + uu];
    }
    if (threadIdx.x == 0) {
        tc::mbar_init(mma_bar, kChains);
        *s_fail = 0;
        tc::fence_mbar_init();
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
    if (a.h_n) {
        for (int idx = threadIdx.x; idx < a.B * kCU; idx += kCT) {
            const int j = idx / kCU, uu = idx - j * kCU;
            if (s_len[j] == 0) {
                const size_t o = ((size_t)dir * a.B + a.perm[j]) * H + u0 + uu;
                a.h_n[o] = 0.f;
                if (a.c_n) a.c_n[o] = 0.f;
            }
        }
    }
    cl.sync();     // every CTA of the cluster is resident before any remote write

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jq = threadIdx.x >> 3, q8 = threadIdx.x & 7;          // cell item: row jq (+32k), units q8*4..+4
    const int nks = (H + 15) / 16;                                   // MMA k-steps
    const int nch = min(kChains, nks);
    for (int s = 0; s < T; ++s) {
        const int t = dir == 0 ? s : T - 1 - s;
        const int n = s_bs[t];
        const int rowbase = s_off[t];
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < T ? s_bs[t + 1] : 0);
        const int NBs = (n + 15) & ~15;
        const int cur = s & 1;
        cstamp(a, false, dir, rank, s, 0, 0);
        // D[gate rows][rows] = R_slice x h_{t-1}^T: chain ch (k-steps ch, ch + kChains, ...) is
        // issued by warp ch into its own accumulator, so the chains overlap
        if (lane == 0 && warp < kChains && !*(volatile int*)s_fail) {
            fence_proxy_async_cta();
            tc::tc_fence_after_sync();
            cstamp(a, false, dir, rank, s, 1, 1);
            const uint32_t idesc = tc::idesc_bf16_f32(kCM, NBs);
            const uint64_t dah = tc::sdesc_sw128(tc::smem_u32(Ahi)), dal = tc::sdesc_sw128(tc::smem_u32(Alo));
            const uint64_t dbh = tc::sdesc_sw128(tc::smem_u32(Bop(cur, 0))), dbl = tc::sdesc_sw128(tc::smem_u32(Bop(cur, 1)));
            const uint32_t d = tmem + (uint32_t)(warp * NBM);
            for (int i = warp; i < nks; i += kChains) {
                const uint32_t ao = (uint32_t)(i >> 2) * kCM * 128 + (uint32_t)(i & 3) * 32;
                const uint32_t bo = (uint32_t)(i >> 2) * NBM * 128 + (uint32_t)(i & 3) * 32;
                const uint32_t acc = i == warp ? 0u : 1u;
                if (SPLIT) {
                    tc::mma_bf16_ss(d, desc_add(dal, ao), desc_add(dbh, bo), idesc, acc);
                    tc::mma_bf16_ss(d, desc_add(dah, ao), desc_add(dbl, bo), idesc, 1u);
                    tc::mma_bf16_ss(d, desc_add(dah, ao), desc_add(dbh, bo), idesc, 1u);
                } else {
                    tc::mma_bf16_ss(d, desc_add(dah, ao), desc_add(dbh, bo), idesc, acc);
                }
            }
            tc::mma_commit(mma_bar);
        }
        if (warp < kChains) __syncwarp();     // the issuing lane's warp does not poll while it issues
        cstamp(a, false, dir, rank, s, 6, 6);
        // meanwhile: the cell items' own operands (gate pre-activations), rows jq and jq + 32
        float pre[2][4][4];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int j = jq + it * 32;
            if (j < n) {
                const float* gr = a.ga + (size_t)(rowbase + j) * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H);
                    pre[it][g][0] = x.x; pre[it][g][1] = x.y; pre[it][g][2] = x.z; pre[it][g][3] = x.w;
                }
            }
        }
        if (s + 1 < T) {   // next step's own rows into L2 (4 gate blocks of this CTA's units)
            const int t2 = dir == 0 ? s + 1 : T - 2 - s;
            for (int g = 0; g < 4; ++g)
                prefetch_rows(a.ga, nd4H, s_off[t2], s_bs[t2], dir * 4 * H + g * H + u0);
        }
        const bool ok = *(volatile int*)s_fail ? false : tc::mbar_wait(mma_bar, (uint32_t)(s & 1), a.wait_limit_ns);
        if (!ok && !*(volatile int*)s_fail) {
            record_failure(a.status, LSTM_ERR_TIMEOUT, 0x40000u | (unsigned)s);
            *(volatile int*)s_fail = 1;
        }
        cstamp(a, false, dir, rank, s, 7, 7);
        tc::tc_fence_after_sync();
        // accumulators -> shared: warp (quarter q = gate, half) reads lanes 32q.. in 16-column blocks
        {
            const int q = warp & 3, half = warp >> 2;
            for (int c0 = half * 16; c0 < NBs; c0 += 32) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = 0.f;
                for (int ch = 0; ch < nch; ++ch) {
                    uint32_t r[16];
                    tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ch * NBM + c0), r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] += __uint_as_float(r[e]);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) accs[(size_t)(c0 + e) * kCM + q * 32 + lane] = v[e];
            }
        }
        tc::tc_fence_before_sync();
        __syncthreads();
        cstamp(a, false, dir, rank, s, 2, 2);
        // cell: row j, units u0 + q8*4 .. +4
        const int nxt = cur ^ 1;
        for (int it = 0; it * 32 < n; ++it) {
            const int j = jq + it * 32;
            if (j >= n) continue;
            const int row = rowbase + j;
            const int len = s_len[j];
            float pv[4][4];
            if (it < 2) {
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < 4; ++e) pv[g][e] = it == 0 ? pre[0][g][e] : pre[1][g][e];
            } else {
                const float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(gr + g * H);
                    pv[g][0] = x.x; pv[g][1] = x.y; pv[g][2] = x.z; pv[g][3] = x.w;
                }
            }
            float hv[4], cv[4], gg[4][4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int uu = q8 * 4 + e;
                const float* ac = accs + (size_t)j * kCM + uu;
                const float cp = j < n_prev ? cst[j * kCU + uu] : 0.f;
                const float ig = sigm_c(pv[0][e] + ac[0] + peep_s[uu] * cp);
                const float fg = sigm_c(pv[1][e] + ac[32] + peep_s[32 + uu] * cp);
                const float zg = tanh_c(pv[2][e] + ac[64]);
                float c = fg * cp + ig * zg;
                const float og = sigm_c(pv[3][e] + ac[96] + peep_s[64 + uu] * c);
                float h = og * tanh_c(c);
                if (a.padded && t >= len) { c = 0.f; h = 0.f; }
                gg[0][e] = ig; gg[1][e] = fg; gg[2][e] = zg; gg[3][e] = og; cv[e] = c; hv[e] = h;
                cst[j * kCU + uu] = c;
            }
            float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + q8 * 4;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<float4*>(gr + g * H) = make_float4(gg[g][0], gg[g][1], gg[g][2], gg[g][3]);
            const size_t yo = (size_t)row * ndH + dir * H + u0 + q8 * 4;
            *reinterpret_cast<float4*>(a.cbuf + yo) = make_float4(cv[0], cv[1], cv[2], cv[3]);
            *reinterpret_cast<float4*>(a.y + yo) = make_float4(hv[0], hv[1], hv[2], hv[3]);
            uint2 hi, lo;
            split4(hv, hi, lo, SPLIT);
            if (a.y_lo) *reinterpret_cast<uint2*>(a.y_lo + yo) = hi;
            if (a.h_n && ((dir == 0 && t == len - 1) || (dir == 1 && t == 0 && len > 0))) {
                const size_t o = ((size_t)dir * a.B + a.perm[j]) * H + u0 + q8 * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a.h_n[o + e] = hv[e];
                    if (a.c_n) a.c_n[o + e] = cv[e];
                }
            }
            if (it == 0) cstamp(a, false, dir, rank, s, 5, 5);
            // h_t into every peer's operand of the next step (row j, columns u0 + q8*4 ..)
            if (s + 1 < T) {
                const uint32_t o = sw_off4(j, u0 + q8 * 4, NBM);
                for (int p2 = 0; p2 < G; ++p2) {
                    *reinterpret_cast<uint2*>(cl.map_shared_rank(Bop(nxt, 0) + o, p2)) = hi;
                    if (SPLIT) *reinterpret_cast<uint2*>(cl.map_shared_rank(Bop(nxt, 1) + o, p2)) = lo;
                }
            }
        }
        fence_proxy_async_cluster();
        cstamp(a, false, dir, rank, s, 3, 3);
        cl.sync();
        cstamp(a, false, dir, rank, s, 4, 4);
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        __syncwarp();
        tc::tc_fence_after_sync();
        if (*(volatile int*)s_fail) tc::mbar_wait(mma_bar, (uint32_t)((T - 1) & 1) ^ 1u, a.wait_limit_ns);
        tc::tmem_dealloc(tmem, tcols);
    }
}

// ------------------------------------------------------------------------- backward
//
// BPTT of the same recurrence ("Single Stream Parallelization...", Sec. 2) in
// the same cluster layout.  The error reaching h_t through R is
// R^T da_{t+1}; CTA c holds its 128 gate rows of R and the gate errors it
// computes for them, so it forms the partial product P_c = R_c^T da_c for
// every unit on the tensor cores, and pushes the part of P_c that belongs to
// CTA c' (its 32 units) into c''s inbox through distributed shared memory.
// At the next step each CTA adds the G partials of its units in CTA order.
// db and dpeep are summed afterwards by lstm_param_sums_kernel.
// RecArgs offsets: off_h = A_hi, off_red = A_lo, off_contrib = B (gate
// errors), off_acc = inbox, off_state = dc carry, off_sums = mbarrier, TMEM
// slot, failure flag, off_peep = peepholes, off_tab = tables.
template <bool SPLIT>
__global__ void __launch_bounds__(kCT, 1) lstm_rec_bwd_cluster_kernel(RecArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    cg::cluster_group cl = cg::this_cluster();
    const int G = a.G;
    const int rank = (int)cl.block_rank();
    const int dir = blockIdx.x / G;
    const int H = a.H, T = a.T, NBM = a.JC;
    const int MT = (H + kCM - 1) / kCM;              // 128-unit tiles of the partial product
    const int AR = MT * kCM;                         // rows of the R^T operand (zero padded)
    const int u0 = rank * kCU;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    uint8_t* Ahi = base + a.off_h;
    uint8_t* Alo = base + a.off_red;
    uint8_t* Bhi = base + a.off_contrib;             // [2 k-blocks][NBM][128 B]
    uint8_t* Blo = Bhi + (size_t)2 * NBM * 128;
    float* inbox = reinterpret_cast<float*>(base + a.off_acc);       // [2][G][NBM][32]
    float* dcc = reinterpret_cast<float*>(base + a.off_state);       // [B][32]
    uint64_t* mma_bar = reinterpret_cast<uint64_t*>(base + a.off_sums);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 1);
    int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
    float* peep_s = reinterpret_cast<float*>(base + a.off_peep);
    int* s_bs = reinterpret_cast<int*>(base + a.off_tab);
    int* s_off = s_bs + T;
    int* s_len = s_off + T + 1;
    const uint32_t tcols = (uint32_t)a.Umax;
    auto inbox_at = [&](int parity, int src, int j) -> float* {
        return inbox + (((size_t)parity * G + src) * NBM + j) * kCU;
    };

    // R^T slice: row u' (any unit), column r = g*32 + uu (this CTA's gate rows)
    const __nv_bfloat16* Rb = reinterpret_cast<const __nv_bfloat16*>(a.R);
    const float* Rf = reinterpret_cast<const float*>(a.R);
    for (int idx = threadIdx.x; idx < AR * 16; idx += kCT) {
        const int up = idx >> 4, r0 = (idx & 15) * 8;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int r = r0 + e, g = r / kCU, uu = r - g * kCU;
            const size_t src = (size_t)dir * 4 * H * H + (size_t)(g * H + u0 + uu) * H + up;
            v[e] = up < H ? (SPLIT ? Rf[src] : __bfloat162float(Rb[src])) : 0.f;
        }
        uint4 hi, lo;
        split8(v, hi, lo, SPLIT);
        const uint32_t o = sw_off(up, r0, AR);
        *reinterpret_cast<uint4*>(Ahi + o) = hi;
        if (SPLIT) *reinterpret_cast<uint4*>(Alo + o) = lo;
    }
    for (int i = threadIdx.x; i < 2 * 2 * NBM * 128 / 16; i += kCT) reinterpret_cast<uint4*>(Bhi)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < 2 * G * NBM * kCU; i += kCT) inbox[i] = 0.f;
    for (int i = threadIdx.x; i < T; i += kCT) s_bs[i] = a.bs[i];
    for (int i = threadIdx.x; i <= T; i += kCT) s_off[i] = a.off[i];
    for (int i = threadIdx.x; i < a.B; i += kCT) s_len[i] = a.slot_len[i];
    for (int i = threadIdx.x; i < 3 * kCU; i += kCT) {
        const int q = i / kCU, uu = i - q * kCU;
        peep_s[i] = a.peep[(size_t)dir * 3 * H + q * H + u0 + uu];
    }
    if (threadIdx.x == 0) {
        tc::mbar_init(mma_bar, kChains);
        *s_fail = 0;
        tc::fence_mbar_init();
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
    cl.sync();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jq = threadIdx.x >> 3, q8 = threadIdx.x & 7;          // cell item: row jq (+32k), units q8*4..+4
    // own operands (gates, c_t, c_{t-1}, dy) of row jq of a step, loaded one step ahead
    float nx[7][4];
    auto load_own = [&](int s2) {
        const int t2 = dir == 0 ? T - 1 - s2 : s2;
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
        const int np2 = dir == 0 ? (t2 >= 1 ? n2 : 0) : (t2 + 1 < T ? s_bs[t2 + 1] : 0);
        if (jq < np2) {
            const int pb2 = dir == 0 ? s_off[t2 - 1] : s_off[t2 + 1];
            const float4 p0 = __ldg(reinterpret_cast<const float4*>(a.cbuf + (size_t)(pb2 + jq) * ndH + dir * H + u0 + q8 * 4));
            nx[5][0] = p0.x; nx[5][1] = p0.y; nx[5][2] = p0.z; nx[5][3] = p0.w;
        } else {
            nx[5][0] = nx[5][1] = nx[5][2] = nx[5][3] = 0.f;
        }
    };
    load_own(0);
    for (int s = 0; s < T; ++s) {
        const int t = dir == 0 ? T - 1 - s : s;
        const int n = s_bs[t];
        const int rowbase = s_off[t];
        const int n_next = dir == 0 ? (t + 1 < T ? s_bs[t + 1] : 0) : (t >= 1 ? n : 0);
        const int prev_base = dir == 0 ? (t >= 1 ? s_off[t - 1] : 0) : (t + 1 < T ? s_off[t + 1] : 0);
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < T ? s_bs[t + 1] : 0);
        const int NBs = (n + 15) & ~15;
        const int cur = s & 1, nxt = cur ^ 1;
        cstamp(a, true, dir, rank, s, 0, 1);
        for (int it = 0; it * 32 < n; ++it) {
            const int j = jq + it * 32;
            if (j >= n) continue;
            const int row = rowbase + j;
            const int uub = q8 * 4;
            float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u0 + uub;
            float gv[4][4], cv[4], cpv[4], dyv[4];
            if (it == 0) {
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
            {
                const float4 c0 = __ldg(reinterpret_cast<const float4*>(a.cbuf + yo));
                cv[0] = c0.x; cv[1] = c0.y; cv[2] = c0.z; cv[3] = c0.w;
                const float4 d0 = __ldg(reinterpret_cast<const float4*>(a.dy + yo));
                dyv[0] = d0.x; dyv[1] = d0.y; dyv[2] = d0.z; dyv[3] = d0.w;
                if (j < n_prev) {
                    const float4 p0 = __ldg(reinterpret_cast<const float4*>(
                        a.cbuf + (size_t)(prev_base + j) * ndH + dir * H + u0 + uub));
                    cpv[0] = p0.x; cpv[1] = p0.y; cpv[2] = p0.z; cpv[3] = p0.w;
                } else {
                    cpv[0] = cpv[1] = cpv[2] = cpv[3] = 0.f;
                }
            }
            }
            const bool has_next = j < n_next;
            const bool real = !a.padded || t < s_len[j];
            float da[4][4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int uu = uub + e;
                float dh_rec = 0.f;
                if (has_next)
                    for (int c2 = 0; c2 < G; ++c2) dh_rec += inbox_at(cur, c2, j)[uu];
                float dai = 0.f, daf = 0.f, daz = 0.f, dao = 0.f, carry_out = 0.f;
                if (real) {
                    const float ig = gv[0][e], fg = gv[1][e], zg = gv[2][e], og = gv[3][e];
                    const float c = cv[e], cp = cpv[e];
                    const float dh = dyv[e] + dh_rec;
                    const float carry = has_next ? dcc[j * kCU + uu] : 0.f;
                    const float tc = tanh_c(c);
                    dao = dh * tc * og * (1.f - og);
                    const float dc = dh * og * (1.f - tc * tc) + dao * peep_s[64 + uu] + carry;
                    dai = dc * zg * ig * (1.f - ig);
                    daf = dc * cp * fg * (1.f - fg);
                    daz = dc * ig * (1.f - zg * zg);
                    carry_out = dc * fg + dai * peep_s[uu] + daf * peep_s[32 + uu];
                }
                da[0][e] = dai; da[1][e] = daf; da[2][e] = daz; da[3][e] = dao;
                dcc[j * kCU + uu] = carry_out;
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                *reinterpret_cast<float4*>(gr + g * H) = make_float4(da[g][0], da[g][1], da[g][2], da[g][3]);
                uint2 hi, lo;
                split4(da[g], hi, lo, SPLIT);
                const uint32_t o = sw_off4(j, g * kCU + uub, NBM);
                *reinterpret_cast<uint2*>(Bhi + o) = hi;
                if (SPLIT) *reinterpret_cast<uint2*>(Blo + o) = lo;
            }
        }
        fence_proxy_async_cta();
        __syncthreads();
        cstamp(a, true, dir, rank, s, 2, 2);
        if (s + 1 < T) {
            // P[u'][j] = sum over this CTA's gate rows r of R[r][u'] da[j][r]; chain ch of the 8
            // k-steps (k = ch, ch + kChains, ...) is issued by warp ch into accumulators (m, ch)
            if (lane == 0 && warp < kChains && !*(volatile int*)s_fail) {
                tc::tc_fence_after_sync();
                const uint32_t idesc = tc::idesc_bf16_f32(kCM, NBs);
                const uint64_t dah = tc::sdesc_sw128(tc::smem_u32(Ahi)), dal = tc::sdesc_sw128(tc::smem_u32(Alo));
                const uint64_t dbh = tc::sdesc_sw128(tc::smem_u32(Bhi)), dbl = tc::sdesc_sw128(tc::smem_u32(Blo));
                for (int i = warp; i < 8; i += kChains) {
                    const uint32_t bo = (uint32_t)(i >> 2) * NBM * 128 + (uint32_t)(i & 3) * 32;
                    const uint32_t acc = i == warp ? 0u : 1u;
                    for (int m = 0; m < MT; ++m) {
                        const uint32_t ao = (uint32_t)(i >> 2) * AR * 128 + (uint32_t)m * kCM * 128 + (uint32_t)(i & 3) * 32;
                        const uint32_t d = tmem + (uint32_t)((m * kChains + warp) * NBM);
                        if (SPLIT) {
                            tc::mma_bf16_ss(d, desc_add(dal, ao), desc_add(dbh, bo), idesc, acc);
                            tc::mma_bf16_ss(d, desc_add(dah, ao), desc_add(dbl, bo), idesc, 1u);
                            tc::mma_bf16_ss(d, desc_add(dah, ao), desc_add(dbh, bo), idesc, 1u);
                        } else {
                            tc::mma_bf16_ss(d, desc_add(dah, ao), desc_add(dbh, bo), idesc, acc);
                        }
                    }
                }
                tc::mma_commit(mma_bar);
            }
            if (warp < kChains) __syncwarp();
            cstamp(a, true, dir, rank, s, 6, 6);
            const bool ok = *(volatile int*)s_fail ? false : tc::mbar_wait(mma_bar, (uint32_t)(s & 1), a.wait_limit_ns);
            if (!ok && !*(volatile int*)s_fail) {
                record_failure(a.status, LSTM_ERR_TIMEOUT, 0x50000u | (unsigned)s);
                *(volatile int*)s_fail = 1;
            }
            tc::tc_fence_after_sync();
            cstamp(a, true, dir, rank, s, 5, 7);
            // tile m, lane quarter q: units u' = 128m + 32q + lane, owned by CTA 4m + q
            for (int pq = warp; pq < MT * 4; pq += kCT / 32) {
                const int m = pq >> 2, q = pq & 3;
                const int owner = 4 * m + q;
                if (owner >= G) continue;
                float* dst_base = cl.map_shared_rank(inbox_at(nxt, rank, 0), owner);
                for (int c0 = 0; c0 < NBs; c0 += 16) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = 0.f;
                    for (int ch = 0; ch < kChains; ++ch) {
                        uint32_t r[16];
                        tc::tmem_ld_32x32b_x16(tmem + ((uint32_t)(q * 32) << 16) +
                                                   (uint32_t)((m * kChains + ch) * NBM + c0), r);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] += __uint_as_float(r[e]);
                    }
                    // lanes are consecutive units: each store is one coalesced 128-byte row
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (c0 + e < n) dst_base[(size_t)(c0 + e) * kCU + lane] = v[e];
                }
            }
            tc::tc_fence_before_sync();
        }
        if (s + 1 < T) load_own(s + 1);       // the next step's own operands, in flight across the barrier
        cstamp(a, true, dir, rank, s, 3, 3);
        cl.sync();
        cstamp(a, true, dir, rank, s, 4, 4);
    }
    tc::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        __syncwarp();
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem, tcols);
    }
}

// db and dpeep from the gate errors: column (direction, quantity q, unit u),
// q = 0..3 -> sum of da_q, 4 -> da_i c_{t-1}, 5 -> da_f c_{t-1}, 6 -> da_o c_t;
// each thread sums its column over one chunk of rows in row order, and the
// chunks are then added in chunk order (bitwise repeatable).
__global__ void lstm_param_sums_kernel(const float* __restrict__ ga, const float* __restrict__ cbuf,
                                       const int32_t* __restrict__ prev_fwd, const int32_t* __restrict__ prev_rev,
                                       int rows, int H, int ndir, int chunk, float* __restrict__ partial)
{
    const int ncols = ndir * 7 * H;
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= ncols) return;
    const int d = col / (7 * H), rem = col - d * 7 * H, q = rem / H, u = rem - q * H;
    const int r0 = blockIdx.y * chunk, r1 = min(rows, r0 + chunk);
    const int nd4H = ndir * 4 * H, ndH = ndir * H;
    const int32_t* prev = d == 0 ? prev_fwd : prev_rev;
    const int gq = q < 4 ? q : (q == 4 ? 0 : (q == 5 ? 1 : 3));
    float s = 0.f;
    for (int r = r0; r < r1; ++r) {
        const float v = __ldg(ga + (size_t)r * nd4H + d * 4 * H + gq * H + u);
        if (q < 4) s += v;
        else if (q < 6) {
            const int pr = __ldg(prev + r);
            s += pr >= 0 ? v * __ldg(cbuf + (size_t)pr * ndH + d * H + u) : 0.f;
        } else {
            s += v * __ldg(cbuf + (size_t)r * ndH + d * H + u);
        }
    }
    partial[(size_t)blockIdx.y * ncols + col] = s;
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

bool rec_cluster_fwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* lay)
{
    if (p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % kCU != 0) return false;
    const int G = H / kCU;
    if (G > 16 || G * ndir > p.num_sms) return false;
    int bmax = 0;
    for (int t = 0; t < p.T; ++t) bmax = std::max(bmax, p.h_bs[t]);
    const int NBM = std::max(16, (bmax + 15) & ~15);
    if (NBM > 128) return false;                   // cell items: 2 rows of 64 per thread
    const int KB = (H + 63) / 64;
    const bool split = !bf16;
    size_t off = 0;
    const size_t abytes = (size_t)KB * kCM * 128;
    const size_t o_ahi = off; off = al(off + abytes, 1024);
    const size_t o_alo = off; if (split) off = al(off + abytes, 1024);
    const size_t o_b = off; off = al(off + 4 * (size_t)KB * NBM * 128, 1024);
    const size_t o_acc = off; off = al(off + (size_t)NBM * kCM * 4, 16);
    const size_t o_cst = off; off = al(off + (size_t)p.B * kCU * 4, 16);
    const size_t o_bar = off; off = al(off + 64, 16);
    const size_t o_peep = off; off = al(off + 3 * kCU * 4, 16);
    const size_t o_tab = off; off = al(off + (size_t)(2 * p.T + 1 + p.B) * 4, 16);
    const size_t smem = off + 1024 + 64;          // 1024 for the base alignment, 64 static
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device) != cudaSuccess) return false;
    if (smem > (size_t)optin) return false;
    uint32_t cols = 32;
    while (cols < (uint32_t)(kChains * NBM)) cols <<= 1;
    if (cols > 512) return false;
    RecConfig c;
    c.G = G; c.Umax = (int)cols; c.JC = NBM; c.smem = smem; c.cluster = 1;
    *out = c;
    lay->off_h = (int)o_ahi; lay->off_red = (int)o_alo; lay->off_contrib = (int)o_b; lay->off_acc = (int)o_acc;
    lay->off_state = (int)o_cst; lay->off_sums = (int)o_bar; lay->off_peep = (int)o_peep; lay->off_tab = (int)o_tab;
    return true;
}

lstm_status rec_cluster_fwd_launch(const Plan& p, const RecConfig& c, RecArgs a, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    void* fn = a.bf16 ? (void*)lstm_rec_fwd_cluster_kernel<false> : (void*)lstm_rec_fwd_cluster_kernel<true>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem) != cudaSuccess)
        return LSTM_ERR_CUDA;
    if (c.G > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return LSTM_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(c.G * a.ndir);
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c.G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin(p, K_REC_FWD, s);
    void* args[] = {&a};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    trace_end(p, K_REC_FWD, s, e == cudaSuccess ? 1 : 0);
    if (e != cudaSuccess) { cudaGetLastError(); return LSTM_ERR_UNSUPPORTED; }
    return LSTM_OK;
}

bool rec_cluster_bwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* lay)
{
    if (p.gemm_engine != 0 || p.forced_ctas != 0) return false;
    if (H % kCU != 0) return false;
    const int G = H / kCU;
    if (G > 16 || G * ndir > p.num_sms) return false;
    int bmax = 0;
    for (int t = 0; t < p.T; ++t) bmax = std::max(bmax, p.h_bs[t]);
    const int NBM = std::max(16, (bmax + 15) & ~15);
    if (NBM > 128) return false;
    const int MT = (H + kCM - 1) / kCM;
    const bool split = !bf16;
    const size_t abytes = (size_t)MT * kCM * 2 * 128;
    size_t off = 0;
    const size_t o_ahi = off; off = al(off + abytes, 1024);
    const size_t o_alo = off; if (split) off = al(off + abytes, 1024);
    const size_t o_b = off; off = al(off + (size_t)2 * 2 * NBM * 128, 1024);
    const size_t o_in = off; off = al(off + (size_t)2 * G * NBM * kCU * 4, 16);
    const size_t o_dcc = off; off = al(off + (size_t)p.B * kCU * 4, 16);
    const size_t o_bar = off; off = al(off + 64, 16);
    const size_t o_peep = off; off = al(off + 3 * kCU * 4, 16);
    const size_t o_tab = off; off = al(off + (size_t)(2 * p.T + 1 + p.B) * 4, 16);
    const size_t smem = off + 1024 + 64;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device) != cudaSuccess) return false;
    if (smem > (size_t)optin) return false;
    uint32_t cols = 32;
    while (cols < (uint32_t)(MT * kChains * NBM)) cols <<= 1;
    if (cols > 512) return false;
    RecConfig c;
    c.G = G; c.Umax = (int)cols; c.JC = NBM; c.smem = smem; c.cluster = 1;
    *out = c;
    lay->off_h = (int)o_ahi; lay->off_red = (int)o_alo; lay->off_contrib = (int)o_b; lay->off_acc = (int)o_in;
    lay->off_state = (int)o_dcc; lay->off_sums = (int)o_bar; lay->off_peep = (int)o_peep; lay->off_tab = (int)o_tab;
    return true;
}

size_t rec_cluster_bwd_sum_floats(int H, int ndir) { return (size_t)kSumChunks * ndir * 7 * H; }

lstm_status rec_cluster_bwd_launch(const Plan& p, const RecConfig& c, RecArgs a, float* sum_scratch, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    void* fn = a.bf16 ? (void*)lstm_rec_bwd_cluster_kernel<false> : (void*)lstm_rec_bwd_cluster_kernel<true>;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem) != cudaSuccess)
        return LSTM_ERR_CUDA;
    if (c.G > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return LSTM_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(c.G * a.ndir);
    cfg.blockDim = dim3(kCT);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c.G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin(p, K_REC_BWD, s);
    void* args[] = {&a};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    int launched = e == cudaSuccess ? 1 : 0;
    if (e == cudaSuccess) {
        const int ncols = a.ndir * 7 * a.H;
        const int rows = (int)p.rows;
        const int chunk = (rows + kSumChunks - 1) / kSumChunks;
        lstm_param_sums_kernel<<<dim3((ncols + 255) / 256, kSumChunks), 256, 0, s>>>(
            a.ga, a.cbuf, p.d_prev_fwd, p.d_prev_rev, rows, a.H, a.ndir, chunk, sum_scratch);
        lstm_param_sums_combine<<<(ncols + 255) / 256, 256, 0, s>>>(sum_scratch, kSumChunks, a.H, a.ndir, a.db,
                                                                    a.dpeep);
        e = cudaGetLastError();
        launched += e == cudaSuccess ? 2 : 0;
    }
    trace_end(p, K_REC_BWD, s, launched);
    if (e != cudaSuccess) { cudaGetLastError(); return LSTM_ERR_UNSUPPORTED; }
    return LSTM_OK;
}

}  // namespace lstm
