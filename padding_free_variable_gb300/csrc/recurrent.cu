// recurrent.cu -- persistent recurrent kernels of the packed LSTM.
//
// "Single Stream Parallelization of Generalized LSTM-Like RNNs on a GPU",
// Sec. 3: once the non-recurrent part is done for all frames, only the
// recurrent node remains sequential; each step computes the delayed
// connection R h_{t-1} and then the cell's element-wise graph.  The backward
// pass runs the same steps in reverse order (BPTT, Sec. 2).
//
// GB300 layout of the work:
//  * One cooperative launch runs every step of both directions.  The CTAs of
//    direction d split the H units; CTA c owns units [c*U, c*U+U) with all
//    four gates, so the cell update is local.  The CTA's rows of R stay in
//    shared memory for the whole launch.
//  * Step s of the forward direction is time t = s; of the reverse direction
//    t = T-1-s.  Step t runs only the bs[t] rows still active: packed rows
//    off[t] .. off[t]+bs[t]-1.  No padded frame is computed.
//  * Forward exchange: every CTA reads the whole h_{t-1} of its direction
//    (written by its peers in the previous step) and multiplies it by its
//    own rows of R.
//  * Backward exchange (reduce-scatter): the error reaching h_t is
//    R^T da_{t+1}.  Each CTA multiplies the gate errors it just computed by
//    its own rows of R, producing a partial sum for every unit, and
//    publishes it; at the next step a CTA adds the G partials of its own
//    units in a fixed order.  The product runs before the barrier, and each
//    CTA reads G*U values per row instead of all 4H gate errors.
//  * Between steps the CTAs of one direction meet at a flag barrier: each CTA
//    publishes its step count with a release store; a CTA reads every peer's
//    count with acquire loads before it reads their outputs.  Every wait has
//    a time limit; a CTA that runs out records LSTM_ERR_TIMEOUT in the
//    plan's status word and the whole launch returns.
//  * The operands of a step that come from the CTA itself or from earlier
//    launches (gate pre-activations, cell states, upstream errors) are
//    loaded before the barrier wait, so their latency overlaps it.
#include <algorithm>

#include "common.cuh"
#include "recurrent.cuh"

namespace lstm {

namespace {

constexpr int kMaxItems = 4;      // cell items per thread held in registers
constexpr int kMaxJC = 32;        // rows per chunk

// Logistic and tanh from the hardware exp2 (relative error of __expf about
// 2^-21; absolute error of both functions below 1e-6 over the whole line).
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float tanhf_(float x)
{
    const float e = __expf(2.0f * fminf(fmaxf(x, -40.0f), 40.0f));
    return 1.0f - __fdividef(2.0f, e + 1.0f);
}

// 8 consecutive matrix elements from shared memory as floats.
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const unsigned w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// ---------------------------------------------------------------- warp-level tensor-core MMA
//
// The per-step product is small (16-32 gate rows per CTA, <= 32 rows of the
// batch per chunk) and on the critical path of every step, so it runs as
// mma.sync with the CTA's R fragments held in registers for the whole launch.
// fp32 operands use three tf32 products (hi*hi + hi*lo + lo*hi, with x = hi +
// lo split at load), which keeps about 22 bits of each product; bf16
// operands use one bf16 product.

constexpr int kFwdMTW = 2, kFwdKTW = 4;    // m-tiles and k-steps per warp, forward
constexpr int kBwdMTW = 4, kBwdKTW = 2;    // backward

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo)
{
    hi = to_tf32(x);
    lo = to_tf32(x - __uint_as_float(hi));
}

// bf16 pair: `lo_k` (the smaller k index) in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo_k, float hi_k)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_k), "f"(lo_k));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragments (m16 x k) of a matrix given element-wise by `at(row, col)`:
// tf32 -> hi/lo of m16n8k8 fragments; bf16 -> m16n8k16 fragments in hi.
template <bool BF16, typename F>
__device__ __forceinline__ void load_a_frag(F at, int mt, int kt, uint32_t (&hi)[4], uint32_t (&lo)[4])
{
    const int lane = threadIdx.x & 31, grp = lane >> 2, tig = lane & 3;
    const int r0 = mt * 16 + grp, r1 = r0 + 8;
    if (!BF16) {
        const int k0 = kt * 8 + tig, k1 = k0 + 4;
        split_tf32(at(r0, k0), hi[0], lo[0]);
        split_tf32(at(r1, k0), hi[1], lo[1]);
        split_tf32(at(r0, k1), hi[2], lo[2]);
        split_tf32(at(r1, k1), hi[3], lo[3]);
    } else {
        const int k0 = kt * 16 + 2 * tig;
        hi[0] = pack_bf16x2(at(r0, k0), at(r0, k0 + 1));
        hi[1] = pack_bf16x2(at(r1, k0), at(r1, k0 + 1));
        hi[2] = pack_bf16x2(at(r0, k0 + 8), at(r0, k0 + 9));
        hi[3] = pack_bf16x2(at(r1, k0 + 8), at(r1, k0 + 9));
        lo[0] = lo[1] = lo[2] = lo[3] = 0u;
    }
}

// One k-step of C(m16 x n8) += A * B where B(k, n) = V[n][k] (V rows of stride ldv floats).
template <bool BF16>
__device__ __forceinline__ void mma_step(float (&acc)[4], const uint32_t (&ahi)[4], const uint32_t (&alo)[4],
                                         const float* __restrict__ V, int ldv, int nt, int kt)
{
    const int lane = threadIdx.x & 31, grp = lane >> 2, tig = lane & 3;
    const float* row = V + (size_t)(nt * 8 + grp) * ldv;
    if (!BF16) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(row[kt * 8 + tig], bh0, bl0);
        split_tf32(row[kt * 8 + tig + 4], bh1, bl1);
        mma_tf32(acc, alo, bh0, bh1);
        mma_tf32(acc, ahi, bl0, bl1);
        mma_tf32(acc, ahi, bh0, bh1);
    } else {
        const int k0 = kt * 16 + 2 * tig;
        const float2 x0 = *reinterpret_cast<const float2*>(row + k0);
        const float2 x1 = *reinterpret_cast<const float2*>(row + k0 + 8);
        mma_bf16(acc, ahi, pack_bf16x2(x0.x, x0.y), pack_bf16x2(x1.x, x1.y));
    }
}

// outs[j][r] = sum_k M[r][k] * V[j][k] for r < RP, j < jn.
// M: RP rows (stride ldm elements), V: JC rows (stride ldv floats), K a
// multiple of 8, RP and JC multiples of 4.  Each (item) owns a 4x4 block of
// (r, j) over one k-slice: rows {rg + i*NRG}, j {jg + q*NJG}; the KS slices
// are summed through `red` in a fixed order (bitwise repeatable).
template <typename MT>
__device__ void smem_matmul(const MT* __restrict__ Ms, int ldm, const float* __restrict__ Vs, int ldv,
                            int RP, int JC, int K, int jn, float* __restrict__ red,
                            float* __restrict__ outs)
{
    const int NRG = RP >> 2, NJG = JC >> 2;
    const int groups = NRG * NJG;
    int KS = kRecThreads / groups;
    if (KS < 1) KS = 1;
    if (KS > (K >> 3)) KS = K >> 3;
    const int KL = (((K + KS - 1) / KS) + 7) & ~7;
    const int tid = threadIdx.x;
    // more (group, slice) items than threads when a CTA owns many units: loop
    for (int item = tid; item < groups * KS; item += kRecThreads) {
        const int ks = item / groups;
        const int g = item - ks * groups;
        const int jg = g % NJG;
        const int rg = g / NJG;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][q] = 0.f;
        const int k0 = ks * KL;
        const int k1 = min(K, k0 + KL);
        if (jg < jn) {
            for (int k = k0; k < k1; k += 8) {
                float m[4][8], v[4][8];
#pragma unroll
                for (int i = 0; i < 4; ++i) load8(Ms + (size_t)(rg + i * NRG) * ldm + k, m[i]);
#pragma unroll
                for (int q = 0; q < 4; ++q) load8(Vs + (size_t)(jg + q * NJG) * ldv + k, v[q]);
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(m[i][e], v[q][e], acc[i][q]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = rg + i * NRG, j = jg + q * NJG;
                red[((size_t)ks * RP + r) * JC + j] = acc[i][q];
            }
    }
    __syncthreads();
    for (int o = tid; o < RP * jn; o += kRecThreads) {
        const int j = o / RP, r = o - j * RP;
        float s = 0.f;
        for (int ks = 0; ks < KS; ++ks) s += red[((size_t)ks * RP + r) * JC + j];
        outs[j * RP + r] = s;
    }
    __syncthreads();
}

// Wait until every CTA of this direction has published step count >= target.
// Returns false (uniformly across the CTA) when the launch must stop.
__device__ bool step_barrier(const unsigned* flags, int G, unsigned target, DeviceStatus* st,
                             unsigned long long limit_ns, int cta_global, int step)
{
    __shared__ int s_fail;
    if (threadIdx.x == 0) s_fail = 0;
    __syncthreads();
    if (threadIdx.x < G) {
        const unsigned* f = flags + threadIdx.x;
        const unsigned long long t0 = global_timer_ns();
        unsigned spins = 0;
        while ((int)(ld_acquire_gpu(f) - target) < 0) {
            if ((++spins & 63u) == 0) {
                if (failure_recorded(st)) { s_fail = 1; break; }
                if (global_timer_ns() - t0 > limit_ns) {
                    record_failure(st, LSTM_ERR_TIMEOUT, ((unsigned)cta_global << 20) | (unsigned)(step & 0xfffff));
                    s_fail = 1;
                    break;
                }
            }
        }
    }
    __syncthreads();
    const bool ok = (s_fail == 0);
    __syncthreads();
    return ok;
}

__device__ __forceinline__ void step_publish(unsigned* flag, unsigned value, bool skip)
{
    __syncthreads();
    if (threadIdx.x == 0 && !skip) {
        __threadfence();
        st_release_gpu(flag, value);
    }
}

struct Tables {
    const int* bs;
    const int* off;
    const int* len;
};

// Step tables, copied to shared memory when they fit (the caller syncs).
__device__ Tables load_tables(const RecArgs& a, int* s_tab)
{
    if (!a.tables_in_smem) return Tables{a.bs, a.off, a.slot_len};
    int* s_bs = s_tab;
    int* s_off = s_tab + a.T;
    int* s_len = s_off + a.T + 1;
    for (int i = threadIdx.x; i < a.T; i += kRecThreads) s_bs[i] = a.bs[i];
    for (int i = threadIdx.x; i <= a.T; i += kRecThreads) s_off[i] = a.off[i];
    for (int i = threadIdx.x; i < a.B; i += kRecThreads) s_len[i] = a.slot_len[i];
    return Tables{s_bs, s_off, s_len};
}

__device__ __forceinline__ void stamp(const RecArgs& a, bool bwd, int dir, int cta, int s, int k)
{
    if (a.trace && cta == 0 && threadIdx.x == 0 && s < a.trace_steps)
        a.trace[(((size_t)(bwd ? 1 : 0) * a.ndir + dir) * a.trace_steps + s) * 8 + k] = clock64();
}

}  // namespace

// ------------------------------------------------------------------------- forward

template <typename RT, bool MMA>
__global__ void __launch_bounds__(kRecThreads, 1) lstm_rec_fwd_kernel(RecArgs a)
{
    constexpr bool BF16 = sizeof(RT) == 2;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int H = a.H, G = a.G, Umax = a.Umax, RP = 4 * Umax, JC = a.JC, T = a.T;
    const int dir = blockIdx.x / G;
    const int cta = blockIdx.x - dir * G;
    const int u0 = cta * Umax;
    const int Uc = max(0, min(Umax, H - u0));
    const int ldr = H + 16 / (int)sizeof(RT);     // padded row stride of R slice (elements)
    const int ldh = H + 4;                         // padded row stride of h chunk (floats)
    RT* Rs = reinterpret_cast<RT*>(smem_raw);
    float* hs = reinterpret_cast<float*>(smem_raw + a.off_h);
    float* red = reinterpret_cast<float*>(smem_raw + a.off_red);
    float* accs = reinterpret_cast<float*>(smem_raw + a.off_acc);
    float* cst = reinterpret_cast<float*>(smem_raw + a.off_state);
    float* peep_s = reinterpret_cast<float*>(smem_raw + a.off_peep);
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const RT* Rg = reinterpret_cast<const RT*>(a.R) + (size_t)dir * 4 * H * H;
    unsigned* myflags = a.flags + dir * kMaxCtasPerDir;
    const bool skip_pub = (a.debug_skip_cta == (int)blockIdx.x);

    // resident R slice: row r = g*Umax + uu holds R[g*H + u0 + uu][:]
    for (int idx = threadIdx.x; idx < RP * H; idx += kRecThreads) {
        const int r = idx / H, k = idx - r * H;
        const int g = r / Umax, uu = r - g * Umax;
        RT v = RT(0.f);
        if (uu < Uc) v = Rg[(size_t)(g * H + u0 + uu) * H + k];
        Rs[(size_t)r * ldr + k] = v;
    }
    for (int idx = threadIdx.x; idx < 3 * Umax; idx += kRecThreads) {
        const int q = idx / Umax, uu = idx - q * Umax;
        peep_s[idx] = uu < Uc ? a.peep[(size_t)dir * 3 * H + q * H + u0 + uu] : 0.f;
    }
    const Tables tb = load_tables(a, reinterpret_cast<int*>(smem_raw + a.off_tab));
    __syncthreads();
    // tensor-core path: this warp's R fragments, resident in registers
    const int warp = threadIdx.x >> 5;
    const int mw = a.mma_mw, kw = a.mma_kw, MT = (RP + 15) / 16, KT = H / (BF16 ? 16 : 8);
    const int ktw = (KT + kw - 1) / kw;
    const int wm = warp / kw, wk = warp - (warp / kw) * kw;
    const bool mma_warp = MMA && warp < mw * kw;
    uint32_t fa_hi[kFwdMTW][kFwdKTW][4], fa_lo[kFwdMTW][kFwdKTW][4];
    if (MMA) {
        auto at = [&](int r, int k) -> float { return r < RP ? to_f32(Rs[(size_t)r * ldr + k]) : 0.f; };
#pragma unroll
        for (int i = 0; i < kFwdMTW; ++i)
#pragma unroll
            for (int q = 0; q < kFwdKTW; ++q) {
                const int mt = wm + i * mw, kt = wk * ktw + q;
                if (mma_warp && mt < MT && q < ktw && kt < KT) load_a_frag<BF16>(at, mt, kt, fa_hi[i][q], fa_lo[i][q]);
                else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) fa_hi[i][q][e] = fa_lo[i][q][e] = 0u;
                }
            }
    }
    // empty sequences end in their initial state (zero without one)
    if (a.h_n) {
        for (int idx = threadIdx.x; idx < a.B * Uc; idx += kRecThreads) {
            const int j = idx / Uc, uu = idx - j * Uc;
            if (tb.len[j] == 0) {
                const size_t o = ((size_t)dir * a.B + a.perm[j]) * H + u0 + uu;
                a.h_n[o] = a.h0 ? a.h0[o] : 0.f;
                if (a.c_n) a.c_n[o] = a.c0 ? a.c0[o] : 0.f;
            }
        }
    }

    for (int s = 0; s < T; ++s) {
        const int t = dir == 0 ? s : T - 1 - s;
        const int n = tb.bs[t];
        const int rowbase = tb.off[t];
        // h_{t-1} of slot j: forward direction row (t-1, j); reverse direction
        // row (t+1, j) when slot j is still active there
        const int prev_base = dir == 0 ? (t >= 1 ? tb.off[t - 1] : 0) : (t + 1 < T ? tb.off[t + 1] : 0);
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < T ? tb.bs[t + 1] : 0);
        stamp(a, false, dir, cta, s, 0);

        // gate pre-activations of this thread's cell items (own data: before the barrier)
        float pre[kMaxItems][4];
        auto prefetch = [&](int j0, int jn) {
#pragma unroll
            for (int k = 0; k < kMaxItems; ++k) {
                const int idx = threadIdx.x + k * kRecThreads;
                if (idx < jn * Uc) {
                    const int jj = idx / Uc, uu = idx - jj * Uc;
                    const float* gr = a.ga + (size_t)(rowbase + j0 + jj) * nd4H + dir * 4 * H + u0 + uu;
#pragma unroll
                    for (int g = 0; g < 4; ++g) pre[k][g] = gr[g * H];
                }
            }
        };
        prefetch(0, min(JC, n));
        if (s > 0 && G > 1) {
            if (!step_barrier(myflags, G, (unsigned)s, a.status, a.wait_limit_ns, blockIdx.x, s)) return;
        }
        stamp(a, false, dir, cta, s, 1);
        for (int j0 = 0; j0 < n; j0 += JC) {
            const int jn = min(JC, n - j0);
            if (j0 > 0) prefetch(j0, jn);
            // stage h_{t-1} of the chunk (zero where the row has no predecessor)
            const int H4 = H >> 2;
            for (int idx = threadIdx.x; idx < jn * H4; idx += kRecThreads) {
                const int jj = idx / H4, k4 = idx - jj * H4;
                const int j = j0 + jj;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < n_prev) {
                    v = __ldcg(reinterpret_cast<const float4*>(a.y + (size_t)(prev_base + j) * ndH + dir * H) + k4);
                    if (a.bf16) { v.x = bf16_round(v.x); v.y = bf16_round(v.y); v.z = bf16_round(v.z); v.w = bf16_round(v.w); }
                }
                *reinterpret_cast<float4*>(hs + (size_t)jj * ldh + 4 * k4) = v;
            }
            __syncthreads();
            if (j0 == 0) stamp(a, false, dir, cta, s, 2);
            if (!MMA) {
                smem_matmul<RT>(Rs, ldr, hs, ldh, RP, JC, H, jn, red, accs);
            } else {
                // accs[j][r] = sum over k-slices (warps wk) of the warps' m16 x n8 tiles
                if (mma_warp) {
                    const int lane = threadIdx.x & 31, grp = lane >> 2, tig = lane & 3;
                    const int NT = (jn + 7) >> 3;
                    float acc[kFwdMTW][4][4];
#pragma unroll
                    for (int i = 0; i < kFwdMTW; ++i)
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[i][nt][e] = 0.f;
#pragma unroll
                    for (int q = 0; q < kFwdKTW; ++q) {
                        const int kt = wk * ktw + q;
                        if (q >= ktw || kt >= KT) continue;
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
                            if (nt >= NT) continue;
#pragma unroll
                            for (int i = 0; i < kFwdMTW; ++i)
                                if (wm + i * mw < MT) mma_step<BF16>(acc[i][nt], fa_hi[i][q], fa_lo[i][q], hs, ldh, nt, kt);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kFwdMTW; ++i) {
                        const int mt = wm + i * mw;
                        if (mt >= MT) continue;
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int r = mt * 16 + grp + ((e & 2) ? 8 : 0);
                                const int j = nt * 8 + 2 * tig + (e & 1);
                                if (r < RP && j < jn) red[((size_t)wk * RP + r) * JC + j] = acc[i][nt][e];
                            }
                        }
                    }
                }
                __syncthreads();
                for (int o = threadIdx.x; o < RP * jn; o += kRecThreads) {
                    const int j = o / RP, r = o - j * RP;
                    float sacc = 0.f;
                    for (int w2 = 0; w2 < kw; ++w2) sacc += red[((size_t)w2 * RP + r) * JC + j];
                    accs[j * RP + r] = sacc;
                }
                __syncthreads();
            }
            if (j0 == 0) stamp(a, false, dir, cta, s, 5);
            // cell update, one (row, unit) per item
#pragma unroll
            for (int k = 0; k < kMaxItems; ++k) {
                const int idx = threadIdx.x + k * kRecThreads;
                if (idx < jn * Uc) {
                    const int jj = idx / Uc, uu = idx - jj * Uc;
                    const int j = j0 + jj, u = u0 + uu;
                    const int row = rowbase + j;
                    const float* ac = accs + jj * RP;
                    const float cp = j < n_prev ? cst[j * Umax + uu]
                                                : (a.c0 ? a.c0[((size_t)dir * a.B + a.perm[j]) * H + u] : 0.f);
                    const float ig = sigmoidf_(pre[k][0] + ac[uu] + peep_s[uu] * cp);
                    const float fg = sigmoidf_(pre[k][1] + ac[Umax + uu] + peep_s[Umax + uu] * cp);
                    const float zg = tanhf_(pre[k][2] + ac[2 * Umax + uu]);
                    float c = fg * cp + ig * zg;
                    const float og = sigmoidf_(pre[k][3] + ac[3 * Umax + uu] + peep_s[2 * Umax + uu] * c);
                    float h = og * tanhf_(c);
                    const int len = tb.len[j];
                    if (a.padded && t >= len) { c = 0.f; h = 0.f; }
                    float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u;
                    gr[0] = ig; gr[H] = fg; gr[2 * H] = zg; gr[3 * H] = og;
                    const size_t yo = (size_t)row * ndH + dir * H + u;
                    a.cbuf[yo] = c;
                    a.y[yo] = h;
                    if (a.y_lo) a.y_lo[yo] = __float2bfloat16_rn(h);
                    cst[j * Umax + uu] = c;
                    if (a.h_n && ((dir == 0 && t == len - 1) || (dir == 1 && t == 0 && len > 0))) {
                        const size_t o = ((size_t)dir * a.B + a.perm[j]) * H + u;
                        a.h_n[o] = h;
                        if (a.c_n) a.c_n[o] = c;
                    }
                }
            }
            __syncthreads();
        }
        stamp(a, false, dir, cta, s, 3);
        if (G > 1) step_publish(myflags + cta, (unsigned)(s + 1), skip_pub);
        stamp(a, false, dir, cta, s, 4);
    }
}

// ------------------------------------------------------------------------- backward

template <typename RT, bool MMA>
__global__ void __launch_bounds__(kRecThreads, 1) lstm_rec_bwd_kernel(RecArgs a)
{
    constexpr bool BF16 = sizeof(RT) == 2;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int H = a.H, G = a.G, Umax = a.Umax, JC = a.JC, T = a.T, B = a.B;
    // R rows padded to a multiple of the MMA k-step (8 tf32, 16 bf16)
    const int RP8 = BF16 ? ((4 * Umax + 15) & ~15) : ((4 * Umax + 7) & ~7);
    const int ldd = RP8 + 4;                       // padded row stride of da_s
    const int dir = blockIdx.x / G;
    const int cta = blockIdx.x - dir * G;
    const int u0 = cta * Umax;
    const int Uc = max(0, min(Umax, H - u0));
    const int ldr = H + 16 / (int)sizeof(RT);
    RT* Rs = reinterpret_cast<RT*>(smem_raw);
    float* da_s = reinterpret_cast<float*>(smem_raw + a.off_h);       // [JC][ldd]
    float* dcc = reinterpret_cast<float*>(smem_raw + a.off_state);    // [B][Umax]
    float* contrib = reinterpret_cast<float*>(smem_raw + a.off_contrib);   // [7][JC][Umax]
    float* sums = reinterpret_cast<float*>(smem_raw + a.off_sums);    // [7][Umax]
    float* peep_s = reinterpret_cast<float*>(smem_raw + a.off_peep);
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const RT* Rg = reinterpret_cast<const RT*>(a.R) + (size_t)dir * 4 * H * H;
    unsigned* myflags = a.flags + dir * kMaxCtasPerDir;
    const bool skip_pub = (a.debug_skip_cta == (int)blockIdx.x);
    // part[parity][dir][j][c][H]
    auto part_at = [&](int parity, int j, int c) -> float* {
        return a.part + ((((size_t)parity * a.ndir + dir) * B + j) * G + c) * H;
    };

    for (int idx = threadIdx.x; idx < RP8 * H; idx += kRecThreads) {
        const int r = idx / H, k = idx - r * H;
        const int g = r / Umax, uu = r - g * Umax;
        RT v = RT(0.f);
        if (g < 4 && uu < Uc) v = Rg[(size_t)(g * H + u0 + uu) * H + k];
        Rs[(size_t)r * ldr + k] = v;
    }
    for (int idx = threadIdx.x; idx < JC * ldd; idx += kRecThreads) da_s[idx] = 0.f;
    for (int idx = threadIdx.x; idx < 7 * Umax; idx += kRecThreads) sums[idx] = 0.f;
    for (int idx = threadIdx.x; idx < 3 * Umax; idx += kRecThreads) {
        const int q = idx / Umax, uu = idx - q * Umax;
        peep_s[idx] = uu < Uc ? a.peep[(size_t)dir * 3 * H + q * H + u0 + uu] : 0.f;
    }
    const Tables tb = load_tables(a, reinterpret_cast<int*>(smem_raw + a.off_tab));
    __syncthreads();
    // tensor-core path: fragments of R^T (rows = units u', cols = this CTA's gate rows)
    const int warp = threadIdx.x >> 5;
    const int MTb = H / 16, KTb = RP8 / (BF16 ? 16 : 8);
    uint32_t fb_hi[kBwdMTW][kBwdKTW][4], fb_lo[kBwdMTW][kBwdKTW][4];
    if (MMA) {
        auto at = [&](int up, int r) -> float { return to_f32(Rs[(size_t)r * ldr + up]); };
#pragma unroll
        for (int i = 0; i < kBwdMTW; ++i)
#pragma unroll
            for (int q = 0; q < kBwdKTW; ++q) {
                const int mt = warp + i * (kRecThreads / 32);
                if (mt < MTb && q < KTb) load_a_frag<BF16>(at, mt, q, fb_hi[i][q], fb_lo[i][q]);
                else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) fb_hi[i][q][e] = fb_lo[i][q][e] = 0u;
                }
            }
    }

    for (int s = 0; s < T; ++s) {
        const int t = dir == 0 ? T - 1 - s : s;
        const int n = tb.bs[t];
        const int rowbase = tb.off[t];
        // rows whose later step (in this direction's order) exists: their partials arrive
        const int n_next = dir == 0 ? (t + 1 < T ? tb.bs[t + 1] : 0) : (t >= 1 ? n : 0);
        // c_{t-1} of slot j (previous step in this direction's forward order)
        const int prev_base = dir == 0 ? (t >= 1 ? tb.off[t - 1] : 0) : (t + 1 < T ? tb.off[t + 1] : 0);
        const int n_prev = dir == 0 ? (t >= 1 ? n : 0) : (t + 1 < T ? tb.bs[t + 1] : 0);
        stamp(a, true, dir, cta, s, 0);

        // own operands of this thread's cell items, loaded before the barrier:
        // gates i f z o, c_t, c_{t-1}, upstream error
        float op[kMaxItems][7];
        auto prefetch = [&](int j0, int jn) {
#pragma unroll
            for (int k = 0; k < kMaxItems; ++k) {
                const int idx = threadIdx.x + k * kRecThreads;
                if (idx < jn * Uc) {
                    const int jj = idx / Uc, uu = idx - jj * Uc;
                    const int j = j0 + jj, u = u0 + uu;
                    const int row = rowbase + j;
                    const float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u;
#pragma unroll
                    for (int g = 0; g < 4; ++g) op[k][g] = gr[g * H];
                    const size_t yo = (size_t)row * ndH + dir * H + u;
                    op[k][4] = __ldg(a.cbuf + yo);
                    op[k][5] = j < n_prev ? __ldg(a.cbuf + (size_t)(prev_base + j) * ndH + dir * H + u)
                                          : (a.c0 ? __ldg(a.c0 + ((size_t)dir * a.B + a.perm[j]) * H + u) : 0.f);
                    op[k][6] = __ldg(a.dy + yo);
                }
            }
        };
        prefetch(0, min(JC, n));
        if (s > 0 && G > 1) {
            if (!step_barrier(myflags, G, (unsigned)s, a.status, a.wait_limit_ns, blockIdx.x, s)) return;
        }
        stamp(a, true, dir, cta, s, 1);
        const int rd = (s - 1) & 1, wr = s & 1;
        for (int j0 = 0; j0 < n; j0 += JC) {
            const int jn = min(JC, n - j0);
            if (j0 > 0) prefetch(j0, jn);
#pragma unroll
            for (int k = 0; k < kMaxItems; ++k) {
                const int idx = threadIdx.x + k * kRecThreads;
                if (idx < jn * Uc) {
                    const int jj = idx / Uc, uu = idx - jj * Uc;
                    const int j = j0 + jj, u = u0 + uu;
                    const int row = rowbase + j;
                    const float ig = op[k][0], fg = op[k][1], zg = op[k][2], og = op[k][3];
                    const float c = op[k][4], cp = op[k][5];
                    const bool has_next = j < n_next;
                    // error reaching h_t through R: the peers' partials, in CTA order
                    float dh_rec = 0.f;
                    const size_t so = ((size_t)dir * a.B + a.perm[j]) * H + u;   // caller-order state
                    if (has_next) {
                        const float* pp = part_at(rd, j, 0) + u;
                        for (int c2 = 0; c2 < G; ++c2) dh_rec += __ldcg(pp + (size_t)c2 * H);
                    } else if (a.dh_n) {
                        dh_rec = __ldg(a.dh_n + so);          // the sequence's last step: the final state's error
                    }
                    float dai = 0.f, daf = 0.f, daz = 0.f, dao = 0.f, carry_out = 0.f;
                    const bool real = !a.padded || t < tb.len[j];
                    if (real) {
                        const float dh = op[k][6] + dh_rec;
                        const float carry = has_next ? dcc[j * Umax + uu] : (a.dc_n ? __ldg(a.dc_n + so) : 0.f);
                        const float tc = tanhf_(c);
                        dao = dh * tc * og * (1.f - og);
                        const float dc = dh * og * (1.f - tc * tc) + dao * peep_s[2 * Umax + uu] + carry;
                        dai = dc * zg * ig * (1.f - ig);
                        daf = dc * cp * fg * (1.f - fg);
                        daz = dc * ig * (1.f - zg * zg);
                        carry_out = dc * fg + dai * peep_s[uu] + daf * peep_s[Umax + uu];
                        if (j >= n_prev && a.dc0) a.dc0[so] = carry_out;   // the sequence's first step
                    }
                    float* gr = a.ga + (size_t)row * nd4H + dir * 4 * H + u;
                    gr[0] = dai; gr[H] = daf; gr[2 * H] = daz; gr[3 * H] = dao;
                    float* dr = da_s + jj * ldd + uu;
                    if (a.bf16) {
                        dr[0] = bf16_round(dai); dr[Umax] = bf16_round(daf);
                        dr[2 * Umax] = bf16_round(daz); dr[3 * Umax] = bf16_round(dao);
                    } else {
                        dr[0] = dai; dr[Umax] = daf; dr[2 * Umax] = daz; dr[3 * Umax] = dao;
                    }
                    dcc[j * Umax + uu] = carry_out;
                    const int cs = JC * Umax;
                    float* cb = contrib + jj * Umax + uu;
                    cb[0 * cs] = dai; cb[1 * cs] = daf; cb[2 * cs] = daz; cb[3 * cs] = dao;
                    cb[4 * cs] = dai * cp; cb[5 * cs] = daf * cp; cb[6 * cs] = dao * c;
                }
            }
            __syncthreads();
            if (j0 == 0) stamp(a, true, dir, cta, s, 2);
            // this CTA's share of R^T da for every unit, read by all peers at the next step
            if (s + 1 < T && MMA) {
                // D(u', j) = sum_r R[r][u'] da[j][r]: m16 tiles of units, n8 tiles of rows
                const int lane = threadIdx.x & 31, grp = lane >> 2, tig = lane & 3;
                const int NT = (jn + 7) >> 3;
#pragma unroll
                for (int i = 0; i < kBwdMTW; ++i) {
                    const int mt = warp + i * (kRecThreads / 32);
                    if (mt >= MTb) continue;
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        if (nt >= NT) continue;
                        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int q = 0; q < kBwdKTW; ++q)
                            if (q < KTb) mma_step<BF16>(acc, fb_hi[i][q], fb_lo[i][q], da_s, ldd, nt, q);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int up = mt * 16 + grp + ((e & 2) ? 8 : 0);
                            const int jj = nt * 8 + 2 * tig + (e & 1);
                            if (jj < jn) part_at(wr, j0 + jj, cta)[up] = acc[e];
                        }
                    }
                }
            }
            if (s + 1 < T && !MMA) {
                for (int up = threadIdx.x; up < H; up += kRecThreads) {
                    float acc[kMaxJC];
#pragma unroll
                    for (int jj = 0; jj < kMaxJC; ++jj) acc[jj] = 0.f;
                    for (int r0 = 0; r0 < RP8; r0 += 8) {
                        float rv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) rv[e] = to_f32(Rs[(size_t)(r0 + e) * ldr + up]);
#pragma unroll
                        for (int jj = 0; jj < kMaxJC; ++jj) {
                            if (jj < jn) {
                                float d[8];
                                load8(da_s + jj * ldd + r0, d);
                                float v = acc[jj];
#pragma unroll
                                for (int e = 0; e < 8; ++e) v = fmaf(rv[e], d[e], v);
                                acc[jj] = v;
                            }
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < kMaxJC; ++jj)
                        if (jj < jn) part_at(wr, j0 + jj, cta)[up] = acc[jj];
                }
            }
            if (j0 == 0) stamp(a, true, dir, cta, s, 5);
            for (int idx = threadIdx.x; idx < 7 * Uc; idx += kRecThreads) {
                const int q = idx / Uc, uu = idx - q * Uc;
                const float* cb = contrib + (size_t)q * JC * Umax + uu;
                float sacc = sums[q * Umax + uu];
                for (int jj = 0; jj < jn; ++jj) sacc += cb[jj * Umax];
                sums[q * Umax + uu] = sacc;
            }
            __syncthreads();
        }
        stamp(a, true, dir, cta, s, 3);
        if (G > 1) step_publish(myflags + cta, (unsigned)(s + 1), skip_pub);
        else __syncthreads();
        stamp(a, true, dir, cta, s, 4);
    }
    for (int idx = threadIdx.x; idx < 7 * Uc; idx += kRecThreads) {
        const int q = idx / Uc, uu = idx - q * Uc;
        const int u = u0 + uu;
        const float v = sums[q * Umax + uu];
        if (q < 4) a.db[(size_t)dir * 4 * H + q * H + u] = v;
        else a.dpeep[(size_t)dir * 3 * H + (q - 4) * H + u] = v;
    }
}

// ------------------------------------------------------------------------- launch

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int matmul_red_floats(int RP, int JC, int K)
{
    const int groups = (RP / 4) * (JC / 4);
    int KS = kRecThreads / groups;
    if (KS < 1) KS = 1;
    if (KS > K / 8) KS = K / 8;
    return KS * RP * JC;
}

// Shared-memory layout for a given configuration; returns total bytes.
static size_t rec_layout(const RecConfig& c, int H, int B, int T, int relem, bool bwd, RecArgs* a)
{
    const int Umax = c.Umax, JC = c.JC;
    size_t off = 0, o_h = 0, o_red = 0, o_acc = 0, o_state = 0, o_contrib = 0, o_sums = 0, o_tab = 0, o_peep;
    if (!bwd) {
        const int RP = 4 * Umax;
        off = align_up((size_t)RP * (H + 16 / relem) * relem, 16);
        o_h = off; off = align_up(off + (size_t)JC * (H + 4) * 4, 16);
        o_red = off;
        off = align_up(off + (size_t)std::max(matmul_red_floats(RP, JC, H), 8 * RP * JC) * 4, 16);
        o_acc = off; off = align_up(off + (size_t)JC * RP * 4, 16);
        o_state = off; off = align_up(off + (size_t)B * Umax * 4, 16);
    } else {
        const int RP8 = relem == 2 ? ((4 * Umax + 15) & ~15) : ((4 * Umax + 7) & ~7);
        off = align_up((size_t)RP8 * (H + 16 / relem) * relem, 16);
        o_h = off; off = align_up(off + (size_t)JC * (RP8 + 4) * 4, 16);
        o_state = off; off = align_up(off + (size_t)B * Umax * 4, 16);
        o_contrib = off; off = align_up(off + (size_t)7 * JC * Umax * 4, 16);
        o_sums = off; off = align_up(off + (size_t)7 * Umax * 4, 16);
    }
    o_peep = off; off = align_up(off + (size_t)3 * Umax * 4, 16);
    if (c.tables) { o_tab = off; off = align_up(off + (size_t)(2 * T + 1 + B) * 4, 16); }
    if (a) {
        a->off_h = (int)o_h; a->off_red = (int)o_red; a->off_acc = (int)o_acc;
        a->off_state = (int)o_state; a->off_contrib = (int)o_contrib; a->off_sums = (int)o_sums;
        a->off_tab = (int)o_tab; a->off_peep = (int)o_peep;
        a->tables_in_smem = c.tables;
    }
    return off + 64;   // room for the barrier's static shared word
}

// Product engine, chunk size and shared-memory layout for c.G / c.Umax; c.JC
// stays 0 when nothing fits.
static void configure_for(const Plan& p, int H, bool bf16, bool bwd, RecConfig& c)
{
    int smem_optin = 0;
    if (cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device) != cudaSuccess)
        return;
    const int relem = bf16 ? 2 : 4;
    const int Umax = c.Umax;
    // tensor-core product when this CTA's fragments fit the per-warp register budget
    const int ksz = bf16 ? 16 : 8;
    if (p.gemm_engine == 1) {
        // CUDA cores only
    } else if (!bwd) {
        const int MT = (4 * Umax + 15) / 16;
        if (H % ksz == 0) {
            const int KT = H / ksz;
            for (int mw = 1; mw <= kRecThreads / 32 && !c.mma; ++mw)
                for (int kw = kRecThreads / 32 / mw; kw >= 1; --kw)
                    if (ceil_div(MT, mw) <= kFwdMTW && ceil_div(KT, kw) <= kFwdKTW) {
                        c.mma = 1; c.mma_mw = mw; c.mma_kw = kw;
                        break;
                    }
        }
    } else {
        const int RPK = bf16 ? ((4 * Umax + 15) & ~15) : ((4 * Umax + 7) & ~7);
        if (H % 16 == 0 && ceil_div(H / 16, kRecThreads / 32) <= kBwdMTW && RPK / ksz <= kBwdKTW) c.mma = 1;
    }
    c.JC = 0;
    for (int tables = 1; tables >= 0 && c.JC == 0; --tables) {
        for (int jc : {32, 16, 8, 4}) {
            if (jc * Umax > kMaxItems * kRecThreads) continue;
            RecConfig t = c;
            t.JC = jc;
            t.tables = tables;
            const size_t bytes = rec_layout(t, H, p.B, p.T, relem, bwd, nullptr);
            if (bytes <= (size_t)smem_optin) { c = t; c.smem = bytes; break; }
        }
    }
}

lstm_status rec_configure(const Plan& p, int H, int ndir, bool bf16, bool bwd, int forced_G,
                          RecConfig* out)
{
    const int per_dir_max = std::min(kMaxCtasPerDir, p.num_sms / ndir);
    if (per_dir_max < 1) return LSTM_ERR_UNSUPPORTED;
    int bmax = 0;
    for (int t = 0; t < p.T; ++t) bmax = std::max(bmax, p.h_bs[t]);
    int G0;
    if (forced_G > 0) G0 = std::min(forced_G, per_dir_max);
    else {
        // one CTA per direction while a step's product is small; otherwise one per SM
        const double fmas = 4.0 * H * (double)H * std::max(1, bmax);
        G0 = (fmas <= 1.5e6 && H <= 256) ? 1 : per_dir_max;
    }
    // automatic choice: fall back to one CTA per SM when the slice does not fit
    const int tries[2] = {G0, per_dir_max};
    RecConfig c;
    for (int attempt = 0; attempt < (forced_G > 0 ? 1 : 2) && c.JC == 0; ++attempt) {
        int G = tries[attempt];
        const int Umax = ceil_div(H, G);
        G = ceil_div(H, Umax);
        c = RecConfig();
        c.G = G; c.Umax = Umax;
        configure_for(p, H, bf16, bwd, c);
    }
    if (c.JC == 0) return LSTM_ERR_UNSUPPORTED;
    *out = c;
    return LSTM_OK;
}

size_t rec_bwd_part_floats(const Plan& p, int H, int ndir, bool bf16, int forced_G)
{
    RecConfig c;
    if (rec_configure(p, H, ndir, bf16, true, forced_G, &c) != LSTM_OK) return 0;
    return (size_t)2 * ndir * p.B * c.G * H;
}

lstm_status rec_launch(const Plan& p, const RecConfig& c, RecArgs a, bool bwd, cudaStream_t s)
{
    a.G = c.G; a.Umax = c.Umax; a.JC = c.JC;
    a.trace = p.d_trace; a.trace_steps = p.trace_steps;
    rec_layout(c, a.H, p.B, p.T, a.bf16 ? 2 : 4, bwd, &a);
    a.mma_mw = c.mma_mw; a.mma_kw = c.mma_kw;
    void* fn;
    if (!bwd) {
        if (c.mma) fn = a.bf16 ? (void*)lstm_rec_fwd_kernel<__nv_bfloat16, true> : (void*)lstm_rec_fwd_kernel<float, true>;
        else fn = a.bf16 ? (void*)lstm_rec_fwd_kernel<__nv_bfloat16, false> : (void*)lstm_rec_fwd_kernel<float, false>;
    } else {
        if (c.mma) fn = a.bf16 ? (void*)lstm_rec_bwd_kernel<__nv_bfloat16, true> : (void*)lstm_rec_bwd_kernel<float, true>;
        else fn = a.bf16 ? (void*)lstm_rec_bwd_kernel<__nv_bfloat16, false> : (void*)lstm_rec_bwd_kernel<float, false>;
    }
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)c.smem) != cudaSuccess)
        return LSTM_ERR_CUDA;
    // fresh step counters for this launch
    if (c.G > 1 && cudaMemsetAsync(p.d_flags, 0, sizeof(unsigned) * 2 * kMaxCtasPerDir, s) != cudaSuccess)
        return LSTM_ERR_CUDA;
    void* args[] = {&a};
    const dim3 grid(c.G * a.ndir), block(kRecThreads);
    cudaError_t e;
    trace_begin(p, bwd ? K_REC_BWD : K_REC_FWD, s);
    if (c.G > 1) e = cudaLaunchCooperativeKernel(fn, grid, block, args, c.smem, s);
    else e = cudaLaunchKernel(fn, grid, block, args, c.smem, s);
    trace_end(p, bwd ? K_REC_BWD : K_REC_FWD, s, e == cudaSuccess ? 1 : 0);
    if (e == cudaErrorCooperativeLaunchTooLarge) { cudaGetLastError(); return LSTM_ERR_UNSUPPORTED; }
    return e == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

}  // namespace lstm
