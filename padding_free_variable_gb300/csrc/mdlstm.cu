// mdlstm.cu -- one 2-D MDLSTM layer over example-packed images (fp32).
//
// "No Padding Please: Efficient Neural Handwriting Recognition":
//  * Sec. III / App. A: a cell of the 2-D grid takes the pixel input and the
//    hidden and memory states of its two predecessors (the previous row and
//    the previous column in its scan order); five input blocks (input gate,
//    two forget gates, input node, output gate) each sum W x + U1 h1 + U2 h2
//    + b; each predecessor state enters the input gate, its own forget gate
//    and the output gate (the output gate reads the previous states, the
//    page's variant):
//        i = sig(a_i + p_i1 S1 + p_i2 S2)   f1 = sig(a_f1 + p_f1 S1)
//        f2 = sig(a_f2 + p_f2 S2)           z = tanh(a_z)
//        o = sig(a_o + p_o1 S1 + p_o2 S2)   c = f1 S1 + f2 S2 + i z
//        h = o tanh(c)
//    A predecessor outside the example gives h = S = 0 (Sec. V's mask).
//  * Sec. IV-A: along a skewed column (an anti-diagonal of the image) the
//    cells depend only on the previous column: one parallel step.
//  * Sec. V: the examples are packed so that one launch covers them all.
//
// Layout: the plan stores the cells of every scan direction in wavefront
// order with their predecessor and successor cells (md_plan.cu).  A layer is
//  1. the input projection of every pixel for all directions, one CUDA-core
//     GEMM: gx[N][ndir*5H] = x W^T + b;
//  2. one cooperative launch over all SMs that walks the steps: a warp per
//     cell, a lane per unit (up to 4 units a lane); the recurrent products
//     U1 h1 + U2 h2 read h1, h2 from L2 and U^T from shared memory (when the
//     layer's weights fit) and the cell writes h, c, the gates and y; a
//     bounded grid barrier separates the steps;
//  3. backward: the same walk in reverse; a cell's h error is its dy plus
//     U1^T da of the cell that takes it as predecessor 1 plus U2^T da of the
//     one that takes it as predecessor 2, and its state error is what those
//     successors left for it; the gate errors overwrite the gates in place;
//  4. dx = dA W from the pixel-order gate errors (one thread a pixel, W in
//     shared memory); dW, dU1,
//     dU2, db and the six peephole sums in one pass over each direction's
//     cells (outer products of the gate errors with [x | h1 | h2 | 1], chunk
//     partials added in chunk order: bitwise repeatable).
#include <cstring>

#include "gemm.cuh"
#include "md_plan.cuh"

namespace lstm {

namespace {

constexpr int kMdThreads = 256;
constexpr int kMdMaxH = 128;                  // 4 units a lane
constexpr size_t kMdSmemCap = 200 * 1024;     // resident recurrent weights up to this size

__device__ __forceinline__ float sg_md(float v) { return __fdividef(1.0f, 1.0f + __expf(-v)); }
__device__ __forceinline__ float th_md(float v)
{
    const float e = __expf(2.0f * fminf(fmaxf(v, -40.0f), 40.0f));
    return 1.0f - __fdividef(2.0f, e + 1.0f);
}

__device__ __forceinline__ void red_release_add_md(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct MdArgs {
    int H, ndir, steps;
    int64_t N;
    const int64_t* step_off;     // [ndir][steps+1]
    const int32_t* src;
    const int32_t* pred1;
    const int32_t* pred2;
    const int32_t* succ1;
    const int32_t* succ2;
    const float* U;              // forward: U^T [ndir][2][H][5H]; backward: U [ndir][2][5H][H]
    const float* peep;           // [ndir][6][H]
    const float* gx;             // [N][ndir*5H]
    float* h;                    // [cells][H]
    float* c;                    // [cells][H]
    float* act;                  // [cells][5H] gates, then gate errors
    float* y;                    // [N][ndir*H]
    const float* dy;             // [N][ndir*H]
    float* dap;                  // [N][ndir*5H] gate errors in pixel order
    float* ds1;                  // [cells][H] state error a cell leaves for its predecessor 1
    float* ds2;
    unsigned* ctr;
    DeviceStatus* status;
    unsigned long long wait_limit_ns;
    int debug_skip_cta;          // test hook (-1 off): this CTA skips its first arrival
    int ngrp;                    // direction groups: CTA b serves directions of group b % ngrp
};

// Every CTA has finished step `done` (steps counted from 1): bounded wait by thread 0.
__device__ __forceinline__ bool md_barrier(const MdArgs& a, unsigned done, unsigned where)
{
    __syncthreads();
    int fail = 0;
    if (threadIdx.x == 0) {
        if (!(done == 1 && (int)blockIdx.x == a.debug_skip_cta)) red_release_add_md(a.ctr, 1u);
        const unsigned target = done * gridDim.x;
        const unsigned long long t0 = global_timer_ns();
        unsigned spins = 0;
        while ((int)(ld_acquire_gpu(a.ctr) - target) < 0) {
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

// The directions a CTA serves (its group's) and its warp's place among the group's warps.
struct MdWork {
    int d0, dn;                  // directions [d0, d0 + dn)
    int64_t gw, warps;
};

__device__ __forceinline__ MdWork md_work(const MdArgs& a)
{
    MdWork w;
    const int g = (int)(blockIdx.x % a.ngrp);
    w.dn = a.ndir / a.ngrp;
    w.d0 = g * w.dn;
    w.warps = (int64_t)(gridDim.x / a.ngrp) * (blockDim.x >> 5);
    w.gw = (int64_t)(blockIdx.x / a.ngrp) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    return w;
}

// the item-th cell of step k over the group's directions: its direction and index
__device__ __forceinline__ bool md_item(const MdArgs& a, const MdWork& w, int k, int64_t item, int& d, int64_t& p)
{
    for (d = w.d0; d < w.d0 + w.dn; ++d) {
        const int64_t* so = a.step_off + (size_t)d * (a.steps + 1);
        const int64_t n = so[k + 1] - so[k];
        if (item < n) { p = so[k] + item; return true; }
        item -= n;
    }
    return false;
}

__device__ __forceinline__ int64_t md_step_cells(const MdArgs& a, const MdWork& w, int k)
{
    int64_t n = 0;
    for (int d = w.d0; d < w.d0 + w.dn; ++d) {
        const int64_t* so = a.step_off + (size_t)d * (a.steps + 1);
        n += so[k + 1] - so[k];
    }
    return n;
}

// One cell's operands in the forward walk: its direction, index, predecessors, pixel and
// input projection (none of which depends on the step before), then the predecessors' h and
// c (which do).
template <int NU>
struct MdCell {
    int d = 0, q1 = -1, q2 = -1;
    int64_t p = -1, px = 0;
    float g[5][NU];
    float h1[NU], h2[NU], s1[NU], s2[NU];
};

template <int NU>
__device__ __forceinline__ void md_fetch(const MdArgs& a, const MdWork& w, int k, int64_t item, int lane,
                                         MdCell<NU>& m)
{
    const int H = a.H, H5 = 5 * H;
    m.p = -1;
    if (k >= a.steps || !md_item(a, w, k, item, m.d, m.p)) return;
    m.q1 = a.pred1[m.p];
    m.q2 = a.pred2[m.p];
    m.px = a.src[m.p];
    const float* gr = a.gx + (size_t)m.px * a.ndir * H5 + (size_t)m.d * H5;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int u = lane + 32 * j;
#pragma unroll
        for (int g = 0; g < 5; ++g) m.g[g][j] = u < H ? __ldg(gr + g * H + u) : 0.f;
    }
}

template <int NU>
__device__ __forceinline__ void md_fetch_states(const MdArgs& a, int lane, MdCell<NU>& m)
{
    const int H = a.H;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int u = lane + 32 * j;
        const bool ok = u < H && m.p >= 0;
        m.h1[j] = ok && m.q1 >= 0 ? __ldcg(a.h + (size_t)m.q1 * H + u) : 0.f;
        m.s1[j] = ok && m.q1 >= 0 ? __ldcg(a.c + (size_t)m.q1 * H + u) : 0.f;
        m.h2[j] = ok && m.q2 >= 0 ? __ldcg(a.h + (size_t)m.q2 * H + u) : 0.f;
        m.s2[j] = ok && m.q2 >= 0 ? __ldcg(a.c + (size_t)m.q2 * H + u) : 0.f;
    }
}

// The forward cell on fetched operands: U1 h1 and U2 h2 in separate accumulators (two short
// dependency chains; h1[kk], h2[kk] broadcast from the lane that holds them), then the gates,
// c and h; writes h, c, the gates (cell order) and y (pixel order).
template <int NU>
__device__ __forceinline__ void md_fwd_cell(const MdArgs& a, const float* UT, int d0, int lane, const MdCell<NU>& m)
{
    const int H = a.H, H5 = 5 * H;
    const int d = m.d;
    float acc1[5][NU], acc2[5][NU];
#pragma unroll
    for (int j = 0; j < NU; ++j)
#pragma unroll
        for (int g = 0; g < 5; ++g) {
            acc1[g][j] = m.g[g][j];
            acc2[g][j] = 0.f;
        }
    const float* U1t = UT + (size_t)(d - d0) * 2 * H * H5;      // UT starts at direction d0
    const float* U2t = U1t + (size_t)H * H5;
    if (m.q1 >= 0 || m.q2 >= 0) {
#pragma unroll
        for (int jj = 0; jj < NU; ++jj)
#pragma unroll(NU == 1 ? 32 : 4)
            for (int l = 0; l < 32; ++l) {          // (full unroll for one unit a lane: compile time)
                const int kk = 32 * jj + l;
                if (kk < H) {                               // (uniform across the warp)
                    const float x1 = __shfl_sync(0xffffffffu, m.h1[jj], l);
                    const float x2 = __shfl_sync(0xffffffffu, m.h2[jj], l);
                    const float* r1 = U1t + (size_t)kk * H5;
                    const float* r2 = U2t + (size_t)kk * H5;
#pragma unroll
                    for (int j = 0; j < NU; ++j) {
                        const int u = lane + 32 * j;
                        if (u < H)
#pragma unroll
                            for (int g = 0; g < 5; ++g) {
                                acc1[g][j] = fmaf(r1[g * H + u], x1, acc1[g][j]);
                                acc2[g][j] = fmaf(r2[g * H + u], x2, acc2[g][j]);
                            }
                    }
                }
            }
    }
    const float* pp = a.peep + (size_t)d * 6 * H;
#pragma unroll
    for (int j = 0; j < NU; ++j) {
        const int u = lane + 32 * j;
        if (u >= H) continue;
        float acc[5];
#pragma unroll
        for (int g = 0; g < 5; ++g) acc[g] = acc1[g][j] + acc2[g][j];
        const float s1 = m.s1[j], s2 = m.s2[j];
        const float ig = sg_md(acc[0] + __ldg(pp + u) * s1 + __ldg(pp + H + u) * s2);
        const float f1 = sg_md(acc[1] + __ldg(pp + 2 * H + u) * s1);
        const float f2 = sg_md(acc[2] + __ldg(pp + 3 * H + u) * s2);
        const float zg = th_md(acc[3]);
        const float og = sg_md(acc[4] + __ldg(pp + 4 * H + u) * s1 + __ldg(pp + 5 * H + u) * s2);
        const float cv = f1 * s1 + f2 * s2 + ig * zg;
        const float hv = og * th_md(cv);
        a.h[(size_t)m.p * H + u] = hv;
        a.c[(size_t)m.p * H + u] = cv;
        float* ar = a.act + (size_t)m.p * H5;
        ar[u] = ig; ar[H + u] = f1; ar[2 * H + u] = f2; ar[3 * H + u] = zg; ar[4 * H + u] = og;
        a.y[(size_t)m.px * a.ndir * H + (size_t)d * H + u] = hv;
    }
}

// Forward walk.  NU = units per lane (ceil(H / 32)); SM = U^T resident in shared memory.
// A warp's cells of a step are software-pipelined: the next cell's operands (and, once the
// barrier has passed, its predecessors' states) load while the current one computes; the
// first cell of the next step fetches its own operands before the barrier.
template <int NU, bool SM>
__global__ void __launch_bounds__(kMdThreads, NU <= 2 ? 2 : 1) md_fwd_kernel(MdArgs a)
{
    extern __shared__ float md_smem[];
    const int H = a.H, H5 = 5 * H;
    const int lane = threadIdx.x & 31;
    const MdWork w = md_work(a);
    const int64_t per = (int64_t)2 * H * H5;                // U^T floats of one direction
    const float* UT = a.U + (size_t)w.d0 * per;
    if (SM) {
        for (int64_t i = threadIdx.x; i < w.dn * per; i += blockDim.x) md_smem[i] = UT[i];
        __syncthreads();
        UT = md_smem;
    }
    MdCell<NU> cur;
    md_fetch<NU>(a, w, 0, w.gw, lane, cur);
    for (int k = 0; k < a.steps; ++k) {
        const int64_t total = md_step_cells(a, w, k);
        md_fetch_states<NU>(a, lane, cur);
        for (int64_t item = w.gw; item < total; item += w.warps) {
            MdCell<NU> nx;
            const bool more = item + w.warps < total;
            if (more) {
                md_fetch<NU>(a, w, k, item + w.warps, lane, nx);
                md_fetch_states<NU>(a, lane, nx);
            }
            md_fwd_cell<NU>(a, UT, w.d0, lane, cur);
            if (more) cur = nx;
        }
        md_fetch<NU>(a, w, k + 1, w.gw, lane, cur);      // the next step's first cell, before the barrier
        if (k + 1 < a.steps && !md_barrier(a, (unsigned)(k + 1), 0xA00000u | (unsigned)k)) return;
    }
}

// Backward walk (steps in reverse).  SM = U resident in shared memory.
template <int NU, bool SM>
__global__ void __launch_bounds__(kMdThreads, 1) md_bwd_kernel(MdArgs a)
{
    extern __shared__ float md_smem[];
    const int H = a.H, H5 = 5 * H;
    constexpr int NR = (5 * 32 * NU + 31) / 32;      // 5H / 32 rounded up, per lane
    const int lane = threadIdx.x & 31;
    const MdWork w = md_work(a);
    const int64_t per = (int64_t)2 * H5 * H;                // U floats of one direction
    const float* Uw = a.U + (size_t)w.d0 * per;
    if (SM) {
        for (int64_t i = threadIdx.x; i < w.dn * per; i += blockDim.x) md_smem[i] = Uw[i];
        __syncthreads();
        Uw = md_smem;
    }
    const int64_t warps = w.warps, gw = w.gw;
    unsigned done = 0;
    for (int k = a.steps - 1; k >= 0; --k) {
        const int64_t total = md_step_cells(a, w, k);
        for (int64_t item = gw; item < total; item += warps) {
            int d;
            int64_t p;
            md_item(a, w, k, item, d, p);
            const int r1 = a.succ1[p], r2 = a.succ2[p];
            const int q1 = a.pred1[p], q2 = a.pred2[p];
            const int64_t px = a.src[p];
            float e[NU], dsin[NU];
#pragma unroll
            for (int j = 0; j < NU; ++j) {
                const int u = lane + 32 * j;
                const bool ok = u < H;
                e[j] = ok ? __ldg(a.dy + (size_t)px * a.ndir * H + (size_t)d * H + u) : 0.f;
                dsin[j] = (ok && r1 >= 0 ? __ldcg(a.ds1 + (size_t)r1 * H + u) : 0.f) +
                          (ok && r2 >= 0 ? __ldcg(a.ds2 + (size_t)r2 * H + u) : 0.f);
            }
            // U1^T da(successor 1) + U2^T da(successor 2): the successors' gate errors are
            // spread over the lanes (element 32 m + lane in slot m) and broadcast one by one
            const float* U1 = Uw + (size_t)(d - w.d0) * 2 * H5 * H;      // Uw starts at direction d0
            const float* U2 = U1 + (size_t)H5 * H;
            if (r1 >= 0 || r2 >= 0) {
                float g1[NR], g2[NR];
#pragma unroll
                for (int m = 0; m < NR; ++m) {
                    const int r = 32 * m + lane;
                    g1[m] = r < H5 && r1 >= 0 ? __ldcg(a.act + (size_t)r1 * H5 + r) : 0.f;
                    g2[m] = r < H5 && r2 >= 0 ? __ldcg(a.act + (size_t)r2 * H5 + r) : 0.f;
                }
#pragma unroll
                for (int m = 0; m < NR; ++m)
                    for (int l = 0; l < 32; ++l) {
                        const int r = 32 * m + l;
                        if (r >= H5) break;                 // (uniform across the warp)
                        const float x1 = __shfl_sync(0xffffffffu, g1[m], l);
                        const float x2 = __shfl_sync(0xffffffffu, g2[m], l);
#pragma unroll
                        for (int j = 0; j < NU; ++j) {
                            const int u = lane + 32 * j;
                            if (u < H) e[j] = fmaf(U1[(size_t)r * H + u], x1, fmaf(U2[(size_t)r * H + u], x2, e[j]));
                        }
                    }
            }
            // every lane has read the successors' errors before any lane of another warp can
            // change them: they were final at the previous barrier, and this cell writes only
            // its own row
            const float* pp = a.peep + (size_t)d * 6 * H;
            float* ar = a.act + (size_t)p * H5;
#pragma unroll
            for (int j = 0; j < NU; ++j) {
                const int u = lane + 32 * j;
                if (u >= H) continue;
                const float S1 = q1 >= 0 ? __ldcg(a.c + (size_t)q1 * H + u) : 0.f;
                const float S2 = q2 >= 0 ? __ldcg(a.c + (size_t)q2 * H + u) : 0.f;
                const float ig = ar[u], f1 = ar[H + u], f2 = ar[2 * H + u], zg = ar[3 * H + u], og = ar[4 * H + u];
                const float cv = __ldcg(a.c + (size_t)p * H + u);
                const float tc = th_md(cv);
                const float dao = e[j] * tc * og * (1.f - og);
                const float dc = e[j] * og * (1.f - tc * tc) + dsin[j];
                const float dai = dc * zg * ig * (1.f - ig);
                const float daf1 = dc * S1 * f1 * (1.f - f1);
                const float daf2 = dc * S2 * f2 * (1.f - f2);
                const float daz = dc * ig * (1.f - zg * zg);
                a.ds1[(size_t)p * H + u] = dc * f1 + __ldg(pp + u) * dai + __ldg(pp + 2 * H + u) * daf1 +
                                           __ldg(pp + 4 * H + u) * dao;
                a.ds2[(size_t)p * H + u] = dc * f2 + __ldg(pp + H + u) * dai + __ldg(pp + 3 * H + u) * daf2 +
                                           __ldg(pp + 5 * H + u) * dao;
                ar[u] = dai; ar[H + u] = daf1; ar[2 * H + u] = daf2; ar[3 * H + u] = daz; ar[4 * H + u] = dao;
                float* dp = a.dap + (size_t)px * a.ndir * H5 + (size_t)d * H5;
                dp[u] = dai; dp[H + u] = daf1; dp[2 * H + u] = daf2; dp[3 * H + u] = daz; dp[4 * H + u] = dao;
            }
        }
        ++done;
        if (k > 0 && !md_barrier(a, done, 0xB00000u | (unsigned)k)) return;
    }
}

// U [ndir][2][5H][H] -> U^T [ndir][2][H][5H]
__global__ void md_transpose_kernel(const float* __restrict__ U1, const float* __restrict__ U2, float* __restrict__ UT,
                                    float* __restrict__ Ucat, int ndir, int H)
{
    const int H5 = 5 * H;
    const int64_t n = (int64_t)ndir * 2 * H5 * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t per = (int64_t)H5 * H;
        const int d = (int)(i / (2 * per));
        const int w = (int)((i / per) & 1);
        const int64_t r = i % per;                   // element of U_w[d]: row r / H, column r % H
        const int row = (int)(r / H), col = (int)(r % H);
        const float v = (w == 0 ? U1 : U2)[(size_t)d * per + r];
        Ucat[i] = v;
        UT[(size_t)d * 2 * per + (size_t)w * per + (size_t)col * H5 + row] = v;
    }
}

// Weight gradients of one direction in one pass over its cells.  Cell p contributes the outer
// product of its gate errors da[p][5H] with its operand row v[p] = [x(pixel) | h(pred 1) |
// h(pred 2) | 1] (D + 2H + 1 columns: dW, dU1, dU2, db), and the six peephole products
// da_g S_d (element-wise).  A CTA takes one chunk of kMdWgCells cells, stages kMdWgTile of them
// at a time in shared memory (gathered rows) and accumulates a register block of RB x CB
// outputs per thread (a 16 x 16 thread grid over an output tile of 16 RB rows x 16 CB
// columns; larger shapes walk several output tiles); every output sums its cells in cell
// order, and the chunks are added in chunk order by md_wgrad_combine (bitwise repeatable).
constexpr int kMdWgTile = 32;
constexpr int kMdWgCells = 1024;
constexpr int kMdWgRB = 10, kMdWgCB = 6;

__global__ void __launch_bounds__(256) md_wgrad_kernel(const float* __restrict__ act, const float* __restrict__ h,
                                                        const float* __restrict__ c, const float* __restrict__ x,
                                                        const int32_t* __restrict__ src,
                                                        const int32_t* __restrict__ pred1,
                                                        const int32_t* __restrict__ pred2, int D, int H, int64_t N,
                                                        float* __restrict__ partial)
{
    extern __shared__ float wg_smem[];
    const int H5 = 5 * H, L = D + 2 * H + 1, nout = H5 * L + 6 * H;
    const int d = blockIdx.y;
    const int64_t lo = (int64_t)blockIdx.x * kMdWgCells, hi = min(N, lo + kMdWgCells);
    const int64_t base = (int64_t)d * N;
    float* sda = wg_smem;                                   // [tile][5H]
    float* sv = sda + kMdWgTile * H5;                       // [tile][L]
    float* ss1 = sv + kMdWgTile * L;                        // [tile][H]
    float* ss2 = ss1 + kMdWgTile * H;
    int* sidx = reinterpret_cast<int*>(ss2 + kMdWgTile * H);   // [3][tile]: pixel, pred 1, pred 2
    const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
    float* out = partial + ((size_t)d * gridDim.x + blockIdx.x) * nout;
    const int rt_n = (H5 + 16 * kMdWgRB - 1) / (16 * kMdWgRB), ct_n = (L + 16 * kMdWgCB - 1) / (16 * kMdWgCB);
    for (int ot = 0; ot < rt_n * ct_n; ++ot) {
        const int r0 = (ot / ct_n) * 16 * kMdWgRB, c0 = (ot % ct_n) * 16 * kMdWgCB;
        const bool peep_pass = ot == 0;
        float acc[kMdWgRB][kMdWgCB];
#pragma unroll
        for (int i = 0; i < kMdWgRB; ++i)
#pragma unroll
            for (int j = 0; j < kMdWgCB; ++j) acc[i][j] = 0.f;
        float pacc[3] = {0.f, 0.f, 0.f};                   // peephole sums: items t, t + 256, t + 512
        for (int64_t p0 = lo; p0 < hi; p0 += kMdWgTile) {
            const int nt = (int)min((int64_t)kMdWgTile, hi - p0);
            __syncthreads();                                // the previous tile has been read
            if (t < kMdWgTile) {                            // the tile's cells: pixel and predecessors
                const bool live = t < nt;
                const int64_t p = base + p0 + t;
                sidx[t] = live ? src[p] : -1;
                sidx[kMdWgTile + t] = live ? pred1[p] : -1;
                sidx[2 * kMdWgTile + t] = live ? pred2[p] : -1;
            }
            __syncthreads();
            // warp w gathers rows w, w + 8, ...: each row's columns by consecutive lanes
            for (int k = t >> 5; k < kMdWgTile; k += 8) {
                const int lane = t & 31;
                const bool live = k < nt;
                const int64_t p = base + p0 + k;
                const int px = sidx[k], q1 = sidx[kMdWgTile + k], q2 = sidx[2 * kMdWgTile + k];
                for (int r = lane; r < H5; r += 32) sda[k * H5 + r] = live ? act[(size_t)p * H5 + r] : 0.f;
                float* vr = sv + k * L;
                for (int col = lane; col < D; col += 32) vr[col] = live ? x[(size_t)px * D + col] : 0.f;
                for (int u = lane; u < H; u += 32) {
                    vr[D + u] = live && q1 >= 0 ? h[(size_t)q1 * H + u] : 0.f;
                    vr[D + H + u] = live && q2 >= 0 ? h[(size_t)q2 * H + u] : 0.f;
                    if (peep_pass) {
                        ss1[k * H + u] = live && q1 >= 0 ? c[(size_t)q1 * H + u] : 0.f;
                        ss2[k * H + u] = live && q2 >= 0 ? c[(size_t)q2 * H + u] : 0.f;
                    }
                }
                if (lane == 0) vr[D + 2 * H] = live ? 1.f : 0.f;
            }
            __syncthreads();
            for (int k = 0; k < nt; ++k) {
                float a[kMdWgRB], v[kMdWgCB];
#pragma unroll
                for (int i = 0; i < kMdWgRB; ++i) {
                    const int r = r0 + ty + 16 * i;
                    a[i] = r < H5 ? sda[k * H5 + r] : 0.f;
                }
#pragma unroll
                for (int j = 0; j < kMdWgCB; ++j) {
                    const int col = c0 + tx + 16 * j;
                    v[j] = col < L ? sv[k * L + col] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < kMdWgRB; ++i)
#pragma unroll
                    for (int j = 0; j < kMdWgCB; ++j) acc[i][j] = fmaf(a[i], v[j], acc[i][j]);
            }
            if (peep_pass)
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const int it = t + 256 * m;            // peephole q = it / H of unit it % H
                    if (it < 6 * H) {
                        const int q = it / H, u = it - q * H;
                        const int gate = q < 2 ? 0 : q == 2 ? 1 : q == 3 ? 2 : 4;   // i, i, f1, f2, o, o
                        const float* S = (q & 1) == 0 ? ss1 : ss2;
                        for (int k = 0; k < nt; ++k) pacc[m] = fmaf(sda[k * H5 + gate * H + u], S[k * H + u], pacc[m]);
                    }
                }
        }
#pragma unroll
        for (int i = 0; i < kMdWgRB; ++i)
#pragma unroll
            for (int j = 0; j < kMdWgCB; ++j) {
                const int r = r0 + ty + 16 * i, col = c0 + tx + 16 * j;
                if (r < H5 && col < L) out[(size_t)r * L + col] = acc[i][j];
            }
        if (peep_pass)
#pragma unroll
            for (int m = 0; m < 3; ++m) {
                const int it = t + 256 * m;
                if (it < 6 * H) out[(size_t)H5 * L + it] = pacc[m];
            }
    }
}

// Chunks added in order; the columns scattered to dW, dU1, dU2, db and the peepholes.
__global__ void md_wgrad_combine(const float* __restrict__ partial, int chunks, int D, int H, int ndir,
                                 float* __restrict__ dW, float* __restrict__ dU1, float* __restrict__ dU2,
                                 float* __restrict__ db, float* __restrict__ dpeep)
{
    const int H5 = 5 * H, L = D + 2 * H + 1, nout = H5 * L + 6 * H;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)ndir * nout) return;
    const int d = (int)(i / nout), e = (int)(i - (int64_t)d * nout);
    float s = 0.f;
    for (int k = 0; k < chunks; ++k) s += partial[((size_t)d * chunks + k) * nout + e];
    if (e >= H5 * L) {
        if (dpeep) dpeep[(size_t)d * 6 * H + (e - H5 * L)] = s;
        return;
    }
    const int r = e / L, col = e - r * L;
    if (col < D) {
        if (dW) dW[((size_t)d * H5 + r) * D + col] = s;
    } else if (col < D + H) {
        if (dU1) dU1[((size_t)d * H5 + r) * H + col - D] = s;
    } else if (col < D + 2 * H) {
        if (dU2) dU2[((size_t)d * H5 + r) * H + col - D - H] = s;
    } else if (db) {
        db[(size_t)d * H5 + r] = s;
    }
}

size_t md_wgrad_smem(int D, int H)
{
    return sizeof(float) * kMdWgTile * (5 * H + (D + 2 * H + 1) + 2 * H) + sizeof(int) * 3 * kMdWgTile;
}

// dx[p][k] = sum over the ndir*5H gate errors of pixel p of dA[p][r] W[r][k]: one thread per
// pixel with its D outputs in registers, W (all directions) staged in shared memory.
template <int DK>
__global__ void __launch_bounds__(128) md_dx_kernel(const float* __restrict__ dap, const float* __restrict__ W, int R,
                                                     int D, int64_t N, float* __restrict__ dx)
{
    extern __shared__ float dx_smem[];
    for (int i = threadIdx.x; i < R * D; i += blockDim.x) dx_smem[i] = W[i];
    __syncthreads();
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= N) return;
    float acc[DK];
#pragma unroll
    for (int k = 0; k < DK; ++k) acc[k] = 0.f;
    const float4* row = reinterpret_cast<const float4*>(dap + (size_t)p * R);
    for (int r4 = 0; r4 < R / 4; ++r4) {
        const float4 a4 = __ldg(row + r4);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float* wr = dx_smem + (size_t)(4 * r4 + e) * D;
#pragma unroll
            for (int k = 0; k < DK; ++k)
                if (k < D) acc[k] = fmaf(av[e], wr[k], acc[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < DK; ++k)
        if (k < D) dx[(size_t)p * D + k] = acc[k];
}

// ---------------------------------------------------------------- workspace layout

struct MdLayout {
    size_t gx, h, c, act, ut, ucat, total;          // byte offsets (workspace)
    size_t ds1, ds2, part, stotal;                  // byte offsets (scratch)
    int chunks = 1;
};

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

MdLayout md_layout(const MdPlan& p, int D, int H)
{
    MdLayout L;
    const size_t N = (size_t)p.pixels, cells = (size_t)p.cells, nd = (size_t)p.ndir, H5 = 5 * (size_t)H;
    size_t o = 0;
    L.gx = o; o = al256(o + 4 * N * nd * H5);
    L.h = o; o = al256(o + 4 * cells * H);
    L.c = o; o = al256(o + 4 * cells * H);
    L.act = o; o = al256(o + 4 * cells * H5);
    L.ut = o; o = al256(o + 4 * nd * 2 * H5 * H);
    L.ucat = o; o = al256(o + 4 * nd * 2 * H5 * H);
    L.total = o;
    // scratch: ds1, ds2, the weight gradients' chunk partials
    o = 0;
    L.ds1 = o; o = al256(o + 4 * cells * H);
    L.ds2 = o; o = al256(o + 4 * cells * H);
    L.chunks = (int)std::max<int64_t>(1, (p.pixels + kMdWgCells - 1) / kMdWgCells);
    L.part = o; o = al256(o + 4 * nd * (size_t)L.chunks * ((size_t)H5 * (D + 2 * H + 1) + 6 * H));
    L.stotal = o;
    return L;
}

bool md_shape_ok(const MdPlan& p, const lstm_md_shape* s)
{
    return s && s->hidden_size >= 1 && s->hidden_size <= kMdMaxH && s->input_size >= 1 &&
           s->num_directions == p.ndir;
}

bool al16(const void* q) { return ((uintptr_t)q & 15) == 0; }

template <bool FWD>
lstm_status md_launch(const MdPlan& p, MdArgs& a, cudaStream_t s)
{
    const int H = a.H;
    const int NU = (H + 31) / 32;
    const size_t per_dir = (size_t)2 * 5 * H * H * 4;             // recurrent weights of one direction
    const void* fn_sm = nullptr;
    const void* fn_gl = nullptr;
#define MD_PICK(nu)                                                                                        \
    if (NU == nu) {                                                                                        \
        fn_sm = FWD ? (const void*)md_fwd_kernel<nu, true> : (const void*)md_bwd_kernel<nu, true>;         \
        fn_gl = FWD ? (const void*)md_fwd_kernel<nu, false> : (const void*)md_bwd_kernel<nu, false>;       \
    }
    MD_PICK(1) MD_PICK(2) MD_PICK(3) MD_PICK(4)
#undef MD_PICK
    if (!fn_sm) return LSTM_ERR_UNSUPPORTED;
    // direction groups (forward): the largest number (dividing ndir) for which a group's weights
    // fit in shared memory and that many CTAs share an SM, so that more warps hide the walk's
    // latency (measured on 4 directions, H = 32: 1.88 against 2.59 ms).  The backward walk
    // measured slower in groups (3.97 against 3.40 ms) and runs as one.  Otherwise one group,
    // weights resident if they fit, else read from L2.
    const void* fn = nullptr;
    size_t smem = 0;
    int ngrp = 1, per_sm = 0;
    for (int g = FWD ? p.ndir : 1; g >= 1; --g) {
        if (p.ndir % g) continue;
        const size_t sm = per_dir * (p.ndir / g);
        if (sm > kMdSmemCap) continue;
        if (cudaFuncSetAttribute(fn_sm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn_sm, kMdThreads, sm) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (per_sm >= g || (g == 1 && per_sm >= 1)) {
            fn = fn_sm; smem = sm; ngrp = g;
            break;
        }
    }
    if (!fn) {
        fn = fn_gl; smem = 0; ngrp = 1;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 0) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kMdThreads, 0) != cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            return LSTM_ERR_UNSUPPORTED;
        }
    }
    const int per = ngrp > 1 ? ngrp : std::min(per_sm, 2);
    const int grid = p.num_sms * per;                           // a multiple of ngrp
    a.ngrp = ngrp;
    if (cudaMemsetAsync(a.ctr, 0, sizeof(unsigned), s) != cudaSuccess) return LSTM_ERR_CUDA;
    void* args[] = {&a};
    tracer_begin(p.tracer, FWD ? MD_FWD : MD_BWD, s);
    const cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kMdThreads), args, smem, s);
    tracer_end(p.tracer, FWD ? MD_FWD : MD_BWD, s, e == cudaSuccess ? 1 : 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LSTM_ERR_CUDA;
    }
    return LSTM_OK;
}

MdArgs md_args(const MdPlan& p, int H)
{
    MdArgs a;
    memset(&a, 0, sizeof(a));
    a.H = H; a.ndir = p.ndir; a.steps = p.steps; a.N = p.pixels;
    a.step_off = p.d_step_off; a.src = p.d_src;
    a.pred1 = p.d_pred1; a.pred2 = p.d_pred2; a.succ1 = p.d_succ1; a.succ2 = p.d_succ2;
    a.ctr = p.d_ctr; a.status = p.d_status; a.wait_limit_ns = p.wait_limit_ns;
    a.debug_skip_cta = p.debug_skip_cta;
    return a;
}

// dx = dA W, dW = dA^T x (pixel order, all directions at once); dU1, dU2 per direction; db and
// the peephole sums.  *launched counts the kernels.
lstm_status md_grads(const MdPlan& p, int D, int H, const lstm_md_params* prm, const float* x, const float* dap,
                     const float* h, const float* c, const float* act, float* dx, const lstm_md_grads* grads,
                     float* part, int chunks, cudaStream_t s, int* launched)
{
    const int nd = p.ndir, H5 = 5 * H;
    lstm_status st = LSTM_OK;
    if (dx) {
        const int R = nd * H5;                         // a multiple of 4 (5H per direction, ndir 1..4: 5H*ndir)
        const size_t wsm = sizeof(float) * (size_t)R * D;
        const void* fn = D <= 16 ? (const void*)md_dx_kernel<16> : D <= 32 ? (const void*)md_dx_kernel<32>
                       : D <= 64 ? (const void*)md_dx_kernel<64> : nullptr;
        if (fn && R % 4 == 0 && wsm <= 200 * 1024 &&
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsm) == cudaSuccess) {
            const unsigned blocks = (unsigned)((p.pixels + 127) / 128);
            if (D <= 16) md_dx_kernel<16><<<blocks, 128, wsm, s>>>(dap, prm->W, R, D, p.pixels, dx);
            else if (D <= 32) md_dx_kernel<32><<<blocks, 128, wsm, s>>>(dap, prm->W, R, D, p.pixels, dx);
            else md_dx_kernel<64><<<blocks, 128, wsm, s>>>(dap, prm->W, R, D, p.pixels, dx);
            if (cudaGetLastError() != cudaSuccess) return LSTM_ERR_CUDA;
        } else {                                       // wide inputs: the CUDA-core GEMM
            cudaGetLastError();
            GemmDesc g;
            g.M = (int)p.pixels; g.N = D; g.K = R;
            g.A = dap; g.sam = R; g.sak = 1;
            g.B = prm->W; g.sbk = D; g.sbn = 1;
            g.C = dx; g.ldc = D;
            if ((st = gemm_simt_run(g, p.num_sms, s)) != LSTM_OK) return st;
        }
        *launched += 1;
    }
    if (grads->W || grads->U1 || grads->U2 || grads->b || grads->peep) {
        const size_t smem = md_wgrad_smem(D, H);
        if (cudaFuncSetAttribute(md_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return LSTM_ERR_UNSUPPORTED;
        }
        md_wgrad_kernel<<<dim3(chunks, nd), 256, smem, s>>>(act, h, c, x, p.d_src, p.d_pred1, p.d_pred2, D, H,
                                                             p.pixels, part);
        const int64_t nout = (int64_t)nd * (H5 * (D + 2 * H + 1) + 6 * H);
        md_wgrad_combine<<<(unsigned)((nout + 255) / 256), 256, 0, s>>>(part, chunks, D, H, nd, grads->W, grads->U1,
                                                                         grads->U2, grads->b, grads->peep);
        if (cudaGetLastError() != cudaSuccess) return LSTM_ERR_CUDA;
        *launched += 2;
    }
    return LSTM_OK;
}

}  // namespace

}  // namespace lstm

using lstm::MdLayout;
using lstm::MdPlan;

extern "C" {

size_t lstm_md_workspace_bytes(const lstm_md_plan* plan, const lstm_md_shape* shape)
{
    if (!plan || !lstm::md_shape_ok(plan->p, shape)) return 0;
    return lstm::md_layout(plan->p, shape->input_size, shape->hidden_size).total;
}

size_t lstm_md_scratch_bytes(const lstm_md_plan* plan, const lstm_md_shape* shape)
{
    if (!plan || !lstm::md_shape_ok(plan->p, shape)) return 0;
    return lstm::md_layout(plan->p, shape->input_size, shape->hidden_size).stotal;
}

lstm_status lstm_md_fwd(const lstm_md_plan* plan, const lstm_md_shape* shape, const lstm_md_params* prm,
                        const float* x, float* y, void* workspace, void* stream)
{
    if (!plan || !prm) return LSTM_ERR_INVALID_ARG;
    const MdPlan& p = plan->p;
    if (!lstm::md_shape_ok(p, shape)) return LSTM_ERR_INVALID_ARG;
    if (!p.d_src) return LSTM_ERR_UNSUPPORTED;                  // a host-only plan
    if (p.pixels == 0) return LSTM_OK;
    if (!x || !y || !workspace || !prm->W || !prm->U1 || !prm->U2 || !prm->b || !prm->peep) return LSTM_ERR_INVALID_ARG;
    if (!lstm::al16(workspace)) return LSTM_ERR_INVALID_ARG;
    const int D = shape->input_size, H = shape->hidden_size, nd = p.ndir, H5 = 5 * H;
    cudaStream_t s = (cudaStream_t)stream;
    const MdLayout L = lstm::md_layout(p, D, H);
    char* ws = (char*)workspace;
    float* gx = (float*)(ws + L.gx);
    // 1. gx = x W^T + b for every pixel and direction
    lstm::GemmDesc g;
    g.M = (int)p.pixels; g.N = nd * H5; g.K = D;
    g.A = x; g.sam = D; g.sak = 1;
    g.B = prm->W; g.sbk = 1; g.sbn = D;
    g.C = gx; g.ldc = nd * H5; g.bias = prm->b;
    lstm::tracer_begin(p.tracer, lstm::MD_INPUT, s);
    lstm_status st = lstm::gemm_simt_run(g, p.num_sms, s);
    // 2. U^T (forward operand) and U (backward operand, kept in the workspace)
    if (st == LSTM_OK) {
        lstm::md_transpose_kernel<<<64, 256, 0, s>>>(prm->U1, prm->U2, (float*)(ws + L.ut), (float*)(ws + L.ucat),
                                                     nd, H);
        if (cudaGetLastError() != cudaSuccess) st = LSTM_ERR_CUDA;
    }
    lstm::tracer_end(p.tracer, lstm::MD_INPUT, s, st == LSTM_OK ? 2 : 0);
    if (st != LSTM_OK) return st;
    lstm::MdArgs a = lstm::md_args(p, H);
    a.U = (const float*)(ws + L.ut);
    a.peep = prm->peep;
    a.gx = gx;
    a.h = (float*)(ws + L.h); a.c = (float*)(ws + L.c); a.act = (float*)(ws + L.act);
    a.y = y;
    return lstm::md_launch<true>(p, a, s);
}

lstm_status lstm_md_bwd(const lstm_md_plan* plan, const lstm_md_shape* shape, const lstm_md_params* prm,
                        const float* x, void* workspace, const float* dy, float* dx, const lstm_md_grads* grads,
                        void* scratch, void* stream)
{
    if (!plan || !prm || !grads) return LSTM_ERR_INVALID_ARG;
    const MdPlan& p = plan->p;
    if (!lstm::md_shape_ok(p, shape)) return LSTM_ERR_INVALID_ARG;
    if (!p.d_src) return LSTM_ERR_UNSUPPORTED;
    const int D = shape->input_size, H = shape->hidden_size, nd = p.ndir, H5 = 5 * H;
    cudaStream_t s = (cudaStream_t)stream;
    if (p.pixels == 0) {      // no pixel: every gradient is zero
        const size_t pc[5] = {(size_t)nd * H5 * D, (size_t)nd * H5 * H, (size_t)nd * H5 * H, (size_t)nd * H5,
                              (size_t)nd * 6 * H};
        float* dst[5] = {grads->W, grads->U1, grads->U2, grads->b, grads->peep};
        for (int i = 0; i < 5; ++i)
            if (dst[i] && cudaMemsetAsync(dst[i], 0, sizeof(float) * pc[i], s) != cudaSuccess) return LSTM_ERR_CUDA;
        return LSTM_OK;
    }
    if (!x || !dy || !workspace || !scratch || !prm->W || !prm->peep) return LSTM_ERR_INVALID_ARG;
    if (!lstm::al16(workspace) || !lstm::al16(scratch)) return LSTM_ERR_INVALID_ARG;
    const MdLayout L = lstm::md_layout(p, D, H);
    char* ws = (char*)workspace;
    char* sc = (char*)scratch;
    float* dap = (float*)(ws + L.gx);             // the pre-activations' region, no longer needed
    float* h = (float*)(ws + L.h);
    float* c = (float*)(ws + L.c);
    float* act = (float*)(ws + L.act);
    float* part = (float*)(sc + L.part);
    lstm::MdArgs a = lstm::md_args(p, H);
    a.U = (const float*)(ws + L.ucat);
    a.peep = prm->peep;
    a.h = h; a.c = c; a.act = act; a.dy = dy; a.dap = dap;
    a.ds1 = (float*)(sc + L.ds1); a.ds2 = (float*)(sc + L.ds2);
    lstm_status st = lstm::md_launch<false>(p, a, s);
    if (st != LSTM_OK) return st;
    lstm::tracer_begin(p.tracer, lstm::MD_GRADS, s);
    int launched = 0;
    st = lstm::md_grads(p, D, H, prm, x, dap, h, c, act, dx, grads, part, L.chunks, s, &launched);
    lstm::tracer_end(p.tracer, lstm::MD_GRADS, s, launched);
    return st;
}

}  // extern "C"
