// stepwise.cu -- cell kernels of the per-step-launch recurrence.
//
// The design the pages describe for their own GPU LSTM ("RETURNN", Sec. 4.2:
// one matrix product for the non-recurrent part, then per time step a product
// with the recurrent weights and a small kernel for the gating): each step of
// each direction is one product launch (R·h_{t-1} over the step's active
// rows) and each step one cell launch for both directions.  With CUDA-core
// products it is the comparator that measures what the persistent, on-chip
// design saves; with tcgen05 products it is the path for bf16 layers whose R
// does not fit one thread-block cluster (each step's product is then a GEMM
// large enough to spread over the whole GPU).
#include <cuda_bf16.h>

#include "common.cuh"
#include "stepwise.cuh"

namespace lstm {

namespace {

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }

}  // namespace

// One thread per (row j, unit u) of one direction (blockIdx.y) at step s.
__global__ void step_cell_fwd_kernel(StepArgs a, int s)
{
    const int dir = blockIdx.y, H = a.H, T = a.T;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = idx / H, u = idx - j * H;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    if (s == 0 && j < a.B && a.slot_len[j] == 0 && a.h_n) {      // empty sequences end in their initial state
        const size_t o = ((size_t)dir * a.B + a.perm[j]) * H + u;
        a.h_n[o] = a.h0 ? a.h0[o] : 0.f;
        if (a.c_n) a.c_n[o] = a.c0 ? a.c0[o] : 0.f;
    }
    const int t = dir == 0 ? s : T - 1 - s;
    const int n = a.bs[t];
    if (j >= n) return;
    const int row = a.off[t] + j;
    const bool has_prev = dir == 0 ? t >= 1 : (t + 1 < T && j < a.bs[t + 1]);
    const int prow = has_prev ? (dir == 0 ? a.off[t - 1] + j : a.off[t + 1] + j) : 0;
    const float* pre = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u;
    const float* rh = a.rh + ((size_t)dir * a.rh_splits * a.B + j) * 4 * H + u;
    const size_t rstride = (size_t)a.B * 4 * H;
    // R h_{t-1}: the slices added in order, the four gates' loads of a slice issued together
    float r[4] = {0.f, 0.f, 0.f, 0.f};
    if (has_prev) {
#pragma unroll
        for (int g = 0; g < 4; ++g) r[g] = rh[g * H];
        for (int z = 1; z < a.rh_splits; ++z) {
#pragma unroll
            for (int g = 0; g < 4; ++g) r[g] += rh[z * rstride + g * H];
        }
    }
    float av[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) av[g] = pre[g * H] + r[g];
    const size_t so = ((size_t)dir * a.B + a.perm[j]) * H + u;     // caller-order state
    const float cp = has_prev ? a.cbuf[(size_t)prow * ndH + dir * H + u] : (a.c0 ? a.c0[so] : 0.f);
    const float* pp = a.peep + (size_t)dir * 3 * H + u;
    const float ig = sigm(av[0] + pp[0] * cp);
    const float fg = sigm(av[1] + pp[H] * cp);
    const float zg = tanhf(av[2]);
    float c = fg * cp + ig * zg;
    const float og = sigm(av[3] + pp[2 * H] * c);
    float h = og * tanhf(c);
    const int len = a.slot_len[j];
    if (a.padded && t >= len) { c = 0.f; h = 0.f; }     // a padding frame: computed, then masked
    float* gw = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u;
    gw[0] = ig; gw[H] = fg; gw[2 * H] = zg; gw[3 * H] = og;
    const size_t yo = (size_t)row * ndH + dir * H + u;
    a.cbuf[yo] = c;
    a.y[yo] = h;
    if (a.y_lo) a.y_lo[yo] = __float2bfloat16_rn(h);
    if (a.hb16) a.hb16[((size_t)dir * a.B + j) * H + u] = __float2bfloat16_rn(h);
    if (a.h_n && ((dir == 0 && t == len - 1) || (dir == 1 && t == 0))) {
        const size_t o = ((size_t)dir * a.B + a.perm[j]) * H + u;
        a.h_n[o] = h;
        if (a.c_n) a.c_n[o] = c;
    }
}

// BPTT of one step: gate errors of the step's rows from dy, the recurrent
// error R^T da of the step after it (in recurrence order) and the cell-state
// error carried from there.
__global__ void step_cell_bwd_kernel(StepArgs a, int s)
{
    const int dir = blockIdx.y, H = a.H, T = a.T;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = idx / H, u = idx - j * H;
    const int ndH = a.ndir * H, nd4H = a.ndir * 4 * H;
    const int t = dir == 0 ? T - 1 - s : s;
    const int n = a.bs[t];
    if (j >= n) return;
    const int row = a.off[t] + j;
    // the step after t in recurrence order, and the step before it (c_{t-1} of the peepholes)
    const bool has_next = dir == 0 ? (t + 1 < T && j < a.bs[t + 1]) : t >= 1;
    const bool has_prev = dir == 0 ? t >= 1 : (t + 1 < T && j < a.bs[t + 1]);
    const int prow = has_prev ? (dir == 0 ? a.off[t - 1] + j : a.off[t + 1] + j) : 0;
    float* gw = a.ga + (size_t)row * nd4H + (size_t)dir * 4 * H + u;
    const float ig = gw[0], fg = gw[H], zg = gw[2 * H], og = gw[3 * H];
    const size_t yo = (size_t)row * ndH + dir * H + u;
    const float c = a.cbuf[yo];
    const size_t st = ((size_t)dir * a.B + a.perm[j]) * H + u;     // caller-order state
    const float cp = has_prev ? a.cbuf[(size_t)prow * ndH + dir * H + u] : (a.c0 ? a.c0[st] : 0.f);
    const size_t so = ((size_t)dir * a.B + j) * H + u;
    float dhr = 0.f;
    if (has_next) {
        const float* dr = a.dh_rec + ((size_t)dir * a.dh_splits * a.B + j) * H + u;
        for (int z = 0; z < a.dh_splits; ++z) dhr += dr[(size_t)z * a.B * H];
    } else if (a.dh_n) {
        dhr = a.dh_n[st];                          // the sequence's last step: the final state's error
    }
    const float dh = a.dy[yo] + dhr;
    const float carry = has_next ? a.dcc[so] : (a.dc_n ? a.dc_n[st] : 0.f);
    const float* pp = a.peep + (size_t)dir * 3 * H + u;
    float dai = 0.f, daf = 0.f, daz = 0.f, dao = 0.f, carry_out = 0.f;
    if (!a.padded || t < a.slot_len[j]) {           // a padding frame passes no gradient
        const float tc = tanhf(c);
        dao = dh * tc * og * (1.f - og);
        const float dc = dh * og * (1.f - tc * tc) + dao * pp[2 * H] + carry;
        dai = dc * zg * ig * (1.f - ig);
        daf = dc * cp * fg * (1.f - fg);
        daz = dc * ig * (1.f - zg * zg);
        carry_out = dc * fg + dai * pp[0] + daf * pp[H];
        if (!has_prev && a.dc0) a.dc0[st] = carry_out;   // the sequence's first step
    }
    gw[0] = dai; gw[H] = daf; gw[2 * H] = daz; gw[3 * H] = dao;
    a.dcc[so] = carry_out;
    if (a.dab16) {
        __nv_bfloat16* db = a.dab16 + ((size_t)dir * a.B + j) * 4 * H + u;
        db[0] = __float2bfloat16_rn(dai); db[H] = __float2bfloat16_rn(daf);
        db[2 * H] = __float2bfloat16_rn(daz); db[3 * H] = __float2bfloat16_rn(dao);
    }
}

lstm_status step_cell_launch(const StepArgs& a, int s, bool backward, cudaStream_t st)
{
    const int threads = 256;
    const dim3 grid((unsigned)ceil_div(a.B * a.H, threads), (unsigned)a.ndir);
    if (backward) step_cell_bwd_kernel<<<grid, threads, 0, st>>>(a, s);
    else step_cell_fwd_kernel<<<grid, threads, 0, st>>>(a, s);
    return cudaGetLastError() == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

}  // namespace lstm
