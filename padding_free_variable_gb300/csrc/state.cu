// state.cu -- initial states and final-state errors of a layer.
//
// RETURNN paper, Sec. 3.2: the final state of one recurrent network can be
// passed on as the initial state of another.  A direction's state before its
// first step enters that step in two places: through the recurrent product
// R h0 and through the cell's previous state c0 (forget gate and the input
// and forget peepholes).  Here R h0 is one product over the batch whose rows
// are added into each sequence's first-step pre-activations before the
// recurrent kernel runs, so the kernels see it as part of the input
// projection; c0 is read by the kernels' cell at a sequence's first step.
// Backward, dL/dh0 = R^T da of the first step is one product over the
// gathered first-step gate errors, the weight gradient gains da h0^T for
// those rows, and dL/dc0 is the cell-state error the first step passes back
// (written by the recurrent kernels).
#include "common.cuh"
#include "gemm.cuh"
#include "state.cuh"

namespace lstm {

namespace {

// packed row of sorted slot j's first step in direction d (forward: t = 0, reverse: t = len - 1)
__device__ __forceinline__ int first_row(const int32_t* off, const int32_t* len, int d, int j)
{
    return d == 0 ? off[0] + j : off[len[j] - 1] + j;
}

// ga[first_row(d, j)][d*4H + r] += rh[d][perm[j]][r] for every slot with frames
__global__ void state_fold_kernel(float* __restrict__ ga, const float* __restrict__ rh, const int32_t* __restrict__ off,
                                  const int32_t* __restrict__ len, const int32_t* __restrict__ perm, int B, int H,
                                  int ndir)
{
    const int G4 = 4 * H;
    const int64_t total = (int64_t)ndir * B * G4;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i % G4);
        const int j = (int)((i / G4) % B);
        const int d = (int)(i / ((int64_t)G4 * B));
        if (len[j] == 0) continue;
        const int row = first_row(off, len, d, j);
        ga[(size_t)row * ndir * G4 + (size_t)d * G4 + r] += rh[((size_t)d * B + perm[j]) * G4 + r];
    }
}

// out[d][perm[j]][r] = ga[first_row(d, j)][d*4H + r] (the first step's gate errors), 0 for
// empty sequences
__global__ void state_gather_kernel(const float* __restrict__ ga, float* __restrict__ out,
                                    const int32_t* __restrict__ off, const int32_t* __restrict__ len,
                                    const int32_t* __restrict__ perm, int B, int H, int ndir)
{
    const int G4 = 4 * H;
    const int64_t total = (int64_t)ndir * B * G4;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i % G4);
        const int j = (int)((i / G4) % B);
        const int d = (int)(i / ((int64_t)G4 * B));
        float v = 0.f;
        if (len[j] > 0) v = ga[(size_t)first_row(off, len, d, j) * ndir * G4 + (size_t)d * G4 + r];
        out[((size_t)d * B + perm[j]) * G4 + r] = v;
    }
}

// empty sequences pass their final-state errors straight to the initial state
__global__ void state_empty_kernel(const int32_t* __restrict__ len, const int32_t* __restrict__ perm, int B, int H,
                                   int ndir, const float* __restrict__ dh_n, const float* __restrict__ dc_n,
                                   float* __restrict__ dh0, float* __restrict__ dc0)
{
    const int64_t total = (int64_t)ndir * B * H;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int u = (int)(i % H);
        const int j = (int)((i / H) % B);
        const int d = (int)(i / ((int64_t)H * B));
        if (len[j] != 0) continue;
        const size_t o = ((size_t)d * B + perm[j]) * H + u;
        if (dh0) dh0[o] = dh_n ? dh_n[o] : 0.f;
        if (dc0) dc0[o] = dc_n ? dc_n[o] : 0.f;
    }
}

int grid_for(int64_t total, int num_sms)
{
    return (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 8));
}

}  // namespace

size_t state_scratch_floats(const Plan& p, int H, int ndir)
{
    return (size_t)ndir * p.B * 4 * H;
}

lstm_status state_fold_input(const Plan& p, int H, int ndir, bool bf16, const void* R, const float* h0, float* ga,
                             float* scratch, cudaStream_t s)
{
    if (!h0 || p.B == 0) return LSTM_OK;
    const size_t esz = bf16 ? 2 : 4;
    lstm_status st;
    for (int d = 0; d < ndir; ++d) {
        // rh[d][b][r] = sum_k h0[d][b][k] R_d[r][k] (bf16 layers: h0 rounded like every h operand)
        GemmDesc g;
        g.M = p.B; g.N = 4 * H; g.K = H;
        g.A = h0 + (size_t)d * p.B * H; g.sam = H; g.sak = 1;
        g.B = (const char*)R + (size_t)d * 4 * H * H * esz; g.sbk = 1; g.sbn = H; g.b_bf16 = bf16;
        g.C = scratch + (size_t)d * p.B * 4 * H; g.ldc = 4 * H;
        g.round_bf16 = bf16; g.k_splits = 1;
        if ((st = gemm_simt(g, p, K_GEMM_IN, s)) != LSTM_OK) return st;
    }
    const int64_t total = (int64_t)ndir * p.B * 4 * H;
    state_fold_kernel<<<grid_for(total, p.num_sms), 256, 0, s>>>(ga, scratch, p.d_off, p.d_len, p.d_perm, p.B, H, ndir);
    return cudaGetLastError() == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

lstm_status state_backward(const Plan& p, int H, int ndir, bool bf16, const void* R, const float* ga, const float* h0,
                           const float* dh_n, const float* dc_n, float* dh0, float* dc0, float* dR, float* scratch,
                           cudaStream_t s)
{
    if (p.B == 0) return LSTM_OK;
    const size_t esz = bf16 ? 2 : 4;
    const int64_t total = (int64_t)ndir * p.B * 4 * H;
    lstm_status st;
    if (dh0 || h0) {
        state_gather_kernel<<<grid_for(total, p.num_sms), 256, 0, s>>>(ga, scratch, p.d_off, p.d_len, p.d_perm, p.B,
                                                                       H, ndir);
        if (cudaGetLastError() != cudaSuccess) return LSTM_ERR_CUDA;
    }
    for (int d = 0; d < ndir; ++d) {
        const float* daf = scratch + (size_t)d * p.B * 4 * H;
        const char* Rd = (const char*)R + (size_t)d * 4 * H * H * esz;
        if (dh0) {
            // dh0[d][b][u] = sum_r da_first[d][b][r] R_d[r][u]
            GemmDesc g;
            g.M = p.B; g.N = H; g.K = 4 * H;
            g.A = daf; g.sam = 4 * H; g.sak = 1;
            g.B = Rd; g.sbk = H; g.sbn = 1; g.b_bf16 = bf16;
            g.C = dh0 + (size_t)d * p.B * H; g.ldc = H;
            g.round_bf16 = bf16; g.k_splits = 1;
            if ((st = gemm_simt(g, p, K_GEMM_DR, s)) != LSTM_OK) return st;
        }
        if (h0) {
            // dR_d[r][k] += sum_b da_first[d][b][r] h0[d][b][k]: the first steps' h_{t-1} is h0
            GemmDesc g;
            g.M = 4 * H; g.N = H; g.K = p.B;
            g.A = daf; g.sam = 1; g.sak = 4 * H;
            g.B = h0 + (size_t)d * p.B * H; g.sbk = H; g.sbn = 1;
            g.C = dR + (size_t)d * 4 * H * H; g.ldc = H;
            g.round_bf16 = bf16; g.k_splits = 1; g.accumulate = 1;
            if ((st = gemm_simt(g, p, K_GEMM_DR, s)) != LSTM_OK) return st;
        }
    }
    if (dh0 || dc0) {
        const int64_t n = (int64_t)ndir * p.B * H;
        state_empty_kernel<<<grid_for(n, p.num_sms), 256, 0, s>>>(p.d_len, p.d_perm, p.B, H, ndir, dh_n, dc_n, dh0,
                                                                  dc0);
        if (cudaGetLastError() != cudaSuccess) return LSTM_ERR_CUDA;
    }
    return LSTM_OK;
}

}  // namespace lstm
