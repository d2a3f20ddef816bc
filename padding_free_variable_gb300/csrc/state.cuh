// state.cuh -- initial states of a layer: the product R h0 folded into the first
// steps' pre-activations, and the backward pass's dL/dh0 and dR term.
#pragma once

#include "common.cuh"

namespace lstm {

// Floats of scratch the two calls below need ([ndir][B][4H]).
size_t state_scratch_floats(const Plan& p, int H, int ndir);

// ga[first row of (d, sequence b)][d*4H + r] += (R_d h0[d][b])[r] for every non-empty
// sequence.  No-op without h0.
lstm_status state_fold_input(const Plan& p, int H, int ndir, bool bf16, const void* R, const float* h0, float* ga,
                             float* scratch, cudaStream_t s);

// After the BPTT kernel (ga holds the gate errors): dh0 = R^T da of each sequence's first
// step; dR += da_first h0^T when h0 is given; empty sequences get dh0 = dh_n, dc0 = dc_n
// (dc0 of the others is written by the recurrent kernels).  Any pointer may be null.
lstm_status state_backward(const Plan& p, int H, int ndir, bool bf16, const void* R, const float* ga, const float* h0,
                           const float* dh_n, const float* dc_n, float* dh0, float* dc0, float* dR, float* scratch,
                           cudaStream_t s);

}  // namespace lstm
