// stepwise.cuh -- per-step cell kernels of the per-step-launch comparator path.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace lstm {

struct StepArgs {
    int T, B, H, ndir;
    const int32_t* bs;        // [T] active rows per step
    const int32_t* off;       // [T+1] first row of each step
    const int32_t* slot_len;  // [B]
    const int32_t* perm;      // [B]
    float* ga;                // [rows][ndir*4H] pre-activations -> gates -> gate errors
    const float* rh;          // forward: [ndir][rh_splits][B][4H] the step's R h_{t-1} (slices added in order)
    const float* peep;        // [ndir][3][H]
    float* y;                 // [rows][ndir*H]
    __nv_bfloat16* y_lo;      // optional bf16 copy of y
    float* cbuf;              // [rows][ndir*H]
    float* h_n;               // [ndir][B][H] caller order, optional
    float* c_n;
    const float* dy;          // backward: [rows][ndir*H]
    const float* dh_rec;      // backward: [ndir][dh_splits][B][H] R^T da of the step after (recurrence order)
    float* dcc;               // backward: [ndir][B][H] cell-state error carry
    __nv_bfloat16* hb16;      // optional, forward: [ndir][B][H] bf16 h of the step's rows (next product's A)
    __nv_bfloat16* dab16;     // optional, backward: [ndir][B][4H] bf16 gate errors of the step's rows
    int rh_splits, dh_splits; // K slices of the per-step products (1 without split)
    int padded;               // the padded comparator's plan: frames t >= length are masked
    // initial states and final-state errors, [ndir][B][H] caller order (NULL = zero / not wanted);
    // R h0 is folded into the first step's pre-activations beforehand
    const float* h0;
    const float* c0;
    const float* dh_n;
    const float* dc_n;
    float* dc0;
};

// Cell of step s (forward, or BPTT in backward order) for both directions.
lstm_status step_cell_launch(const StepArgs& a, int s, bool backward, cudaStream_t st);

}  // namespace lstm
