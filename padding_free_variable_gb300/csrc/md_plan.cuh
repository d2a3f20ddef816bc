// md_plan.cuh -- the 2-D (MDLSTM) layer's plan: example placement on a packed
// canvas and the wavefront schedule of its cells.
#pragma once

#include "common.cuh"

namespace lstm {

struct MdPlan {
    int32_t n = 0;                // examples
    int32_t ndir = 0;             // scan directions (1..4)
    int32_t schedule = 0;         // 0 canvas, 1 per-example diagonals
    int64_t pixels = 0;           // N: pixels of all examples
    int64_t cells = 0;            // ndir * N
    int32_t steps = 0;            // wavefront steps
    int32_t canvas_h = 0, canvas_w = 0;
    int32_t rows = 0;             // packed rows of the canvas
    int device = 0;
    int num_sms = 0;
    uint64_t wait_limit_ns = 2000000000ull;
    int32_t debug_skip_cta = -1;  // test hook: this CTA never arrives at the first barrier
    // host tables
    int32_t* h_y0 = nullptr;      // [n] canvas row of the example's top-left pixel (-1: empty)
    int32_t* h_x0 = nullptr;      // [n]
    int64_t* h_pix_off = nullptr; // [n+1] first pixel of each example (caller order)
    int64_t* h_step_off = nullptr;  // [ndir][steps+1] first cell of each step (cell order)
    // device tables (cell order: direction, step, packing order, row within the diagonal)
    int64_t* d_step_off = nullptr;
    int32_t* d_src = nullptr;     // [cells] pixel of the cell
    int32_t* d_pred1 = nullptr;   // [cells] cell holding predecessor 1 (previous row in scan order), -1 none
    int32_t* d_pred2 = nullptr;   // [cells] predecessor 2 (previous column in scan order)
    int32_t* d_succ1 = nullptr;   // [cells] the cell whose predecessor 1 this is, -1 none
    int32_t* d_succ2 = nullptr;
    unsigned* d_ctr = nullptr;    // grid barrier counter
    DeviceStatus* d_status = nullptr;
    Tracer* tracer = nullptr;     // owned: launch count and optional per-phase CUDA-event timing
};

// Phases the 2-D plan's tracer times (lstm_md_plan_read_timing order).
enum MdKind { MD_INPUT = 0, MD_FWD, MD_BWD, MD_GRADS, MD_NUM };

}  // namespace lstm

struct lstm_md_plan {
    lstm::MdPlan p;
};
