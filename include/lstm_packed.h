/*
 * lstm_packed.h -- C ABI of the padding-free (bi)LSTM library for sm_103a.
 *
 * The library computes the forward pass and the BPTT backward pass of LSTM
 * layers with forget gates and peephole connections over a batch of
 * variable-length sequences without computing any padded frame.
 *
 * Sources for what is computed:
 *  - "No Padding Please: Efficient Neural Handwriting Recognition", Sec. V
 *    (example-packing) and Appendix B (Algorithm 1): a list of variable-size
 *    examples is packed, the layer runs on the packed tensor, and unpacking
 *    extracts each example's activations with the original example indices.
 *    Here the packing is the one-dimensional form: sequences are sorted by
 *    length (longest first, ties keep the caller's order) and laid out time
 *    major, so the rows of time step t are the first bs[t] sorted sequences.
 *  - "Single Stream Parallelization of Generalized LSTM-Like RNNs on a GPU",
 *    Sec. 2-3 and Fig. 1: the LSTM with forget gates and peepholes built from
 *    additive and multiplicative layers, its BPTT training equations, and the
 *    split into a non-recurrent part computed in parallel over all frames and
 *    a recurrent part computed step by step.
 *  - RETURNN paper, Sec. 4.2: the non-recurrent part of the forward pass is
 *    one matrix product over the whole batch of sequences, and so are the
 *    weight and input gradients after the recurrent part has been
 *    back-propagated; the gating runs in custom kernels.
 *
 * The cell (one direction; the page's equations were lost, this is the
 * standard reading of its graph):
 *     a_t = W x_t + R h_{t-1} + b          gate blocks (i, f, z, o) along 4H
 *     i = sig(a_i + p_i c_{t-1}),  f = sig(a_f + p_f c_{t-1}),  z = tanh(a_z)
 *     c_t = f c_{t-1} + i z,   o = sig(a_o + p_o c_t),   h_t = o tanh(c_t)
 * with h_0 = c_0 = 0.  The reverse direction runs its own cell over
 * x_L..x_1; its output at position t is its state after consuming x_t.
 *
 * Conventions shared by every entry point:
 *  - All device buffers are allocated, owned and freed by the caller.  The
 *    library owns only what lstm_plan_create allocates (small index tables,
 *    step flags and a status word), freed by lstm_plan_destroy.
 *  - Every call is asynchronous on the caller's CUDA stream, passed as
 *    `void* stream` (a cudaStream_t; NULL = legacy default stream).  A plan
 *    may be used by one stream at a time and must outlive its queued work.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call launches nothing and returns LSTM_ERR_INVALID_ARG (bad
 *    pointer, size or alignment) or LSTM_ERR_UNSUPPORTED (a shape or device
 *    the kernels do not cover).  LSTM_ERR_CUDA reports a failed CUDA call.
 *  - Device-side failures (a step barrier that waited longer than the
 *    plan's limit, an index out of range) are recorded in the plan's device
 *    status word; kernels then stop early instead of hanging or trapping.
 *    lstm_status_poll reads and clears it.
 *  - Row-major everywhere.  Packed tensors have N = sum of lengths rows in
 *    the packed order; "cat" tensors have N rows in the caller's order
 *    (sequence 0's frames, then sequence 1's, ...).
 *  - Pointers to device arrays must be 16-byte aligned.
 *  - Nothing throws across this boundary.
 */
#ifndef LSTM_PACKED_H
#define LSTM_PACKED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LSTM_OK = 0,
    LSTM_ERR_INVALID_ARG = 1,
    LSTM_ERR_UNSUPPORTED = 2,
    LSTM_ERR_CUDA = 3,
    LSTM_ERR_TIMEOUT = 4,   /* a per-step barrier wait ran past the plan's limit */
    LSTM_ERR_BOUNDS = 5     /* a kernel found an index outside its buffer */
} lstm_status;

/* Element type of the GEMM operands x, W and R.  Biases, peepholes, states,
 * gates, outputs and all gradients are fp32 in both cases.  With LSTM_BF16
 * the products W x, R h, and the gradient products take bf16 operands
 * (h and the gate errors are rounded to bf16 before they enter a product)
 * and accumulate in fp32. */
typedef enum { LSTM_F32 = 0, LSTM_BF16 = 1 } lstm_dtype;

typedef struct lstm_plan lstm_plan;

typedef struct {
    int32_t input_size;      /* D: width of one input frame, >= 1 */
    int32_t hidden_size;     /* H: units per direction, multiple of 8, 8..2048 */
    int32_t num_directions;  /* 1 (forward only) or 2 (forward and reverse) */
    int32_t dtype;           /* lstm_dtype of x, W and R */
} lstm_layer_shape;

/* Parameters of one layer, device pointers, ndir = num_directions:
 *   W    [ndir][4H][D]   dtype   input weights, gate blocks (i, f, z, o)
 *   R    [ndir][4H][H]   dtype   recurrent weights, same blocks
 *   b    [ndir][4H]      fp32    one bias per gate unit
 *   peep [ndir][3][H]    fp32    diagonal peepholes p_i, p_f, p_o           */
typedef struct {
    const void*  W;
    const void*  R;
    const float* b;
    const float* peep;
} lstm_layer_params;

/* Gradients of one layer, fp32, same shapes as lstm_layer_params.
 * Each is overwritten (not accumulated). */
typedef struct {
    float* dW;
    float* dR;
    float* db;
    float* dpeep;
} lstm_layer_grads;

/*
 * Build the packing plan of one batch ("No Padding Please", Sec. V-A and
 * Algorithm 1: bucket and order the examples, keep the original example
 * indices; here a stable sort by decreasing length).
 *   lengths_host[B]  frames per sequence, each >= 0 (host memory, read only
 *                    during the call); B >= 1; sum <= 2^31 - 1.
 *   out              receives the plan.
 * Allocates the plan's device tables with cudaMalloc and uploads them
 * synchronously on the current device.
 */
lstm_status lstm_plan_create(const int32_t* lengths_host, int32_t B, lstm_plan** out);

/*
 * The padded comparator's plan: the same batch laid out as a right-padded
 * time x batch grid (RETURNN paper, Sec. 5: an index tensor marks which
 * frames of the time x batch tensor belong to a sequence; "No Padding
 * Please", Sec. V: a binary mask blocks state input from padding cells).
 * Every one of the T_max steps runs all B sequences in the caller's order;
 * frames past a sequence's end are computed and then masked: their state
 * and output are set to zero, and they pass no gradient.  Packed buffers of
 * this plan have B * T_max rows.
 */
lstm_status lstm_plan_create_padded(const int32_t* lengths_host, int32_t B, lstm_plan** out);

/*
 * Host-only form of the plan (no device, no allocation): the tables
 * lstm_plan_create uploads.  lstm_plan_dims gives the sizes to allocate:
 * steps T and rows (N packed, or B*T padded).  lstm_plan_compute_host fills
 * every non-NULL output:
 *   batch_sizes[T]  active rows of step t
 *   offsets[T+1]    first row of step t
 *   perm[B]         caller index of the sequence in slot j (longest first;
 *                   equal lengths keep the caller's order)
 *   slot_len[B]     its length
 *   row_src[rows]   caller-order frame of each row (-1: padding row)
 *   prev_fwd[rows]  row holding the forward direction's h_{t-1} (-1: none)
 *   prev_rev[rows]  row holding the reverse direction's state of step t+1
 *                   (-1: the sequence starts there)
 * padded != 0 gives the padded comparator's tables.
 */
lstm_status lstm_plan_dims(const int32_t* lengths_host, int32_t B, int32_t padded, int32_t* steps,
                           int64_t* rows);
lstm_status lstm_plan_compute_host(const int32_t* lengths_host, int32_t B, int32_t padded,
                                   int32_t* batch_sizes, int32_t* offsets, int32_t* perm,
                                   int32_t* slot_len, int32_t* row_src, int32_t* prev_fwd,
                                   int32_t* prev_rev);

/*
 * Segment plan (RETURNN paper, Sec. 4: sequences are cut into possibly
 * overlapping segments of constant length, each trained as a sequence of its
 * own, which trades context for far less padding).  Sequence b of lengths_host
 * yields segments starting at frames 0, step, 2*step, ... of min(chunk,
 * L_b - start) frames, up to the first segment that reaches the sequence's
 * end; an empty sequence yields one empty segment.  1 <= step <= chunk.
 * The plan's sequences ("caller order") are the segments in that order
 * (sequence-major): h_n, c_n and states are per segment.  lstm_pack reads the
 * caller's concatenated frames of the ORIGINAL sequences (frames overlapped by
 * two segments are read by both); lstm_unpack writes each original frame once,
 * from the segment that owns it (a segment owns its frames up to the next
 * segment's start, the last one to the sequence's end).  lstm_plan_info
 * reports the segments as the batch and sum(L_b) as the frames.
 */
lstm_status lstm_plan_create_segments(const int32_t* lengths_host, int32_t B, int32_t chunk,
                                      int32_t step, lstm_plan** out);

/* Host-only listing of the same segments (no device, no allocation):
 * *num_segments receives their count; with capacity >= that count the arrays
 * (any may be NULL) receive each segment's sequence, start frame and length.
 * LSTM_ERR_INVALID_ARG when the arrays are too short. */
lstm_status lstm_segments_host(const int32_t* lengths_host, int32_t B, int32_t chunk, int32_t step,
                               int32_t* num_segments, int32_t* seg_seq, int32_t* seg_start,
                               int32_t* seg_len, int32_t capacity);

/*
 * Window plan for truncated back-propagation through time ("Single Stream
 * Parallelization...", Sec. 4, BPTT(h; h'): the network steps h' frames at a
 * time, and the errors of those frames are back-propagated through them only).
 * The plan covers frames [start, start + width) of every sequence (fewer, or
 * none, near and past its end) with all B sequences in the caller's order, so
 * lstm_fwd_state started from the previous window's h_n / c_n continues each
 * sequence exactly, and lstm_bwd_state truncates its errors at the window's
 * start.  lstm_pack reads and lstm_unpack writes the caller's full
 * concatenated tensors (sum(L_b) rows): only the window's frames are touched.
 */
lstm_status lstm_plan_create_window(const int32_t* lengths_host, int32_t B, int32_t start, int32_t width,
                                    lstm_plan** out);

/*
 * Dynamic (frame-budget) batch formation ("On batching variable size
 * inputs...", Sec. 2: a dynamic batch size is a total length of the batch's
 * sequences rather than a number of sequences, so that batches of short
 * sequences hold more of them).  Sequences are taken in the given order (the
 * caller's batching strategy -- random, sorted or bucketed -- fixes that
 * order); each joins the current batch while the batch stays within `budget`,
 * else it starts the next batch.  budget_kind 0 counts packed frames (sum of
 * the batch's lengths: what the packed kernels compute); 1 counts padded
 * frames (sequences x longest length: the page's definition).  A sequence that
 * alone exceeds the budget forms a batch of its own (cut it first with
 * lstm_plan_create_segments to bound it).  Writes batch_of[i] (batches
 * numbered from 0 in order) and *num_batches.  Host only.
 */
lstm_status lstm_form_batches(const int32_t* lengths_host, int32_t n, int64_t budget, int32_t budget_kind,
                              int32_t* batch_of, int32_t* num_batches);

/* Free the plan and its device tables.  NULL is accepted. */
lstm_status lstm_plan_destroy(lstm_plan* plan);

/* Sizes of the plan: rows of a packed tensor (N, or B*T_max when padded),
 * number of steps T (the longest length), batch B, sum of lengths. */
lstm_status lstm_plan_info(const lstm_plan* plan, int64_t* rows, int32_t* steps, int32_t* batch,
                           int64_t* frames);

/* Host copies of the plan's tables, owned by the plan:
 *   batch_sizes[T]  rows of step t (the active sequences)
 *   offsets[T+1]    first packed row of step t
 *   perm[B]         caller index of the sequence in sorted slot j
 *   slot_len[B]     length of the sequence in slot j                         */
lstm_status lstm_plan_tables(const lstm_plan* plan, const int32_t** batch_sizes,
                             const int32_t** offsets, const int32_t** perm,
                             const int32_t** slot_len);

/* Set the barrier wait limit in nanoseconds (default 2 s).  A step whose
 * barrier waits longer records LSTM_ERR_TIMEOUT and the kernel returns. */
lstm_status lstm_plan_set_wait_limit(lstm_plan* plan, uint64_t nanoseconds);

/*
 * Bytes of the per-layer workspace that lstm_fwd fills and lstm_bwd reads
 * (the saved activations of BPTT: gate activations [rows][ndir*4H] and cell
 * states [rows][ndir*H], fp32).  lstm_bwd overwrites the gate part with the
 * gate errors.  0 on a bad argument.
 */
size_t lstm_workspace_bytes(const lstm_plan* plan, const lstm_layer_shape* shape);

/* Bytes of the transient scratch lstm_bwd needs: the recurrent kernel's
 * exchange of partial products R^T da between CTAs, and (reusing the same
 * bytes afterwards) the split-K partial sums of the weight-gradient
 * products.  Depends on the plan's CTA count: size it after
 * lstm_plan_set_ctas_per_direction.  0 on a bad argument. */
size_t lstm_scratch_bytes(const lstm_plan* plan, const lstm_layer_shape* shape);

/*
 * Pack ("No Padding Please", Sec. V-A): x_packed[row] = x_cat[source(row)]
 * for every packed row; rows of the padded plan past a sequence's end are
 * zero-filled.
 *   x_cat     [frames][width] elements of elem_bytes (2 or 4) in caller order
 *   x_packed  [rows][width]
 * width * elem_bytes must be a multiple of 16.
 */
lstm_status lstm_pack(const lstm_plan* plan, const void* x_cat, int32_t width, int32_t elem_bytes,
                      void* x_packed, void* stream);

/*
 * Unpack ("No Padding Please", Sec. V-A: extract each example's activations
 * using the original example indices): y_cat[source(row)] = y_packed[row];
 * padding rows are dropped.  Exact inverse of lstm_pack (bitwise).
 */
lstm_status lstm_unpack(const lstm_plan* plan, const void* y_packed, int32_t width,
                        int32_t elem_bytes, void* y_cat, void* stream);

/*
 * Forward pass of one layer ("Single Stream Parallelization...", Sec. 3:
 * the non-recurrent part over all frames at once, then the recurrent part
 * step by step; RETURNN, Sec. 4.2).
 *   x_packed   [rows][D] dtype         layer input in packed order
 *   y_packed   [rows][ndir*H] fp32     output [h_fwd | h_rev] per row
 *   y_lo       [rows][ndir*H] bf16     optional bf16 copy of y (the next
 *                                      bf16 layer's input); NULL to skip
 *   h_n, c_n   [ndir][B][H] fp32       final states in caller order (zero
 *                                      for empty sequences); NULL to skip
 *   workspace  lstm_workspace_bytes    saved activations for lstm_bwd
 */
lstm_status lstm_fwd(const lstm_plan* plan, const lstm_layer_shape* shape,
                     const lstm_layer_params* params, const void* x_packed, float* y_packed,
                     void* y_lo, float* h_n, float* c_n, void* workspace, void* stream);

/*
 * BPTT of one layer ("Single Stream Parallelization...", Sec. 3; RETURNN,
 * Sec. 4.2: the weight and input gradients as single products after the
 * recurrent part is back-propagated through time).
 *   x_packed, y_packed, workspace   as left by lstm_fwd of this layer
 *   dy_packed  [rows][ndir*H] fp32  dL/dy of this layer (read only)
 *   dx_packed  [rows][D] fp32       dL/dx, overwritten; NULL to skip
 *   grads                           overwritten
 *   scratch    lstm_scratch_bytes
 */
lstm_status lstm_bwd(const lstm_plan* plan, const lstm_layer_shape* shape,
                     const lstm_layer_params* params, const void* x_packed,
                     const float* y_packed, void* workspace, const float* dy_packed,
                     float* dx_packed, const lstm_layer_grads* grads, void* scratch,
                     void* stream);

/*
 * Initial states and final-state errors of one layer (RETURNN paper, Sec. 3.2:
 * the final state of one recurrent network passed on as the initial state of
 * another).  Every array is [ndir][B][H] fp32 in caller order (direction d,
 * sequence b at [d][b]), device memory, 16-byte aligned; any pointer may be
 * NULL, meaning zero (inputs) or not wanted (outputs).
 *   h0, c0      the state a direction starts from: the forward direction's
 *               state before frame 0, the reverse direction's before frame
 *               L-1 (it consumes x_L .. x_1).  They enter the first step as
 *               h_{t-1} and c_{t-1}: a = W x + R h0 + b, and c0 in the forget
 *               gate and the input and forget peepholes.
 *   dh_n, dc_n  (backward inputs) dL/dh_n and dL/dc_n from outside the layer,
 *               for a loss that reads the final states as well as y.
 *   dh0, dc0    (backward outputs) dL/dh0 and dL/dc0.
 * A sequence of length 0 consumes nothing: h_n = h0, c_n = c0, dh0 = dh_n,
 * dc0 = dc_n.  Padded plans (lstm_plan_create_padded) take no state: a call
 * with any non-NULL state pointer on one returns LSTM_ERR_UNSUPPORTED.
 */
typedef struct {
    const float* h0;
    const float* c0;
} lstm_state;

typedef struct {
    const float* dh_n;
    const float* dc_n;
    float* dh0;
    float* dc0;
} lstm_state_grads;

/* Bytes of the scratch lstm_fwd_state / lstm_bwd_state need (the product
 * R h0 over the batch, and the first steps' gate errors): [ndir][B][4H] fp32.
 * Needed when h0 is given (forward) or h0 or dh0 is (backward).  0 on a bad
 * argument. */
size_t lstm_state_scratch_bytes(const lstm_plan* plan, const lstm_layer_shape* shape);

/*
 * lstm_fwd starting from the initial states in `state` (NULL = both zero):
 * same arguments, results and errors as lstm_fwd, plus `state_scratch`
 * (lstm_state_scratch_bytes, caller-owned, 16-byte aligned; NULL allowed when
 * h0 is NULL).  h_n / c_n are the states after each sequence's last frame.
 */
lstm_status lstm_fwd_state(const lstm_plan* plan, const lstm_layer_shape* shape,
                           const lstm_layer_params* params, const lstm_state* state,
                           const void* x_packed, float* y_packed, void* y_lo, float* h_n,
                           float* c_n, void* workspace, void* state_scratch, void* stream);

/*
 * lstm_bwd of a layer run by lstm_fwd_state with the same `state`: the loss
 * is L = sum <y, dy> + <h_n, dh_n> + <c_n, dc_n>.  Same arguments, results
 * and errors as lstm_bwd (the weight gradients include the first steps'
 * terms through h0 and c0), plus `state_grads` (NULL = no final-state errors,
 * no initial-state gradients) and `state_scratch` as for lstm_fwd_state.
 */
lstm_status lstm_bwd_state(const lstm_plan* plan, const lstm_layer_shape* shape,
                           const lstm_layer_params* params, const lstm_state* state,
                           const void* x_packed, const float* y_packed, void* workspace,
                           const float* dy_packed, float* dx_packed, const lstm_layer_grads* grads,
                           const lstm_state_grads* state_grads, void* scratch, void* state_scratch,
                           void* stream);

/*
 * lstm_bwd without device allocation.  (The pages have no counterpart: this
 * serves callers that cannot call cudaMalloc -- a host framework whose
 * memory pool owns the device memory and forbids allocations from outside
 * it, or a real-time loop that must not allocate once it has started.)
 *
 * Same arguments and results as lstm_bwd, minus `scratch`: the scratch comes
 * from one array of LSTM_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library's
 * own device memory, which every GPU that loads the library holds until the
 * process exits.  The caller still passes all inputs and outputs.
 *   - Returns LSTM_ERR_UNSUPPORTED, launching nothing, when
 *     lstm_scratch_bytes(plan, shape) exceeds LSTM_NOALLOC_SCRATCH_BYTES.
 *   - The plan's device must be the current device; otherwise
 *     LSTM_ERR_INVALID_ARG and nothing is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture begins.  Later calls only read the cached
 *     address.  Neither calls cudaMalloc, cudaFree or an allocating library
 *     routine.  The cached address does not survive cudaDeviceReset: after a
 *     reset this entry point must not be called again in the process.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; nothing in it needs to start at zero.  Calls whose
 *     work overlaps on the GPU (other streams, other host threads) race on
 *     it: serialise them.
 */
#define LSTM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
lstm_status lstm_bwd_noalloc(const lstm_plan* plan, const lstm_layer_shape* shape,
                             const lstm_layer_params* params, const void* x_packed,
                             const float* y_packed, void* workspace, const float* dy_packed,
                             float* dx_packed, const lstm_layer_grads* grads, void* stream);

/* Synchronise the stream, then return and clear the plan's device status
 * word (LSTM_OK, LSTM_ERR_TIMEOUT or LSTM_ERR_BOUNDS). */
lstm_status lstm_status_poll(lstm_plan* plan, void* stream);

/* Static description of a status code. */
const char* lstm_status_string(lstm_status status);

/* Number of CTAs per direction of the recurrent kernels (0 = automatic:
 * one CTA while a step's product is small, otherwise one per SM).  Each
 * CTA owns ceil(H / ctas) units; the count is capped at the SMs available. */
lstm_status lstm_plan_set_ctas_per_direction(lstm_plan* plan, int32_t ctas);

/* Engine of the matrix products.  0 (default): tensor cores.  The input
 * projection and the backward's dX, dW and dR run on the tcgen05 GEMM
 * (TMA-fed, fp32 accumulation in tensor memory); fp32 operands are split
 * into three bf16 pieces and the six piece products above 2^-24 of the
 * leading one are accumulated, over K slices of at most 1024 whose partial
 * sums are added on CUDA cores, so the products keep fp32 accuracy.  The
 * recurrent products run on tcgen05 in the cluster kernels (fp32 as the
 * same three pieces) and in the persistent kernels and per-step launches of
 * bf16 layers wider than a cluster, and on warp-level mma.sync in the grid
 * kernels that cover the remaining shapes (fp32 as three tf32 products).  1: CUDA-core FFMA for
 * every product, a comparator: the GEMMs on CUDA cores and the recurrence
 * in the grid kernels.  LSTM_ERR_INVALID_ARG outside 0..1. */
lstm_status lstm_plan_set_gemm_engine(lstm_plan* plan, int32_t engine);

/* Test hook: only the forward input projection of lstm_fwd,
 * out[rows][ndir*4H] = x_packed W^T + b (fp32), with the plan's engine. */
lstm_status lstm_debug_input_projection(const lstm_plan* plan, const lstm_layer_shape* shape,
                                        const lstm_layer_params* params, const void* x_packed, float* out,
                                        void* stream);

/* Kinds of launch the plan's tracer times. */
typedef enum {
    LSTM_KERNEL_PACK = 0,       /* lstm_pack gather */
    LSTM_KERNEL_UNPACK = 1,     /* lstm_unpack scatter */
    LSTM_KERNEL_INPUT_GEMM = 2, /* forward: X W^T + b for both directions */
    LSTM_KERNEL_REC_FWD = 3,    /* forward: persistent recurrent kernel */
    LSTM_KERNEL_REC_BWD = 4,    /* backward: persistent BPTT kernel */
    LSTM_KERNEL_GEMM_DX = 5,    /* backward: dX = dA W */
    LSTM_KERNEL_GEMM_DW = 6,    /* backward: dW = dA^T X (with its split-K sum) */
    LSTM_KERNEL_GEMM_DR = 7,    /* backward: dR = dA^T H_prev (with its split-K sum) */
    LSTM_KERNEL_CONVERT = 8,    /* backward, bf16: transposed bf16 operands of dX, dW, dR */
    LSTM_KERNEL_KINDS = 9
} lstm_kernel_kind;

/* Tracing ("CUDA events around each launch"): with timing enabled every
 * launch sequence of the plan is bracketed by two CUDA events on the
 * caller's stream.  Enabling (or disabling) clears the sums.
 * lstm_plan_read_timing waits for the recorded events and returns, per
 * kind, the summed milliseconds and the number of timed calls (either
 * array may be NULL; each has LSTM_KERNEL_KINDS entries). */
lstm_status lstm_plan_enable_timing(lstm_plan* plan, int32_t enable);
lstm_status lstm_plan_read_timing(lstm_plan* plan, double* ms, int64_t* calls);

/* Per-step-launch path (a comparator, not the fast path).  The design the
 * RETURNN paper describes for its GPU LSTM (Sec. 4.2): after the one
 * non-recurrent product, every time step is one product launch per direction
 * (R h_{t-1} over the step's active rows: tcgen05 for bf16 layers, CUDA cores
 * for fp32) and one cell launch for both directions; the backward pass
 * mirrors it (one cell launch and one R^T da product per direction per
 * step), then the same db/dpeep sums and
 * dX/dW/dR products as lstm_bwd.  Same arguments, layouts, results (within
 * the fp32 / bf16 tolerances) and errors as lstm_fwd / lstm_bwd, plus
 * `scratch` (device, 16-byte aligned, lstm_stepwise_scratch_bytes, owned by
 * the caller; the forward pass also needs it).  Padded plans run with the
 * same masking as lstm_fwd / lstm_bwd.  2·T·ndir + T launches per layer and
 * pass. */
size_t lstm_stepwise_scratch_bytes(const lstm_plan* plan, const lstm_layer_shape* shape);
lstm_status lstm_fwd_stepwise(const lstm_plan* plan, const lstm_layer_shape* shape,
                              const lstm_layer_params* params, const void* x_packed, float* y_packed,
                              void* y_lo, float* h_n, float* c_n, void* workspace, void* scratch, void* stream);
lstm_status lstm_bwd_stepwise(const lstm_plan* plan, const lstm_layer_shape* shape,
                              const lstm_layer_params* params, const void* x_packed, const float* y_packed,
                              void* workspace, const float* dy_packed, float* dx_packed,
                              const lstm_layer_grads* grads, void* scratch, void* stream);

/* Kernels launched through this plan since it was created (traced or not);
 * -1 for a NULL plan. */
int64_t lstm_plan_launch_count(const lstm_plan* plan);

/* Launch configuration of the last recurrent kernel run through this plan:
 * `pass` 0 = forward (lstm_fwd), 1 = backward (lstm_bwd / lstm_bwd_noalloc).
 * kind: 0 none yet, 1 grid-wide persistent kernel with flag barriers,
 *       2 one thread-block cluster per direction and sequence group, 3 per-step
 *       launches of a tcgen05 product over the whole GPU and a cell kernel,
 *       4 the persistent kernel of bf16 layers whose R does not fit one cluster
 *       (H > 512): R or R^T resident in the shared memory of H/16 CTAs per
 *       direction, tcgen05 products, a grid barrier per step;
 * ctas_per_direction: CTAs that hold one direction's recurrent weights;
 * product: 0 CUDA cores, 1 warp-level mma.sync, 2 tcgen05 with TMEM accumulators;
 * variant (cluster kernels): bit 0 = operands exchanged by bulk copies into
 * double buffers (else DSMEM stores between cluster-barrier halves), bit 1 =
 * the cell's operands arrive as TMA tiles.
 * Any output pointer may be NULL.  LSTM_ERR_INVALID_ARG for a NULL plan or a
 * pass other than 0 or 1.  Host only; no device work. */
lstm_status lstm_plan_recurrent_config(const lstm_plan* plan, int32_t pass, int32_t* kind,
                                       int32_t* ctas_per_direction, int32_t* product, int32_t* variant);

/* Sequence groups of the last cluster recurrent kernel run through this plan
 * (`pass` as above): the sorted slots are cut into `groups` contiguous groups
 * of `slots_per_group` slots (the last may be shorter), and each (direction,
 * group) pair runs as its own thread-block cluster.  Sequences never interact
 * in the recurrence, so the groups exchange nothing; each group runs only as
 * many steps as its longest sequence.  Other recurrent kernels report one
 * group of B slots; 0 before any recurrent launch.  Host only.
 * LSTM_ERR_INVALID_ARG for a NULL plan or a pass other than 0 or 1. */
lstm_status lstm_plan_recurrent_groups(const lstm_plan* plan, int32_t pass, int32_t* groups,
                                       int32_t* slots_per_group);

/* Test hook for bf16 layers wider than one cluster (H > 512): -1 = automatic
 * (the persistent kernels with R, resp. R^T, resident across H/16 CTAs per
 * direction where they apply -- H a multiple of 64 up to 1024, at most 256
 * sequences -- the backward only in its form with clusters of four CTAs that
 * split the gate errors between them; else per-step launches), 0 = per-step
 * launches both ways, 1 = the persistent kernels both ways where they apply
 * (either form), 2 = the persistent kernels without thread-block clusters
 * (forward: every CTA reads each operand tile from L2 itself instead of
 * sharing it by multicast; backward: every CTA streams all 4H gate errors).
 * lstm_plan_recurrent_config reports the persistent kernels' cluster size in
 * `variant`.  LSTM_ERR_INVALID_ARG outside -1..2. */
lstm_status lstm_debug_wide_recurrence(lstm_plan* plan, int32_t mode);

/* Tuning hook of the persistent kernels of layers wider than a cluster: caps
 * the depth of the operand ring each CTA streams the step's operand tiles
 * through (`max_stages` >= 2; 0 = no cap, as many 16 KB stages as the shared
 * memory beside the resident weights holds, at most 8; -1 = leave the cap as
 * it is), and reports the depths the last forward and backward persistent
 * launches used (0 when none ran).  Results do not depend on the depth.
 * Either output pointer may be NULL.  LSTM_ERR_INVALID_ARG for a NULL plan or
 * max_stages outside -1, 0, 2..64. */
lstm_status lstm_debug_wide_stages(lstm_plan* plan, int32_t max_stages, int32_t* used_fwd, int32_t* used_bwd);

/* Test hook: slots per sequence group of the cluster recurrent kernels (0 =
 * automatic: the smallest multiple of 8 that gives every cluster an SM of its
 * own; 1..128 forces that many).  Results do not depend on it.
 * LSTM_ERR_INVALID_ARG outside 0..128. */
lstm_status lstm_debug_sequence_groups(lstm_plan* plan, int32_t slots);

/* Per-step phase stamps of the recurrent kernels (diagnostics).  With a
 * device buffer of 2 * ndir * steps * 8 int64 set, CTA 0 of each direction
 * writes clock64() stamps for its first `steps` steps at
 * [kernel (0 fwd, 1 bwd)][direction][step][k]: k = 0 step start, 1 after the
 * barrier, 2 after the exchanged operands are staged, 3 after the cell
 * update (and, backward, the partial product), 4 after publishing.  The
 * buffer is the caller's; steps = 0 turns the stamps off. */
lstm_status lstm_debug_trace_steps(lstm_plan* plan, int64_t* device_buffer, int32_t steps);

/* Test hook (-1 = off).  Grid recurrent kernels, and the persistent kernels of
 * layers wider than a cluster: CTA `cta` (of direction 0) never announces its
 * (first) step, so the others' barrier waits run out.  Cluster recurrent
 * kernels: CTA `cta` of the first direction's cluster withholds the
 * completion signal of its first tensor-core product, so its own bounded wait
 * runs out (and, with the bulk exchange, its peers' waits for its operand).
 * Either way the launch returns and LSTM_ERR_TIMEOUT is reported: the failure
 * path runs without a GPU fault. */
lstm_status lstm_debug_skip_arrival(lstm_plan* plan, int32_t cta);

/* Test hook: restricts the cluster recurrent kernels to one variant (-1 =
 * automatic choice; else bit 0 = bulk-copy exchange, bit 1 = TMA operand
 * tiles, as lstm_plan_recurrent_config reports them).  When the forced
 * variant does not fit (shared memory, co-residency), the plan falls back to
 * the grid kernel exactly as when no cluster variant fits.  Lets parity tests
 * reach every variant at small sizes.  LSTM_ERR_INVALID_ARG outside -1..3. */
lstm_status lstm_debug_cluster_variant(lstm_plan* plan, int32_t variant);

/* ======================================================================
 * 2-D example-packing for MDLSTM layers ("No Padding Please: Efficient
 * Neural Handwriting Recognition", Sec. III-V, App. A-B).  fp32 throughout.
 *
 * Examples are images of h x w pixels with D features each, given in caller
 * order: pixels of example 0 row by row, then example 1, ... (N pixels).  The
 * plan places them on a canvas with the page's packing algorithm (App. B,
 * Algorithm 1): bucket by height (descending), fill rows greedily with the
 * widest example that still fits beside the row's examples and one separator
 * pixel (ties: lower index; an empty row takes the widest example left even
 * if it is wider than the row; a bucket's last row closes when the bucket runs
 * out), stack the rows with one separator row between them.  The row width
 * is the caller's, or the widest example when 0.
 *
 * A layer scans the image from num_directions corners (direction d flips x
 * when d & 1 and y when d & 2; Sec. III's 4-directional layer stacks all
 * four).  Cell of a direction at scan position (ys, xs): predecessor 1 is
 * (ys - 1, xs), predecessor 2 is (ys, xs - 1), absent outside the example
 * (the mask of Sec. V: zero state input).  With gates a_g = W_g x + U1_g h1
 * + U2_g h2 + b_g, g in (i, f1, f2, z, o):
 *   i = sig(a_i + p_i1 S1 + p_i2 S2), f1 = sig(a_f1 + p_f1 S1),
 *   f2 = sig(a_f2 + p_f2 S2), z = tanh(a_z), o = sig(a_o + p_o1 S1 + p_o2 S2),
 *   c = f1 S1 + f2 S2 + i z, h = o tanh(c)
 * (App. A: five products per hidden state, three per memory state; Sec. III:
 * the output gate reads the previous states).  Output y[N][ndir*H], the
 * direction d in columns [dH, dH + H).
 *
 * Schedule (Sec. IV-A, input skewing): the cells of one skewed column depend
 * only on the previous column and run as one parallel step.  schedule 0 =
 * the canvas's skewed columns (height + width - 1 steps); 1 = every example
 * from step 0 along its own anti-diagonals (longest h + w - 1 steps).  The
 * results do not depend on the schedule; separator and padding cells are
 * never computed under either.
 * ====================================================================== */

typedef struct lstm_md_plan lstm_md_plan;

typedef struct {
    int32_t input_size;      /* D */
    int32_t hidden_size;     /* H, 1..128 */
    int32_t num_directions;  /* must equal the plan's */
} lstm_md_shape;

/* Device pointers, fp32, 16-byte aligned: W[ndir][5H][D], U1[ndir][5H][H]
 * (predecessor 1), U2[ndir][5H][H], b[ndir][5H], peep[ndir][6][H] in the order
 * p_i1, p_i2, p_f1, p_f2, p_o1, p_o2; gate blocks of 5H in the order i, f1,
 * f2, z, o. */
typedef struct {
    const float* W;
    const float* U1;
    const float* U2;
    const float* b;
    const float* peep;
} lstm_md_params;

/* Gradients in the same layouts (overwritten; any pointer may be NULL). */
typedef struct {
    float* W;
    float* U1;
    float* U2;
    float* b;
    float* peep;
} lstm_md_grads;

/* Pack n examples (heights[i] x widths[i], either may be 0) and build the
 * schedule's tables on the current device.  row_width >= 0 (0 = widest),
 * num_directions 1..4, schedule 0 or 1.  Host and device memory are owned by
 * the plan.  LSTM_ERR_INVALID_ARG for bad arguments, LSTM_ERR_UNSUPPORTED when
 * ndir x N reaches 2^31 cells, LSTM_ERR_CUDA when the device tables cannot be
 * made. */
lstm_status lstm_md_plan_create(const int32_t* heights, const int32_t* widths, int32_t n, int32_t row_width,
                                int32_t num_directions, int32_t schedule, lstm_md_plan** out);
void lstm_md_plan_destroy(lstm_md_plan* plan);

/* The same packing and schedule on the host only (no device work), for
 * checking: info = {steps, canvas height, canvas width, packed rows}; y0, x0
 * [n] = each example's top-left canvas pixel (-1 without pixels); step_off
 * [ndir][steps + 1] = first cell of each step (cells are numbered direction by
 * direction, step by step, examples in packing order, then by scan row); per
 * cell [ndir * N]: src = its pixel (caller order), pred1 / pred2 = its
 * predecessor cells, succ1 / succ2 = the cells it is predecessor 1 / 2 of (-1
 * none).  Any output pointer may be NULL. */
lstm_status lstm_md_plan_compute_host(const int32_t* heights, const int32_t* widths, int32_t n, int32_t row_width,
                                      int32_t num_directions, int32_t schedule, int32_t* info, int32_t* y0,
                                      int32_t* x0, int64_t* step_off, int32_t* src, int32_t* pred1, int32_t* pred2,
                                      int32_t* succ1, int32_t* succ2);

lstm_status lstm_md_plan_info(const lstm_md_plan* plan, int64_t* pixels, int32_t* steps, int32_t* canvas_height,
                              int32_t* canvas_width, int32_t* rows);
lstm_status lstm_md_plan_placement(const lstm_md_plan* plan, int32_t* y0, int32_t* x0);
/* step_off[ndir][steps + 1], as lstm_md_plan_compute_host. */
lstm_status lstm_md_plan_step_cells(const lstm_md_plan* plan, int64_t* step_off);
/* Bound on each grid-barrier wait of the layer kernels (default 2 s). */
lstm_status lstm_md_plan_set_wait_limit(lstm_md_plan* plan, uint64_t ns);
/* Synchronise the stream, then return and clear the plan's device status word
 * (LSTM_OK or LSTM_ERR_TIMEOUT). */
lstm_status lstm_md_status_poll(lstm_md_plan* plan, void* stream);
/* Test hook (-1 = off): CTA `cta` of the layer kernels never arrives at the
 * first grid barrier, so every CTA's bounded wait runs out; the launch
 * returns and LSTM_ERR_TIMEOUT is reported without a GPU fault. */
lstm_status lstm_md_debug_skip_arrival(lstm_md_plan* plan, int32_t cta);
/* Kernels launched through this plan; -1 for a NULL plan. */
int64_t lstm_md_plan_launch_count(const lstm_md_plan* plan);
/* Optional CUDA-event timing of the layer's phases (diagnostics; enabling
 * clears the totals): read_timing fills ms[4] and calls[4] in the order input
 * projection (GEMM and weight transpose), forward walk, backward walk,
 * gradient products and sums.  Either output may be NULL; reading waits for
 * the recorded events. */
lstm_status lstm_md_plan_enable_timing(lstm_md_plan* plan, int32_t enable);
lstm_status lstm_md_plan_read_timing(lstm_md_plan* plan, double* ms, int64_t* calls);

/* Device bytes the caller provides: the workspace (kept from lstm_md_fwd to
 * lstm_md_bwd) and the backward scratch.  0 for an invalid shape. */
size_t lstm_md_workspace_bytes(const lstm_md_plan* plan, const lstm_md_shape* shape);
size_t lstm_md_scratch_bytes(const lstm_md_plan* plan, const lstm_md_shape* shape);

/* Forward of one layer: x[N][D] (caller order) -> y[N][ndir*H]; stream-ordered
 * on `stream`.  The workspace keeps the cells' h, c and gates for the
 * backward pass.  A barrier wait that runs out is reported by
 * lstm_md_status_poll. */
lstm_status lstm_md_fwd(const lstm_md_plan* plan, const lstm_md_shape* shape, const lstm_md_params* params,
                        const float* x, float* y, void* workspace, void* stream);

/* Backward of the last lstm_md_fwd on this workspace (it is consumed: a
 * second backward needs a new forward): dy[N][ndir*H] = dL/dy; writes dx[N][D]
 * (NULL: skipped) and the parameter gradients (bitwise repeatable: every sum
 * runs in a fixed order). */
lstm_status lstm_md_bwd(const lstm_md_plan* plan, const lstm_md_shape* shape, const lstm_md_params* params,
                        const float* x, void* workspace, const float* dy, float* dx, const lstm_md_grads* grads,
                        void* scratch, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LSTM_PACKED_H */
