// api.cu -- lstm_fwd / lstm_bwd: argument checks and the order of launches.
//
// Forward of one layer ("Single Stream Parallelization...", Sec. 3; RETURNN,
// Sec. 4.2):  (1) one product for the non-recurrent part of every frame and
// both directions at once, A_in = X [W_fwd; W_rev]^T + b ("No Padding
// Please", Sec. IV-B: all gate projections of one input in one grouped
// operation); (2) the persistent recurrent kernel over the steps.
// Backward:  (1) the persistent BPTT kernel (gate errors, db, dpeep);
// (2) one product each for dX, dW and dR over all frames.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "gemm.cuh"
#include "recurrent.cuh"
#include "state.cuh"
#include "stepwise.cuh"

namespace lstm {

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Initial states and final-state errors of one call (all [ndir][B][H] caller order; null =
// zero / not wanted) and the scratch their products use.
struct StateIO {
    const float* h0 = nullptr;
    const float* c0 = nullptr;
    const float* dh_n = nullptr;
    const float* dc_n = nullptr;
    float* dh0 = nullptr;
    float* dc0 = nullptr;
    float* scratch = nullptr;
    bool any() const { return h0 || c0 || dh_n || dc_n || dh0 || dc0; }
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

lstm_status check_shape(const lstm_layer_shape* s)
{
    if (!s) return LSTM_ERR_INVALID_ARG;
    if (s->input_size < 1 || s->hidden_size < 8 || s->hidden_size % 8 != 0) return LSTM_ERR_INVALID_ARG;
    if (s->num_directions != 1 && s->num_directions != 2) return LSTM_ERR_INVALID_ARG;
    if (s->dtype != LSTM_F32 && s->dtype != LSTM_BF16) return LSTM_ERR_INVALID_ARG;
    if (s->hidden_size > 2048 || s->input_size > 65536) return LSTM_ERR_UNSUPPORTED;
    return LSTM_OK;
}

// fp32 layers whose products can run on tcgen05 as six bf16 products of three-piece splits
// concatenated along K: the K extents (D, ndir*4H, frames) must be TMA-addressable.
bool f32_split_shape(const lstm_layer_shape& s) { return s.dtype == LSTM_F32 && s.input_size % 8 == 0; }

// bf16 layers wider than one thread-block cluster can hold (one direction's R of more than 16
// CTAs x 32 units): the recurrence runs as per-step tcgen05 products over the whole GPU.
bool wide_bf16(const lstm_layer_shape& s) { return s.dtype == LSTM_BF16 && s.hidden_size > 512; }

// K splits of a bf16 layer's per-step tensor-core products (a function of the shape only, so
// that the buffers holding their slices have a fixed layout): forward R h, N = 4H, K = H;
// backward R^T da, N = H, K = 4H; both directions in one launch.
int step_splits(const Plan& p, const lstm_layer_shape& s, bool bwd)
{
    if (s.dtype != LSTM_BF16) return 1;
    const int H = s.hidden_size;
    return gemm_tc_pair_splits(p.B, bwd ? H : 4 * H, bwd ? 4 * H : H, s.num_directions, p.num_sms);
}

struct Layout {
    size_t ga_off, c_off, xs_off, ws_off, rh_off, hb_off, total;   // workspace
};

// gates/errors, cell states, then (fp32 split shapes) the input projection's split operands:
// X as [rows][6D] and W as [ndir*4H][6D] bf16 (six K segments, kSplitSegments)
Layout workspace_layout(const Plan& p, const lstm_layer_shape& s)
{
    Layout l;
    const size_t rows = (size_t)p.rows, H = (size_t)s.hidden_size, nd = (size_t)s.num_directions;
    const size_t D = (size_t)s.input_size;
    l.ga_off = 0;
    l.c_off = align256(rows * nd * 4 * H * sizeof(float));
    l.xs_off = l.c_off + align256(rows * nd * H * sizeof(float));
    const size_t ns = kSplitSegments;
    l.ws_off = l.xs_off + (f32_split_shape(s) ? align256(rows * ns * D * 2) : 0);
    l.rh_off = l.ws_off + (f32_split_shape(s) ? align256(nd * 4 * H * ns * D * 2) : 0);
    // wide bf16 layers: a step's R h_{t-1} [ndir][B][4H] fp32 and bf16 h [ndir][2][B][H] (the per-step
    // products use parity 0; the persistent kernel exchanges h through both)
    const size_t B = (size_t)p.B;
    l.hb_off = l.rh_off + (wide_bf16(s) ? align256(nd * (size_t)step_splits(p, s, false) * B * 4 * H * 4) : 0);
    l.total = l.hb_off + (wide_bf16(s) ? align256(2 * nd * B * H * 2) : 0);
    return l;
}

// The three gradient products of lstm_bwd (shapes only).
void bwd_gemm_shapes(const Plan& p, const lstm_layer_shape& s, GemmDesc* dW, GemmDesc* dR, GemmDesc* dX)
{
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size;
    dW->M = nd * 4 * H; dW->N = D; dW->K = (int)p.rows; dW->k_splits = 32;
    dR->M = 4 * H; dR->N = H; dR->K = (int)p.rows; dR->k_splits = 32;
    dX->M = (int)p.rows; dX->N = D; dX->K = nd * 4 * H; dX->k_splits = 8;
}

constexpr int kMaxTcSplits = 16;
// fp32 layers: the longest K range one tensor-memory accumulator sums (64 MMAs of K = 16).
// The accumulator's additions lose about 2^-23 of the running sum each (measured on the
// frame-reduced products dW and dR: the element-wise error grows linearly with the MMAs
// per accumulator), so long K ranges are cut into splits whose partial sums are added in
// fp32 on the CUDA cores, in split order.
constexpr int kF32SplitK = 1024;

// K splits of a tensor-core product of the backward pass.
int bwd_tc_splits(const Plan& p, int M, int N, int K, bool f32)
{
    const int sp = gemm_tc_splits(M, N, K, p.num_sms, kMaxTcSplits);
    return f32 ? std::max(sp, (K + kF32SplitK - 1) / kF32SplitK) : sp;
}

// Scratch of lstm_bwd.  Region U holds the recurrent kernel's partial-product
// exchange, later the split-K partial sums (never live at the same time).  The
// bf16 path adds its tensor-core operands: dA (row-major and transposed), X^T,
// H_prev^T and W^T, all bf16, the frame dimension padded to a multiple of 8.
struct BwdScratch {
    size_t u_bytes = 0, dA16 = 0, dAT16 = 0, XT16 = 0, HpT16 = 0, WT16 = 0, total = 0;
    int64_t ldr = 0;   // padded frame count (row pitch of the transposes)
};

BwdScratch bwd_scratch(const Plan& p, const lstm_layer_shape& s)
{
    BwdScratch b;
    GemmDesc dW, dR, dX;
    bwd_gemm_shapes(p, s, &dW, &dR, &dX);
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size;
    size_t gemm = std::max(std::max(gemm_partial_floats(dW, p.num_sms), gemm_partial_floats(dR, p.num_sms)),
                           gemm_partial_floats(dX, p.num_sms));
    const size_t part = std::max(rec_bwd_part_floats(p, H, nd, s.dtype == LSTM_BF16, p.forced_ctas),
                                 rec_cluster_bwd_sum_floats(H, nd));
    const bool tc_shape = s.dtype == LSTM_BF16 || f32_split_shape(s);
    const int ns = s.dtype == LSTM_BF16 ? 1 : kSplitSegments;   // K segments of the tensor-core operands
    const int64_t ldr = (int64_t)(((size_t)p.rows + 7) / 8 * 8);
    if (tc_shape) {
        const bool f32 = ns > 1;
        const int kr = ns == 1 ? (int)p.rows : (int)(ns * ldr);
        size_t tc = std::max((size_t)bwd_tc_splits(p, nd * 4 * H, D, kr, f32) * nd * 4 * H * D,
                             (size_t)bwd_tc_splits(p, 4 * H, H, kr, f32) * 4 * H * H);
        const int sx = f32 ? bwd_tc_splits(p, (int)p.rows, D, ns * nd * 4 * H, true) : 1;
        if (sx > 1) tc = std::max(tc, (size_t)sx * (size_t)p.rows * D);
        gemm = std::max(gemm, tc);
    }
    b.u_bytes = align256(std::max<size_t>(1, std::max(gemm, part)) * sizeof(float));
    size_t off = b.u_bytes;
    if (tc_shape) {
        const size_t rows = (size_t)p.rows, G4 = (size_t)nd * 4 * H;
        b.ldr = ldr;
        b.dA16 = off; off += align256(rows * ns * G4 * 2);
        b.dAT16 = off; off += align256(G4 * ns * (size_t)b.ldr * 2);
        b.XT16 = off; off += align256((size_t)D * ns * b.ldr * 2);
        b.HpT16 = off; off += align256((size_t)nd * H * ns * b.ldr * 2);
        b.WT16 = off; off += align256((size_t)D * ns * G4 * 2);
    }
    b.total = off;
    return b;
}

struct StepScratch;
size_t step_scratch_total(const Plan& p, const lstm_layer_shape& s);

size_t scratch_floats(const Plan& p, const lstm_layer_shape& s)
{
    return (wide_bf16(s) ? step_scratch_total(p, s) : bwd_scratch(p, s).total) / sizeof(float);
}

RecArgs base_args(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm, float* ga,
                  float* cbuf)
{
    RecArgs a;
    memset(&a, 0, sizeof(a));
    a.T = p.T; a.B = p.B; a.H = s.hidden_size; a.ndir = s.num_directions;
    a.bf16 = s.dtype == LSTM_BF16; a.padded = p.padded ? 1 : 0;
    a.debug_skip_cta = p.debug_skip_cta;
    a.wait_limit_ns = p.wait_limit_ns;
    a.bs = p.d_bs; a.off = p.d_off; a.slot_len = p.d_len; a.perm = p.d_perm;
    a.ga = ga; a.R = prm.R; a.peep = prm.peep; a.cbuf = cbuf;
    a.flags = p.d_flags; a.status = p.d_status;
    return a;
}

bool encode_ready();

// A_in[rows][ndir*4H] = X W^T + b for both directions at once; tcgen05 for bf16 operands, and
// for fp32 operands as six bf16 products of three-piece splits (X in split pattern 1, W in
// pattern 2, six K segments each, in the workspace's split region `split_ws`, when given).
lstm_status input_projection(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm,
                             const void* x_packed, float* out, void* split_ws, cudaStream_t cs)
{
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size;
    const bool bf16 = s.dtype == LSTM_BF16;
    if (bf16 && p.gemm_engine == 0 && gemm_tc_supported((int)p.rows, nd * 4 * H, D, x_packed, prm.W))
        return gemm_tc_bf16_nt(p, K_GEMM_IN, x_packed, prm.W, out, (int64_t)nd * 4 * H, prm.b, (int)p.rows,
                               nd * 4 * H, D, cs);
    if (!bf16 && split_ws && p.gemm_engine == 0 && f32_split_shape(s) && encode_ready()) {
        const int rows = (int)p.rows, G4 = nd * 4 * H;
        char* xs = (char*)split_ws;
        const int ns = kSplitSegments;
        char* ws = xs + align256((size_t)rows * ns * D * 2);
        lstm_status st;
        if ((st = transpose_to_bf16_split(p, x_packed, false, D, 0, nullptr, rows, rows, D, 1, nullptr, 0, 0, xs,
                                          (int64_t)ns * D, D, cs)) != LSTM_OK)
            return st;
        if ((st = transpose_to_bf16_split(p, prm.W, false, D, 0, nullptr, G4, G4, D, 2, nullptr, 0, 0, ws,
                                          (int64_t)ns * D, D, cs)) != LSTM_OK)
            return st;
        return gemm_tc_bf16_nt(p, K_GEMM_IN, xs, ws, out, G4, prm.b, rows, G4, ns * D, cs);
    }
    GemmDesc g;
    g.M = (int)p.rows; g.N = nd * 4 * H; g.K = D;
    g.A = x_packed; g.sam = D; g.sak = 1; g.a_bf16 = bf16;
    g.B = prm.W; g.sbk = 1; g.sbn = D; g.b_bf16 = bf16;
    g.C = out; g.ldc = nd * 4 * H; g.bias = prm.b;
    return gemm_simt(g, p, K_GEMM_IN, cs);
}

bool encode_ready() { return gemm_tc_supported(1, 1, 8, nullptr, nullptr); }

// dX, dW and dR on tcgen05, from the gate errors dA (fp32, in the workspace) and bf16
// operands built in the scratch: transposes (frames innermost, padded to a multiple of 8
// with zeros) and a row-major copy of dA.  bf16 layers use one bf16 copy of each operand;
// fp32 layers six K segments per operand (dA in split pattern 1; X, H_prev and W in pattern
// 2), so that each product is the sum of the six piece products in one launch.
lstm_status bwd_products_tc(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm,
                            const void* x_packed, const float* y_packed, const float* ga, float* dx_packed,
                            const lstm_layer_grads& g, void* scratch, cudaStream_t cs)
{
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size, rows = (int)p.rows;
    const int G4 = nd * 4 * H;
    const bool bf16 = s.dtype == LSTM_BF16;
    const int ns = bf16 ? 1 : kSplitSegments;
    const int pa = bf16 ? 0 : 1, pb = bf16 ? 0 : 2;      // split patterns of the two operand sides
    const BwdScratch b = bwd_scratch(p, s);
    const int64_t ldr = b.ldr, kt = (int64_t)ns * ldr;    // transposed operands: row pitch = K extent
    const int kr = bf16 ? rows : (int)kt;                 // K of the frame-reduced products
    char* base = (char*)scratch;
    float* partial = (float*)base;
    void* dA16 = base + b.dA16;
    char* dAT16 = base + b.dAT16;
    void* XT16 = base + b.XT16;
    char* HpT16 = base + b.HpT16;
    void* WT16 = base + b.WT16;
    lstm_status st;
    // operands: dA as bf16 columns and rows, X^T, H_prev^T per direction, W^T
    if ((st = transpose_to_bf16_split(p, ga, false, G4, 0, nullptr, rows, (int)ldr, G4, pa, dAT16, kt, ldr, dA16,
                                      (int64_t)ns * G4, G4, cs)) != LSTM_OK)
        return st;
    if ((st = transpose_to_bf16_split(p, x_packed, bf16, D, 0, nullptr, rows, (int)ldr, D, pb, XT16, kt, ldr,
                                      nullptr, 0, 0, cs)) != LSTM_OK)
        return st;
    for (int d = 0; d < nd; ++d)
        if ((st = transpose_to_bf16_split(p, y_packed, false, (int64_t)nd * H, d * H, d == 0 ? p.d_prev_fwd : p.d_prev_rev,
                                          rows, (int)ldr, H, pb, HpT16 + (size_t)d * H * kt * 2, kt, ldr, nullptr, 0, 0,
                                          cs)) != LSTM_OK)
            return st;
    if ((st = transpose_to_bf16_split(p, prm.W, bf16, D, 0, nullptr, G4, G4, D, pb, WT16, (int64_t)ns * G4, G4,
                                      nullptr, 0, 0, cs)) != LSTM_OK)
        return st;
    // dX[rows][D] = dA[rows][G4] W[G4][D]
    const int sx = bf16 ? 1 : bwd_tc_splits(p, rows, D, ns * G4, true);
    if (dx_packed && (st = gemm_tc_bf16(p, K_GEMM_DX, dA16, (int64_t)ns * G4, WT16, (int64_t)ns * G4, rows, D, ns * G4,
                                        dx_packed, D, nullptr, sx, partial, cs)) != LSTM_OK)
        return st;
    // dW[G4][D] = dA^T X, K = frames
    int sp = bwd_tc_splits(p, G4, D, kr, !bf16);
    if ((st = gemm_tc_bf16(p, K_GEMM_DW, dAT16, kt, XT16, kt, G4, D, kr, g.dW, D, nullptr, sp, partial, cs)) != LSTM_OK)
        return st;
    // dR_d[4H][H] = dA_d^T H_prev_d, K = frames
    sp = bwd_tc_splits(p, 4 * H, H, kr, !bf16);
    for (int d = 0; d < nd; ++d)
        if ((st = gemm_tc_bf16(p, K_GEMM_DR, dAT16 + (size_t)d * 4 * H * kt * 2, kt, HpT16 + (size_t)d * H * kt * 2, kt,
                               4 * H, H, kr, g.dR + (size_t)d * 4 * H * H, H, nullptr, sp, partial, cs)) != LSTM_OK)
            return st;
    return LSTM_OK;
}

// dX, dW and dR of a layer from its gate errors (ga) after the recurrence.
lstm_status bwd_products(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm,
                         const void* x_packed, const float* y_packed, const float* ga, float* dx_packed,
                         const lstm_layer_grads& grads, void* scratch, cudaStream_t cs)
{
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size;
    const bool bf16 = s.dtype == LSTM_BF16;
    lstm_status st;
    const int nd4H = nd * 4 * H;
    if ((bf16 || f32_split_shape(s)) && p.gemm_engine == 0 && D % 8 == 0 && encode_ready())
        return bwd_products_tc(p, s, prm, x_packed, y_packed, ga, dx_packed, grads, scratch, cs);
    GemmDesc gw, gr, gx;
    bwd_gemm_shapes(p, s, &gw, &gr, &gx);
    if (dx_packed) {
        GemmDesc g = gx;
        g.partial = (float*)scratch;
        g.A = ga; g.sam = nd4H; g.sak = 1;
        g.B = prm.W; g.sbk = D; g.sbn = 1; g.b_bf16 = bf16;
        g.C = dx_packed; g.ldc = D; g.round_bf16 = bf16;
        if ((st = gemm_simt(g, p, K_GEMM_DX, cs)) != LSTM_OK) return st;
    }
    gw.A = ga; gw.sam = 1; gw.sak = nd4H;
    gw.B = x_packed; gw.sbk = D; gw.sbn = 1; gw.b_bf16 = bf16;
    gw.C = grads.dW; gw.ldc = D; gw.round_bf16 = bf16; gw.partial = (float*)scratch;
    if ((st = gemm_simt(gw, p, K_GEMM_DW, cs)) != LSTM_OK) return st;
    for (int d = 0; d < nd; ++d) {
        GemmDesc g = gr;
        g.A = ga + (size_t)d * 4 * H; g.sam = 1; g.sak = nd4H;
        g.B = y_packed + (size_t)d * H; g.sbk = nd * H; g.sbn = 1;
        g.b_rows = d == 0 ? p.d_prev_fwd : p.d_prev_rev;
        g.C = grads.dR + (size_t)d * 4 * H * H; g.ldc = H; g.round_bf16 = bf16;
        g.partial = (float*)scratch;
        if ((st = gemm_simt(g, p, K_GEMM_DR, cs)) != LSTM_OK) return st;
    }
    return LSTM_OK;
}

// Scratch of the per-step path: the gradient products' scratch (whose first
// region also holds the db / dpeep partials), then R h_{t-1} of a step
// [ndir][B][4H], R^T da of a step [ndir][B][H] and the cell-state error carry
// [ndir][B][H].
// bf16 layers, the per-step products on tcgen05: bf16 h of a step's rows [ndir][B][H], bf16
// gate errors [ndir][B][4H] and R^T [ndir][H][4H] bf16.
struct StepScratch {
    size_t rh = 0, dh = 0, dcc = 0, hb = 0, dab = 0, rt = 0, total = 0;
};

StepScratch step_scratch(const Plan& p, const lstm_layer_shape& s)
{
    StepScratch q;
    const size_t B = (size_t)p.B, H = (size_t)s.hidden_size, nd = (size_t)s.num_directions;
    size_t off = align256(bwd_scratch(p, s).total);
    q.rh = off; off += align256(nd * (size_t)step_splits(p, s, false) * B * 4 * H * sizeof(float));
    q.dh = off; off += align256(nd * (size_t)step_splits(p, s, true) * B * H * sizeof(float));
    q.dcc = off; off += align256(nd * B * H * sizeof(float));
    if (s.dtype == LSTM_BF16) {
        q.hb = off; off += align256(nd * B * H * 2);
        q.dab = off; off += align256(2 * nd * B * 4 * H * 2);      // [ndir][2][B][4H]: both parities (persistent kernel)
        q.rt = off; off += align256(nd * H * 4 * H * 2);
    }
    q.total = off;
    return q;
}

size_t step_scratch_total(const Plan& p, const lstm_layer_shape& s) { return step_scratch(p, s).total; }

bool step_tc(const Plan& p, const lstm_layer_shape& s);

// Whether lstm_fwd / lstm_bwd run this layer's recurrence as per-step tcgen05 products.
bool wide_step_path(const Plan& p, const lstm_layer_shape& s)
{
    return wide_bf16(s) && p.forced_ctas == 0 && step_tc(p, s);
}

StepArgs step_args(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm, float* ga,
                   float* cbuf)
{
    StepArgs a;
    memset(&a, 0, sizeof(a));
    a.T = p.T; a.B = p.B; a.H = s.hidden_size; a.ndir = s.num_directions;
    a.bs = p.d_bs; a.off = p.d_off; a.slot_len = p.d_len; a.perm = p.d_perm;
    a.ga = ga; a.cbuf = cbuf; a.peep = prm.peep;
    a.padded = p.padded ? 1 : 0;
    return a;
}

// Per-step tensor-core products for this layer (bf16 operands, tcgen05 available).
bool step_tc(const Plan& p, const lstm_layer_shape& s)
{
    return s.dtype == LSTM_BF16 && p.gemm_engine == 0 && encode_ready();
}

// The forward recurrence as per-step launches: per direction one product R h_{t-1} over the
// step's rows with a previous state (tcgen05 from the bf16 copy hb16 when given, else CUDA
// cores from y), then one cell launch for both directions.
lstm_status stepwise_fwd_core(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm, float* y,
                              void* y_lo, float* h_n, float* c_n, float* ga, float* cbuf, float* rh,
                              __nv_bfloat16* hb16, cudaStream_t cs, const StateIO& sio = StateIO())
{
    const int H = s.hidden_size, nd = s.num_directions, ndH = nd * H;
    const bool bf16 = s.dtype == LSTM_BF16;
    const size_t esz = bf16 ? 2 : 4;
    StepArgs a = step_args(p, s, prm, ga, cbuf);
    a.h0 = sio.h0; a.c0 = sio.c0;
    a.rh = rh; a.hb16 = hb16;
    a.y = y; a.y_lo = (__nv_bfloat16*)y_lo; a.h_n = h_n; a.c_n = c_n;
    lstm_status st = LSTM_OK;
    // tcgen05: both directions' products of a step in one launch, tensor maps encoded once, K
    // split into S slices of rh that the cell adds; the CUDA-core products write one slice
    TcOperands op[2];
    bool pair = hb16 != nullptr;
    int S = pair ? step_splits(p, s, false) : 1;
    for (int d = 0; d < nd && pair; ++d)
        pair = gemm_tc_prepare(&op[d], hb16 + (size_t)d * p.B * H, H, p.B, (const char*)prm.R + (size_t)d * 4 * H * H * esz,
                               H, 4 * H, H, rh + (size_t)d * S * p.B * 4 * H, 4 * H, S);
    if (!pair) S = 1;
    a.rh_splits = S;
    trace_begin(p, K_REC_FWD, cs);
    int launches = 0;
    for (int step = 0; step < p.T && st == LSTM_OK; ++step) {
        int Md[2] = {0, 0};
        for (int d = 0; d < nd; ++d) {
            const int t = d == 0 ? step : p.T - 1 - step;
            Md[d] = d == 0 ? (t >= 1 ? p.h_bs[t] : 0) : (t + 1 < p.T ? p.h_bs[t + 1] : 0);
        }
        if (pair && (Md[0] > 0 || Md[1] > 0))
            st = gemm_tc_pair(p, -1, op[0], Md[0], nd == 2 ? &op[1] : nullptr, Md[1], cs);
        for (int d = 0; d < nd && st == LSTM_OK && !pair; ++d) {
            // R h_{t-1} of the step's rows that have a previous state (the first M rows)
            const int t = d == 0 ? step : p.T - 1 - step;
            const int M = Md[d];
            if (M == 0) continue;
            const char* Rd = (const char*)prm.R + (size_t)d * 4 * H * H * esz;
            float* C = rh + (size_t)d * S * p.B * 4 * H;
            if (hb16) {
                st = gemm_tc_bf16(p, -1, hb16 + (size_t)d * p.B * H, H, Rd, H, M, 4 * H, H, C, 4 * H, nullptr, 1,
                                  nullptr, cs);
            } else {
                const int prow0 = d == 0 ? p.h_off[t - 1] : p.h_off[t + 1];
                GemmDesc g;
                g.M = M; g.N = 4 * H; g.K = H;
                g.A = y + (size_t)prow0 * ndH + (size_t)d * H; g.sam = ndH; g.sak = 1;
                g.B = Rd; g.sbk = 1; g.sbn = H; g.b_bf16 = bf16;
                g.C = C; g.ldc = 4 * H;
                g.round_bf16 = bf16; g.k_splits = 1;
                st = gemm_simt_run(g, p.num_sms, cs);
                ++launches;
            }
        }
        if (st == LSTM_OK) st = step_cell_launch(a, step, false, cs);
        ++launches;
    }
    trace_end(p, K_REC_FWD, cs, launches);
    return st;
}

// The BPTT recurrence as per-step launches (one cell launch, then per direction one product
// R^T da of the step's rows, tcgen05 when dab16 / rt16 are given), the db / dpeep sums, and
// the dX / dW / dR products.
lstm_status stepwise_bwd_core(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm,
                              const void* x_packed, const float* y_packed, float* ga, float* cbuf,
                              const float* dy_packed, float* dx_packed, const lstm_layer_grads& grads, void* scratch,
                              float* dh_rec, float* dcc, __nv_bfloat16* dab16, __nv_bfloat16* rt16, cudaStream_t cs,
                              const StateIO& sio = StateIO())
{
    const int H = s.hidden_size, nd = s.num_directions;
    const bool bf16 = s.dtype == LSTM_BF16;
    const int nd4H = nd * 4 * H;
    const size_t esz = bf16 ? 2 : 4;
    StepArgs a = step_args(p, s, prm, ga, cbuf);
    a.dy = dy_packed; a.dh_rec = dh_rec; a.dcc = dcc; a.dab16 = dab16;
    a.c0 = sio.c0; a.dh_n = sio.dh_n; a.dc_n = sio.dc_n; a.dc0 = sio.dc0;
    lstm_status st = LSTM_OK;
    if (rt16)   // R_d^T [H][4H] bf16: the B operand (K-major) of the per-step R^T da products
        for (int d = 0; d < nd && st == LSTM_OK; ++d)
            st = transpose_to_bf16_split(p, (const char*)prm.R + (size_t)d * 4 * H * H * esz, bf16, H, 0, nullptr,
                                         4 * H, 4 * H, H, 0, rt16 + (size_t)d * H * 4 * H, 4 * H, 0, nullptr, 0, 0,
                                         cs);
    if (st != LSTM_OK) return st;
    TcOperands op[2];
    bool pair = rt16 != nullptr;
    int S = pair ? step_splits(p, s, true) : 1;
    for (int d = 0; d < nd && pair; ++d)
        pair = gemm_tc_prepare(&op[d], dab16 + (size_t)d * p.B * 4 * H, 4 * H, p.B, rt16 + (size_t)d * H * 4 * H,
                               4 * H, H, 4 * H, dh_rec + (size_t)d * S * p.B * H, H, S);
    if (!pair) S = 1;
    a.dh_splits = S;
    trace_begin(p, K_REC_BWD, cs);     // (no traced call may nest inside this bracket)
    int launches = 0;
    for (int step = 0; step < p.T && st == LSTM_OK; ++step) {
        st = step_cell_launch(a, step, true, cs);
        ++launches;
        if (step + 1 == p.T) break;
        if (pair && st == LSTM_OK) {
            const int M0 = p.h_bs[p.T - 1 - step], M1 = nd == 2 ? p.h_bs[step] : 0;
            st = gemm_tc_pair(p, -1, op[0], M0, nd == 2 ? &op[1] : nullptr, M1, cs);
            continue;
        }
        for (int d = 0; d < nd && st == LSTM_OK; ++d) {
            // R^T da of every row of the step, for the step after it in recurrence order
            const int t = d == 0 ? p.T - 1 - step : step;
            float* C = dh_rec + (size_t)d * S * p.B * H;
            if (rt16) {
                st = gemm_tc_bf16(p, -1, dab16 + (size_t)d * p.B * 4 * H, 4 * H, rt16 + (size_t)d * H * 4 * H, 4 * H,
                                  p.h_bs[t], H, 4 * H, C, H, nullptr, 1, nullptr, cs);
            } else {
                GemmDesc g;
                g.M = p.h_bs[t]; g.N = H; g.K = 4 * H;
                g.A = ga + (size_t)p.h_off[t] * nd4H + (size_t)d * 4 * H; g.sam = nd4H; g.sak = 1;
                g.B = (const char*)prm.R + (size_t)d * 4 * H * H * esz; g.sbk = H; g.sbn = 1; g.b_bf16 = bf16;
                g.C = C; g.ldc = H;
                g.round_bf16 = bf16; g.k_splits = 1;
                st = gemm_simt_run(g, p.num_sms, cs);
                ++launches;
            }
        }
    }
    if (st == LSTM_OK) {
        st = param_sums_launch(p, ga, cbuf, H, nd, grads.db, grads.dpeep, (float*)scratch, cs, sio.c0);
        launches += 2;
    }
    trace_end(p, K_REC_BWD, cs, launches);
    if (st != LSTM_OK) return st;
    return bwd_products(p, s, prm, x_packed, y_packed, ga, dx_packed, grads, scratch, cs);
}

WideArgs wide_args(const Plan& p, const lstm_layer_shape& s, const lstm_layer_params& prm, float* ga, float* cbuf,
                   const StateIO& sio)
{
    WideArgs w;
    memset(&w, 0, sizeof(w));
    w.T = p.T; w.B = p.B; w.H = s.hidden_size; w.ndir = s.num_directions;
    w.padded = p.padded ? 1 : 0;
    w.bs = p.d_bs; w.off = p.d_off; w.len = p.d_len; w.perm = p.d_perm;
    w.ga = ga; w.peep = prm.peep; w.cbuf = cbuf;
    w.h0 = sio.h0; w.c0 = sio.c0; w.dh_n = sio.dh_n; w.dc_n = sio.dc_n; w.dc0 = sio.dc0;
    w.status = p.d_status; w.wait_limit_ns = p.wait_limit_ns;
    w.debug_skip_cta = p.debug_skip_cta;
    return w;
}

// Argument checks of the state pointers (16-byte aligned: the kernels read them as float4).
lstm_status check_state(const Plan& p, const StateIO& sio, bool need_scratch)
{
    if (!sio.any()) return LSTM_OK;
    if (p.padded) return LSTM_ERR_UNSUPPORTED;   // the padded comparator runs from the zero state
    for (const void* q : {(const void*)sio.h0, (const void*)sio.c0, (const void*)sio.dh_n, (const void*)sio.dc_n,
                          (const void*)sio.dh0, (const void*)sio.dc0})
        if (q && !aligned16(q)) return LSTM_ERR_INVALID_ARG;
    if (need_scratch && (!sio.scratch || !aligned16(sio.scratch))) return LSTM_ERR_INVALID_ARG;
    return LSTM_OK;
}

lstm_status check_params(const lstm_layer_params* prm)
{
    if (!prm || !prm->W || !prm->R || !prm->b || !prm->peep) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(prm->W) || !aligned16(prm->R) || !aligned16(prm->b) || !aligned16(prm->peep))
        return LSTM_ERR_INVALID_ARG;
    return LSTM_OK;
}

lstm_status fwd_impl(const lstm_plan* plan, const lstm_layer_shape* shape,
                            const lstm_layer_params* params, const void* x_packed, float* y_packed,
                            void* y_lo, float* h_n, float* c_n, void* workspace, const StateIO& sio, void* stream)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    lstm_status st = check_shape(shape);
    if (st != LSTM_OK) return st;
    if ((st = check_params(params)) != LSTM_OK) return st;
    const Plan& p = plan->p;
    const lstm_layer_shape& s = *shape;
    const int H = s.hidden_size, nd = s.num_directions;
    const bool bf16 = s.dtype == LSTM_BF16;
    cudaStream_t cs = (cudaStream_t)stream;
    if ((h_n && !aligned16(h_n)) || (c_n && !aligned16(c_n))) return LSTM_ERR_INVALID_ARG;
    if ((st = check_state(p, sio, sio.h0 != nullptr && p.rows > 0)) != LSTM_OK) return st;
    if (p.rows == 0) {      // every sequence is empty: its final state is its initial state
        const size_t bytes = sizeof(float) * nd * p.B * H;
        if (h_n) LSTM_CUDA_TRY(sio.h0 ? cudaMemcpyAsync(h_n, sio.h0, bytes, cudaMemcpyDeviceToDevice, cs)
                                      : cudaMemsetAsync(h_n, 0, bytes, cs));
        if (c_n) LSTM_CUDA_TRY(sio.c0 ? cudaMemcpyAsync(c_n, sio.c0, bytes, cudaMemcpyDeviceToDevice, cs)
                                      : cudaMemsetAsync(c_n, 0, bytes, cs));
        return LSTM_OK;
    }
    if (!x_packed || !y_packed || !workspace) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(x_packed) || !aligned16(y_packed) || !aligned16(workspace) || (y_lo && !aligned16(y_lo)))
        return LSTM_ERR_INVALID_ARG;
    const Layout L = workspace_layout(p, s);
    float* ga = (float*)((char*)workspace + L.ga_off);
    float* cbuf = (float*)((char*)workspace + L.c_off);

    if (wide_step_path(p, s)) {
        if ((st = input_projection(p, s, *params, x_packed, ga, (char*)workspace + L.xs_off, cs)) != LSTM_OK)
            return st;
        if ((st = state_fold_input(p, H, nd, bf16, params->R, sio.h0, ga, sio.scratch, cs)) != LSTM_OK) return st;
        if (p.wide_mode != 0 && rec_wide_supported(p, H, nd, bf16)) {
            WideArgs w = wide_args(p, s, *params, ga, cbuf, sio);
            w.y = y_packed; w.y_lo = (__nv_bfloat16*)y_lo; w.h_n = h_n; w.c_n = c_n;
            w.xbuf = (__nv_bfloat16*)((char*)workspace + L.hb_off);
            p.last_rec_kind[0] = 4; p.last_rec_ctas[0] = H / 16; p.last_rec_mma[0] = 2; p.last_rec_variant[0] = 0;
            p.last_rec_groups[0] = 1; p.last_rec_grp_rows[0] = p.B;
            // a launch the device cannot co-schedule falls back to per-step launches (nothing ran)
            if ((st = rec_wide_fwd_launch(p, w, params->R, cs)) != LSTM_ERR_UNSUPPORTED) return st;
        }
        p.last_rec_kind[0] = 3; p.last_rec_ctas[0] = 0; p.last_rec_mma[0] = 2; p.last_rec_variant[0] = 0;
        p.last_rec_groups[0] = 1; p.last_rec_grp_rows[0] = p.B;
        return stepwise_fwd_core(p, s, *params, y_packed, y_lo, h_n, c_n, ga, cbuf,
                                 (float*)((char*)workspace + L.rh_off), (__nv_bfloat16*)((char*)workspace + L.hb_off),
                                 cs, sio);
    }
    RecConfig rc, rcc;
    RecArgs cl_layout;
    memset(&cl_layout, 0, sizeof(cl_layout));
    const bool cluster = rec_cluster_fwd_configure(p, H, nd, bf16, &rcc, &cl_layout);
    if (!cluster && (st = rec_configure(p, H, nd, bf16, false, p.forced_ctas, &rc)) != LSTM_OK) return st;

    if ((st = input_projection(p, s, *params, x_packed, ga, (char*)workspace + L.xs_off, cs)) != LSTM_OK) return st;
    if ((st = state_fold_input(p, H, nd, bf16, params->R, sio.h0, ga, sio.scratch, cs)) != LSTM_OK) return st;

    RecArgs a = base_args(p, s, *params, ga, cbuf);
    a.y = y_packed; a.y_lo = (__nv_bfloat16*)y_lo; a.h_n = h_n; a.c_n = c_n;
    a.h0 = sio.h0; a.c0 = sio.c0;
    if (cluster) {
        a.off_h = cl_layout.off_h; a.off_red = cl_layout.off_red; a.off_contrib = cl_layout.off_contrib;
        a.off_acc = cl_layout.off_acc; a.off_state = cl_layout.off_state; a.off_sums = cl_layout.off_sums;
        a.off_peep = cl_layout.off_peep; a.off_tab = cl_layout.off_tab;
        p.last_rec_kind[0] = 2; p.last_rec_ctas[0] = rcc.G; p.last_rec_mma[0] = 2;
        p.last_rec_variant[0] = (rcc.bulk ? 1 : 0) | (rcc.tma_pre ? 2 : 0);
        p.last_rec_groups[0] = rcc.ngroups; p.last_rec_grp_rows[0] = rcc.grp_rows;
        return rec_cluster_fwd_launch(p, rcc, a, cs);
    }
    p.last_rec_kind[0] = 1; p.last_rec_ctas[0] = rc.G; p.last_rec_mma[0] = rc.mma;
    p.last_rec_groups[0] = 1; p.last_rec_grp_rows[0] = p.B;
    return rec_launch(p, rc, a, false, cs);
}

lstm_status bwd_impl(const lstm_plan* plan, const lstm_layer_shape* shape,
                            const lstm_layer_params* params, const void* x_packed, const float* y_packed,
                            void* workspace, const float* dy_packed, float* dx_packed,
                            const lstm_layer_grads* grads, void* scratch, const StateIO& sio, void* stream)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    lstm_status st = check_shape(shape);
    if (st != LSTM_OK) return st;
    if ((st = check_params(params)) != LSTM_OK) return st;
    if (!grads || !grads->dW || !grads->dR || !grads->db || !grads->dpeep) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(grads->dW) || !aligned16(grads->dR) || !aligned16(grads->db) || !aligned16(grads->dpeep))
        return LSTM_ERR_INVALID_ARG;
    const Plan& p = plan->p;
    const lstm_layer_shape& s = *shape;
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size;
    const bool bf16 = s.dtype == LSTM_BF16;
    cudaStream_t cs = (cudaStream_t)stream;
    if ((st = check_state(p, sio, (sio.h0 || sio.dh0) && p.rows > 0)) != LSTM_OK) return st;
    if (p.rows == 0) {
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->dW, 0, sizeof(float) * nd * 4 * H * D, cs));
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->dR, 0, sizeof(float) * nd * 4 * H * H, cs));
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->db, 0, sizeof(float) * nd * 4 * H, cs));
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->dpeep, 0, sizeof(float) * nd * 3 * H, cs));
        // every sequence is empty: the final-state errors are the initial-state errors
        const size_t bytes = sizeof(float) * nd * p.B * H;
        if (sio.dh0) LSTM_CUDA_TRY(sio.dh_n ? cudaMemcpyAsync(sio.dh0, sio.dh_n, bytes, cudaMemcpyDeviceToDevice, cs)
                                            : cudaMemsetAsync(sio.dh0, 0, bytes, cs));
        if (sio.dc0) LSTM_CUDA_TRY(sio.dc_n ? cudaMemcpyAsync(sio.dc0, sio.dc_n, bytes, cudaMemcpyDeviceToDevice, cs)
                                            : cudaMemsetAsync(sio.dc0, 0, bytes, cs));
        return LSTM_OK;
    }
    if (!x_packed || !y_packed || !workspace || !dy_packed) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(x_packed) || !aligned16(y_packed) || !aligned16(workspace) || !aligned16(dy_packed) ||
        (dx_packed && !aligned16(dx_packed)))
        return LSTM_ERR_INVALID_ARG;
    const size_t need_scratch = scratch_floats(p, s);
    if (need_scratch > 0 && (!scratch || !aligned16(scratch))) return LSTM_ERR_INVALID_ARG;
    const Layout L = workspace_layout(p, s);
    float* ga = (float*)((char*)workspace + L.ga_off);
    float* cbuf = (float*)((char*)workspace + L.c_off);

    if (wide_step_path(p, s)) {
        const StepScratch q = step_scratch(p, s);
        char* sc = (char*)scratch;
        // the persistent backward (automatic: only its K-split cluster form; when that cannot
        // be launched, the per-step launches below)
        if (p.wide_mode != 0 && rec_wide_supported(p, H, nd, bf16)) {
            // R^T [ndir][H][4H] bf16: the resident B operand of each CTA's R^T da product
            __nv_bfloat16* rt16 = (__nv_bfloat16*)(sc + q.rt);
            for (int d = 0; d < nd; ++d)
                if ((st = transpose_to_bf16_split(p, (const char*)params->R + (size_t)d * 4 * H * H * 2, true, H, 0,
                                                  nullptr, 4 * H, 4 * H, H, 0, rt16 + (size_t)d * H * 4 * H, 4 * H, 0,
                                                  nullptr, 0, 0, cs)) != LSTM_OK)
                    return st;
            WideArgs w = wide_args(p, s, *params, ga, cbuf, sio);
            w.dy = dy_packed;
            w.xbuf = (__nv_bfloat16*)(sc + q.dab);
            p.last_rec_kind[1] = 4; p.last_rec_ctas[1] = H / 16; p.last_rec_mma[1] = 2; p.last_rec_variant[1] = 0;
            p.last_rec_groups[1] = 1; p.last_rec_grp_rows[1] = p.B;
            st = rec_wide_bwd_launch(p, w, rt16, (float*)scratch, grads->db, grads->dpeep, cs);
            if (st == LSTM_OK) {
                if ((st = bwd_products(p, s, *params, x_packed, y_packed, ga, dx_packed, *grads, scratch, cs)) != LSTM_OK)
                    return st;
                return sio.any() ? state_backward(p, H, nd, bf16, params->R, ga, sio.h0, sio.dh_n, sio.dc_n, sio.dh0,
                                                  sio.dc0, grads->dR, sio.scratch, cs)
                                 : LSTM_OK;
            }
            if (st != LSTM_ERR_UNSUPPORTED) return st;   // not co-schedulable: per-step launches below
        }
        p.last_rec_kind[1] = 3; p.last_rec_ctas[1] = 0; p.last_rec_mma[1] = 2; p.last_rec_variant[1] = 0;
        p.last_rec_groups[1] = 1; p.last_rec_grp_rows[1] = p.B;
        if ((st = stepwise_bwd_core(p, s, *params, x_packed, y_packed, ga, cbuf, dy_packed, dx_packed, *grads, scratch,
                                    (float*)(sc + q.dh), (float*)(sc + q.dcc), (__nv_bfloat16*)(sc + q.dab),
                                    (__nv_bfloat16*)(sc + q.rt), cs, sio)) != LSTM_OK)
            return st;
        return sio.any() ? state_backward(p, H, nd, bf16, params->R, ga, sio.h0, sio.dh_n, sio.dc_n, sio.dh0, sio.dc0,
                                          grads->dR, sio.scratch, cs)
                         : LSTM_OK;
    }
    RecConfig rc, rcc;
    RecArgs cl_layout;
    memset(&cl_layout, 0, sizeof(cl_layout));
    const bool cluster = rec_cluster_bwd_configure(p, H, nd, bf16, &rcc, &cl_layout);
    if (!cluster && (st = rec_configure(p, H, nd, bf16, true, p.forced_ctas, &rc)) != LSTM_OK) return st;
    RecArgs a = base_args(p, s, *params, ga, cbuf);
    a.y = const_cast<float*>(y_packed); a.dy = dy_packed; a.db = grads->db; a.dpeep = grads->dpeep;
    a.part = (float*)scratch;
    a.c0 = sio.c0; a.dh_n = sio.dh_n; a.dc_n = sio.dc_n; a.dc0 = sio.dc0;
    if (cluster) {
        a.off_h = cl_layout.off_h; a.off_red = cl_layout.off_red; a.off_contrib = cl_layout.off_contrib;
        a.off_acc = cl_layout.off_acc; a.off_state = cl_layout.off_state; a.off_sums = cl_layout.off_sums;
        a.off_peep = cl_layout.off_peep; a.off_tab = cl_layout.off_tab;
        p.last_rec_kind[1] = 2; p.last_rec_ctas[1] = rcc.G; p.last_rec_mma[1] = 2;
        p.last_rec_variant[1] = (rcc.bulk ? 1 : 0) | (rcc.tma_pre ? 2 : 0);
        p.last_rec_groups[1] = rcc.ngroups; p.last_rec_grp_rows[1] = rcc.grp_rows;
        if ((st = rec_cluster_bwd_launch(p, rcc, a, (float*)scratch, cs)) != LSTM_OK) return st;
    } else {
        p.last_rec_kind[1] = 1; p.last_rec_ctas[1] = rc.G; p.last_rec_mma[1] = rc.mma; p.last_rec_variant[1] = 0;
        p.last_rec_groups[1] = 1; p.last_rec_grp_rows[1] = p.B;
        if ((st = rec_launch(p, rc, a, true, cs)) != LSTM_OK) return st;
    }

    if ((st = bwd_products(p, s, *params, x_packed, y_packed, ga, dx_packed, *grads, scratch, cs)) != LSTM_OK)
        return st;
    return sio.any() ? state_backward(p, H, nd, bf16, params->R, ga, sio.h0, sio.dh_n, sio.dc_n, sio.dh0, sio.dc0,
                                      grads->dR, sio.scratch, cs)
                     : LSTM_OK;
}

}  // namespace

}  // namespace lstm

using namespace lstm;

extern "C" {

size_t lstm_workspace_bytes(const lstm_plan* plan, const lstm_layer_shape* shape)
{
    if (!plan || check_shape(shape) != LSTM_OK) return 0;
    return workspace_layout(plan->p, *shape).total;
}

size_t lstm_scratch_bytes(const lstm_plan* plan, const lstm_layer_shape* shape)
{
    if (!plan || check_shape(shape) != LSTM_OK) return 0;
    return align256(std::max<size_t>(1, scratch_floats(plan->p, *shape)) * sizeof(float));
}

lstm_status lstm_fwd(const lstm_plan* plan, const lstm_layer_shape* shape,
                     const lstm_layer_params* params, const void* x_packed, float* y_packed,
                     void* y_lo, float* h_n, float* c_n, void* workspace, void* stream)
{
    return fwd_impl(plan, shape, params, x_packed, y_packed, y_lo, h_n, c_n, workspace, StateIO(), stream);
}

lstm_status lstm_bwd(const lstm_plan* plan, const lstm_layer_shape* shape,
                     const lstm_layer_params* params, const void* x_packed, const float* y_packed,
                     void* workspace, const float* dy_packed, float* dx_packed,
                     const lstm_layer_grads* grads, void* scratch, void* stream)
{
    return bwd_impl(plan, shape, params, x_packed, y_packed, workspace, dy_packed, dx_packed, grads, scratch,
                    StateIO(), stream);
}

size_t lstm_state_scratch_bytes(const lstm_plan* plan, const lstm_layer_shape* shape)
{
    if (!plan || check_shape(shape) != LSTM_OK) return 0;
    return align256(std::max<size_t>(1, state_scratch_floats(plan->p, shape->hidden_size, shape->num_directions)) *
                    sizeof(float));
}

lstm_status lstm_fwd_state(const lstm_plan* plan, const lstm_layer_shape* shape, const lstm_layer_params* params,
                           const lstm_state* state, const void* x_packed, float* y_packed, void* y_lo, float* h_n,
                           float* c_n, void* workspace, void* state_scratch, void* stream)
{
    StateIO sio;
    if (state) { sio.h0 = state->h0; sio.c0 = state->c0; }
    sio.scratch = (float*)state_scratch;
    return fwd_impl(plan, shape, params, x_packed, y_packed, y_lo, h_n, c_n, workspace, sio, stream);
}

lstm_status lstm_bwd_state(const lstm_plan* plan, const lstm_layer_shape* shape, const lstm_layer_params* params,
                           const lstm_state* state, const void* x_packed, const float* y_packed, void* workspace,
                           const float* dy_packed, float* dx_packed, const lstm_layer_grads* grads,
                           const lstm_state_grads* state_grads, void* scratch, void* state_scratch, void* stream)
{
    StateIO sio;
    if (state) { sio.h0 = state->h0; sio.c0 = state->c0; }
    if (state_grads) {
        sio.dh_n = state_grads->dh_n; sio.dc_n = state_grads->dc_n;
        sio.dh0 = state_grads->dh0; sio.dc0 = state_grads->dc0;
    }
    sio.scratch = (float*)state_scratch;
    return bwd_impl(plan, shape, params, x_packed, y_packed, workspace, dy_packed, dx_packed, grads, scratch, sio,
                    stream);
}

size_t lstm_stepwise_scratch_bytes(const lstm_plan* plan, const lstm_layer_shape* shape)
{
    if (!plan || check_shape(shape) != LSTM_OK) return 0;
    return step_scratch(plan->p, *shape).total;
}

lstm_status lstm_fwd_stepwise(const lstm_plan* plan, const lstm_layer_shape* shape,
                              const lstm_layer_params* params, const void* x_packed, float* y_packed,
                              void* y_lo, float* h_n, float* c_n, void* workspace, void* scratch, void* stream)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    lstm_status st = check_shape(shape);
    if (st != LSTM_OK) return st;
    if ((st = check_params(params)) != LSTM_OK) return st;
    const Plan& p = plan->p;
    const lstm_layer_shape& s = *shape;
    const int H = s.hidden_size, nd = s.num_directions;
    cudaStream_t cs = (cudaStream_t)stream;
    if ((h_n && !aligned16(h_n)) || (c_n && !aligned16(c_n))) return LSTM_ERR_INVALID_ARG;
    if (p.rows == 0) {
        if (h_n) LSTM_CUDA_TRY(cudaMemsetAsync(h_n, 0, sizeof(float) * nd * p.B * H, cs));
        if (c_n) LSTM_CUDA_TRY(cudaMemsetAsync(c_n, 0, sizeof(float) * nd * p.B * H, cs));
        return LSTM_OK;
    }
    if (!x_packed || !y_packed || !workspace || !scratch) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(x_packed) || !aligned16(y_packed) || !aligned16(workspace) || !aligned16(scratch) ||
        (y_lo && !aligned16(y_lo)))
        return LSTM_ERR_INVALID_ARG;
    const Layout L = workspace_layout(p, s);
    float* ga = (float*)((char*)workspace + L.ga_off);
    float* cbuf = (float*)((char*)workspace + L.c_off);
    if ((st = input_projection(p, s, *params, x_packed, ga, (char*)workspace + L.xs_off, cs)) != LSTM_OK) return st;
    const StepScratch q = step_scratch(p, s);
    char* sc = (char*)scratch;
    return stepwise_fwd_core(p, s, *params, y_packed, y_lo, h_n, c_n, ga, cbuf, (float*)(sc + q.rh),
                             step_tc(p, s) ? (__nv_bfloat16*)(sc + q.hb) : nullptr, cs);
}

lstm_status lstm_bwd_stepwise(const lstm_plan* plan, const lstm_layer_shape* shape,
                              const lstm_layer_params* params, const void* x_packed, const float* y_packed,
                              void* workspace, const float* dy_packed, float* dx_packed,
                              const lstm_layer_grads* grads, void* scratch, void* stream)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    lstm_status st = check_shape(shape);
    if (st != LSTM_OK) return st;
    if ((st = check_params(params)) != LSTM_OK) return st;
    if (!grads || !grads->dW || !grads->dR || !grads->db || !grads->dpeep) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(grads->dW) || !aligned16(grads->dR) || !aligned16(grads->db) || !aligned16(grads->dpeep))
        return LSTM_ERR_INVALID_ARG;
    const Plan& p = plan->p;
    const lstm_layer_shape& s = *shape;
    const int H = s.hidden_size, nd = s.num_directions, D = s.input_size;
    cudaStream_t cs = (cudaStream_t)stream;
    if (p.rows == 0) {
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->dW, 0, sizeof(float) * nd * 4 * H * D, cs));
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->dR, 0, sizeof(float) * nd * 4 * H * H, cs));
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->db, 0, sizeof(float) * nd * 4 * H, cs));
        LSTM_CUDA_TRY(cudaMemsetAsync(grads->dpeep, 0, sizeof(float) * nd * 3 * H, cs));
        return LSTM_OK;
    }
    if (!x_packed || !y_packed || !workspace || !dy_packed || !scratch) return LSTM_ERR_INVALID_ARG;
    if (!aligned16(x_packed) || !aligned16(y_packed) || !aligned16(workspace) || !aligned16(dy_packed) ||
        !aligned16(scratch) || (dx_packed && !aligned16(dx_packed)))
        return LSTM_ERR_INVALID_ARG;
    const Layout L = workspace_layout(p, s);
    float* ga = (float*)((char*)workspace + L.ga_off);
    float* cbuf = (float*)((char*)workspace + L.c_off);
    const StepScratch q = step_scratch(p, s);
    char* sc = (char*)scratch;
    const bool tc = step_tc(p, s);
    return stepwise_bwd_core(p, s, *params, x_packed, y_packed, ga, cbuf, dy_packed, dx_packed, *grads, scratch,
                             (float*)(sc + q.dh), (float*)(sc + q.dcc), tc ? (__nv_bfloat16*)(sc + q.dab) : nullptr,
                             tc ? (__nv_bfloat16*)(sc + q.rt) : nullptr, cs);
}

lstm_status lstm_debug_input_projection(const lstm_plan* plan, const lstm_layer_shape* shape,
                                        const lstm_layer_params* params, const void* x_packed, float* out,
                                        void* stream)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    lstm_status st = check_shape(shape);
    if (st != LSTM_OK) return st;
    if ((st = check_params(params)) != LSTM_OK) return st;
    if (plan->p.rows == 0) return LSTM_OK;
    if (!x_packed || !out || !aligned16(x_packed) || !aligned16(out)) return LSTM_ERR_INVALID_ARG;
    return input_projection(plan->p, *shape, *params, x_packed, out, nullptr, (cudaStream_t)stream);
}

}  // extern "C"
