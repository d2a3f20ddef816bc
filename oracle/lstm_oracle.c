/*
 * lstm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of what the packed (bi)LSTM
 * path computes.  It exists to check the CUDA library against; nothing in the
 * product calls it.  It shares no code, header or table with the CUDA path.
 *
 * What it computes, and where that comes from:
 *
 *  - The cell.  "Single Stream Parallelization of Generalized LSTM-Like RNNs
 *    on a GPU", Sec. 2 and Fig. 1, builds an LSTM that has forget gates and
 *    peepholes out of additive layers (sum of the incoming
 *    connections, then an activation) and multiplicative layers (element-wise
 *    products).  The page's equations did not survive extraction, so this
 *    file uses the standard reading of that graph: for one direction,
 *        a_t = W x_t + R h_{t-1} + b            (blocks i, f, z, o)
 *        i_t = sig(a_i + p_i * c_{t-1})
 *        f_t = sig(a_f + p_f * c_{t-1})
 *        z_t = tanh(a_z)
 *        c_t = f_t * c_{t-1} + i_t * z_t
 *        o_t = sig(a_o + p_o * c_t)
 *        h_t = o_t * tanh(c_t)
 *    with h_0 = c_0 = 0, diagonal peepholes and one bias per gate.
 *  - The backward pass is BPTT ("Single Stream Parallelization...", Sec. 3):
 *    the error is carried back through the additive and multiplicative nodes
 *    in reverse time, and each connection's gradient is the sum over frames
 *    of its back-propagated error times its source activation.
 *  - Padding-free evaluation ("No Padding Please", Sec. V): every sequence is
 *    computed on its own frames only, so the packed result must equal the
 *    result of running every example on its own (Sec. V-B).  This oracle
 *    therefore loops over each sequence alone.
 *  - The padded comparator (RETURNN paper, Sec. 5: an index tensor marks which
 *    time-batch frames belong to a sequence; "No Padding Please", Sec. V: a
 *    binary mask blocks state input from padding cells): a separate batch-
 *    vector code path over a right-padded [T][B] grid in which masked frames
 *    carry the state unchanged and emit zero output.
 *
 * Bidirectional layers run a second cell with its own parameters over
 * x_L ... x_1; its output at position t is its state after consuming x_t.
 * The layer output is [h_fwd ; h_bwd].  Layer l+1 reads layer l's output.
 *
 * Loss: L = sum over frames of <y_top, G>, so dL/dy_top = G (given).
 *
 * Parameter layout of one layer (ndir directions, D inputs, H units):
 *   W[ndir][4H][D], R[ndir][4H][H], b[ndir][4H], p[ndir][3][H] (p_i,p_f,p_o),
 *   stored back to back in that order.  Gradients use the same layout.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double sigm(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * Diagnostic mode (off by default; never the parity reference): round the
 * state h and the gate errors to bfloat16 before they enter a product, as a
 * bf16-operand implementation does.  Comparing against this mode separates
 * a wrong bf16 kernel from the expected bf16 rounding.
 */
static int g_bf16_products = 0;

void oracle_set_bf16_products(int on) { g_bf16_products = on ? 1 : 0; }

static double to_bf16(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof(u));
    if ((u & 0x7f800000u) == 0x7f800000u) return v;
    u = (u + (((u >> 16) & 1u) + 0x7fffu)) & 0xffff0000u;
    memcpy(&f, &u, sizeof(f));
    return (double)f;
}

static double rb(double v) { return g_bf16_products ? to_bf16(v) : v; }

/* The diagnostic mode's rounding, exported for its pin: v rounded to fp32,
 * then to the nearest bfloat16 (ties to even); Inf and NaN pass through. */
double oracle_round_bf16(double v) { return to_bf16(v); }

static size_t layer_param_count(int ndir, int D, int H)
{
    return (size_t)ndir * ((size_t)4 * H * D + (size_t)4 * H * H + (size_t)4 * H + (size_t)3 * H);
}

/* Number of doubles in one layer's parameter block. */
long oracle_layer_param_count(int ndir, int D, int H) { return (long)layer_param_count(ndir, D, H); }

/*
 * One direction of one layer over one sequence of L frames.
 * x[L][D]; h, c [L][H] and g [L][4H] (post-activation i, f, z, o) are indexed
 * by frame position: h[t] is the state after consuming x[t].
 * reverse = 0 walks t = 0..L-1, reverse = 1 walks t = L-1..0.
 * h0, c0 [H]: the state before the first step (NULL = zero; RETURNN paper,
 * Sec. 3.2: one RNN's final state passed on as another's initial state).
 */
void oracle_dir_forward(int L, int D, int H, const double* x,
                        const double* W, const double* R, const double* b, const double* p,
                        int reverse, const double* h0, const double* c0, double* h, double* c, double* g)
{
    double* a = (double*)malloc(sizeof(double) * 4 * (size_t)H);
    for (int s = 0; s < L; ++s) {
        const int t = reverse ? L - 1 - s : s;
        const int tp = reverse ? t + 1 : t - 1;          /* previous step's position */
        const double* hp = (s == 0) ? h0 : h + (size_t)tp * H;
        const double* cp = (s == 0) ? c0 : c + (size_t)tp * H;
        for (int r = 0; r < 4 * H; ++r) {
            double acc = b[r];
            for (int k = 0; k < D; ++k) acc += W[(size_t)r * D + k] * x[(size_t)t * D + k];
            if (hp)
                for (int k = 0; k < H; ++k) acc += R[(size_t)r * H + k] * rb(hp[k]);
            a[r] = acc;
        }
        for (int u = 0; u < H; ++u) {
            const double cprev = cp ? cp[u] : 0.0;
            const double ig = sigm(a[u] + p[u] * cprev);
            const double fg = sigm(a[H + u] + p[H + u] * cprev);
            const double zg = tanh(a[2 * H + u]);
            const double cn = fg * cprev + ig * zg;
            const double og = sigm(a[3 * H + u] + p[2 * H + u] * cn);
            h[(size_t)t * H + u] = og * tanh(cn);
            c[(size_t)t * H + u] = cn;
            double* gt = g + (size_t)t * 4 * H;
            gt[u] = ig;
            gt[H + u] = fg;
            gt[2 * H + u] = zg;
            gt[3 * H + u] = og;
        }
    }
    free(a);
}

/*
 * BPTT for one direction over one sequence, given the forward results.
 * dy[L][H] is dL/dh_t from outside the recurrence (the layer above, or G).
 * h0, c0 [H]: the initial state of the forward pass (NULL = zero).
 * dhn, dcn [H]: dL/dh and dL/dc of the final state from outside (NULL = zero).
 * Accumulates into dx[L][D], dW[4H][D], dR[4H][H], db[4H], dp[3][H]; writes
 * dh0, dc0 [H] (dL/d of the initial state; either may be NULL).
 */
void oracle_dir_backward(int L, int D, int H, const double* x,
                         const double* W, const double* R, const double* p, int reverse,
                         const double* h0, const double* c0, const double* dhn, const double* dcn,
                         const double* h, const double* c, const double* g, const double* dy,
                         double* dx, double* dW, double* dR, double* db, double* dp,
                         double* dh0, double* dc0)
{
    const size_t G4 = 4 * (size_t)H;
    double* da = (double*)malloc(sizeof(double) * G4);
    double* da_next = (double*)calloc(G4, sizeof(double));
    double* dc_next = (double*)calloc((size_t)H, sizeof(double));
    double* f_next = (double*)calloc((size_t)H, sizeof(double));
    double* dc_cur = (double*)malloc(sizeof(double) * H);
    double* dh = (double*)malloc(sizeof(double) * H);
    int have_next = 0;
    for (int s = L - 1; s >= 0; --s) {
        const int t = reverse ? L - 1 - s : s;
        const int tp = reverse ? t + 1 : t - 1;
        const double* gt = g + (size_t)t * G4;
        /* error reaching h_t: from outside, and from every gate of the next step through R
         * (the last step: from the final state's own gradient instead) */
        for (int u = 0; u < H; ++u) {
            double acc = dy[(size_t)t * H + u];
            if (have_next)
                for (size_t r = 0; r < G4; ++r) acc += R[r * H + u] * rb(da_next[r]);
            else if (dhn)
                acc += dhn[u];
            dh[u] = acc;
        }
        for (int u = 0; u < H; ++u) {
            const double ig = gt[u], fg = gt[H + u], zg = gt[2 * H + u], og = gt[3 * H + u];
            const double cn = c[(size_t)t * H + u];
            const double cprev = (s > 0) ? c[(size_t)tp * H + u] : (c0 ? c0[u] : 0.0);
            const double tc = tanh(cn);
            const double da_o = dh[u] * tc * og * (1.0 - og);
            double dc = dh[u] * og * (1.0 - tc * tc) + da_o * p[2 * H + u];
            if (have_next)
                dc += dc_next[u] * f_next[u] + da_next[u] * p[u] + da_next[H + u] * p[H + u];
            else if (dcn)
                dc += dcn[u];
            const double da_i = dc * zg * ig * (1.0 - ig);
            const double da_f = dc * cprev * fg * (1.0 - fg);
            const double da_z = dc * ig * (1.0 - zg * zg);
            da[u] = da_i;
            da[H + u] = da_f;
            da[2 * H + u] = da_z;
            da[3 * H + u] = da_o;
            dp[u] += da_i * cprev;
            dp[H + u] += da_f * cprev;
            dp[2 * H + u] += da_o * cn;
            dc_cur[u] = dc;
        }
        for (size_t r = 0; r < G4; ++r) {
            db[r] += da[r];
            for (int k = 0; k < D; ++k) dW[r * D + k] += rb(da[r]) * x[(size_t)t * D + k];
            if (s > 0)
                for (int k = 0; k < H; ++k) dR[r * H + k] += rb(da[r]) * rb(h[(size_t)tp * H + k]);
            else if (h0)
                for (int k = 0; k < H; ++k) dR[r * H + k] += rb(da[r]) * rb(h0[k]);
        }
        if (s == 0) {
            /* the initial state: dh0 through R from the first step's gates, dc0 as the carry
             * the first step passes back (forget gate and the i, f peepholes read c0) */
            for (int u = 0; u < H; ++u) {
                if (dh0) {
                    double acc = 0.0;
                    for (size_t r = 0; r < G4; ++r) acc += R[r * H + u] * rb(da[r]);
                    dh0[u] = acc;
                }
                if (dc0) dc0[u] = dc_cur[u] * gt[H + u] + da[u] * p[u] + da[H + u] * p[H + u];
            }
        }
        for (int k = 0; k < D; ++k) {
            double acc = 0.0;
            for (size_t r = 0; r < G4; ++r) acc += W[r * D + k] * rb(da[r]);
            dx[(size_t)t * D + k] += acc;
        }
        memcpy(da_next, da, sizeof(double) * G4);
        memcpy(dc_next, dc_cur, sizeof(double) * H);
        for (int u = 0; u < H; ++u) f_next[u] = gt[H + u];
        have_next = 1;
    }
    free(da); free(da_next); free(dc_next); free(f_next); free(dc_cur); free(dh);
}

/* Per-layer views into a flat parameter (or gradient) block. */
typedef struct { double *W, *R, *b, *p; } dir_view;

static dir_view view_of(double* base, int ndir, int dir, int D, int H)
{
    dir_view v;
    double* W0 = base;
    double* R0 = W0 + (size_t)ndir * 4 * H * D;
    double* b0 = R0 + (size_t)ndir * 4 * H * H;
    double* p0 = b0 + (size_t)ndir * 4 * H;
    v.W = W0 + (size_t)dir * 4 * H * D;
    v.R = R0 + (size_t)dir * 4 * H * H;
    v.b = b0 + (size_t)dir * 4 * H;
    v.p = p0 + (size_t)dir * 3 * H;
    return v;
}

/*
 * A stack of num_layers layers over B sequences given in the caller's order.
 *   lengths[B]          frames per sequence (0 allowed)
 *   x_cat[N][D0]        sequences concatenated frame after frame, N = sum(lengths)
 *   layer_params[l]     flat block, layout above; D_l = D0 for l = 0 else ndir*H
 *   dy_cat[N][ndir*H]   dL/dy of the top layer (NULL: forward only)
 * Outputs (any may be NULL):
 *   y_cat[N][ndir*H]                  top-layer output
 *   h_n, c_n [num_layers][ndir][B][H] final states (zero for empty sequences)
 *   dx_cat[N][D0]                     dL/dx
 *   layer_grads[l]                    overwritten with dL/dparams
 * nthreads > 1 splits the sequences over OpenMP threads; per-thread gradient
 * sums are then added in thread order.
 * Returns 0 on success, -1 on a bad argument or allocation failure.
 */
int oracle_lstm_stack_state(int B, const int* lengths, int num_layers, int ndir, int H, int D0,
                            const double* x_cat, double* const* layer_params, const double* dy_cat,
                            const double* h0, const double* c0, const double* dh_n, const double* dc_n,
                            double* y_cat, double* h_n, double* c_n, double* dx_cat,
                            double* const* layer_grads, double* dh0, double* dc0, int nthreads);

int oracle_lstm_stack(int B, const int* lengths, int num_layers, int ndir, int H, int D0,
                      const double* x_cat, double* const* layer_params, const double* dy_cat,
                      double* y_cat, double* h_n, double* c_n, double* dx_cat,
                      double* const* layer_grads, int nthreads)
{
    return oracle_lstm_stack_state(B, lengths, num_layers, ndir, H, D0, x_cat, layer_params, dy_cat, NULL, NULL,
                                   NULL, NULL, y_cat, h_n, c_n, dx_cat, layer_grads, NULL, NULL, nthreads);
}

/*
 * The same stack with initial states and final-state gradients (all
 * [num_layers][ndir][B][H], caller order, NULL = zero):
 *   h0, c0       state of every layer and direction before its first step
 *   dh_n, dc_n   dL/dh_n, dL/dc_n from outside (a loss that reads the final states)
 *   dh0, dc0     outputs: dL/dh0, dL/dc0 (NULL: not wanted)
 * A sequence of length 0 consumes nothing: h_n = h0, c_n = c0, dh0 = dh_n, dc0 = dc_n.
 */
int oracle_lstm_stack_state(int B, const int* lengths, int num_layers, int ndir, int H, int D0,
                            const double* x_cat, double* const* layer_params, const double* dy_cat,
                            const double* h0, const double* c0, const double* dh_n, const double* dc_n,
                            double* y_cat, double* h_n, double* c_n, double* dx_cat,
                            double* const* layer_grads, double* dh0, double* dc0, int nthreads)
{
    if (B < 0 || num_layers < 1 || (ndir != 1 && ndir != 2) || H < 1 || D0 < 1) return -1;
    long long* start = (long long*)malloc(sizeof(long long) * (size_t)(B + 1));
    start[0] = 0;
    for (int b = 0; b < B; ++b) {
        if (lengths[b] < 0) { free(start); return -1; }
        start[b + 1] = start[b] + lengths[b];
    }
    const int Hout = ndir * H;
    const int do_bwd = (dy_cat != NULL);
    if (nthreads < 1) nthreads = 1;
    size_t* gsize = (size_t*)malloc(sizeof(size_t) * num_layers);
    size_t gtotal = 0;
    for (int l = 0; l < num_layers; ++l) {
        gsize[l] = layer_param_count(ndir, l == 0 ? D0 : Hout, H);
        gtotal += gsize[l];
    }
    /* private gradient sums, one set per thread */
    double* gpriv = do_bwd ? (double*)calloc(gtotal * (size_t)nthreads, sizeof(double)) : NULL;
    const size_t nst = (size_t)num_layers * ndir * B * H;
    if (h_n) { if (h0) memcpy(h_n, h0, sizeof(double) * nst); else memset(h_n, 0, sizeof(double) * nst); }
    if (c_n) { if (c0) memcpy(c_n, c0, sizeof(double) * nst); else memset(c_n, 0, sizeof(double) * nst); }
    if (dh0) { if (dh_n) memcpy(dh0, dh_n, sizeof(double) * nst); else memset(dh0, 0, sizeof(double) * nst); }
    if (dc0) { if (dc_n) memcpy(dc0, dc_n, sizeof(double) * nst); else memset(dc0, 0, sizeof(double) * nst); }

    int err = 0;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int b = 0; b < B; ++b) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        const int L = lengths[b];
        if (L == 0) continue;
        const int Dmax = D0 > Hout ? D0 : Hout;
        /* acts[l] = input of layer l ([L][D_l]); acts[num_layers] = top output */
        double** acts = (double**)malloc(sizeof(double*) * (num_layers + 1));
        double** hs = (double**)malloc(sizeof(double*) * num_layers * ndir);
        double** cs = (double**)malloc(sizeof(double*) * num_layers * ndir);
        double** gs = (double**)malloc(sizeof(double*) * num_layers * ndir);
        acts[0] = (double*)malloc(sizeof(double) * (size_t)L * D0);
        memcpy(acts[0], x_cat + (size_t)start[b] * D0, sizeof(double) * (size_t)L * D0);
        for (int l = 0; l < num_layers; ++l) {
            const int D = (l == 0) ? D0 : Hout;
            acts[l + 1] = (double*)malloc(sizeof(double) * (size_t)L * Hout);
            for (int d = 0; d < ndir; ++d) {
                dir_view v = view_of(layer_params[l], ndir, d, D, H);
                double* h = hs[l * ndir + d] = (double*)malloc(sizeof(double) * (size_t)L * H);
                double* c = cs[l * ndir + d] = (double*)malloc(sizeof(double) * (size_t)L * H);
                double* g = gs[l * ndir + d] = (double*)malloc(sizeof(double) * (size_t)L * 4 * H);
                const size_t so = (((size_t)l * ndir + d) * B + b) * H;     /* this state's offset */
                oracle_dir_forward(L, D, H, acts[l], v.W, v.R, v.b, v.p, d == 1, h0 ? h0 + so : NULL,
                                   c0 ? c0 + so : NULL, h, c, g);
                for (int t = 0; t < L; ++t)
                    memcpy(acts[l + 1] + (size_t)t * Hout + (size_t)d * H, h + (size_t)t * H,
                           sizeof(double) * H);
                if (g_bf16_products && l + 1 < num_layers)   /* next layer's operand */
                    for (int t = 0; t < L; ++t)
                        for (int u = 0; u < H; ++u) {
                            double* v = acts[l + 1] + (size_t)t * Hout + (size_t)d * H + u;
                            *v = to_bf16(*v);
                        }
                const int tl = (d == 0) ? L - 1 : 0;      /* last position consumed */
                const size_t o = (((size_t)l * ndir + d) * B + b) * H;
                if (h_n) memcpy(h_n + o, h + (size_t)tl * H, sizeof(double) * H);
                if (c_n) memcpy(c_n + o, c + (size_t)tl * H, sizeof(double) * H);
            }
        }
        if (y_cat)
            memcpy(y_cat + (size_t)start[b] * Hout, acts[num_layers], sizeof(double) * (size_t)L * Hout);
        if (do_bwd) {
            double* dout = (double*)malloc(sizeof(double) * (size_t)L * Dmax);
            double* din = (double*)malloc(sizeof(double) * (size_t)L * Dmax);
            double* dyd = (double*)malloc(sizeof(double) * (size_t)L * H);
            memcpy(dout, dy_cat + (size_t)start[b] * Hout, sizeof(double) * (size_t)L * Hout);
            double* gbase = gpriv + (size_t)tid * gtotal;
            size_t goff[64];
            goff[0] = 0;
            for (int l = 1; l < num_layers && l < 64; ++l) goff[l] = goff[l - 1] + gsize[l - 1];
            for (int l = num_layers - 1; l >= 0; --l) {
                const int D = (l == 0) ? D0 : Hout;
                memset(din, 0, sizeof(double) * (size_t)L * D);
                for (int d = 0; d < ndir; ++d) {
                    dir_view v = view_of(layer_params[l], ndir, d, D, H);
                    dir_view gv = view_of(gbase + goff[l], ndir, d, D, H);
                    for (int t = 0; t < L; ++t)
                        memcpy(dyd + (size_t)t * H, dout + (size_t)t * Hout + (size_t)d * H,
                               sizeof(double) * H);
                    const size_t so = (((size_t)l * ndir + d) * B + b) * H;
                    oracle_dir_backward(L, D, H, acts[l], v.W, v.R, v.p, d == 1, h0 ? h0 + so : NULL,
                                        c0 ? c0 + so : NULL, dh_n ? dh_n + so : NULL, dc_n ? dc_n + so : NULL,
                                        hs[l * ndir + d], cs[l * ndir + d], gs[l * ndir + d], dyd,
                                        din, gv.W, gv.R, gv.b, gv.p, dh0 ? dh0 + so : NULL,
                                        dc0 ? dc0 + so : NULL);
                }
                double* tmp = dout; dout = din; din = tmp;   /* dout now holds dL/d(input of l) */
            }
            if (dx_cat) memcpy(dx_cat + (size_t)start[b] * D0, dout, sizeof(double) * (size_t)L * D0);
            free(dout); free(din); free(dyd);
        }
        for (int l = 0; l <= num_layers; ++l) free(acts[l]);
        for (int i = 0; i < num_layers * ndir; ++i) { free(hs[i]); free(cs[i]); free(gs[i]); }
        free(acts); free(hs); free(cs); free(gs);
    }
    if (num_layers > 64) err = -1;
    if (do_bwd && layer_grads) {
        size_t off = 0;
        for (int l = 0; l < num_layers; ++l) {
            if (layer_grads[l]) {
                memset(layer_grads[l], 0, sizeof(double) * gsize[l]);
                for (int th = 0; th < nthreads; ++th) {
                    const double* src = gpriv + (size_t)th * gtotal + off;
                    for (size_t i = 0; i < gsize[l]; ++i) layer_grads[l][i] += src[i];
                }
            }
            off += gsize[l];
        }
    }
    free(gpriv); free(gsize); free(start);
    return err;
}

/*
 * The padded comparator: one layer over a right-padded, time-major batch.
 *   x_pad[T][B][D], mask[T][B] (1 = frame of a sequence, 0 = padding),
 *   params: flat block (layout above), dy_pad[T][B][ndir*H] (NULL: forward only).
 * Masked frames carry (h, c) unchanged, emit y = 0, and their upstream
 * gradient is ignored; the backward direction starts from the zero state at
 * t = T-1 and carries it through trailing padding.
 * Outputs: y_pad[T][B][ndir*H], h_n/c_n [ndir][B][H], dx_pad[T][B][D],
 * grads (flat block, overwritten).  Any output may be NULL.
 */
int oracle_lstm_padded_layer(int T, int B, int D, int H, int ndir,
                             const double* x_pad, const unsigned char* mask, const double* params,
                             const double* dy_pad, double* y_pad, double* h_n, double* c_n,
                             double* dx_pad, double* grads)
{
    if (T < 0 || B < 0 || D < 1 || H < 1 || (ndir != 1 && ndir != 2)) return -1;
    const int Hout = ndir * H;
    const size_t G4 = 4 * (size_t)H;
    const size_t TB = (size_t)T * B;
    if (y_pad) memset(y_pad, 0, sizeof(double) * TB * Hout);
    if (dx_pad) memset(dx_pad, 0, sizeof(double) * TB * D);
    if (grads) memset(grads, 0, sizeof(double) * layer_param_count(ndir, D, H));
    double* hs = (double*)malloc(sizeof(double) * B * H);      /* carried state */
    double* cs = (double*)malloc(sizeof(double) * B * H);
    /* saved per (t, b): state before the step, gates and new c */
    double* h_before = (double*)malloc(sizeof(double) * TB * H);
    double* c_before = (double*)malloc(sizeof(double) * TB * H);
    double* c_after = (double*)malloc(sizeof(double) * TB * H);
    double* gates = (double*)malloc(sizeof(double) * TB * G4);
    double* a = (double*)malloc(sizeof(double) * G4);
    double* dhs = (double*)malloc(sizeof(double) * B * H);
    double* dcs = (double*)malloc(sizeof(double) * B * H);
    double* da = (double*)malloc(sizeof(double) * G4);
    double* dcv = (double*)malloc(sizeof(double) * H);
    for (int d = 0; d < ndir; ++d) {
        dir_view v = view_of((double*)params, ndir, d, D, H);
        memset(hs, 0, sizeof(double) * B * H);
        memset(cs, 0, sizeof(double) * B * H);
        for (int s = 0; s < T; ++s) {
            const int t = d ? T - 1 - s : s;
            for (int b = 0; b < B; ++b) {
                const size_t tb = (size_t)t * B + b;
                if (!mask[tb]) continue;                           /* padding: carry */
                memcpy(h_before + tb * H, hs + (size_t)b * H, sizeof(double) * H);
                memcpy(c_before + tb * H, cs + (size_t)b * H, sizeof(double) * H);
                for (size_t r = 0; r < G4; ++r) {
                    double acc = v.b[r];
                    for (int k = 0; k < D; ++k) acc += v.W[r * D + k] * x_pad[tb * D + k];
                    for (int k = 0; k < H; ++k) acc += v.R[r * H + k] * hs[(size_t)b * H + k];
                    a[r] = acc;
                }
                for (int u = 0; u < H; ++u) {
                    const double cprev = cs[(size_t)b * H + u];
                    const double ig = sigm(a[u] + v.p[u] * cprev);
                    const double fg = sigm(a[H + u] + v.p[H + u] * cprev);
                    const double zg = tanh(a[2 * H + u]);
                    const double cn = fg * cprev + ig * zg;
                    const double og = sigm(a[3 * H + u] + v.p[2 * H + u] * cn);
                    const double hn = og * tanh(cn);
                    gates[tb * G4 + u] = ig;
                    gates[tb * G4 + H + u] = fg;
                    gates[tb * G4 + 2 * H + u] = zg;
                    gates[tb * G4 + 3 * H + u] = og;
                    c_after[tb * H + u] = cn;
                    cs[(size_t)b * H + u] = cn;
                    hs[(size_t)b * H + u] = hn;
                    if (y_pad) y_pad[tb * Hout + (size_t)d * H + u] = hn;
                }
            }
        }
        for (int b = 0; b < B; ++b) {
            if (h_n) memcpy(h_n + ((size_t)d * B + b) * H, hs + (size_t)b * H, sizeof(double) * H);
            if (c_n) memcpy(c_n + ((size_t)d * B + b) * H, cs + (size_t)b * H, sizeof(double) * H);
        }
        if (!dy_pad) continue;
        dir_view gv = view_of(grads, ndir, d, D, H);
        /* dhs/dcs: dL/d(state after the step being undone), from later steps */
        memset(dhs, 0, sizeof(double) * B * H);
        memset(dcs, 0, sizeof(double) * B * H);
        for (int s = T - 1; s >= 0; --s) {
            const int t = d ? T - 1 - s : s;
            for (int b = 0; b < B; ++b) {
                const size_t tb = (size_t)t * B + b;
                if (!mask[tb]) continue;                           /* identity carry */
                for (int u = 0; u < H; ++u) {
                    const double ig = gates[tb * G4 + u], fg = gates[tb * G4 + H + u];
                    const double zg = gates[tb * G4 + 2 * H + u], og = gates[tb * G4 + 3 * H + u];
                    const double cn = c_after[tb * H + u], cprev = c_before[tb * H + u];
                    const double dh = dy_pad[tb * Hout + (size_t)d * H + u] + dhs[(size_t)b * H + u];
                    const double tc = tanh(cn);
                    const double da_o = dh * tc * og * (1.0 - og);
                    const double dc = dh * og * (1.0 - tc * tc) + da_o * v.p[2 * H + u]
                                      + dcs[(size_t)b * H + u];
                    da[u] = dc * zg * ig * (1.0 - ig);
                    da[H + u] = dc * cprev * fg * (1.0 - fg);
                    da[2 * H + u] = dc * ig * (1.0 - zg * zg);
                    da[3 * H + u] = da_o;
                    dcv[u] = dc;
                }
                for (int u = 0; u < H; ++u) {
                    const double cprev = c_before[tb * H + u];
                    gv.p[u] += da[u] * cprev;
                    gv.p[H + u] += da[H + u] * cprev;
                    gv.p[2 * H + u] += da[3 * H + u] * c_after[tb * H + u];
                    /* state error handed to the previous step */
                    dcs[(size_t)b * H + u] = dcv[u] * gates[tb * G4 + H + u]
                                             + da[u] * v.p[u] + da[H + u] * v.p[H + u];
                }
                for (int k = 0; k < H; ++k) {
                    double acc = 0.0;
                    for (size_t r = 0; r < G4; ++r) acc += v.R[r * H + k] * da[r];
                    dhs[(size_t)b * H + k] = acc;
                }
                for (size_t r = 0; r < G4; ++r) {
                    gv.b[r] += da[r];
                    for (int k = 0; k < D; ++k) gv.W[r * D + k] += da[r] * x_pad[tb * D + k];
                    for (int k = 0; k < H; ++k) gv.R[r * H + k] += da[r] * h_before[tb * H + k];
                }
                if (dx_pad)
                    for (int k = 0; k < D; ++k) {
                        double acc = 0.0;
                        for (size_t r = 0; r < G4; ++r) acc += v.W[r * D + k] * da[r];
                        dx_pad[tb * D + k] += acc;
                    }
            }
        }
    }
    free(hs); free(cs); free(h_before); free(c_before); free(c_after); free(gates); free(a);
    free(dhs); free(dcs); free(da); free(dcv);
    return 0;
}
