/*
 * mdlstm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of one 2-D MDLSTM layer, for
 * checking the CUDA library's 2-D example-packing path against.  Nothing in
 * the product calls it; it shares no code, header or table with the CUDA path.
 *
 * What it computes, and where that comes from ("No Padding Please: Efficient
 * Neural Handwriting Recognition"):
 *
 *  - The cell (Sec. III, Fig. 4(a); App. A).  Every cell of a 2-D grid takes
 *    the pixel input and the <hidden, state> pairs of two predecessor cells:
 *    the one before it along the rows (index 1, "above" for the top-left scan)
 *    and the one before it along the columns (index 2, "left").  Five input
 *    blocks come from x, h1 and h2 (input gate, two forget gates, input node,
 *    output gate: App. A's five matrix products per hidden state); each
 *    predecessor state S_d enters three of them (App. A: three products per
 *    memory state) -- the input gate, its own forget gate and the output gate,
 *    the output gate reading the previous states rather than the new one
 *    (Sec. III's variant).  The pages print no equations; this file uses the
 *    plain reading of that description, with element-wise peepholes:
 *        a_g = W_g x + U1_g h1 + U2_g h2 + b_g        g in (i, f1, f2, z, o)
 *        i   = sig(a_i  + p_i1 S1 + p_i2 S2)
 *        f1  = sig(a_f1 + p_f1 S1)
 *        f2  = sig(a_f2 + p_f2 S2)
 *        z   = tanh(a_z)
 *        o   = sig(a_o  + p_o1 S1 + p_o2 S2)
 *        c   = f1 S1 + f2 S2 + i z
 *        h   = o tanh(c)
 *    A predecessor outside the example contributes h = S = 0 (Sec. V: the
 *    mask blocks state input from padding and separator cells, so a packed
 *    example computes exactly what it computes alone).
 *  - Scan directions (Sec. III: a 4-directional layer stacks four MDLSTMs,
 *    one per corner the grid is scanned from): direction d scans the image
 *    flipped along x when d & 1 and along y when d & 2; its output at pixel
 *    (y, x) is the cell state after that pixel in its own scan order.
 *  - The backward pass is back-propagation through the 2-D recurrence in the
 *    reverse scan order: a cell's h and S errors collect from the two cells
 *    that take it as predecessor 1 and 2.
 *
 * Parameter block of one direction (D inputs, H units), back to back:
 *   W[5H][D], U1[5H][H], U2[5H][H], b[5H], p[6][H] (p_i1, p_i2, p_f1, p_f2,
 *   p_o1, p_o2); gate blocks of 5H in the order i, f1, f2, z, o.  A layer is
 *   ndir such blocks.  Gradients use the same layout.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static double sg(double v) { return 1.0 / (1.0 + exp(-v)); }

long oracle_md_param_count(int D, int H) { return 5L * H * D + 2L * 5 * H * H + 5L * H + 6L * H; }

/* pixel index (row-major, caller layout) of scan position (ys, xs) */
static int pix(int h, int w, int fy, int fx, int ys, int xs)
{
    const int y = fy ? h - 1 - ys : ys;
    const int x = fx ? w - 1 - xs : xs;
    return y * w + x;
}

typedef struct {
    const double *W, *U1, *U2, *b, *p;
} md_params;

static md_params md_view(const double* blk, int D, int H)
{
    md_params m;
    m.W = blk;
    m.U1 = m.W + 5 * H * D;
    m.U2 = m.U1 + 5 * H * H;
    m.b = m.U2 + 5 * H * H;
    m.p = m.b + 5 * H;
    return m;
}

/*
 * Forward of one example (h x w pixels, x[h*w][D]) in direction d.  Writes the
 * output y[h*w][H] (pixel order) and, when given, the gate activations
 * act[h*w][5H] (i, f1, f2, z, o) and the states cst[h*w][H].
 */
void oracle_md_forward(int h, int w, int D, int H, int d, const double* x, const double* blk, double* y, double* act,
                       double* cst)
{
    const md_params m = md_view(blk, D, H);
    const int fx = d & 1, fy = (d >> 1) & 1;
    double* a = (double*)malloc(sizeof(double) * 5 * H);
    double* cs = cst ? cst : (double*)calloc((size_t)h * w * H, sizeof(double));
    for (int ys = 0; ys < h; ++ys)
        for (int xs = 0; xs < w; ++xs) {
            const int q = pix(h, w, fy, fx, ys, xs);
            const int q1 = ys > 0 ? pix(h, w, fy, fx, ys - 1, xs) : -1;    /* predecessor 1 */
            const int q2 = xs > 0 ? pix(h, w, fy, fx, ys, xs - 1) : -1;    /* predecessor 2 */
            const double* xv = x + (size_t)q * D;
            for (int r = 0; r < 5 * H; ++r) {
                double s = m.b[r];
                for (int k = 0; k < D; ++k) s += m.W[(size_t)r * D + k] * xv[k];
                if (q1 >= 0)
                    for (int k = 0; k < H; ++k) s += m.U1[(size_t)r * H + k] * y[(size_t)q1 * H + k];
                if (q2 >= 0)
                    for (int k = 0; k < H; ++k) s += m.U2[(size_t)r * H + k] * y[(size_t)q2 * H + k];
                a[r] = s;
            }
            for (int u = 0; u < H; ++u) {
                const double S1 = q1 >= 0 ? cs[(size_t)q1 * H + u] : 0.0;
                const double S2 = q2 >= 0 ? cs[(size_t)q2 * H + u] : 0.0;
                const double ig = sg(a[u] + m.p[u] * S1 + m.p[H + u] * S2);
                const double f1 = sg(a[H + u] + m.p[2 * H + u] * S1);
                const double f2 = sg(a[2 * H + u] + m.p[3 * H + u] * S2);
                const double zg = tanh(a[3 * H + u]);
                const double og = sg(a[4 * H + u] + m.p[4 * H + u] * S1 + m.p[5 * H + u] * S2);
                const double c = f1 * S1 + f2 * S2 + ig * zg;
                cs[(size_t)q * H + u] = c;
                y[(size_t)q * H + u] = og * tanh(c);
                if (act) {
                    double* ar = act + (size_t)q * 5 * H;
                    ar[u] = ig; ar[H + u] = f1; ar[2 * H + u] = f2; ar[3 * H + u] = zg; ar[4 * H + u] = og;
                }
            }
        }
    free(a);
    if (!cst) free(cs);
}

/*
 * Backward of one example in direction d: dy[h*w][H] is dL/dy; adds dL/dx into
 * dx[h*w][D] and the parameter gradients into gblk (same layout as blk).
 */
void oracle_md_backward(int h, int w, int D, int H, int d, const double* x, const double* blk, const double* dy,
                        double* dx, double* gblk)
{
    const md_params m = md_view(blk, D, H);
    double* gW = gblk;
    double* gU1 = gW + 5 * H * D;
    double* gU2 = gU1 + 5 * H * H;
    double* gb = gU2 + 5 * H * H;
    double* gp = gb + 5 * H;
    const int fx = d & 1, fy = (d >> 1) & 1;
    const size_t n = (size_t)h * w;
    double* y = (double*)calloc(n * H, sizeof(double));
    double* act = (double*)calloc(n * 5 * H, sizeof(double));
    double* cs = (double*)calloc(n * H, sizeof(double));
    double* dh = (double*)calloc(n * H, sizeof(double));     /* errors reaching h from successors */
    double* dS = (double*)calloc(n * H, sizeof(double));     /* errors reaching the state from successors */
    double* da = (double*)malloc(sizeof(double) * 5 * H);
    oracle_md_forward(h, w, D, H, d, x, blk, y, act, cs);
    for (int ys = h - 1; ys >= 0; --ys)
        for (int xs = w - 1; xs >= 0; --xs) {
            const int q = pix(h, w, fy, fx, ys, xs);
            const int q1 = ys > 0 ? pix(h, w, fy, fx, ys - 1, xs) : -1;
            const int q2 = xs > 0 ? pix(h, w, fy, fx, ys, xs - 1) : -1;
            const double* ar = act + (size_t)q * 5 * H;
            for (int u = 0; u < H; ++u) {
                const double S1 = q1 >= 0 ? cs[(size_t)q1 * H + u] : 0.0;
                const double S2 = q2 >= 0 ? cs[(size_t)q2 * H + u] : 0.0;
                const double ig = ar[u], f1 = ar[H + u], f2 = ar[2 * H + u], zg = ar[3 * H + u], og = ar[4 * H + u];
                const double c = cs[(size_t)q * H + u];
                const double tc = tanh(c);
                const double e = dy[(size_t)q * H + u] + dh[(size_t)q * H + u];
                const double dao = e * tc * og * (1.0 - og);
                const double dc = e * og * (1.0 - tc * tc) + dS[(size_t)q * H + u];
                const double dai = dc * zg * ig * (1.0 - ig);
                const double daf1 = dc * S1 * f1 * (1.0 - f1);
                const double daf2 = dc * S2 * f2 * (1.0 - f2);
                const double daz = dc * ig * (1.0 - zg * zg);
                da[u] = dai; da[H + u] = daf1; da[2 * H + u] = daf2; da[3 * H + u] = daz; da[4 * H + u] = dao;
                /* the predecessors' states: through f1 / f2 and the three peepholes each */
                if (q1 >= 0)
                    dS[(size_t)q1 * H + u] += dc * f1 + m.p[u] * dai + m.p[2 * H + u] * daf1 + m.p[4 * H + u] * dao;
                if (q2 >= 0)
                    dS[(size_t)q2 * H + u] += dc * f2 + m.p[H + u] * dai + m.p[3 * H + u] * daf2 + m.p[5 * H + u] * dao;
                gp[u] += dai * S1;
                gp[H + u] += dai * S2;
                gp[2 * H + u] += daf1 * S1;
                gp[3 * H + u] += daf2 * S2;
                gp[4 * H + u] += dao * S1;
                gp[5 * H + u] += dao * S2;
            }
            const double* xv = x + (size_t)q * D;
            for (int r = 0; r < 5 * H; ++r) {
                gb[r] += da[r];
                for (int k = 0; k < D; ++k) {
                    gW[(size_t)r * D + k] += da[r] * xv[k];
                    dx[(size_t)q * D + k] += m.W[(size_t)r * D + k] * da[r];
                }
                if (q1 >= 0)
                    for (int k = 0; k < H; ++k) {
                        gU1[(size_t)r * H + k] += da[r] * y[(size_t)q1 * H + k];
                        dh[(size_t)q1 * H + k] += m.U1[(size_t)r * H + k] * da[r];
                    }
                if (q2 >= 0)
                    for (int k = 0; k < H; ++k) {
                        gU2[(size_t)r * H + k] += da[r] * y[(size_t)q2 * H + k];
                        dh[(size_t)q2 * H + k] += m.U2[(size_t)r * H + k] * da[r];
                    }
            }
        }
    free(y); free(act); free(cs); free(dh); free(dS); free(da);
}

/*
 * One layer over a list of examples, each on its own: n examples of heights
 * hs[i] and widths ws[i], pixels concatenated in example order (x[N][D],
 * N = sum hs*ws), ndir directions with parameter blocks back to back in blk.
 * Output y[N][ndir*H] (direction d in columns [dH, dH+H)).  With dy
 * ([N][ndir*H]) also dx[N][D] and the gradients gblk (zeroed here).
 */
int oracle_md_layer(int n, const int* hs, const int* ws, int D, int H, int ndir, const double* x, const double* blk,
                    const double* dy, double* y, double* dx, double* gblk)
{
    const long pc = oracle_md_param_count(D, H);
    size_t N = 0;
    for (int i = 0; i < n; ++i) {
        if (hs[i] < 0 || ws[i] < 0) return 1;
        N += (size_t)hs[i] * ws[i];
    }
    if (dy) {
        memset(dx, 0, sizeof(double) * N * D);
        memset(gblk, 0, sizeof(double) * pc * ndir);
    }
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
        const size_t np = (size_t)hs[i] * ws[i];
        for (int d = 0; d < ndir; ++d) {
            double* yd = (double*)calloc(np * H, sizeof(double));
            oracle_md_forward(hs[i], ws[i], D, H, d, x + off * D, blk + pc * d, yd, NULL, NULL);
            for (size_t q = 0; q < np; ++q)
                for (int u = 0; u < H; ++u) y[(off + q) * ndir * H + (size_t)d * H + u] = yd[q * H + u];
            if (dy) {
                double* dyd = (double*)malloc(sizeof(double) * np * H);
                for (size_t q = 0; q < np; ++q)
                    for (int u = 0; u < H; ++u) dyd[q * H + u] = dy[(off + q) * ndir * H + (size_t)d * H + u];
                oracle_md_backward(hs[i], ws[i], D, H, d, x + off * D, blk + pc * d, dyd, dx + off * D,
                                   gblk + pc * d);
                free(dyd);
            }
            free(yd);
        }
        off += np;
    }
    return 0;
}
