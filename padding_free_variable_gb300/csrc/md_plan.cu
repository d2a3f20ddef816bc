// md_plan.cu -- host side of the 2-D (MDLSTM) path: example-packing onto a
// canvas and the wavefront schedule of the cells.
//
// "No Padding Please: Efficient Neural Handwriting Recognition", Sec. V-A and
// App. B (Algorithm 1): the examples are bucketed by height, each bucket fills
// rows greedily with the widest example that still fits, and the rows are
// tiled with one separator pixel between neighbouring examples and between
// rows; Sec. IV-A: after the input-skewing trick (row r shifted by r pixels),
// the cells of one skewed column depend only on the previous column, so a
// column is one parallel step.
//
// On the GPU nothing of the canvas is materialised.  The cells of every
// example and scan direction are stored in wavefront order -- the skewed
// canvas read column by column, without its padding, separator and corner
// cells -- and each cell carries the indices of its two predecessor cells
// (-1 where the mask would block the input: the example's border).  Two
// schedules of the same cells:
//  * canvas (the page's packing): a cell runs at its skewed canvas column,
//    y'0 + x'0 + ys + xs for an example placed at (y'0, x'0) of the canvas
//    scanned from the direction's corner;
//  * diagonal: every example starts at step 0 and a cell runs at its own
//    anti-diagonal ys + xs, so the step count is the longest example's
//    h + w - 1 instead of the canvas's height + width - 1.
// Both compute every pixel from the same predecessors: results are identical.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "md_plan.cuh"

using lstm::MdPlan;

namespace {

template <typename T>
T* host_copy(const std::vector<T>& v)
{
    T* p = new (std::nothrow) T[v.size() > 0 ? v.size() : 1];
    if (p && !v.empty()) std::memcpy(p, v.data(), v.size() * sizeof(T));
    return p;
}

// Algorithm 1 ("No Padding Please", App. B): placement (y0, x0) of every example; -1 for
// examples without pixels.  Buckets in descending height; in a bucket, the widest example
// that fits beside the row's examples and a separator (ties: lower index), an empty row
// taking the widest left even when it is wider than the row; a bucket's last row closes
// when the bucket runs out.
struct Packing {
    std::vector<int32_t> y0, x0;
    int32_t height = 0, width = 0, rows = 0;
    std::vector<int32_t> order;      // examples in packing order (row by row, left to right)
};

Packing pack_examples(const int32_t* hs, const int32_t* ws, int n, int row_width)
{
    Packing pk;
    pk.y0.assign(n, -1);
    pk.x0.assign(n, -1);
    std::vector<int> live;
    int widest = 0;
    for (int i = 0; i < n; ++i)
        if (hs[i] > 0 && ws[i] > 0) {
            live.push_back(i);
            widest = std::max(widest, (int)ws[i]);
        }
    const int W = row_width > 0 ? row_width : widest;
    std::vector<int> heights;
    for (int i : live) heights.push_back(hs[i]);
    std::sort(heights.begin(), heights.end(), [](int a, int b) { return a > b; });
    heights.erase(std::unique(heights.begin(), heights.end()), heights.end());
    std::vector<std::vector<int>> rows;
    for (int hgt : heights) {
        std::vector<int> bucket;                       // widest first, then lower index
        for (int i : live)
            if (hs[i] == hgt) bucket.push_back(i);
        std::stable_sort(bucket.begin(), bucket.end(), [&](int a, int b) { return ws[a] > ws[b]; });
        std::vector<int> row;
        int used = 0;
        while (!bucket.empty()) {
            const int room = W - used - (row.empty() ? 0 : 1);
            int pick = -1;
            for (size_t k = 0; k < bucket.size(); ++k)
                if (ws[bucket[k]] <= room) { pick = (int)k; break; }
            if (pick < 0 && row.empty()) pick = 0;
            if (pick >= 0) {
                const int e = bucket[pick];
                bucket.erase(bucket.begin() + pick);
                used += ws[e] + (row.empty() ? 0 : 1);
                row.push_back(e);
            } else {
                rows.push_back(row);
                row.clear();
                used = 0;
            }
        }
        if (!row.empty()) rows.push_back(row);
    }
    int top = 0;
    for (size_t r = 0; r < rows.size(); ++r) {
        if (r > 0) top += 1;                           // separator row
        int left = 0;
        for (size_t k = 0; k < rows[r].size(); ++k) {
            const int e = rows[r][k];
            if (k > 0) left += 1;                      // separator column
            pk.y0[e] = top;
            pk.x0[e] = left;
            left += ws[e];
            pk.order.push_back(e);
        }
        pk.width = std::max(pk.width, left);
        top += hs[rows[r][0]];
    }
    pk.height = top;
    pk.rows = (int)rows.size();
    return pk;
}

void free_tracer(MdPlan& p)
{
    if (!p.tracer) return;
    lstm::tracer_flush(p.tracer);
    free(p.tracer->pending);
    delete p.tracer;
    p.tracer = nullptr;
}

void free_host(MdPlan& p)
{
    delete[] p.h_y0; delete[] p.h_x0; delete[] p.h_pix_off; delete[] p.h_step_off;
    p.h_y0 = p.h_x0 = nullptr;
    p.h_pix_off = nullptr;
    p.h_step_off = nullptr;
}

void free_device(MdPlan& p)
{
    cudaFree(p.d_step_off); cudaFree(p.d_src); cudaFree(p.d_pred1); cudaFree(p.d_pred2);
    cudaFree(p.d_succ1); cudaFree(p.d_succ2); cudaFree(p.d_ctr); cudaFree(p.d_status);
    p.d_step_off = nullptr;
    p.d_src = p.d_pred1 = p.d_pred2 = p.d_succ1 = p.d_succ2 = nullptr;
    p.d_ctr = nullptr;
    p.d_status = nullptr;
}

// the schedule's tables on the host: step offsets [ndir][steps+1] and, per cell, its pixel
// and its predecessor / successor cells
struct Tables {
    std::vector<int64_t> step_off;
    std::vector<int32_t> src, pred1, pred2, succ1, succ2;
};

void build_tables(const MdPlan& p, const int32_t* hs, const int32_t* ws, const Packing& pk, Tables& t)
{
    const int64_t N = p.pixels;
    const int S = p.steps;
    t.step_off.assign((size_t)p.ndir * (S + 1), 0);
    t.src.assign((size_t)p.cells, 0);
    t.pred1.assign((size_t)p.cells, -1);
    t.pred2.assign((size_t)p.cells, -1);
    t.succ1.assign((size_t)p.cells, -1);
    t.succ2.assign((size_t)p.cells, -1);
    std::vector<int32_t> cell_of((size_t)N);
    for (int d = 0; d < p.ndir; ++d) {
        const int fx = d & 1, fy = (d >> 1) & 1;
        int64_t* off = t.step_off.data() + (size_t)d * (S + 1);
        auto origin = [&](int e) -> int {             // the example's first step
            if (p.schedule != 0) return 0;
            const int yy = fy ? p.canvas_h - pk.y0[e] - hs[e] : pk.y0[e];
            const int xx = fx ? p.canvas_w - pk.x0[e] - ws[e] : pk.x0[e];
            return yy + xx;
        };
        // cells per step: the example's anti-diagonal lengths
        std::vector<int64_t> cnt((size_t)S, 0);
        for (int e : pk.order) {
            const int o = origin(e), h = hs[e], w = ws[e];
            for (int dd = 0; dd <= h + w - 2; ++dd)
                cnt[(size_t)(o + dd)] += std::min(dd, h - 1) - std::max(0, dd - w + 1) + 1;
        }
        off[0] = (int64_t)d * N;
        for (int k = 0; k < S; ++k) off[k + 1] = off[k] + cnt[(size_t)k];
        std::vector<int64_t> cur(off, off + S);
        for (int e : pk.order) {
            const int o = origin(e), h = hs[e], w = ws[e];
            const int64_t base = p.h_pix_off[e];
            for (int dd = 0; dd <= h + w - 2; ++dd)
                for (int ys = std::max(0, dd - w + 1); ys <= std::min(dd, h - 1); ++ys) {
                    const int xs = dd - ys;
                    const int y = fy ? h - 1 - ys : ys, x = fx ? w - 1 - xs : xs;
                    const int64_t c = cur[(size_t)(o + dd)]++;
                    t.src[(size_t)c] = (int32_t)(base + (int64_t)y * w + x);
                    cell_of[(size_t)(base + (int64_t)y * w + x)] = (int32_t)c;
                }
        }
        for (int e : pk.order) {
            const int h = hs[e], w = ws[e];
            const int64_t base = p.h_pix_off[e];
            auto cell = [&](int ys, int xs) -> int32_t {
                const int y = fy ? h - 1 - ys : ys, x = fx ? w - 1 - xs : xs;
                return cell_of[(size_t)(base + (int64_t)y * w + x)];
            };
            for (int ys = 0; ys < h; ++ys)
                for (int xs = 0; xs < w; ++xs) {
                    const int32_t c = cell(ys, xs);
                    if (ys > 0) {
                        t.pred1[(size_t)c] = cell(ys - 1, xs);
                        t.succ1[(size_t)cell(ys - 1, xs)] = c;
                    }
                    if (xs > 0) {
                        t.pred2[(size_t)c] = cell(ys, xs - 1);
                        t.succ2[(size_t)cell(ys, xs - 1)] = c;
                    }
                }
        }
    }
}

template <typename T>
bool upload(T** dst, const std::vector<T>& v)
{
    if (cudaMalloc(dst, sizeof(T) * (v.empty() ? 1 : v.size())) != cudaSuccess) return false;
    return v.empty() || cudaMemcpy(*dst, v.data(), sizeof(T) * v.size(), cudaMemcpyHostToDevice) == cudaSuccess;
}

lstm_status create(const int32_t* heights, const int32_t* widths, int32_t n, int32_t row_width, int32_t ndir,
                   int32_t schedule, bool device, Tables* keep, lstm_md_plan** out)
{
    if (!out || n < 0 || (n > 0 && (!heights || !widths)) || ndir < 1 || ndir > 4 || schedule < 0 ||
        schedule > 1 || row_width < 0)
        return LSTM_ERR_INVALID_ARG;
    *out = nullptr;
    int64_t N = 0;
    for (int i = 0; i < n; ++i) {
        if (heights[i] < 0 || widths[i] < 0) return LSTM_ERR_INVALID_ARG;
        N += (int64_t)heights[i] * widths[i];
    }
    if (N * ndir >= ((int64_t)1 << 31)) return LSTM_ERR_UNSUPPORTED;   // cell indices are int32
    lstm_md_plan* plan = new (std::nothrow) lstm_md_plan;
    if (!plan) return LSTM_ERR_CUDA;
    MdPlan& p = plan->p;
    p.n = n; p.ndir = ndir; p.schedule = schedule;
    p.pixels = N; p.cells = N * ndir;
    const Packing pk = pack_examples(heights, widths, n, row_width);
    p.canvas_h = pk.height; p.canvas_w = pk.width; p.rows = pk.rows;
    int steps = 0;
    for (int i = 0; i < n; ++i)
        if (heights[i] > 0 && widths[i] > 0) steps = std::max(steps, heights[i] + widths[i] - 1);
    if (schedule == 0 && N > 0) steps = p.canvas_h + p.canvas_w - 1;
    p.steps = steps;
    std::vector<int64_t> pix_off((size_t)n + 1, 0);
    for (int i = 0; i < n; ++i) pix_off[(size_t)i + 1] = pix_off[(size_t)i] + (int64_t)heights[i] * widths[i];
    p.h_y0 = host_copy(pk.y0);
    p.h_x0 = host_copy(pk.x0);
    p.h_pix_off = host_copy(pix_off);
    Tables t;
    build_tables(p, heights, widths, pk, t);
    p.h_step_off = host_copy(t.step_off);
    p.tracer = new (std::nothrow) lstm::Tracer;
    if (!p.h_y0 || !p.h_x0 || !p.h_pix_off || !p.h_step_off || !p.tracer) {
        free_tracer(p);
        free_host(p);
        delete plan;
        return LSTM_ERR_CUDA;
    }
    if (device) {
        if (cudaGetDevice(&p.device) != cudaSuccess ||
            cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess ||
            !upload(&p.d_step_off, t.step_off) || !upload(&p.d_src, t.src) || !upload(&p.d_pred1, t.pred1) ||
            !upload(&p.d_pred2, t.pred2) || !upload(&p.d_succ1, t.succ1) || !upload(&p.d_succ2, t.succ2) ||
            cudaMalloc(&p.d_ctr, sizeof(unsigned) * 4) != cudaSuccess ||
            cudaMalloc(&p.d_status, sizeof(lstm::DeviceStatus)) != cudaSuccess ||
            cudaMemset(p.d_status, 0, sizeof(lstm::DeviceStatus)) != cudaSuccess) {
            cudaGetLastError();
            free_device(p);
            free_host(p);
            free_tracer(p);
            delete plan;
            return LSTM_ERR_CUDA;
        }
    }
    if (keep) *keep = std::move(t);
    *out = plan;
    return LSTM_OK;
}

}  // namespace

extern "C" {

lstm_status lstm_md_plan_create(const int32_t* heights, const int32_t* widths, int32_t n, int32_t row_width,
                                int32_t num_directions, int32_t schedule, lstm_md_plan** out)
{
    return create(heights, widths, n, row_width, num_directions, schedule, true, nullptr, out);
}

lstm_status lstm_md_plan_compute_host(const int32_t* heights, const int32_t* widths, int32_t n, int32_t row_width,
                                      int32_t num_directions, int32_t schedule, int32_t* info, int32_t* y0,
                                      int32_t* x0, int64_t* step_off, int32_t* src, int32_t* pred1, int32_t* pred2,
                                      int32_t* succ1, int32_t* succ2)
{
    lstm_md_plan* plan = nullptr;
    Tables t;
    const lstm_status st = create(heights, widths, n, row_width, num_directions, schedule, false, &t, &plan);
    if (st != LSTM_OK) return st;
    const MdPlan& p = plan->p;
    if (info) {
        info[0] = p.steps; info[1] = p.canvas_h; info[2] = p.canvas_w; info[3] = p.rows;
    }
    if (y0 && n > 0) std::memcpy(y0, p.h_y0, sizeof(int32_t) * n);
    if (x0 && n > 0) std::memcpy(x0, p.h_x0, sizeof(int32_t) * n);
    if (step_off) std::memcpy(step_off, t.step_off.data(), sizeof(int64_t) * t.step_off.size());
    auto put = [](int32_t* dst, const std::vector<int32_t>& v) {
        if (dst && !v.empty()) std::memcpy(dst, v.data(), sizeof(int32_t) * v.size());
    };
    put(src, t.src); put(pred1, t.pred1); put(pred2, t.pred2); put(succ1, t.succ1); put(succ2, t.succ2);
    free_host(plan->p);
    free_tracer(plan->p);
    delete plan;
    return LSTM_OK;
}

void lstm_md_plan_destroy(lstm_md_plan* plan)
{
    if (!plan) return;
    free_tracer(plan->p);
    free_device(plan->p);
    free_host(plan->p);
    delete plan;
}

lstm_status lstm_md_plan_info(const lstm_md_plan* plan, int64_t* pixels, int32_t* steps, int32_t* canvas_height,
                              int32_t* canvas_width, int32_t* rows)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    const MdPlan& p = plan->p;
    if (pixels) *pixels = p.pixels;
    if (steps) *steps = p.steps;
    if (canvas_height) *canvas_height = p.canvas_h;
    if (canvas_width) *canvas_width = p.canvas_w;
    if (rows) *rows = p.rows;
    return LSTM_OK;
}

lstm_status lstm_md_plan_placement(const lstm_md_plan* plan, int32_t* y0, int32_t* x0)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    const MdPlan& p = plan->p;
    if (y0 && p.n > 0) std::memcpy(y0, p.h_y0, sizeof(int32_t) * p.n);
    if (x0 && p.n > 0) std::memcpy(x0, p.h_x0, sizeof(int32_t) * p.n);
    return LSTM_OK;
}

lstm_status lstm_md_plan_step_cells(const lstm_md_plan* plan, int64_t* step_off)
{
    if (!plan || !step_off) return LSTM_ERR_INVALID_ARG;
    const MdPlan& p = plan->p;
    std::memcpy(step_off, p.h_step_off, sizeof(int64_t) * (size_t)p.ndir * (p.steps + 1));
    return LSTM_OK;
}

lstm_status lstm_md_plan_set_wait_limit(lstm_md_plan* plan, uint64_t ns)
{
    if (!plan || ns == 0) return LSTM_ERR_INVALID_ARG;
    plan->p.wait_limit_ns = ns;
    return LSTM_OK;
}

lstm_status lstm_md_debug_skip_arrival(lstm_md_plan* plan, int32_t cta)
{
    if (!plan || cta < -1) return LSTM_ERR_INVALID_ARG;
    plan->p.debug_skip_cta = cta;
    return LSTM_OK;
}

lstm_status lstm_md_status_poll(lstm_md_plan* plan, void* stream)
{
    if (!plan || !plan->p.d_status) return LSTM_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LSTM_ERR_CUDA;
    lstm::DeviceStatus st;
    if (cudaMemcpy(&st, plan->p.d_status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return LSTM_ERR_CUDA;
    if (cudaMemset(plan->p.d_status, 0, sizeof(st)) != cudaSuccess) return LSTM_ERR_CUDA;
    return (lstm_status)(uint32_t)(st.word & 0xffffffffu);
}

int64_t lstm_md_plan_launch_count(const lstm_md_plan* plan)
{
    return plan && plan->p.tracer ? (int64_t)plan->p.tracer->launches : -1;
}

lstm_status lstm_md_plan_enable_timing(lstm_md_plan* plan, int32_t enable)
{
    if (!plan || !plan->p.tracer) return LSTM_ERR_INVALID_ARG;
    lstm::Tracer* t = plan->p.tracer;
    lstm::tracer_flush(t);
    for (int k = 0; k < lstm::K_NUM; ++k) { t->ms[k] = 0.0; t->calls[k] = 0; }
    t->enabled = enable != 0;
    return LSTM_OK;
}

lstm_status lstm_md_plan_read_timing(lstm_md_plan* plan, double* ms, int64_t* calls)
{
    if (!plan || !plan->p.tracer) return LSTM_ERR_INVALID_ARG;
    lstm::Tracer* t = plan->p.tracer;
    lstm::tracer_flush(t);
    for (int k = 0; k < lstm::MD_NUM; ++k) {
        if (ms) ms[k] = t->ms[k];
        if (calls) calls[k] = t->calls[k];
    }
    return LSTM_OK;
}

}  // extern "C"
