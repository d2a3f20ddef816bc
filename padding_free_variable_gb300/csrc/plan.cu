// plan.cu -- the packing plan (host) and the pack / unpack gather kernels.
//
// "No Padding Please", Sec. V-A and Appendix B (Algorithm 1): examples are
// ordered, tiled into the packed tensor, and their original indices are kept
// so that unpacking can extract each example's activations.  In one
// dimension the tiling is a stable sort by decreasing length and a
// time-major layout: the rows of step t are the first bs[t] sorted
// sequences, so each step runs only the sequences still active.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <vector>

#include "common.cuh"

namespace lstm {

// One thread moves one 16-byte vector of a row.  Pack reads the source row
// named by row_src (zero-fills padding rows); unpack writes it.
__global__ void pack_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                 const int32_t* __restrict__ row_src, int64_t rows, int vecs_per_row,
                                 int unpack)
{
    const int64_t total = rows * (int64_t)vecs_per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / vecs_per_row;
        const int v = (int)(i - row * vecs_per_row);
        const int32_t s = __ldg(row_src + row);
        if (!unpack) {
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (s >= 0) val = __ldg(src + (int64_t)s * vecs_per_row + v);
            dst[i] = val;
        } else if (s >= 0) {
            dst[(int64_t)s * vecs_per_row + v] = __ldg(src + i);
        }
    }
}

lstm_status launch_pack(const Plan& p, const void* src, int width, int elem_bytes, void* dst,
                        bool unpack, cudaStream_t s)
{
    const int64_t rowbytes = (int64_t)width * elem_bytes;
    const int vecs = (int)(rowbytes / 16);
    const int64_t total = p.rows * vecs;
    if (total == 0) return LSTM_OK;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)p.num_sms * 8;
    if (blocks > cap) blocks = cap;
    trace_begin(p, unpack ? K_UNPACK : K_PACK, s);
    // segment and window plans unpack through their own map (frames that several segments
    // read are written back by the one segment that owns them)
    const int32_t* map = unpack && p.d_row_dst ? p.d_row_dst : p.d_row_src;
    pack_rows_kernel<<<(unsigned)blocks, threads, 0, s>>>((const uint4*)src, (uint4*)dst, map, p.rows, vecs,
                                                          unpack ? 1 : 0);
    trace_end(p, unpack ? K_UNPACK : K_PACK, s, 1);
    return cudaGetLastError() == cudaSuccess ? LSTM_OK : LSTM_ERR_CUDA;
}

void tracer_begin(Tracer* t, int kind, cudaStream_t s)
{
    if (!t || !t->enabled || kind < 0) return;     // kind < 0: counted, not timed (inside another kind)
    if (t->npending == t->cap) {
        int ncap = t->cap ? 2 * t->cap : 64;
        Tracer::Rec* n = (Tracer::Rec*)realloc(t->pending, sizeof(Tracer::Rec) * ncap);
        if (!n) return;
        t->pending = n;
        t->cap = ncap;
    }
    Tracer::Rec& r = t->pending[t->npending];
    r.kind = kind;
    if (cudaEventCreate(&r.a) != cudaSuccess) return;
    if (cudaEventCreate(&r.b) != cudaSuccess) { cudaEventDestroy(r.a); return; }
    cudaEventRecord(r.a, s);
    ++t->npending;
}

void tracer_end(Tracer* t, int kind, cudaStream_t s, int kernels)
{
    if (!t) return;
    t->launches += kernels;
    if (!t->enabled || t->npending == 0 || kind < 0) return;
    Tracer::Rec& r = t->pending[t->npending - 1];
    if (r.kind == kind) cudaEventRecord(r.b, s);
}

void trace_begin(const Plan& p, int kind, cudaStream_t s) { tracer_begin(p.tracer, kind, s); }

void trace_end(const Plan& p, int kind, cudaStream_t s, int kernels) { tracer_end(p.tracer, kind, s, kernels); }

void tracer_flush(Tracer* t)
{
    for (int i = 0; i < t->npending; ++i) {
        Tracer::Rec& r = t->pending[i];
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
            t->ms[r.kind] += ms;
            t->calls[r.kind] += 1;
        } else {
            cudaGetLastError();   // an unmatched bracket: drop the record, leave no error behind
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    t->npending = 0;
}

static void free_plan(Plan& p)
{
    if (p.tracer) {
        tracer_flush(p.tracer);
        free(p.tracer->pending);
        delete p.tracer;
    }
    free(p.h_bs); free(p.h_off); free(p.h_perm); free(p.h_len); free(p.h_cstart);
    cudaFree(p.d_bs); cudaFree(p.d_off); cudaFree(p.d_perm); cudaFree(p.d_len);
    cudaFree(p.d_row_src); cudaFree(p.d_prev_fwd); cudaFree(p.d_prev_rev); cudaFree(p.d_row_slot);
    cudaFree(p.d_row_dst);
    cudaFree(p.d_flags); cudaFree(p.d_status);
    p = Plan();
}

template <typename T>
static cudaError_t upload(T** dptr, const T* host, size_t n)
{
    size_t bytes = sizeof(T) * (n > 0 ? n : 1);
    cudaError_t e = cudaMalloc((void**)dptr, bytes);
    if (e != cudaSuccess) return e;
    if (n > 0) e = cudaMemcpy(*dptr, host, sizeof(T) * n, cudaMemcpyHostToDevice);
    return e;
}

// Host tables of a plan.  Fills whichever outputs are non-null.
static lstm_status compute_tables(const int32_t* lengths, int32_t B, bool padded, int32_t* T_out,
                                  int64_t* rows_out, int64_t* frames_out, int32_t* bs, int32_t* off,
                                  int32_t* perm, int32_t* slot_len, int32_t* cstart, int32_t* row_src,
                                  int32_t* prev_fwd, int32_t* prev_rev)
{
    if (!lengths || B < 1) return LSTM_ERR_INVALID_ARG;
    int64_t frames = 0;
    int32_t T = 0;
    for (int32_t b = 0; b < B; ++b) {
        if (lengths[b] < 0) return LSTM_ERR_INVALID_ARG;
        frames += lengths[b];
        T = std::max(T, lengths[b]);
    }
    const int64_t rows = padded ? (int64_t)B * T : frames;
    if (rows > INT32_MAX || frames > INT32_MAX) return LSTM_ERR_INVALID_ARG;
    if (T_out) *T_out = T;
    if (rows_out) *rows_out = rows;
    if (frames_out) *frames_out = frames;
    if (!bs && !off && !perm && !slot_len && !cstart && !row_src && !prev_fwd && !prev_rev) return LSTM_OK;

    std::vector<int32_t> cst(B + 1), order(B), len(B), nb(T + 1), of(T + 1);
    cst[0] = 0;
    for (int32_t b = 0; b < B; ++b) cst[b + 1] = cst[b] + lengths[b];
    std::iota(order.begin(), order.end(), 0);
    if (!padded)   // longest first; equal lengths keep the caller's order
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return lengths[a] > lengths[b]; });
    for (int32_t j = 0; j < B; ++j) len[j] = lengths[order[j]];
    for (int32_t t = 0; t < T; ++t) {
        int32_t n = 0;
        if (padded) n = B;
        else
            while (n < B && len[n] > t) ++n;
        nb[t] = n;
    }
    of[0] = 0;
    for (int32_t t = 0; t < T; ++t) of[t + 1] = of[t] + nb[t];
    if (bs) std::copy(nb.begin(), nb.begin() + T, bs);
    if (off) std::copy(of.begin(), of.end(), off);
    if (perm) std::copy(order.begin(), order.end(), perm);
    if (slot_len) std::copy(len.begin(), len.end(), slot_len);
    if (cstart) std::copy(cst.begin(), cst.end(), cstart);
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < nb[t]; ++j) {
            const int64_t r = (int64_t)of[t] + j;
            if (row_src) row_src[r] = (t < len[j]) ? cst[order[j]] + t : -1;
            if (prev_fwd) prev_fwd[r] = (t >= 1) ? of[t - 1] + j : -1;
            if (prev_rev) prev_rev[r] = (t + 1 < T && j < nb[t + 1]) ? of[t + 1] + j : -1;
        }
    }
    return LSTM_OK;
}

// Frame map of a plan whose units are pieces of the caller's sequences (segments, windows):
// unit u covers caller frames src_start[u] .. + length - 1; unpack writes back only its first
// own_len[u] frames; the caller's tensors have `frames` rows.
struct FrameMap {
    const int32_t* src_start = nullptr;
    const int32_t* own_len = nullptr;
    int64_t frames = 0;
};

static lstm_status create_plan(const int32_t* lengths, int32_t B, bool padded, lstm_plan** out,
                               const FrameMap* fm = nullptr)
{
    if (!out) return LSTM_ERR_INVALID_ARG;
    *out = nullptr;
    int32_t T = 0;
    int64_t rows = 0, frames = 0;
    lstm_status st = compute_tables(lengths, B, padded, &T, &rows, &frames, nullptr, nullptr, nullptr,
                                    nullptr, nullptr, nullptr, nullptr, nullptr);
    if (st != LSTM_OK) return st;
    if (fm) frames = fm->frames;

    lstm_plan* hp = new lstm_plan();
    Plan& p = hp->p;
    p.B = B; p.T = T; p.rows = rows; p.frames = frames; p.padded = padded;
    p.tracer = new Tracer();
    if (cudaGetDevice(&p.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess) {
        delete p.tracer;
        delete hp;
        return LSTM_ERR_CUDA;
    }
    p.h_bs = (int32_t*)malloc(sizeof(int32_t) * (T + 1));
    p.h_off = (int32_t*)malloc(sizeof(int32_t) * (T + 1));
    p.h_perm = (int32_t*)malloc(sizeof(int32_t) * B);
    p.h_len = (int32_t*)malloc(sizeof(int32_t) * B);
    p.h_cstart = (int32_t*)malloc(sizeof(int32_t) * (B + 1));
    std::vector<int32_t> row_src(rows), prev_fwd(rows), prev_rev(rows), row_dst;
    compute_tables(lengths, B, padded, nullptr, nullptr, nullptr, p.h_bs, p.h_off, p.h_perm, p.h_len,
                   p.h_cstart, row_src.data(), prev_fwd.data(), prev_rev.data());
    if (fm) {   // rows read (and write back) the caller's frames through the frame map
        row_dst.resize(rows);
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < p.h_bs[t]; ++j) {
                const int64_t r = (int64_t)p.h_off[t] + j;
                const int u = p.h_perm[j];
                row_src[r] = fm->src_start[u] + t;
                row_dst[r] = t < fm->own_len[u] ? fm->src_start[u] + t : -1;
            }
    }
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = upload(&p.d_bs, p.h_bs, (size_t)T);
    if (e == cudaSuccess) e = upload(&p.d_off, p.h_off, (size_t)T + 1);
    if (e == cudaSuccess) e = upload(&p.d_perm, p.h_perm, (size_t)B);
    if (e == cudaSuccess) e = upload(&p.d_len, p.h_len, (size_t)B);
    if (e == cudaSuccess) e = upload(&p.d_row_src, row_src.data(), (size_t)rows);
    if (e == cudaSuccess && fm) e = upload(&p.d_row_dst, row_dst.data(), (size_t)rows);
    if (e == cudaSuccess) e = upload(&p.d_prev_fwd, prev_fwd.data(), (size_t)rows);
    if (e == cudaSuccess) e = upload(&p.d_prev_rev, prev_rev.data(), (size_t)rows);
    {   // sorted slot of each packed row (row off[t] + j holds slot j)
        std::vector<int32_t> row_slot(rows);
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < p.h_bs[t]; ++j) row_slot[(size_t)p.h_off[t] + j] = j;
        if (e == cudaSuccess) e = upload(&p.d_row_slot, row_slot.data(), (size_t)rows);
    }
    if (e == cudaSuccess) e = cudaMalloc((void**)&p.d_flags, sizeof(unsigned) * 2 * kMaxCtasPerDir);
    if (e == cudaSuccess) e = cudaMemset(p.d_flags, 0, sizeof(unsigned) * 2 * kMaxCtasPerDir);
    if (e == cudaSuccess) e = cudaMalloc((void**)&p.d_status, sizeof(DeviceStatus));
    if (e == cudaSuccess) e = cudaMemset(p.d_status, 0, sizeof(DeviceStatus));
    if (e != cudaSuccess) {
        free_plan(p);
        delete hp;
        return LSTM_ERR_CUDA;
    }
    *out = hp;
    return LSTM_OK;
}

// Segments of RETURNN-style chunking (RETURNN paper, Sec. 4: sequences cut into possibly
// overlapping segments of constant length, each then trained as a sequence of its own):
// sequence b yields segments starting at 0, step, 2 step, ... of min(chunk, L_b - start)
// frames, up to the first segment that reaches the sequence's end; an empty sequence yields
// one empty segment.  Segment u owns (unpacks) its frames up to the next segment's start.
static lstm_status make_segments(const int32_t* lengths, int32_t B, int32_t chunk, int32_t step,
                                 std::vector<int32_t>* seq, std::vector<int32_t>* start, std::vector<int32_t>* len,
                                 std::vector<int32_t>* own, int64_t* frames)
{
    if (!lengths || B < 1 || chunk < 1 || step < 1 || step > chunk) return LSTM_ERR_INVALID_ARG;
    int64_t f = 0;
    for (int32_t b = 0; b < B; ++b) {
        if (lengths[b] < 0) return LSTM_ERR_INVALID_ARG;
        const int32_t L = lengths[b];
        for (int32_t s0 = 0;; s0 += step) {
            const int32_t e = std::min(s0 + chunk, L);
            seq->push_back(b);
            start->push_back(s0);
            len->push_back(std::max(0, e - s0));
            own->push_back(e == L ? std::max(0, e - s0) : step);
            if (e >= L) break;
        }
        f += L;
    }
    if (f > INT32_MAX || seq->size() > (size_t)INT32_MAX) return LSTM_ERR_INVALID_ARG;
    *frames = f;
    return LSTM_OK;
}

}  // namespace lstm

using lstm::Plan;

extern "C" {

lstm_status lstm_plan_create(const int32_t* lengths_host, int32_t B, lstm_plan** out)
{
    return lstm::create_plan(lengths_host, B, false, out);
}

lstm_status lstm_plan_create_padded(const int32_t* lengths_host, int32_t B, lstm_plan** out)
{
    return lstm::create_plan(lengths_host, B, true, out);
}

lstm_status lstm_segments_host(const int32_t* lengths_host, int32_t B, int32_t chunk, int32_t step,
                               int32_t* num_segments, int32_t* seg_seq, int32_t* seg_start, int32_t* seg_len,
                               int32_t capacity)
{
    std::vector<int32_t> seq, start, len, own;
    int64_t frames = 0;
    const lstm_status st = lstm::make_segments(lengths_host, B, chunk, step, &seq, &start, &len, &own, &frames);
    if (st != LSTM_OK) return st;
    const int32_t n = (int32_t)seq.size();
    if (num_segments) *num_segments = n;
    if (!seg_seq && !seg_start && !seg_len) return LSTM_OK;
    if (capacity < n) return LSTM_ERR_INVALID_ARG;
    for (int32_t u = 0; u < n; ++u) {
        if (seg_seq) seg_seq[u] = seq[u];
        if (seg_start) seg_start[u] = start[u];
        if (seg_len) seg_len[u] = len[u];
    }
    return LSTM_OK;
}

lstm_status lstm_plan_create_segments(const int32_t* lengths_host, int32_t B, int32_t chunk, int32_t step,
                                      lstm_plan** out)
{
    std::vector<int32_t> seq, start, len, own;
    int64_t frames = 0;
    lstm_status st = lstm::make_segments(lengths_host, B, chunk, step, &seq, &start, &len, &own, &frames);
    if (st != LSTM_OK) return st;
    std::vector<int32_t> cst(B + 1, 0), src(seq.size());
    for (int32_t b = 0; b < B; ++b) cst[b + 1] = cst[b] + lengths_host[b];
    for (size_t u = 0; u < seq.size(); ++u) src[u] = cst[seq[u]] + start[u];
    lstm::FrameMap fm;
    fm.src_start = src.data(); fm.own_len = own.data(); fm.frames = frames;
    return lstm::create_plan(len.data(), (int32_t)len.size(), false, out, &fm);
}

lstm_status lstm_plan_create_window(const int32_t* lengths_host, int32_t B, int32_t start, int32_t width,
                                    lstm_plan** out)
{
    if (!lengths_host || B < 1 || start < 0 || width < 1) return LSTM_ERR_INVALID_ARG;
    std::vector<int32_t> len(B), src(B);
    int64_t frames = 0;
    for (int32_t b = 0; b < B; ++b) {
        if (lengths_host[b] < 0) return LSTM_ERR_INVALID_ARG;
        len[b] = std::max(0, std::min(lengths_host[b] - start, width));
        src[b] = (int32_t)frames + std::min(start, lengths_host[b]);
        frames += lengths_host[b];
    }
    if (frames > INT32_MAX) return LSTM_ERR_INVALID_ARG;
    lstm::FrameMap fm;
    fm.src_start = src.data(); fm.own_len = len.data(); fm.frames = frames;
    return lstm::create_plan(len.data(), B, false, out, &fm);
}

lstm_status lstm_form_batches(const int32_t* lengths_host, int32_t n, int64_t budget, int32_t budget_kind,
                              int32_t* batch_of, int32_t* num_batches)
{
    if (n < 0 || (n > 0 && (!lengths_host || !batch_of)) || budget < 1 || (budget_kind != 0 && budget_kind != 1))
        return LSTM_ERR_INVALID_ARG;
    int32_t b = 0, count = 0, longest = 0;
    int64_t sum = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t L = lengths_host[i];
        if (L < 0) return LSTM_ERR_INVALID_ARG;
        const int64_t size = budget_kind == 0 ? sum + L : (int64_t)(count + 1) * std::max(longest, L);
        if (count > 0 && size > budget) { ++b; count = 0; sum = 0; longest = 0; }
        batch_of[i] = b;
        ++count;
        sum += L;
        longest = std::max(longest, L);
    }
    if (num_batches) *num_batches = n > 0 ? b + 1 : 0;
    return LSTM_OK;
}

lstm_status lstm_plan_dims(const int32_t* lengths_host, int32_t B, int32_t padded, int32_t* steps,
                           int64_t* rows)
{
    return lstm::compute_tables(lengths_host, B, padded != 0, steps, rows, nullptr, nullptr, nullptr,
                                nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
}

lstm_status lstm_plan_compute_host(const int32_t* lengths_host, int32_t B, int32_t padded,
                                   int32_t* batch_sizes, int32_t* offsets, int32_t* perm,
                                   int32_t* slot_len, int32_t* row_src, int32_t* prev_fwd,
                                   int32_t* prev_rev)
{
    return lstm::compute_tables(lengths_host, B, padded != 0, nullptr, nullptr, nullptr, batch_sizes,
                                offsets, perm, slot_len, nullptr, row_src, prev_fwd, prev_rev);
}

lstm_status lstm_plan_destroy(lstm_plan* plan)
{
    if (!plan) return LSTM_OK;
    lstm::free_plan(plan->p);
    delete plan;
    return LSTM_OK;
}

lstm_status lstm_plan_info(const lstm_plan* plan, int64_t* rows, int32_t* steps, int32_t* batch,
                           int64_t* frames)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    if (rows) *rows = plan->p.rows;
    if (steps) *steps = plan->p.T;
    if (batch) *batch = plan->p.B;
    if (frames) *frames = plan->p.frames;
    return LSTM_OK;
}

lstm_status lstm_plan_tables(const lstm_plan* plan, const int32_t** batch_sizes,
                             const int32_t** offsets, const int32_t** perm, const int32_t** slot_len)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    if (batch_sizes) *batch_sizes = plan->p.h_bs;
    if (offsets) *offsets = plan->p.h_off;
    if (perm) *perm = plan->p.h_perm;
    if (slot_len) *slot_len = plan->p.h_len;
    return LSTM_OK;
}

lstm_status lstm_plan_set_wait_limit(lstm_plan* plan, uint64_t nanoseconds)
{
    if (!plan || nanoseconds == 0) return LSTM_ERR_INVALID_ARG;
    plan->p.wait_limit_ns = nanoseconds;
    return LSTM_OK;
}

lstm_status lstm_plan_enable_timing(lstm_plan* plan, int32_t enable)
{
    if (!plan || !plan->p.tracer) return LSTM_ERR_INVALID_ARG;
    lstm::Tracer* t = plan->p.tracer;
    lstm::tracer_flush(t);
    for (int k = 0; k < lstm::K_NUM; ++k) { t->ms[k] = 0.0; t->calls[k] = 0; }
    t->enabled = enable != 0;
    return LSTM_OK;
}

lstm_status lstm_plan_read_timing(lstm_plan* plan, double* ms, int64_t* calls)
{
    if (!plan || !plan->p.tracer) return LSTM_ERR_INVALID_ARG;
    lstm::Tracer* t = plan->p.tracer;
    lstm::tracer_flush(t);
    for (int k = 0; k < lstm::K_NUM; ++k) {
        if (ms) ms[k] = t->ms[k];
        if (calls) calls[k] = t->calls[k];
    }
    return LSTM_OK;
}

int64_t lstm_plan_launch_count(const lstm_plan* plan)
{
    return (plan && plan->p.tracer) ? (int64_t)plan->p.tracer->launches : -1;
}

lstm_status lstm_plan_recurrent_config(const lstm_plan* plan, int32_t pass, int32_t* kind,
                                       int32_t* ctas_per_direction, int32_t* product, int32_t* variant)
{
    if (!plan || pass < 0 || pass > 1) return LSTM_ERR_INVALID_ARG;
    if (kind) *kind = plan->p.last_rec_kind[pass];
    if (ctas_per_direction) *ctas_per_direction = plan->p.last_rec_ctas[pass];
    if (product) *product = plan->p.last_rec_mma[pass];
    if (variant) *variant = plan->p.last_rec_variant[pass];
    return LSTM_OK;
}

lstm_status lstm_plan_recurrent_groups(const lstm_plan* plan, int32_t pass, int32_t* groups, int32_t* slots_per_group)
{
    if (!plan || pass < 0 || pass > 1) return LSTM_ERR_INVALID_ARG;
    if (groups) *groups = plan->p.last_rec_groups[pass];
    if (slots_per_group) *slots_per_group = plan->p.last_rec_grp_rows[pass];
    return LSTM_OK;
}

lstm_status lstm_debug_wide_recurrence(lstm_plan* plan, int32_t mode)
{
    if (!plan || mode < -1 || mode > 2) return LSTM_ERR_INVALID_ARG;
    plan->p.wide_mode = mode;
    return LSTM_OK;
}

lstm_status lstm_debug_wide_stages(lstm_plan* plan, int32_t max_stages, int32_t* used_fwd, int32_t* used_bwd)
{
    if (!plan || max_stages < -1 || max_stages == 1 || max_stages > 64) return LSTM_ERR_INVALID_ARG;
    if (max_stages >= 0) plan->p.wide_stages = max_stages;
    if (used_fwd) *used_fwd = plan->p.last_rec_stages[0];
    if (used_bwd) *used_bwd = plan->p.last_rec_stages[1];
    return LSTM_OK;
}

lstm_status lstm_debug_sequence_groups(lstm_plan* plan, int32_t slots)
{
    if (!plan || slots < 0 || slots > 128) return LSTM_ERR_INVALID_ARG;
    plan->p.forced_group_rows = slots;
    return LSTM_OK;
}

lstm_status lstm_debug_trace_steps(lstm_plan* plan, int64_t* device_buffer, int32_t steps)
{
    if (!plan || steps < 0 || (steps > 0 && !device_buffer)) return LSTM_ERR_INVALID_ARG;
    plan->p.d_trace = steps > 0 ? (long long*)device_buffer : nullptr;
    plan->p.trace_steps = steps;
    return LSTM_OK;
}

lstm_status lstm_plan_set_gemm_engine(lstm_plan* plan, int32_t engine)
{
    if (!plan || engine < 0 || engine > 1) return LSTM_ERR_INVALID_ARG;
    plan->p.gemm_engine = engine;
    return LSTM_OK;
}

lstm_status lstm_plan_set_ctas_per_direction(lstm_plan* plan, int32_t ctas)
{
    if (!plan || ctas < 0) return LSTM_ERR_INVALID_ARG;
    plan->p.forced_ctas = ctas;
    return LSTM_OK;
}

lstm_status lstm_debug_skip_arrival(lstm_plan* plan, int32_t cta)
{
    if (!plan || cta < -1) return LSTM_ERR_INVALID_ARG;
    plan->p.debug_skip_cta = cta;
    return LSTM_OK;
}

lstm_status lstm_debug_cluster_variant(lstm_plan* plan, int32_t variant)
{
    if (!plan || variant < -1 || variant > 3) return LSTM_ERR_INVALID_ARG;
    plan->p.forced_variant = variant;
    return LSTM_OK;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

lstm_status lstm_pack(const lstm_plan* plan, const void* x_cat, int32_t width, int32_t elem_bytes,
                      void* x_packed, void* stream)
{
    if (!plan || width < 1 || (elem_bytes != 2 && elem_bytes != 4)) return LSTM_ERR_INVALID_ARG;
    if (((int64_t)width * elem_bytes) % 16 != 0) return LSTM_ERR_INVALID_ARG;
    if (plan->p.rows > 0 && (!x_packed || !aligned16(x_packed))) return LSTM_ERR_INVALID_ARG;
    if (plan->p.frames > 0 && (!x_cat || !aligned16(x_cat))) return LSTM_ERR_INVALID_ARG;
    return lstm::launch_pack(plan->p, x_cat, width, elem_bytes, x_packed, false, (cudaStream_t)stream);
}

lstm_status lstm_unpack(const lstm_plan* plan, const void* y_packed, int32_t width, int32_t elem_bytes,
                        void* y_cat, void* stream)
{
    if (!plan || width < 1 || (elem_bytes != 2 && elem_bytes != 4)) return LSTM_ERR_INVALID_ARG;
    if (((int64_t)width * elem_bytes) % 16 != 0) return LSTM_ERR_INVALID_ARG;
    if (plan->p.rows > 0 && (!y_packed || !aligned16(y_packed))) return LSTM_ERR_INVALID_ARG;
    if (plan->p.frames > 0 && (!y_cat || !aligned16(y_cat))) return LSTM_ERR_INVALID_ARG;
    return lstm::launch_pack(plan->p, y_packed, width, elem_bytes, y_cat, true, (cudaStream_t)stream);
}

lstm_status lstm_status_poll(lstm_plan* plan, void* stream)
{
    if (!plan) return LSTM_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LSTM_ERR_CUDA;
    lstm::DeviceStatus st;
    if (cudaMemcpy(&st, plan->p.d_status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LSTM_ERR_CUDA;
    if (st.word == 0) return LSTM_OK;
    if (cudaMemset(plan->p.d_status, 0, sizeof(st)) != cudaSuccess) return LSTM_ERR_CUDA;
    return (lstm_status)(unsigned)(st.word & 0xffffffffu);
}

const char* lstm_status_string(lstm_status s)
{
    switch (s) {
    case LSTM_OK: return "ok";
    case LSTM_ERR_INVALID_ARG: return "invalid argument";
    case LSTM_ERR_UNSUPPORTED: return "unsupported shape or device";
    case LSTM_ERR_CUDA: return "CUDA call failed";
    case LSTM_ERR_TIMEOUT: return "step barrier wait exceeded the plan's limit";
    case LSTM_ERR_BOUNDS: return "index out of range in a kernel";
    }
    return "unknown status";
}

}  // extern "C"
