// recurrent.cuh -- launch interface of the persistent recurrent kernels.
#pragma once

#include "common.cuh"

namespace lstm {

struct RecArgs {
    int T, B, H, ndir, G, Umax, JC;
    int bf16, padded, debug_skip_cta;
    unsigned long long wait_limit_ns;
    const int32_t* bs;        // [T] active rows per step
    const int32_t* off;       // [T+1] first row of each step
    const int32_t* slot_len;  // [B] length of the sequence in slot j
    const int32_t* perm;      // [B] caller index of slot j
    float* ga;                // [rows][ndir*4H] gate pre-activations -> gates -> gate errors
    const void* R;            // [ndir][4H][H]
    const float* peep;        // [ndir][3][H]
    float* y;                 // [rows][ndir*H]
    __nv_bfloat16* y_lo;      // optional bf16 copy of y
    float* cbuf;              // [rows][ndir*H] cell states
    float* h_n;               // [ndir][B][H] caller order, optional
    float* c_n;
    const float* dy;          // backward: [rows][ndir*H]
    // initial states ([ndir][B][H] fp32, caller order; NULL = zero).  The product R h0 is
    // folded into the first step's pre-activations before the recurrent kernels run, so
    // they read h0 only as the final state of an empty sequence.
    const float* h0;
    const float* c0;
    const float* dh_n;        // backward: dL/dh_n from outside (NULL = zero)
    const float* dc_n;        // backward: dL/dc_n from outside (NULL = zero)
    float* dc0;               // backward: dL/dc0, written at each sequence's first step (NULL: not wanted)
    float* db;                // backward: [ndir][4H]
    float* dpeep;             // backward: [ndir][3][H]
    float* part;              // backward: [2][ndir][B][G][H] partial R^T da exchange
    unsigned* flags;
    DeviceStatus* status;
    long long* trace;         // optional [ndir][trace_steps][8] clock64 stamps of each direction's CTA 0
    int trace_steps;
    int tables_in_smem;
    int mma_mw, mma_kw;       // forward tensor-core product: warps along rows and along k
    int tm_chains, tm_acol;   // cluster kernels: TMEM accumulator chains, first column of the R operand
    int tma_pre;              // cluster kernels: the cell's operands arrive as TMA tiles (at off_red)
    int grp_rows, ngroups;    // cluster kernels: sorted slots per sequence group, groups (one cluster each per direction)
    // dynamic shared-memory layout (byte offsets)
    int off_h, off_red, off_acc, off_state, off_contrib, off_sums, off_tab, off_peep;
};

struct RecConfig {
    int G = 0;          // CTAs per direction
    int Umax = 0;       // units per CTA
    int JC = 0;         // rows per staged chunk
    int tables = 0;     // step tables copied to shared memory
    int mma = 0;        // 1: warp-level tensor-core product (mma.sync), 0: CUDA cores
    int mma_mw = 1, mma_kw = 1;
    int cluster = 0;    // 1: one thread-block cluster per direction (recurrent_cluster.cu)
    int chains = 0;     // cluster kernels: accumulator chains (issuing warps per M tile)
    int acol = 0;       // cluster kernels: TMEM column of the R operand
    int bulk = 0;       // cluster forward kernel: 1 = bulk-copy exchange into a double-buffered operand
    int tma_pre = 0;    // cluster forward kernel: 1 = pre-activation tiles loaded by TMA
    int grp_rows = 0;   // cluster kernels: sorted slots per sequence group
    int ngroups = 1;    // cluster kernels: sequence groups (one cluster per direction each)
    size_t smem = 0;    // dynamic shared memory bytes
};

// Launch configuration of the recurrent kernels.  The per-step product runs
// on warp-level tensor cores when the CTA's fragments fit and the plan's
// engine allows it (gemm_engine 0), otherwise on CUDA cores.
lstm_status rec_configure(const Plan& p, int H, int ndir, bool bf16, bool bwd, int forced_G,
                          RecConfig* out);
lstm_status rec_launch(const Plan& p, const RecConfig& c, RecArgs a, bool bwd, cudaStream_t s);

// Cluster-resident forward kernel: configured when one direction's R fits a
// cluster of H/32 CTAs (<= 16) with its operand buffers; false otherwise.
// The batch's sorted slots are cut into sequence groups, one cluster per
// (direction, group).
bool rec_cluster_fwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* layout);
lstm_status rec_cluster_fwd_launch(const Plan& p, const RecConfig& c, RecArgs a, cudaStream_t s);

// Cluster-resident BPTT kernel (and the db / dpeep sums after it, which need
// rec_cluster_bwd_sum_floats floats of scratch).
bool rec_cluster_bwd_configure(const Plan& p, int H, int ndir, bool bf16, RecConfig* out, RecArgs* layout);
size_t rec_cluster_bwd_sum_floats(int H, int ndir);
lstm_status rec_cluster_bwd_launch(const Plan& p, const RecConfig& c, RecArgs a, float* sum_scratch,
                                   cudaStream_t s);

// Persistent kernels of bf16 layers wider than a cluster (recurrent_wide.cu): H/16 CTAs per
// direction, each holding its slice of R (forward) or R^T (backward) in shared memory; the
// previous step's operand (bf16 h, or bf16 gate errors) is exchanged through a double-
// buffered global array read back with TMA; a bounded grid barrier per step.
struct WideArgs {
    int T, B, H, ndir, NC;                 // NC: CTAs per direction (set by the launchers)
    int stages;                            // operand-ring depth (set by the launchers)
    int padded;
    const int32_t* bs;
    const int32_t* off;
    const int32_t* len;
    const int32_t* perm;
    float* ga;                             // [rows][ndir*4H] pre-activations -> gates -> gate errors
    const float* peep;
    float* y;                              // forward
    __nv_bfloat16* y_lo;                   // forward, optional
    float* cbuf;
    float* h_n;                            // forward, optional
    float* c_n;
    const float* dy;                       // backward
    const float* h0;                       // initial states and final-state errors (optional)
    const float* c0;
    const float* dh_n;
    const float* dc_n;
    float* dc0;
    __nv_bfloat16* xbuf;                   // forward [ndir][2][B][H], backward [ndir][2][B][4H] bf16
    unsigned* ctr;                         // [ndir] step counters (set by the launchers)
    DeviceStatus* status;
    unsigned long long wait_limit_ns;
    long long* trace;                      // optional phase stamps of CTA 0 of each direction (as RecArgs)
    int trace_steps;
    int debug_skip_cta;                    // test hook: this CTA of direction 0 never publishes step 0 (-1 off)
};

bool rec_wide_supported(const Plan& p, int H, int ndir, bool bf16);
size_t rec_wide_xbuf_bytes(const Plan& p, int H, int ndir, bool bwd);
lstm_status rec_wide_fwd_launch(const Plan& p, WideArgs a, const void* R, cudaStream_t s);
// RT: R^T as [ndir][H][4H] bf16.  Runs the db / dpeep sums after the kernel.
lstm_status rec_wide_bwd_launch(const Plan& p, WideArgs a, const void* RT, float* sum_scratch, float* db,
                                float* dpeep, cudaStream_t s);

// Floats of the backward kernel's partial-product exchange buffer.
size_t rec_bwd_part_floats(const Plan& p, int H, int ndir, bool bf16, int forced_G);

// db and dpeep of a layer from its gate errors (ga) and cell states, summed in
// a fixed row-chunk order (bitwise repeatable); sum_scratch holds
// rec_cluster_bwd_sum_floats(H, ndir) floats.
lstm_status param_sums_launch(const Plan& p, const float* ga, const float* cbuf, int H, int ndir, float* db,
                              float* dpeep, float* sum_scratch, cudaStream_t s, const float* c0 = nullptr);

}  // namespace lstm
