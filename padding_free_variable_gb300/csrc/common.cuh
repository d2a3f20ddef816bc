// common.cuh -- internals shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "lstm_packed.h"

namespace lstm {

constexpr int kMaxCtasPerDir = 160;     // > 152 SMs; one flag per CTA
constexpr int kRecThreads = 256;        // block size of the recurrent kernels

// Device status word layout (one int64 per plan):
//   low 32 bits  lstm_status of the first failure (0 = none)
//   high 32 bits detail (CTA index and step for a timeout)
struct DeviceStatus {
    unsigned long long word;
};

// Kinds of work the tracer times (matches lstm_kernel_kind in the header).
enum KernelKind {
    K_PACK = 0, K_UNPACK, K_GEMM_IN, K_REC_FWD, K_REC_BWD, K_GEMM_DX, K_GEMM_DW, K_GEMM_DR, K_CONVERT, K_NUM
};

// Optional CUDA-event timing of every library launch, and a launch counter.
struct Tracer {
    bool enabled = false;
    long long launches = 0;                 // kernels launched through the plan
    struct Rec { int kind; cudaEvent_t a, b; };
    Rec* pending = nullptr;
    int npending = 0, cap = 0;
    double ms[K_NUM] = {};
    long long calls[K_NUM] = {};
};

struct Plan {
    int32_t B = 0;            // sequences
    int32_t T = 0;            // steps (longest length)
    int64_t rows = 0;         // rows of a packed tensor
    int64_t frames = 0;       // sum of lengths
    bool padded = false;
    uint64_t wait_limit_ns = 2000000000ull;
    int32_t debug_skip_cta = -1;
    int32_t forced_ctas = 0;        // 0 = automatic
    int32_t forced_variant = -1;    // cluster kernels: -1 automatic, else bit 0 bulk exchange, bit 1 TMA tiles
    int32_t forced_group_rows = 0;  // cluster kernels: sorted slots per sequence group (0 = automatic)
    int32_t wide_mode = -1;         // bf16 layers wider than a cluster: -1 automatic, 0 per-step launches,
                                    // 1 the persistent kernel where it applies
    int32_t wide_stages = 0;        // persistent wide kernels: cap on the operand-ring depth (0 = none)
    int32_t gemm_engine = 0;        // 0 = tensor cores for bf16 operands, 1 = CUDA cores
    int device = 0;
    int num_sms = 0;
    // host tables
    int32_t* h_bs = nullptr;        // [T]
    int32_t* h_off = nullptr;       // [T+1]
    int32_t* h_perm = nullptr;      // [B]  caller index of slot j
    int32_t* h_len = nullptr;       // [B]  length of slot j
    int32_t* h_cstart = nullptr;    // [B+1] caller-order frame offsets
    // device tables
    int32_t* d_bs = nullptr;
    int32_t* d_off = nullptr;
    int32_t* d_perm = nullptr;
    int32_t* d_len = nullptr;
    int32_t* d_row_src = nullptr;   // [rows] caller-order frame of packed row (-1 = padding)
    int32_t* d_prev_fwd = nullptr;  // [rows] row holding h_{t-1} for the forward direction (-1 none)
    int32_t* d_prev_rev = nullptr;  // [rows] row holding the reverse direction's previous state
    int32_t* d_row_slot = nullptr;  // [rows] sorted slot j of packed row (row off[t] + j)
    int32_t* d_row_dst = nullptr;   // segment / window plans: [rows] caller frame unpack writes (-1 none)
    unsigned* d_flags = nullptr;    // [2 * kMaxCtasPerDir] step counters
    DeviceStatus* d_status = nullptr;
    Tracer* tracer = nullptr;       // owned; mutable through const plans
    long long* d_trace = nullptr;   // caller's phase-stamp buffer (not owned)
    int32_t trace_steps = 0;
    // launch configuration of the last recurrent launch: [0] forward, [1] backward
    mutable int32_t last_rec_kind[2] = {0, 0};   // 0 none, 1 grid kernel, 2 cluster kernel
    mutable int32_t last_rec_ctas[2] = {0, 0};   // CTAs per direction
    mutable int32_t last_rec_mma[2] = {0, 0};    // 0 CUDA cores, 1 mma.sync, 2 tcgen05
    mutable int32_t last_rec_variant[2] = {0, 0}; // cluster kernels: bit 0 bulk exchange, bit 1 TMA tiles
    mutable int32_t last_rec_groups[2] = {0, 0};  // cluster kernels: sequence groups
    mutable int32_t last_rec_grp_rows[2] = {0, 0}; // cluster kernels: sorted slots per group
    mutable int32_t last_rec_stages[2] = {0, 0};   // persistent wide kernels: operand-ring depth
};

// Bracket a launch sequence of `kind`; `kernels` = launches it issued.  A
// negative kind counts the launches without timing them (a sequence inside
// another kind's bracket).
void trace_begin(const Plan& p, int kind, cudaStream_t s);
void trace_end(const Plan& p, int kind, cudaStream_t s, int kernels);
// The same on a tracer of its own (the 2-D plan's); flush = wait for and add up the pending records.
void tracer_begin(Tracer* t, int kind, cudaStream_t s);
void tracer_end(Tracer* t, int kind, cudaStream_t s, int kernels);
void tracer_flush(Tracer* t);

// ---------------------------------------------------------------- helpers

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ float bf16_round(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Record the first failure; later ones are dropped.
__device__ __forceinline__ void record_failure(DeviceStatus* st, int code, unsigned detail) {
    unsigned long long w = ((unsigned long long)detail << 32) | (unsigned)code;
    atomicCAS(&st->word, 0ull, w);
}

__device__ __forceinline__ bool failure_recorded(const DeviceStatus* st) {
    return ld_relaxed_gpu_u64(&st->word) != 0ull;
}

// ---------------------------------------------------------------- launchers (defined per .cu)

lstm_status launch_pack(const Plan& p, const void* src, int width, int elem_bytes, void* dst,
                        bool unpack, cudaStream_t s);

}  // namespace lstm

struct lstm_plan {
    lstm::Plan p;
};

#define LSTM_CUDA_TRY(expr)                                 \
    do {                                                    \
        cudaError_t _e = (expr);                            \
        if (_e != cudaSuccess) return LSTM_ERR_CUDA;        \
    } while (0)
