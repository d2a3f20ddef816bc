// noalloc.cu -- lstm_bwd_noalloc: the backward pass of one layer without any
// device allocation by the caller or the library.
//
// Some callers cannot call cudaMalloc: a host framework whose memory pool
// owns the device memory and forbids allocations from outside it, or a
// real-time loop that must not allocate once it has started.  lstm_bwd needs
// a transient scratch buffer (the recurrent kernel's exchange of partial
// products between CTAs, then the split-K partial sums of the gradient
// products).  This entry point takes that scratch from one fixed array in
// the library's own device memory instead of from the caller.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds LSTM_NOALLOC_SCRATCH_BYTES for it until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and keeps it for later calls on that device.  The
// plan's device must be the current device.  A cudaDeviceReset destroys the
// array together with the context; the kept address is then stale, so no call
// may follow a reset in the same process.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[LSTM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on device `dev`, which must be the current device (looked up
// once per device).
lstm_status noalloc_scratch(int dev, void** out)
{
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return LSTM_ERR_CUDA;
    if (cur != dev) return LSTM_ERR_INVALID_ARG;     // the plan's tables live on another device
    if (dev < 0 || dev >= kMaxDevices) return LSTM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return LSTM_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return LSTM_OK;
}

}  // namespace

extern "C" lstm_status lstm_bwd_noalloc(const lstm_plan* plan, const lstm_layer_shape* shape,
                                        const lstm_layer_params* params, const void* x_packed,
                                        const float* y_packed, void* workspace, const float* dy_packed,
                                        float* dx_packed, const lstm_layer_grads* grads, void* stream)
{
    if (!plan || !shape) return LSTM_ERR_INVALID_ARG;
    const size_t need = lstm_scratch_bytes(plan, shape);
    if (need == 0) return LSTM_ERR_INVALID_ARG;
    if (need > (size_t)LSTM_NOALLOC_SCRATCH_BYTES) return LSTM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    lstm_status st = noalloc_scratch(plan->p.device, &scratch);
    if (st != LSTM_OK) return st;
    // Nothing in the array has to start at zero: every scratch byte lstm_bwd
    // reads was written earlier in the same call.
    return lstm_bwd(plan, shape, params, x_packed, y_packed, workspace, dy_packed, dx_packed, grads,
                    scratch, stream);
}
