// kla_chunk_bwd_noalloc: the backward pass with its scratch (the state at
// every chunk start and dL/dS at every chunk end) held in a fixed device
// array of this library, for callers that cannot allocate device memory.
//
// The array is file-scope and static: every GPU that loads the library holds
// its kNoAllocScratchBytes until the process exits.  In host code its name is
// only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress while the device is current, and that address is what
// the kernels receive.
#include <mutex>

#include "kla_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB

static __device__ __align__(256) float
    g_bwd_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device.  Outside a stream
// capture it is looked up on every call (so that an address from before a
// cudaDeviceReset, which unloads the module, is never reused) and kept;
// while `stream` is being captured the kept address is used, since the
// lookup may load the module, which a capture does not allow.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    } else if (!g_scratch_addr[dev]) {
        return cudaErrorStreamCaptureUnsupported;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kla_status kla_chunk_bwd_noalloc(
    const void* q, const void* k, const void* v, const float* log_alpha,
    const float* eta, float eps, const float* h0, const void* o_grad,
    const float* hT_grad, void* q_grad, void* k_grad, void* v_grad,
    float* log_alpha_grad, float* eta_grad, float* h0_grad, int B, int T,
    int H, int dk, int dv, int C, kla_dtype dtype, kla_step_rule rule,
    kla_stream_t stream) {
    // the argument checks of kla_chunk_bwd come first, then the size limit
    if (rule != KLA_STEP_KACZMARZ && rule != KLA_STEP_GIVEN)
        return KLA_ERR_INVALID_ARG;
    const kla::BwdArgs a{q, k, v, log_alpha, eta, eps, 0, h0, o_grad, hT_grad,
                         q_grad, k_grad, v_grad, log_alpha_grad, eta_grad,
                         h0_grad, nullptr, nullptr, B, T, H, dk, dv, C, dtype};
    kla_status st = kla::check_chunk_bwd_args(a);
    if (st != KLA_OK) return st;
    size_t need = 0;
    st = kla_chunk_bwd_workspace_size(B, T, H, dk, dv, C, &need);
    if (st != KLA_OK) return st;
    if (need > kNoAllocScratchBytes) return KLA_ERR_UNSUPPORTED_SHAPE;
    void* ws = nullptr;
    if (need > 0 &&
        scratch_address(reinterpret_cast<cudaStream_t>(stream), &ws) !=
            cudaSuccess)
        return KLA_ERR_CUDA;
    // Nothing in the array has to start at zero: every element the kernels
    // read is written earlier in the same call.
    return kla_chunk_bwd(q, k, v, log_alpha, eta, eps, h0, o_grad, hT_grad,
                         q_grad, k_grad, v_grad, log_alpha_grad, eta_grad,
                         h0_grad, B, T, H, dk, dv, C, dtype, rule, ws,
                         kNoAllocScratchBytes, stream);
}
