// Internal launchers of libkla.so (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "kla.h"

namespace kla {

// Element load/store helpers for the two I/O types.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) {
    return x;
}
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(
    float x) {
    return __float2bfloat16_rn(x);
}

struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* eta;
    float eps;
    int gdn;           // 1: beta = eta (learned step), 0: Kaczmarz step
    const float* h0;   // may be null
    void* o;
    float* hT;         // may be null
    int B, T, H, dk, dv, C;
    kla_dtype dtype;
    // may be null: the state at the start of every chunk, fp32
    // [B, H, ceil(T / C), dk, dv] (the tensor-core kernel takes exactly one
    // of o and ckpt)
    float* ckpt = nullptr;
    // may be null: separate write keys [B, T, H, dk]; null means the write
    // key is k
    const void* kw = nullptr;
    // tensor-core kernel only: v is a zeroed [1, 64, H, dv] tile standing
    // for an all-zero V (every other load falls outside it and reads zeros)
    bool v_zero = false;
    // two-kernel path only, may be null: the pre-pass also writes the
    // backward's per-chunk records (bwdrec layout) here
    uint8_t* bwd_rec = nullptr;
};

struct PrecondArgs {
    const void* k;      // [B, T, H, dk]
    const float* A0;    // [B, H, dk] or null (zero)
    void* kw;           // [B, T, H, dk] write keys
    float* AT;          // [B, H, dk] or null
    int B, T, H, dk;
    float x, delta;
    kla_dtype dtype;
};

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* eta;
    float eps;
    int gdn;
    const float* h0;     // may be null
    const void* dout;    // like o
    const float* dhT;    // may be null (zero)
    void* dq;            // like q
    void* dk_;           // like k
    void* dv_;           // like v
    float* dlog_alpha;   // [B, T, H]
    float* deta;         // [B, T, H]
    float* dh0;          // may be null
    float* ckpt;         // workspace: state at every chunk start
    float* dsck;         // workspace: dL/dS at every chunk end
    int B, T, H, dk, dv, C;
    kla_dtype dtype;
    uint8_t* rec = nullptr;   // workspace: per-chunk records (tensor-core path)
    uint8_t* fwd_rec = nullptr;   // workspace: the forward pre-pass's records
    bool rec_ready = false;   // rec written by the checkpointing forward
};

// Per-chunk record of the backward's tensor-core kernels (bytes): T = A^{-1}
// and P (bf16, 64 x 64, rows of 64, zeros above the diagonal), the
// cumulative log decay g (natural log), beta and ||k||^2 (fp32).
namespace bwdrec {
constexpr int T_OFF = 0, P_OFF = 8192, G_OFF = 16384, B_OFF = 16640,
              N_OFF = 16896, BYTES = 17152;
}  // namespace bwdrec

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* eta;
    float eps;
    int gdn;
    float* S;
    void* o;
    int N, H, dk, dv;
    kla_dtype dtype;
    const void* kw = nullptr;   // separate write keys [N, H, dk] or null
};

// Each returns cudaSuccess or the launch error.  Shapes are validated by the
// caller (kla_api.cu); a launcher returning cudaErrorInvalidValue means the
// shape has no instantiation.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_simt(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_tc(const FwdArgs& a, cudaStream_t stream);
bool chunk_tc_eligible(const FwdArgs& a);
// Two-kernel tensor-core forward (chunk-parallel pre-pass, then the state
// pass): bf16, dk = dv = 128, C = 64, no separate write keys.  The workspace
// (chunk_tc2_workspace_bytes(B, T, H) bytes, 16-byte aligned) holds the
// pre-pass records (chunk_tc2_record_bytes(B, T, H) bytes), then one ready
// flag per record and the pre-pass's work counters.  Takes exactly one of
// a.o and a.ckpt.
bool chunk_tc2_eligible(const FwdArgs& a);
size_t chunk_tc2_record_bytes(int B, int T, int H);
size_t chunk_tc2_workspace_bytes(int B, int T, int H);
cudaError_t launch_chunk_tc2(const FwdArgs& a, void* workspace,
                             cudaStream_t stream);
// Its two launches apart: the pre-pass writes the records of a.q, a.k and
// the gates (a.v, a.o, a.h0 unused) into the workspace ws, each followed by
// its ready flag; the state pass reads them.  Two state passes may share
// one pre-pass when they differ only in v, h0, o, hT (the second may start
// at a later sequence of the first: rec and ready then point there).
// ready: the flags of rec's records when the state pass follows the
// pre-pass (or another state pass that follows it) directly on this
// stream; it is then launched as a programmatic dependent and reads each
// record as soon as its flag is up.  Null: the records are complete (stream
// order), and the launch is a plain one.  state_ctas: CTAs of the state
// passes launched with flags (the pre-pass hands its last chunks to the SMs
// they leave free); 0 when none is.
cudaError_t launch_prep_tc2(const FwdArgs& a, void* ws, cudaStream_t stream,
                            int state_ctas);
cudaError_t launch_state_tc2(const FwdArgs& a, const void* rec,
                             const unsigned int* ready, cudaStream_t stream);
// The flags of the records in a workspace of chunk_tc2_workspace_bytes(B,
// T, H) bytes, and the CTAs of one state pass over B sequences of H heads.
const unsigned int* chunk_tc2_ready(const void* ws, int B, int T, int H);
int chunk_tc2_state_ctas(int B, int H);
cudaError_t read_and_clear_fault2(unsigned int* word);
// One CTA of the state-pass kernel whose producer issues no copy and whose
// waits give up after 1 ms: it takes the kernel's abort path and sets the
// fault word.
cudaError_t launch_state_selftest(cudaStream_t stream);
// Backward pass: the checkpointing forward, the reverse state-gradient
// recurrence and the per-chunk gradients (CUDA cores, fp32).
cudaError_t launch_chunk_bwd(const BwdArgs& a, cudaStream_t stream);
// Write keys: the cluster kernel (any supported dk, no workspace) ...
cudaError_t launch_precond_keys(const PrecondArgs& a, cudaStream_t stream);
// ... and the chunked form (dk = 128, k and kw 16-byte aligned), which takes
// precond_chunked_bytes of fp32 workspace (the per-chunk sums of k^2 and A
// before each chunk; none when T <= 64) and fills every SM.
bool precond_chunked_eligible(const PrecondArgs& a);
size_t precond_chunked_bytes(int B, int T, int H);
cudaError_t launch_precond_chunked(const PrecondArgs& a, void* workspace,
                                   cudaStream_t stream);
// Workspace of kla_chunk_bwd: the fp32 states at every chunk start and
// dL/dS at every chunk end (chunk_bwd_state_floats each), then, for dk = 128
// and C = 64, the tensor-core kernels' per-chunk records.
size_t chunk_bwd_state_floats(int B, int T, int H, int dk, int dv, int C);
size_t chunk_bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int C);
// Every argument check of kla_chunk_bwd except those on the workspace and
// the step rule (a.ckpt, a.dsck are not looked at).
kla_status check_chunk_bwd_args(const BwdArgs& a);
// SM count of the current device (cached per device).
int device_sm_count();

// cuTensorMapEncodeTiled from the driver (looked up once); false if absent.
bool get_encoder();
// Tensor map of a [B, T, H, 128] bf16 tensor with 128-byte swizzle and boxes
// of 64 features x 1 head x 64 tokens x 1 batch (zero fill out of range).
bool make_map(CUtensorMap* m, const void* base, int B, int T, int H);

// Device fault word of the tensor-core kernels (bounded waits that gave up).
// read_and_clear_fault synchronises the stream first.
cudaError_t read_and_clear_fault(cudaStream_t stream, unsigned int* word);

}  // namespace kla
