// C ABI of libkla.so: argument validation and kernel dispatch.
// Every check runs on the host before any launch; no exception crosses the
// interface.  See include/kla.h for the contract of each entry point.
#include <cmath>
#include <cstdint>

#include "kla_internal.cuh"

namespace {

bool supported_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool supported_chunk(int c) { return c == 16 || c == 32 || c == 64; }

bool aligned(const void* p, size_t n) {
    return (reinterpret_cast<uintptr_t>(p) % n) == 0;
}

kla_status from_cuda(cudaError_t e) {
    return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

// A buffer of the call: start and length in bytes (null or empty: none).
struct Span {
    const void* p;
    size_t n;
};

// True when the byte ranges of a and b share at least one byte.
bool overlap(Span a, Span b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// True when any written span overlaps any read span, or two written spans
// overlap each other.
template <size_t NI, size_t NO>
bool any_overlap(const Span (&ins)[NI], const Span (&outs)[NO]) {
    for (size_t i = 0; i < NO; ++i) {
        for (size_t j = 0; j < NI; ++j)
            if (overlap(outs[i], ins[j])) return true;
        for (size_t j = i + 1; j < NO; ++j)
            if (overlap(outs[i], outs[j])) return true;
    }
    return false;
}

}  // namespace

// Whether KLA_ALGO_AUTO takes the two-kernel tensor-core path where it is
// eligible (else the fused kernel): the faster of the two on GB300.
constexpr bool kAutoTwoKernel = true;

// Bytes of workspace the two-kernel tensor-core path needs for these sizes
// (0 when the shape or the algorithm does not take that path).
static size_t fwd_workspace_bytes(int B, int T, int H, int dk, int dv, int C,
                                  kla_dtype dtype, kla_algo algo) {
    if (dtype != KLA_BF16 || dk != 128 || dv != 128 || C != 64) return 0;
    if (algo != KLA_ALGO_TC && !(algo == KLA_ALGO_AUTO && kAutoTwoKernel))
        return 0;
    return kla::chunk_tc2_workspace_bytes(B, T, H);
}

// Forward pass with optional separate write keys kw (null: the keys) and an
// optional caller workspace (null: stream-ordered scratch when needed).
static kla_status chunk_fwd_impl(const void* q, const void* k, const void* kw,
                                 const void* v, const float* log_alpha,
                                 const float* eta, float eps, const float* h0,
                                 void* o, float* hT, int B, int T, int H,
                                 int dk, int dv, int C, kla_dtype dtype,
                                 kla_algo algo, kla_step_rule rule,
                                 void* workspace, size_t workspace_bytes,
                                 kla_stream_t stream) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || C <= 0)
        return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_F32 && dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (algo != KLA_ALGO_AUTO && algo != KLA_ALGO_SIMT &&
        algo != KLA_ALGO_TC && algo != KLA_ALGO_TC_FUSED)
        return KLA_ERR_INVALID_ARG;
    if (rule != KLA_STEP_KACZMARZ && rule != KLA_STEP_GIVEN)
        return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return KLA_ERR_INVALID_ARG;
    if (!supported_dim(dk) || !supported_dim(dv) || !supported_chunk(C))
        return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H > 0x7fffffffLL) return KLA_ERR_UNSUPPORTED_SHAPE;

    const size_t elt = dtype == KLA_BF16 ? 2 : 4;
    const bool empty = (long long)B * H == 0;
    if (!empty && T > 0) {
        if (!q || !k || !v || !log_alpha || !eta || !o)
            return KLA_ERR_INVALID_ARG;
        if (!aligned(q, elt) || !aligned(k, elt) || !aligned(v, elt) ||
            !aligned(o, elt) || !aligned(log_alpha, 4) || !aligned(eta, 4) ||
            (kw && !aligned(kw, elt)))
            return KLA_ERR_INVALID_ARG;
        // o must not overlap any input or hT (hT may alias h0 exactly: the
        // state is read before it is written)
        const size_t tok = (size_t)B * T * H;
        const size_t st = sizeof(float) * (size_t)B * H * dk * dv;
        const Span ins[] = {{q, tok * dk * elt}, {k, tok * dk * elt},
                            {v, tok * dv * elt}, {log_alpha, tok * 4},
                            {eta, tok * 4}, {kw, tok * dk * elt}, {h0, st}};
        const Span outs[] = {{o, tok * dv * elt}};
        if (any_overlap(ins, outs) || overlap({o, tok * dv * elt}, {hT, st}))
            return KLA_ERR_INVALID_ARG;
        if (hT && (const void*)hT != (const void*)h0) {
            const Span ins2[] = {{q, tok * dk * elt}, {k, tok * dk * elt},
                                 {v, tok * dv * elt}, {log_alpha, tok * 4},
                                 {eta, tok * 4}, {kw, tok * dk * elt},
                                 {h0, st}};
            const Span outs2[] = {{hT, st}};
            if (any_overlap(ins2, outs2)) return KLA_ERR_INVALID_ARG;
        }
    }
    if ((h0 && !aligned(h0, 4)) || (hT && !aligned(hT, 4)))
        return KLA_ERR_INVALID_ARG;
    if (empty) return KLA_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (!hT) return KLA_OK;
        const size_t bytes = sizeof(float) * (size_t)B * H * dk * dv;
        if (h0 == hT) return KLA_OK;
        if (h0)
            return from_cuda(
                cudaMemcpyAsync(hT, h0, bytes, cudaMemcpyDeviceToDevice, s));
        return from_cuda(cudaMemsetAsync(hT, 0, bytes, s));
    }

    kla::FwdArgs a{q, k, v, log_alpha, eta, eps,
                   rule == KLA_STEP_GIVEN ? 1 : 0, h0, o, hT,
                   B, T, H, dk, dv, C, dtype};
    a.kw = kw;
    const bool tc2_ok = kla::chunk_tc2_eligible(a);
    const bool tc_ok = kla::chunk_tc_eligible(a);
    if ((algo == KLA_ALGO_TC || (algo == KLA_ALGO_AUTO && kAutoTwoKernel)) &&
        tc2_ok) {
        const size_t need = kla::chunk_tc2_workspace_bytes(B, T, H);
        if (workspace) {
            if (workspace_bytes < need || !aligned(workspace, 16))
                return KLA_ERR_INVALID_ARG;
            const Span bufs[] = {{q, (size_t)B * T * H * dk * 2},
                                 {k, (size_t)B * T * H * dk * 2},
                                 {v, (size_t)B * T * H * dv * 2},
                                 {o, (size_t)B * T * H * dv * 2},
                                 {log_alpha, (size_t)B * T * H * 4},
                                 {eta, (size_t)B * T * H * 4},
                                 {h0, sizeof(float) * B * H * dk * dv},
                                 {hT, sizeof(float) * B * H * dk * dv},
                                 {kw, (size_t)B * T * H * dk * 2}};
            const Span ws[] = {{workspace, need}};
            if (any_overlap(bufs, ws)) return KLA_ERR_INVALID_ARG;
            return from_cuda(kla::launch_chunk_tc2(a, workspace, s));
        }
        // stream-ordered scratch from the device's current memory pool
        void* scratch = nullptr;
        if (cudaMallocAsync(&scratch, need, s) != cudaSuccess)
            return KLA_ERR_CUDA;
        const cudaError_t e = kla::launch_chunk_tc2(a, scratch, s);
        const cudaError_t f = cudaFreeAsync(scratch, s);
        return from_cuda(e != cudaSuccess ? e : f);
    }
    if (algo == KLA_ALGO_TC || algo == KLA_ALGO_TC_FUSED) {
        if (!tc_ok) return KLA_ERR_UNSUPPORTED_SHAPE;
        return from_cuda(kla::launch_chunk_tc(a, s));
    }
    if (algo == KLA_ALGO_AUTO && tc_ok)
        return from_cuda(kla::launch_chunk_tc(a, s));
    return from_cuda(kla::launch_chunk_simt(a, s));
}

extern "C" kla_status kla_chunk_fwd_workspace_size(int B, int T, int H,
                                                   int dk, int dv, int C,
                                                   kla_dtype dtype,
                                                   kla_algo algo,
                                                   size_t* bytes) {
    if (!bytes || B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || C <= 0)
        return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_F32 && dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (algo != KLA_ALGO_AUTO && algo != KLA_ALGO_SIMT &&
        algo != KLA_ALGO_TC && algo != KLA_ALGO_TC_FUSED)
        return KLA_ERR_INVALID_ARG;
    if (!supported_dim(dk) || !supported_dim(dv) || !supported_chunk(C))
        return KLA_ERR_UNSUPPORTED_SHAPE;
    *bytes = fwd_workspace_bytes(B, T, H, dk, dv, C, dtype, algo);
    return KLA_OK;
}

extern "C" kla_status kla_chunk_fwd_ws(const void* q, const void* k,
                                       const void* v, const float* log_alpha,
                                       const float* eta, float eps,
                                       const float* h0, void* o, float* hT,
                                       int B, int T, int H, int dk, int dv,
                                       int C, kla_dtype dtype, kla_algo algo,
                                       kla_step_rule rule, void* workspace,
                                       size_t workspace_bytes,
                                       kla_stream_t stream) {
    if (!workspace && fwd_workspace_bytes(B, T, H, dk, dv, C, dtype, algo) &&
        (long long)B * H > 0 && T > 0)
        return KLA_ERR_INVALID_ARG;
    return chunk_fwd_impl(q, k, nullptr, v, log_alpha, eta, eps, h0, o, hT, B,
                          T, H, dk, dv, C, dtype, algo, rule, workspace,
                          workspace_bytes, stream);
}

extern "C" kla_status kla_chunk_fwd_ex(const void* q, const void* k,
                                       const void* v, const float* log_alpha,
                                       const float* eta, float eps,
                                       const float* h0, void* o, float* hT,
                                       int B, int T, int H, int dk, int dv,
                                       int C, kla_dtype dtype, kla_algo algo,
                                       kla_step_rule rule,
                                       kla_stream_t stream) {
    return chunk_fwd_impl(q, k, nullptr, v, log_alpha, eta, eps, h0, o, hT, B,
                          T, H, dk, dv, C, dtype, algo, rule, nullptr, 0,
                          stream);
}

extern "C" kla_status kla_chunk_fwd_kw(const void* q, const void* k,
                                       const void* k_write, const void* v,
                                       const float* log_alpha,
                                       const float* eta, float eps,
                                       const float* h0, void* o, float* hT,
                                       int B, int T, int H, int dk, int dv,
                                       int C, kla_dtype dtype,
                                       kla_step_rule rule,
                                       kla_stream_t stream) {
    return kla_chunk_fwd_kw_ex(q, k, k_write, v, log_alpha, eta, eps, h0, o,
                               hT, B, T, H, dk, dv, C, dtype, KLA_ALGO_AUTO,
                               rule, nullptr, 0, stream);
}

extern "C" kla_status kla_chunk_fwd_kw_ex(const void* q, const void* k,
                                          const void* k_write, const void* v,
                                          const float* log_alpha,
                                          const float* eta, float eps,
                                          const float* h0, void* o, float* hT,
                                          int B, int T, int H, int dk, int dv,
                                          int C, kla_dtype dtype,
                                          kla_algo algo, kla_step_rule rule,
                                          void* workspace,
                                          size_t workspace_bytes,
                                          kla_stream_t stream) {
    if (!k_write && (long long)B * H > 0 && T > 0) return KLA_ERR_INVALID_ARG;
    return chunk_fwd_impl(q, k, k_write, v, log_alpha, eta, eps, h0, o, hT, B,
                          T, H, dk, dv, C, dtype, algo, rule, workspace,
                          workspace_bytes, stream);
}

extern "C" kla_status kla_precond_keys_workspace_size(int B, int T, int H,
                                                      int dk, kla_dtype dtype,
                                                      size_t* bytes) {
    if (!bytes) return KLA_ERR_INVALID_ARG;
    *bytes = 0;
    if (B < 0 || T < 0 || H < 0 || dk <= 0) return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_F32 && dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (!supported_dim(dk)) return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H > 0x7fffffffLL) return KLA_ERR_UNSUPPORTED_SHAPE;
    if (dk == 128) *bytes = kla::precond_chunked_bytes(B, T, H);
    return KLA_OK;
}

extern "C" kla_status kla_precond_keys_ex(const void* k, const float* A0,
                                          void* k_write, float* AT, int B,
                                          int T, int H, int dk, float x,
                                          float delta, kla_dtype dtype,
                                          void* workspace,
                                          size_t workspace_bytes,
                                          kla_stream_t stream) {
    if (B < 0 || T < 0 || H < 0 || dk <= 0) return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_F32 && dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (!(x > 1.f) || !std::isfinite(x) || !(delta >= 0.f) ||
        !std::isfinite(delta))
        return KLA_ERR_INVALID_ARG;
    if (!supported_dim(dk)) return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H > 0x7fffffffLL) return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H == 0) return KLA_OK;
    const size_t elt = dtype == KLA_BF16 ? 2 : 4;
    if (T > 0 && (!k || !k_write || !aligned(k, elt) ||
                  !aligned(k_write, elt)))
        return KLA_ERR_INVALID_ARG;
    if ((A0 && !aligned(A0, 4)) || (AT && !aligned(AT, 4)))
        return KLA_ERR_INVALID_ARG;
    {   // k_write must not overlap k, A0 or AT; AT may equal A0 exactly
        const size_t kb = (size_t)B * T * H * dk * elt;
        const size_t ab = sizeof(float) * (size_t)B * H * dk;
        const Span ins[] = {{k, kb}, {A0, ab}};
        const Span outs[] = {{T > 0 ? k_write : nullptr, kb}};
        if (any_overlap(ins, outs) || overlap({T > 0 ? k_write : nullptr, kb},
                                              {AT, ab}))
            return KLA_ERR_INVALID_ARG;
        if ((const void*)AT != (const void*)A0 &&
            (overlap({AT, ab}, {A0, ab}) || overlap({AT, ab}, {k, kb})))
            return KLA_ERR_INVALID_ARG;
    }
    kla::PrecondArgs a{k, A0, k_write, AT, B, T, H, dk, x, delta, dtype};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!kla::precond_chunked_eligible(a))
        return from_cuda(kla::launch_precond_keys(a, s));
    const size_t need = kla::precond_chunked_bytes(B, T, H);
    if (workspace) {
        if (workspace_bytes < need || !aligned(workspace, 16))
            return KLA_ERR_INVALID_ARG;
        const size_t kb = (size_t)B * T * H * dk * elt;
        const size_t ab = sizeof(float) * (size_t)B * H * dk;
        const Span bufs[] = {{k, kb}, {T > 0 ? k_write : nullptr, kb},
                             {A0, ab}, {AT, ab}};
        const Span ws[] = {{workspace, need}};
        if (any_overlap(bufs, ws)) return KLA_ERR_INVALID_ARG;
        return from_cuda(kla::launch_precond_chunked(a, workspace, s));
    }
    if (need == 0)   // T <= 64: no scan, no workspace
        return from_cuda(kla::launch_precond_chunked(a, nullptr, s));
    // stream-ordered scratch from the device's current memory pool
    void* scratch = nullptr;
    if (cudaMallocAsync(&scratch, need, s) != cudaSuccess) return KLA_ERR_CUDA;
    const cudaError_t e = kla::launch_precond_chunked(a, scratch, s);
    const cudaError_t f = cudaFreeAsync(scratch, s);
    return from_cuda(e != cudaSuccess ? e : f);
}

extern "C" kla_status kla_precond_keys(const void* k, const float* A0,
                                       void* k_write, float* AT, int B, int T,
                                       int H, int dk, float x, float delta,
                                       kla_dtype dtype, kla_stream_t stream) {
    return kla_precond_keys_ex(k, A0, k_write, AT, B, T, H, dk, x, delta,
                               dtype, nullptr, 0, stream);
}

extern "C" kla_status kla_chunk_fwd(const void* q, const void* k,
                                    const void* v, const float* log_alpha,
                                    const float* eta, float eps,
                                    const float* h0, void* o, float* hT,
                                    int B, int T, int H, int dk, int dv,
                                    int C, kla_dtype dtype,
                                    kla_stream_t stream) {
    return kla_chunk_fwd_ex(q, k, v, log_alpha, eta, eps, h0, o, hT, B, T, H,
                            dk, dv, C, dtype, KLA_ALGO_AUTO, KLA_STEP_KACZMARZ,
                            stream);
}

static kla_status decode_impl(const void* q, const void* k, const void* kw,
                              const void* v, const float* log_alpha,
                              const float* eta, float eps, float* S, void* o,
                              int N, int H, int dk, int dv, kla_dtype dtype,
                              kla_step_rule rule, kla_stream_t stream) {
    if (N < 0 || H < 0 || dk <= 0 || dv <= 0) return KLA_ERR_INVALID_ARG;
    if (rule != KLA_STEP_KACZMARZ && rule != KLA_STEP_GIVEN)
        return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_F32 && dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return KLA_ERR_INVALID_ARG;
    if (!supported_dim(dk) || !supported_dim(dv))
        return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)N * H > 0x7fffffffLL) return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)N * H == 0) return KLA_OK;
    if (!q || !k || !v || !log_alpha || !eta || !S || !o)
        return KLA_ERR_INVALID_ARG;
    const size_t elt = dtype == KLA_BF16 ? 2 : 4;
    if (!aligned(q, elt) || !aligned(k, elt) || !aligned(v, elt) ||
        !aligned(o, elt) || !aligned(log_alpha, 4) || !aligned(eta, 4) ||
        !aligned(S, 16) || (kw && !aligned(kw, elt)))
        return KLA_ERR_INVALID_ARG;
    {   // o must not overlap S or any input; S is updated in place and
        // must not overlap the token inputs either
        const size_t nh = (size_t)N * H;
        const Span ins[] = {{q, nh * dk * elt}, {k, nh * dk * elt},
                            {v, nh * dv * elt}, {log_alpha, nh * 4},
                            {eta, nh * 4}, {kw, nh * dk * elt}};
        const Span outs[] = {{o, nh * dv * elt},
                             {S, sizeof(float) * nh * dk * dv}};
        if (any_overlap(ins, outs)) return KLA_ERR_INVALID_ARG;
    }
    kla::DecodeArgs a{q, k, v, log_alpha, eta, eps,
                      rule == KLA_STEP_GIVEN ? 1 : 0, S, o, N, H, dk, dv,
                      dtype};
    a.kw = kw;
    return from_cuda(
        kla::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" kla_status kla_decode_step_ex(const void* q, const void* k,
                                         const void* v, const float* log_alpha,
                                         const float* eta, float eps, float* S,
                                         void* o, int N, int H, int dk, int dv,
                                         kla_dtype dtype, kla_step_rule rule,
                                         kla_stream_t stream) {
    return decode_impl(q, k, nullptr, v, log_alpha, eta, eps, S, o, N, H, dk,
                       dv, dtype, rule, stream);
}

extern "C" kla_status kla_decode_step_kw(const void* q, const void* k,
                                         const void* k_write, const void* v,
                                         const float* log_alpha,
                                         const float* eta, float eps, float* S,
                                         void* o, int N, int H, int dk, int dv,
                                         kla_dtype dtype, kla_step_rule rule,
                                         kla_stream_t stream) {
    if (!k_write && (long long)N * H > 0) return KLA_ERR_INVALID_ARG;
    return decode_impl(q, k, k_write, v, log_alpha, eta, eps, S, o, N, H, dk,
                       dv, dtype, rule, stream);
}

extern "C" kla_status kla_decode_step(const void* q, const void* k,
                                      const void* v, const float* log_alpha,
                                      const float* eta, float eps, float* S,
                                      void* o, int N, int H, int dk, int dv,
                                      kla_dtype dtype, kla_stream_t stream) {
    return kla_decode_step_ex(q, k, v, log_alpha, eta, eps, S, o, N, H, dk, dv,
                              dtype, KLA_STEP_KACZMARZ, stream);
}

extern "C" kla_status kla_chunk_bwd_workspace_size(int B, int T, int H,
                                                   int dk, int dv, int C,
                                                   size_t* bytes) {
    if (!bytes || B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || C <= 0)
        return KLA_ERR_INVALID_ARG;
    *bytes = kla::chunk_bwd_workspace_bytes(B, T, H, dk, dv, C);
    return KLA_OK;
}

namespace kla {

// Every check of kla_chunk_bwd except those on the workspace.
kla_status check_chunk_bwd_args(const BwdArgs& a) {
    const int B = a.B, T = a.T, H = a.H, dk = a.dk, dv = a.dv, C = a.C;
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || C <= 0)
        return KLA_ERR_INVALID_ARG;
    if (a.dtype != KLA_F32 && a.dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (!(a.eps >= 0.f) || !std::isfinite(a.eps)) return KLA_ERR_INVALID_ARG;
    if (!supported_dim(dk) || !supported_dim(dv) || !supported_chunk(C))
        return KLA_ERR_UNSUPPORTED_SHAPE;
    const long long nch = ((long long)T + C - 1) / C;
    if ((long long)B * H > 0x7fffffffLL ||
        (long long)B * H * nch > 0x7fffffffLL)
        return KLA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * H > 0 && T > 0) {
        if (!a.q || !a.k || !a.v || !a.log_alpha || !a.eta || !a.dout ||
            !a.dq || !a.dk_ || !a.dv_ || !a.dlog_alpha || !a.deta)
            return KLA_ERR_INVALID_ARG;
        const size_t elt = a.dtype == KLA_BF16 ? 2 : 4;
        if (!aligned(a.q, elt) || !aligned(a.k, elt) || !aligned(a.v, elt) ||
            !aligned(a.dout, elt) || !aligned(a.dq, elt) ||
            !aligned(a.dk_, elt) || !aligned(a.dv_, elt) ||
            !aligned(a.log_alpha, 4) || !aligned(a.eta, 4) ||
            !aligned(a.dlog_alpha, 4) || !aligned(a.deta, 4))
            return KLA_ERR_INVALID_ARG;
        const size_t tok = (size_t)B * T * H;
        const size_t st = sizeof(float) * (size_t)B * H * dk * dv;
        const Span ins[] = {{a.q, tok * dk * elt}, {a.k, tok * dk * elt},
                            {a.v, tok * dv * elt}, {a.log_alpha, tok * 4},
                            {a.eta, tok * 4}, {a.h0, st},
                            {a.dout, tok * dv * elt}, {a.dhT, st}};
        const Span outs[] = {{a.dq, tok * dk * elt}, {a.dk_, tok * dk * elt},
                             {a.dv_, tok * dv * elt}, {a.dlog_alpha, tok * 4},
                             {a.deta, tok * 4}, {a.dh0, st}};
        if (any_overlap(ins, outs)) return KLA_ERR_INVALID_ARG;
    }
    if ((a.h0 && !aligned(a.h0, 4)) || (a.dhT && !aligned(a.dhT, 4)) ||
        (a.dh0 && !aligned(a.dh0, 4)))
        return KLA_ERR_INVALID_ARG;
    return KLA_OK;
}

}  // namespace kla

extern "C" kla_status kla_chunk_bwd(
    const void* q, const void* k, const void* v, const float* log_alpha,
    const float* eta, float eps, const float* h0, const void* o_grad,
    const float* hT_grad, void* q_grad, void* k_grad, void* v_grad,
    float* log_alpha_grad, float* eta_grad, float* h0_grad, int B, int T,
    int H, int dk, int dv, int C, kla_dtype dtype, kla_step_rule rule,
    void* workspace, size_t workspace_bytes, kla_stream_t stream) {
    if (rule != KLA_STEP_KACZMARZ && rule != KLA_STEP_GIVEN)
        return KLA_ERR_INVALID_ARG;
    kla::BwdArgs a{q, k, v, log_alpha, eta, eps,
                   rule == KLA_STEP_GIVEN ? 1 : 0, h0, o_grad, hT_grad,
                   q_grad, k_grad, v_grad, log_alpha_grad, eta_grad, h0_grad,
                   nullptr, nullptr, B, T, H, dk, dv, C, dtype};
    const kla_status st = kla::check_chunk_bwd_args(a);
    if (st != KLA_OK) return st;
    const bool empty = (long long)B * H == 0;
    if (!empty && T > 0) {
        if (!workspace || !aligned(workspace, 16)) return KLA_ERR_INVALID_ARG;
        const size_t need = kla::chunk_bwd_workspace_bytes(B, T, H, dk, dv, C);
        if (workspace_bytes < need) return KLA_ERR_INVALID_ARG;
        const size_t elt = dtype == KLA_BF16 ? 2 : 4;
        const size_t tok = (size_t)B * T * H;
        const size_t st = sizeof(float) * (size_t)B * H * dk * dv;
        const Span bufs[] = {{q, tok * dk * elt}, {k, tok * dk * elt},
                             {v, tok * dv * elt}, {log_alpha, tok * 4},
                             {eta, tok * 4}, {h0, st},
                             {o_grad, tok * dv * elt}, {hT_grad, st},
                             {q_grad, tok * dk * elt}, {k_grad, tok * dk * elt},
                             {v_grad, tok * dv * elt},
                             {log_alpha_grad, tok * 4}, {eta_grad, tok * 4},
                             {h0_grad, st}};
        const Span ws[] = {{workspace, need}};
        if (any_overlap(bufs, ws)) return KLA_ERR_INVALID_ARG;
    }
    if (empty) return KLA_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {   // L depends on h0 only through hT = h0
        if (!h0_grad) return KLA_OK;
        const size_t bytes = sizeof(float) * (size_t)B * H * dk * dv;
        if (hT_grad)
            return from_cuda(cudaMemcpyAsync(h0_grad, hT_grad, bytes,
                                             cudaMemcpyDeviceToDevice, s));
        return from_cuda(cudaMemsetAsync(h0_grad, 0, bytes, s));
    }
    const size_t nst = kla::chunk_bwd_state_floats(B, T, H, dk, dv, C);
    float* ws = static_cast<float*>(workspace);
    a.ckpt = ws;
    a.dsck = ws + nst;
    if (dk == 128 && C == 64) {   // the tensor-core kernels' records
        const size_t nch = ((size_t)T + C - 1) / C;
        a.rec = reinterpret_cast<uint8_t*>(ws + 2 * nst);   // 16-byte aligned
        if (dv == 128)   // and the two-kernel forward's, for the checkpoints
            a.fwd_rec = a.rec + (size_t)B * H * nch * kla::bwdrec::BYTES;
    }
    return from_cuda(kla::launch_chunk_bwd(a, s));
}

extern "C" kla_status kla_device_status(kla_stream_t stream) {
    unsigned int word = 0;
    cudaError_t e = kla::read_and_clear_fault(
        reinterpret_cast<cudaStream_t>(stream), &word);
    if (e != cudaSuccess) return KLA_ERR_CUDA;
    return word ? KLA_ERR_TIMEOUT : KLA_OK;
}

extern "C" kla_status kla_selftest_wait_timeout(kla_stream_t stream) {
    return from_cuda(kla::launch_state_selftest(
        reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" const char* kla_status_string(kla_status status) {
    switch (status) {
        case KLA_OK: return "ok";
        case KLA_ERR_INVALID_ARG: return "invalid argument";
        case KLA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape or dtype";
        case KLA_ERR_CUDA: return "CUDA runtime error";
        case KLA_ERR_TIMEOUT: return "device-side wait timed out";
        case KLA_ERR_NOT_IMPLEMENTED: return "not implemented";
    }
    return "unknown status";
}
