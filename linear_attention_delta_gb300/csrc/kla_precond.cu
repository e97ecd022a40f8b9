// Write keys of the diagonal-preconditioned delta rule.
//
// Per (batch, head) and key dimension i, with the running second moments
// A_t,i = A_{t-1},i + k_t,i^2 (A_0 given or zero):
//   z_i   = mean_j log(A_t,j + delta) - log(A_t,i + delta)
//   P_t,i = exp(log(x) tanh(z_i / log(x)))        in [1/x, x]
//   kw_t  = P_t (.) k_t
// (the diagonal approximation of the inverse key Gram matrix, squashed in
// log space onto [1/x, x], applied to the write key: gist.science
// "preconditioned DeltaNet" page, section "Aproximacion Diagonal"; the tanh
// squash centred on the mean log second moment is this library's reading).
//
// One CTA per (batch, head), one thread per key dimension, tokens in order
// (A_t is a running sum); the mean over the key dimensions is a block
// reduction per token.
#include "kla_internal.cuh"

namespace kla {
namespace {

constexpr int kPrecondThreads = 128;   // >= dk, a multiple of 32

template <typename IO>
__global__ void __launch_bounds__(kPrecondThreads)
kla_precond_keys_kernel(PrecondArgs a) {
    __shared__ float part[kPrecondThreads / 32];
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
    const int dk = a.dk, T = a.T, H = a.H;
    const int nwarps = (dk + 31) / 32;
    const bool live = i < dk;
    const float lx = logf(a.x);
    float A = (live && a.A0) ? a.A0[(size_t)bh * dk + i] : 0.f;
    const IO* k = static_cast<const IO*>(a.k);
    IO* kw = static_cast<IO*>(a.kw);

    for (int t = 0; t < T; ++t) {
        const size_t off = (((size_t)b * T + t) * H + h) * dk + i;
        const float kv = live ? to_f32(k[off]) : 0.f;
        A = fmaf(kv, kv, A);
        const float l = live ? logf(A + a.delta) : 0.f;
        float s = l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0 && warp < nwarps) part[warp] = s;
        __syncthreads();
        float tot = 0.f;
        for (int w = 0; w < nwarps; ++w) tot += part[w];
        __syncthreads();
        if (live) {
            const float z = tot / (float)dk - l;
            kw[off] = from_f32<IO>(expf(lx * tanhf(z / lx)) * kv);
        }
    }
    if (live && a.AT) a.AT[(size_t)bh * dk + i] = A;
}

}  // namespace

cudaError_t launch_precond_keys(const PrecondArgs& a, cudaStream_t stream) {
    const long bhs = (long)a.B * a.H;
    if (bhs == 0) return cudaSuccess;
    if (a.dk > kPrecondThreads) return cudaErrorInvalidValue;
    if (a.dtype == KLA_BF16)
        kla_precond_keys_kernel<__nv_bfloat16>
            <<<(unsigned)bhs, kPrecondThreads, 0, stream>>>(a);
    else
        kla_precond_keys_kernel<float>
            <<<(unsigned)bhs, kPrecondThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kla
