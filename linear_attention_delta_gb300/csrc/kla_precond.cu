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
// The running sum is a prefix sum over tokens, so the sequence is split
// into pieces whose sums of k^2 are added up first, and each piece then
// walks its tokens in order from the A before it.  A lane holds dk / 32 key
// dimensions (one when dk = 16), so the mean over the key dimensions is a
// warp reduction.  Two forms:
//  * dk = 128 with 16-byte aligned k and kw (the models' shape): the
//    chunked form below, three launches over (batch, head, 64-token chunk)
//    items that fill every SM, with a workspace of per-chunk sums;
//  * any other shape: one cluster of kClusterCtas CTAs per (batch, head),
//    each CTA one contiguous slice of the tokens and each of its warps one
//    sub-slice; the sums that precede a warp come from shared memory
//    (earlier warps) and over the cluster's distributed shared memory
//    (earlier CTAs).  No workspace, one launch.
// The logarithm, the exponentials and the reciprocal are the hardware
// approximations (PTX lg2/ex2/rcp .approx.ftz, a few ulp: they move kw by a
// few 1e-6 relative, far inside the 1e-4 bound), in base 2 with the
// constants folded (Squash below); tanh is written through the exponential.
#include <cooperative_groups.h>
#include <cstdint>
#include <type_traits>

#include "kla_internal.cuh"

namespace kla {
namespace {

namespace cg = cooperative_groups;

constexpr int kClusterCtas = 8;
constexpr int kPrecondWarps = 32;
constexpr int kPrecondThreads = kPrecondWarps * 32;
constexpr int kTokBatch = 4;   // tokens loaded ahead of their use

// A lane's DPL consecutive key dimensions: one 16-byte (fp32) or 8-byte
// (bf16) access when VEC (DPL == 4, tensors 16-byte aligned), else DPL
// scalar ones.
template <bool VEC, int DPL, typename IO>
__device__ __forceinline__ void ld_dims(const IO* p, float (&x)[DPL]) {
    if constexpr (VEC && DPL == 4) {
        if constexpr (std::is_same<IO, float>::value) {
            const float4 v = *reinterpret_cast<const float4*>(p);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else {
            const uint2 v = *reinterpret_cast<const uint2*>(p);
            x[0] = __uint_as_float(v.x << 16);
            x[1] = __uint_as_float(v.x & 0xffff0000u);
            x[2] = __uint_as_float(v.y << 16);
            x[3] = __uint_as_float(v.y & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int d = 0; d < DPL; ++d) x[d] = to_f32(p[d]);
    }
}

template <bool VEC, int DPL, typename IO>
__device__ __forceinline__ void st_dims(IO* p, const float (&x)[DPL]) {
    if constexpr (VEC && DPL == 4) {
        if constexpr (std::is_same<IO, float>::value) {
            *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
        } else {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(x[2], x[3]);
            *reinterpret_cast<uint2*>(p) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                           *reinterpret_cast<const uint32_t*>(&hi));
        }
    } else {
#pragma unroll
        for (int d = 0; d < DPL; ++d) p[d] = from_f32<IO>(x[d]);
    }
}

// Four consecutive key dimensions of one token as loaded (the VEC case):
// one 16-byte fp32 or 8-byte bf16 access, unpacked only where it is used.
template <typename IO>
using Raw4 = typename std::conditional<std::is_same<IO, float>::value,
                                       float4, uint2>::type;

template <typename IO>
__device__ __forceinline__ void unpack4(const Raw4<IO>& r, float (&x)[4]) {
    if constexpr (std::is_same<IO, float>::value) {
        x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
    } else {
        x[0] = __uint_as_float(r.x << 16);
        x[1] = __uint_as_float(r.x & 0xffff0000u);
        x[2] = __uint_as_float(r.y << 16);
        x[3] = __uint_as_float(r.y & 0xffff0000u);
    }
}

__device__ __forceinline__ float lg2_approx(float v) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float ex2_approx(float v) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float rcp_approx(float v) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// The squash in base 2.  With l_i = log2(A_i + delta) and m their mean,
// z_i = ln 2 (m - l_i) and y_i = z_i / ln x = (m - l_i) / log2 x, so
//   e^{2 y_i} = 2^{E_i},  E_i = c (m - l_i),  c = 2 log2(e) / log2(x)
//   tanh y_i  = 1 - 2 / (2^{E_i} + 1)
//   P_i       = x^{tanh y_i} = 2^{log2(x) - 2 log2(x) / (2^{E_i} + 1)}
// E is clamped to [-64, 64] (tanh is +-1 to fp32 beyond; a NaN from
// delta = 0 and A_i = 0 becomes -64, P = 1/x).
struct Squash {
    float delta, c, c_mean, lx2, m2lx2;   // c_mean = c / dk, m2lx2 = -2 log2 x
    __device__ Squash(float x, float d, int dk) {
        lx2 = log2f(x);
        c = 2.f * 1.44269504088896341f / lx2;
        c_mean = c / (float)dk;
        m2lx2 = -2.f * lx2;
        delta = d;
    }
};

// One token: A += k^2, then kw = P (.) k.
template <int DPL>
__device__ __forceinline__ void weigh_token(float (&A)[DPL],
                                            const float (&kv)[DPL], bool live,
                                            const Squash& q,
                                            float (&w)[DPL]) {
    float l[DPL], s = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
        A[d] = fmaf(kv[d], kv[d], A[d]);
        l[d] = live ? lg2_approx(A[d] + q.delta) : 0.f;
        s += l[d];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float cm = s * q.c_mean;   // c m
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
        const float E = fminf(fmaxf(fmaf(-l[d], q.c, cm), -64.f), 64.f);
        const float r = rcp_approx(ex2_approx(E) + 1.f);
        w[d] = ex2_approx(fmaf(r, q.m2lx2, q.lx2)) * kv[d];
    }
}

template <int DK, typename IO, bool VEC>
__global__ void __cluster_dims__(kClusterCtas, 1, 1)
    __launch_bounds__(kPrecondThreads, 1)
    kla_precond_keys_kernel(PrecondArgs a) {
    constexpr int DPL = DK >= 32 ? DK / 32 : 1;   // dimensions per lane
    constexpr int LANES = DK / DPL;               // lanes holding dimensions
    __shared__ float wsum[kPrecondWarps][DK];     // sum of k^2 per sub-slice
    __shared__ float ctot[DK];                    // ... per CTA slice
    __shared__ float base[DK];                    // A before this CTA's slice

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int bh = blockIdx.x / kClusterCtas;
    const int b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, H = a.H;
    const bool live = lane < LANES;
    const int d0 = lane * DPL;

    // this warp's tokens [t_lo, t_hi)
    const int per_cta = (T + kClusterCtas - 1) / kClusterCtas;
    const int per_warp = (per_cta + kPrecondWarps - 1) / kPrecondWarps;
    const int c_lo = min(T, rank * per_cta);
    const int c_hi = min(T, c_lo + per_cta);
    const int t_lo = min(c_hi, c_lo + warp * per_warp);
    const int t_hi = min(c_hi, t_lo + per_warp);

    // this lane's dimensions of the warp's first token; a token is H DK
    // elements further
    const size_t tstride = (size_t)H * DK;
    const size_t first = (((size_t)b * T + t_lo) * H + h) * DK + d0;
    const IO* kb = static_cast<const IO*>(a.k) + first;
    IO* wb = static_cast<IO*>(a.kw) + first;

    // ---- pass 1: sum of k^2 over the sub-slice ----
    float sq[DPL] = {};
    for (int t = t_lo; t < t_hi; t += kTokBatch) {
        float kv[kTokBatch][DPL];
#pragma unroll
        for (int u = 0; u < kTokBatch; ++u) {
            if (live && t + u < t_hi) {
                ld_dims<VEC>(kb + (size_t)(t + u - t_lo) * tstride, kv[u]);
            } else {
#pragma unroll
                for (int d = 0; d < DPL; ++d) kv[u][d] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kTokBatch; ++u)
#pragma unroll
            for (int d = 0; d < DPL; ++d) sq[d] = fmaf(kv[u][d], kv[u][d], sq[d]);
    }
    if (live) {
#pragma unroll
        for (int d = 0; d < DPL; ++d) wsum[warp][d0 + d] = sq[d];
    }
    __syncthreads();
    if (tid < DK) {
        float s = 0.f;
        for (int w = 0; w < kPrecondWarps; ++w) s += wsum[w][tid];
        ctot[tid] = s;
    }
    cluster.sync();   // every CTA's slice total is visible cluster-wide
    if (tid < DK) {
        float s = a.A0 ? a.A0[(size_t)bh * DK + tid] : 0.f;
        for (int r = 0; r < rank; ++r) s += cluster.map_shared_rank(ctot, r)[tid];
        base[tid] = s;
        if (rank == kClusterCtas - 1 && a.AT)
            a.AT[(size_t)bh * DK + tid] = s + ctot[tid];
    }
    cluster.sync();   // remote reads done (no CTA leaves while read); base set

    // ---- pass 2: the sub-slice's tokens in order ----
    float A[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
        float s = live ? base[d0 + d] : 0.f;
        for (int w = 0; w < warp; ++w) s += live ? wsum[w][d0 + d] : 0.f;
        A[d] = s;
    }
    const Squash q(a.x, a.delta, DK);
    for (int t = t_lo; t < t_hi; t += kTokBatch) {
        float kv[kTokBatch][DPL];
#pragma unroll
        for (int u = 0; u < kTokBatch; ++u) {
            if (live && t + u < t_hi) {
                ld_dims<VEC>(kb + (size_t)(t + u - t_lo) * tstride, kv[u]);
            } else {
#pragma unroll
                for (int d = 0; d < DPL; ++d) kv[u][d] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kTokBatch; ++u) {
            if (t + u >= t_hi) break;   // warp-uniform
            float w[DPL];
            weigh_token<DPL>(A, kv[u], live, q, w);
            if (live) st_dims<VEC>(wb + (size_t)(t + u - t_lo) * tstride, w);
        }
    }
}

template <int DK, typename IO>
cudaError_t launch_io(const PrecondArgs& a, cudaStream_t stream) {
    const unsigned grid = (unsigned)((long)a.B * a.H * kClusterCtas);
    auto al16 = [](const void* p) {
        return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    };
    if constexpr (DK == 128) {
        if (al16(a.k) && al16(a.kw)) {
            kla_precond_keys_kernel<DK, IO, true>
                <<<grid, kPrecondThreads, 0, stream>>>(a);
            return cudaGetLastError();
        }
    }
    kla_precond_keys_kernel<DK, IO, false>
        <<<grid, kPrecondThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// ---- the chunked form (dk = 128, 16-byte aligned k and kw) ----
//
// The cluster kernel above runs a few waves of one 1024-thread CTA per SM
// (clusters of 8 on one GPC), each a load, a cluster exchange and the
// weighting in turn, so it is bound by latency.  The chunked form spreads
// the same steps over (batch, head, 64-token chunk) items that fill every
// SM, in three launches on the stream, each later one a programmatic
// dependent of the one before:
//   sums   per item, the sum of k^2 over its tokens        -> sums[item]
//   scan   per (batch, head), bases[item] = A0 + the sums of its earlier
//          chunks (A before the chunk), and A_T
//   weigh  per item, the keys and per-warp sums first, then (after the scan)
//          A before each warp's tokens and the tokens in order
// The workspace is two fp32 rows of dk per item (sums, bases).  A sequence
// of one chunk
// (T <= 64: a decode step) needs no scan: the weighting kernel alone
// starts from A0 and writes A_T, without a workspace.
constexpr int kPcTok = 64;                    // tokens per item
constexpr int kPcWarps = 8;                   // warps per item
constexpr int kPcWarpTok = kPcTok / kPcWarps; // tokens per warp
constexpr int kPcThreads = kPcWarps * 32;
constexpr int kPcDk = 128;

// this warp's first token (clamped to T) and its count (0..kPcWarpTok), and
// the element offset of the lane's four dimensions of that token
template <typename IO>
struct WarpTokens {
    int t0, n;
    size_t off;
};

template <typename IO>
__device__ __forceinline__ WarpTokens<IO> warp_tokens(const PrecondArgs& a,
                                                      int item, int nchunks,
                                                      int warp, int lane) {
    const int bh = item / nchunks, c = item - bh * nchunks;
    const int b = bh / a.H, h = bh - b * a.H;
    WarpTokens<IO> w;
    w.t0 = min(a.T, c * kPcTok + warp * kPcWarpTok);
    w.n = min(kPcWarpTok, a.T - w.t0);
    w.off = (((size_t)b * a.T + w.t0) * a.H + h) * kPcDk + lane * 4;
    return w;
}

template <typename IO>
__device__ __forceinline__ void load_tokens(const PrecondArgs& a,
                                            const WarpTokens<IO>& w,
                                            Raw4<IO> (&kr)[kPcWarpTok]) {
    const IO* kb = static_cast<const IO*>(a.k) + w.off;
    const size_t tstride = (size_t)a.H * kPcDk;
#pragma unroll
    for (int u = 0; u < kPcWarpTok; ++u)
        kr[u] = u < w.n ? *reinterpret_cast<const Raw4<IO>*>(kb + u * tstride)
                        : Raw4<IO>{};
}

template <typename IO>
__device__ __forceinline__ void sum_squares(const Raw4<IO> (&kr)[kPcWarpTok],
                                            float (&sq)[4]) {
#pragma unroll
    for (int u = 0; u < kPcWarpTok; ++u) {
        float kv[4];
        unpack4<IO>(kr[u], kv);
#pragma unroll
        for (int d = 0; d < 4; ++d) sq[d] = fmaf(kv[d], kv[d], sq[d]);
    }
}

template <typename IO>
__global__ void __launch_bounds__(kPcThreads)
    kla_precond_sums_kernel(PrecondArgs a, float* ws, int nchunks) {
    __shared__ float wsum[kPcWarps][kPcDk];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int item = blockIdx.x;
    const WarpTokens<IO> w = warp_tokens<IO>(a, item, nchunks, warp, lane);
    Raw4<IO> kr[kPcWarpTok];
    load_tokens<IO>(a, w, kr);
    // the scan may be scheduled once every CTA of this grid has started; it
    // waits for this grid's memory before reading the sums
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float sq[4] = {};
    sum_squares<IO>(kr, sq);
#pragma unroll
    for (int d = 0; d < 4; ++d) wsum[warp][lane * 4 + d] = sq[d];
    __syncthreads();
    if (tid < kPcDk) {
        float s = 0.f;
#pragma unroll
        for (int v = 0; v < kPcWarps; ++v) s += wsum[v][tid];
        ws[(size_t)item * kPcDk + tid] = s;
    }
}

__global__ void __launch_bounds__(kPcDk)
    kla_precond_scan_kernel(PrecondArgs a, const float* sums, float* bases,
                            int nchunks) {
    // the weighting may be scheduled now; it waits for this grid's memory
    // before reading what this writes.  Everything here waits for the sums
    // (and for earlier work on the stream, which may write A0 or read AT).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int bh = blockIdx.x, d = threadIdx.x;
    float s = a.A0 ? a.A0[(size_t)bh * kPcDk + d] : 0.f;
    const size_t row = (size_t)bh * nchunks * kPcDk + d;
    // all loads of a batch in flight at once (one round trip to T = 4096);
    // the bases go to their own array, so that no store can be taken for
    // one to the address of a later load
    constexpr int kAhead = 64;
    for (int c0 = 0; c0 < nchunks; c0 += kAhead) {
        float v[kAhead];
#pragma unroll
        for (int j = 0; j < kAhead; ++j)
            v[j] = c0 + j < nchunks ? sums[row + (size_t)(c0 + j) * kPcDk]
                                    : 0.f;
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            if (c0 + j < nchunks) {
                bases[row + (size_t)(c0 + j) * kPcDk] = s;
                s += v[j];
            }
        }
    }
    if (a.AT) a.AT[(size_t)bh * kPcDk + d] = s;
}

// kSingle: one chunk per sequence (nchunks == 1), an ordinary launch that
// reads A0 for the chunk's start and writes A_T; else a dependent of the
// scan, reading A before the chunk from bases.
template <typename IO, bool kSingle>
__global__ void __launch_bounds__(kPcThreads)
    kla_precond_weigh_kernel(PrecondArgs a, const float* bases,
                             int nchunks) {
    __shared__ float wsum[kPcWarps][kPcDk];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int item = blockIdx.x;
    const WarpTokens<IO> w = warp_tokens<IO>(a, item, nchunks, warp, lane);
    // k is ready (the sums kernel, or this one when kSingle, was an ordinary
    // launch after every earlier piece of work); the chunk's start A is
    // not, until the scan completes
    Raw4<IO> kr[kPcWarpTok];
    load_tokens<IO>(a, w, kr);
    float sq[4] = {};
    sum_squares<IO>(kr, sq);
#pragma unroll
    for (int d = 0; d < 4; ++d) wsum[warp][lane * 4 + d] = sq[d];
    if constexpr (!kSingle) asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    float A[4];
#pragma unroll
    for (int d = 0; d < 4; ++d) {
        const size_t i = (size_t)item * kPcDk + lane * 4 + d;
        float s = kSingle ? (a.A0 ? a.A0[i] : 0.f) : bases[i];
        for (int v = 0; v < warp; ++v) s += wsum[v][lane * 4 + d];
        A[d] = s;
    }
    if constexpr (kSingle) {
        // A_T = A0 + the chunk's sum, added as the scan would; AT may be A0,
        // so only once every thread has read A0
        __syncthreads();
        if (a.AT && tid < kPcDk) {
            float s = 0.f;
#pragma unroll
            for (int v = 0; v < kPcWarps; ++v) s += wsum[v][tid];
            const size_t i = (size_t)item * kPcDk + tid;
            a.AT[i] = (a.A0 ? a.A0[i] : 0.f) + s;
        }
    }
    const Squash q(a.x, a.delta, kPcDk);
    IO* wb = static_cast<IO*>(a.kw) + w.off;
    const size_t tstride = (size_t)a.H * kPcDk;
#pragma unroll
    for (int u = 0; u < kPcWarpTok; ++u) {
        if (u >= w.n) break;   // warp-uniform
        float kv[4], kwv[4];
        unpack4<IO>(kr[u], kv);
        weigh_token<4>(A, kv, true, q, kwv);
        st_dims<true>(wb + u * tstride, kwv);
    }
}

template <typename K, typename... Args>
cudaError_t launch_dependent(K kern, unsigned grid, unsigned block,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename IO>
cudaError_t launch_chunked_io(const PrecondArgs& a, float* ws,
                              cudaStream_t stream) {
    const int nchunks = (a.T + kPcTok - 1) / kPcTok;
    const unsigned items = (unsigned)((long)a.B * a.H * nchunks);
    if (nchunks == 1) {
        kla_precond_weigh_kernel<IO, true><<<items, kPcThreads, 0, stream>>>(
            a, nullptr, nchunks);
        return cudaGetLastError();
    }
    float* sums = ws;
    float* bases = ws ? ws + (size_t)items * kPcDk : nullptr;
    if (items) {
        kla_precond_sums_kernel<IO><<<items, kPcThreads, 0, stream>>>(
            a, sums, nchunks);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_dependent(kla_precond_scan_kernel,
                                     (unsigned)((long)a.B * a.H), kPcDk,
                                     stream, a, (const float*)sums, bases,
                                     nchunks);
    if (e != cudaSuccess || !items) return e;
    return launch_dependent(kla_precond_weigh_kernel<IO, false>, items,
                            kPcThreads, stream, a, (const float*)bases,
                            nchunks);
}

template <int DK>
cudaError_t launch_dk(const PrecondArgs& a, cudaStream_t stream) {
    if (a.dtype == KLA_BF16) return launch_io<DK, __nv_bfloat16>(a, stream);
    return launch_io<DK, float>(a, stream);
}

}  // namespace

bool precond_chunked_eligible(const PrecondArgs& a) {
    auto al16 = [](const void* p) {
        return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    };
    return a.dk == kPcDk && (a.T == 0 || (al16(a.k) && al16(a.kw))) &&
           (long)a.B * a.H * ((a.T + kPcTok - 1) / kPcTok) <= 0x7fffffffL;
}

size_t precond_chunked_bytes(int B, int T, int H) {
    const size_t nchunks = (size_t)((T + kPcTok - 1) / kPcTok);
    return nchunks > 1 ? 2 * sizeof(float) * kPcDk * (size_t)B * H * nchunks
                       : 0;
}

cudaError_t launch_precond_chunked(const PrecondArgs& a, void* workspace,
                                   cudaStream_t stream) {
    if ((long)a.B * a.H == 0) return cudaSuccess;
    if (!precond_chunked_eligible(a)) return cudaErrorInvalidValue;
    float* ws = static_cast<float*>(workspace);
    if (a.dtype == KLA_BF16)
        return launch_chunked_io<__nv_bfloat16>(a, ws, stream);
    return launch_chunked_io<float>(a, ws, stream);
}

cudaError_t launch_precond_keys(const PrecondArgs& a, cudaStream_t stream) {
    const long bhs = (long)a.B * a.H;
    if (bhs == 0) return cudaSuccess;
    if (bhs * kClusterCtas > 0x7fffffffL) return cudaErrorInvalidValue;
    switch (a.dk) {
        case 16: return launch_dk<16>(a, stream);
        case 32: return launch_dk<32>(a, stream);
        case 64: return launch_dk<64>(a, stream);
        case 128: return launch_dk<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kla
