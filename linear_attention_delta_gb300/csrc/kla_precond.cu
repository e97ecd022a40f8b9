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
// The running sum is a prefix sum over tokens, so the sequence is split:
// one cluster of kClusterCtas CTAs per (batch, head), each CTA taking one
// contiguous slice of the tokens and each of its warps one sub-slice.  Pass 1
// sums k^2 over every sub-slice; the sums that precede a warp (earlier warps
// of the CTA from shared memory, earlier CTAs of the cluster from their
// shared memory over the cluster's distributed shared memory) give its
// starting A; pass 2 walks its tokens in order.  A lane holds dk / 32 key
// dimensions (one when dk = 16), so the mean over the key dimensions is a
// warp reduction.  No global scratch, one launch.  The logarithm and the
// exponentials are the hardware approximations (__logf, __expf, a few ulp:
// they move kw by a few 1e-6 relative, far inside the 1e-4 bound), with
// tanh written through the exponential.
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
    const float lx = logf(a.x);
    const float inv_lx = 1.f / lx;
    const float inv_dk = 1.f / (float)DK;
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
            float l[DPL], s = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) {
                A[d] = fmaf(kv[u][d], kv[u][d], A[d]);
                l[d] = live ? __logf(A[d] + a.delta) : 0.f;
                s += l[d];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, o);
            if (live) {
                const float mean = s * inv_dk;
                float w[DPL];
#pragma unroll
                for (int d = 0; d < DPL; ++d) {
                    // tanh(y) = 1 - 2 / (e^{2y} + 1), 2y kept in [-40, 40]
                    // (tanh is +-1 to fp32 there)
                    const float y2 = fminf(fmaxf(2.f * (mean - l[d]) * inv_lx,
                                                 -40.f), 40.f);
                    const float th = 1.f - __fdividef(2.f, __expf(y2) + 1.f);
                    w[d] = __expf(lx * th) * kv[u][d];
                }
                st_dims<VEC>(wb + (size_t)(t + u - t_lo) * tstride, w);
            }
        }
    }
}

template <int DK, typename IO>
cudaError_t launch_io(const PrecondArgs& a, cudaStream_t stream) {
    const unsigned grid = (unsigned)((long)a.B * a.H * kClusterCtas);
    auto al16 = [](const void* p) {
        return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    };
    if (DK == 128 && al16(a.k) && al16(a.kw))
        kla_precond_keys_kernel<DK, IO, true>
            <<<grid, kPrecondThreads, 0, stream>>>(a);
    else
        kla_precond_keys_kernel<DK, IO, false>
            <<<grid, kPrecondThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const PrecondArgs& a, cudaStream_t stream) {
    if (a.dtype == KLA_BF16) return launch_io<DK, __nv_bfloat16>(a, stream);
    return launch_io<DK, float>(a, stream);
}

}  // namespace

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
