// Single-token KLA decode step: one read and one write of every recurrent
// state, fused with the key norm, the Kaczmarz step and the read-out.
//
// Per (sequence, head), with S the dk x dv fp32 state (row = key dim):
//   alpha = exp(log_alpha),  beta = eta / (||k||^2 + eps)      (0 if denom 0)
//   a = S^T k,  b = S^T q                    (reductions over the key dim)
//   e = v - alpha a                          residual against the decayed state
//   o = alpha b + beta (q.k) e               = S_new^T q
//   S_new = alpha S + beta k e^T
// (gist.science/es/paper/2605.08587, section "La Regla de Actualizacion KLA";
// the scalar decay and the read-out after the write are this library's
// reading of the "decayed previous state" and of the output.)
//
// o is formed from the OLD state, so the new state is never re-read: the
// kernel moves exactly 2 * dk * dv * 4 bytes of state per head.
//
// Layout of work: one CTA per (head, dv tile).  A thread owns one float4
// column group of the tile and dk/RS rows (row r = slice + i*RS), so a warp
// reads whole 512-byte row segments.  Every state load is issued before any
// reduction so that each CTA keeps its whole tile in flight.
//
// Each step is launched as a programmatic dependent of the previous kernel
// on the stream: its CTAs may be scheduled while the previous grid's last
// CTAs run, and every CTA waits for that grid (and its memory) before it
// touches memory, so the ordering is that of plain stream order.
#include "kla_internal.cuh"

namespace kla {
namespace {

template <int DK, int DVT>
struct DecodeShape {
    static constexpr int CG = DVT / 4;                  // float4 groups
    static constexpr int RS_CAP = 256 / CG;
    static constexpr int RS = RS_CAP < DK ? RS_CAP : DK;  // row slices
    static constexpr int NT = CG * RS;                  // threads
    static constexpr int ROWS = DK / RS;                // rows per thread
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <int DK, int DVT, typename T>
__global__ void __launch_bounds__(DecodeShape<DK, DVT>::NT)
kla_decode_kernel(DecodeArgs a) {
    using Sh = DecodeShape<DK, DVT>;
    const int head = blockIdx.x;              // n * H + h
    const int dv = a.dv;
    const int j0 = blockIdx.y * DVT;
    const int tid = threadIdx.x;
    const int cg = tid % Sh::CG;
    const int rs = tid / Sh::CG;

    // launched as a programmatic dependent of the previous kernel on the
    // stream: wait for it (and its memory) before touching memory, and let
    // the next one be scheduled as this grid's last CTAs start
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float* S = a.S + (size_t)head * DK * dv + j0 + 4 * cg;

    float4 s[Sh::ROWS];
#pragma unroll
    for (int i = 0; i < Sh::ROWS; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4*>(
            S + (size_t)(rs + i * Sh::RS) * dv));

    __shared__ float ks[DK];
    __shared__ float kws[DK];   // write key (= ks without separate keys)
    __shared__ float qs[DK];
    __shared__ float4 red_a[Sh::RS][Sh::CG];
    __shared__ float4 red_b[Sh::RS][Sh::CG];
    __shared__ float nk_s, qk_s;

    const T* qp = static_cast<const T*>(a.q) + (size_t)head * DK;
    const T* kp = static_cast<const T*>(a.k) + (size_t)head * DK;
    const T* kwp = a.kw ? static_cast<const T*>(a.kw) + (size_t)head * DK
                        : kp;
    for (int i = tid; i < DK; i += Sh::NT) {
        ks[i] = to_f32(kp[i]);
        kws[i] = to_f32(kwp[i]);
        qs[i] = to_f32(qp[i]);
    }
    __syncthreads();

    if (tid < 32) {
        float nk = 0.f, qk = 0.f;
        for (int i = tid; i < DK; i += 32) {
            nk = fmaf(ks[i], kws[i], nk);     // k . (write key)
            qk = fmaf(qs[i], kws[i], qk);
        }
        nk = warp_sum(nk);
        qk = warp_sum(qk);
        if (tid == 0) {
            nk_s = nk;
            qk_s = qk;
        }
    }

    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 pb = pa;
#pragma unroll
    for (int i = 0; i < Sh::ROWS; ++i) {
        const int r = rs + i * Sh::RS;
        const float kr = ks[r], qr = qs[r];
        pa.x = fmaf(s[i].x, kr, pa.x); pa.y = fmaf(s[i].y, kr, pa.y);
        pa.z = fmaf(s[i].z, kr, pa.z); pa.w = fmaf(s[i].w, kr, pa.w);
        pb.x = fmaf(s[i].x, qr, pb.x); pb.y = fmaf(s[i].y, qr, pb.y);
        pb.z = fmaf(s[i].z, qr, pb.z); pb.w = fmaf(s[i].w, qr, pb.w);
    }
    red_a[rs][cg] = pa;
    red_b[rs][cg] = pb;
    __syncthreads();

    float4 ta = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 tb = ta;
#pragma unroll
    for (int r = 0; r < Sh::RS; ++r) {
        const float4 x = red_a[r][cg], y = red_b[r][cg];
        ta.x += x.x; ta.y += x.y; ta.z += x.z; ta.w += x.w;
        tb.x += y.x; tb.y += y.y; tb.z += y.z; tb.w += y.w;
    }

    const float alpha = expf(a.log_alpha[head]);
    const float denom = nk_s + a.eps;
    const float beta =
        a.gdn ? a.eta[head] : (denom == 0.f ? 0.f : a.eta[head] / denom);
    const float bqk = beta * qk_s;

    const T* vp = static_cast<const T*>(a.v) + (size_t)head * dv + j0 + 4 * cg;
    float4 e;
    e.x = to_f32(vp[0]) - alpha * ta.x;
    e.y = to_f32(vp[1]) - alpha * ta.y;
    e.z = to_f32(vp[2]) - alpha * ta.z;
    e.w = to_f32(vp[3]) - alpha * ta.w;

    if (rs == 0) {
        T* op = static_cast<T*>(a.o) + (size_t)head * dv + j0 + 4 * cg;
        op[0] = from_f32<T>(fmaf(alpha, tb.x, bqk * e.x));
        op[1] = from_f32<T>(fmaf(alpha, tb.y, bqk * e.y));
        op[2] = from_f32<T>(fmaf(alpha, tb.z, bqk * e.z));
        op[3] = from_f32<T>(fmaf(alpha, tb.w, bqk * e.w));
    }

#pragma unroll
    for (int i = 0; i < Sh::ROWS; ++i) {
        const int r = rs + i * Sh::RS;
        const float bk = beta * kws[r];
        float4 n;
        n.x = fmaf(alpha, s[i].x, bk * e.x);
        n.y = fmaf(alpha, s[i].y, bk * e.y);
        n.z = fmaf(alpha, s[i].z, bk * e.z);
        n.w = fmaf(alpha, s[i].w, bk * e.w);
        __stcs(reinterpret_cast<float4*>(S + (size_t)r * dv), n);
    }
}

template <int DK, int DVT, typename T>
cudaError_t launch_shape(const DecodeArgs& a, cudaStream_t stream) {
    using Sh = DecodeShape<DK, DVT>;
    const long heads = (long)a.N * a.H;
    if (heads == 0) return cudaSuccess;
    dim3 grid((unsigned)heads, (unsigned)(a.dv / DVT));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Sh::NT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kla_decode_kernel<DK, DVT, T>, a);
}

template <typename T>
cudaError_t launch_dtype(const DecodeArgs& a, cudaStream_t stream) {
    // dv tile = min(dv, 128); dv in {16, 32, 64, 128}.
#define KLA_DECODE_DK(DKV)                                                  \
    if (a.dk == DKV) {                                                      \
        switch (a.dv) {                                                     \
            case 16: return launch_shape<DKV, 16, T>(a, stream);            \
            case 32: return launch_shape<DKV, 32, T>(a, stream);            \
            case 64: return launch_shape<DKV, 64, T>(a, stream);            \
            case 128: return launch_shape<DKV, 128, T>(a, stream);          \
            default: return cudaErrorInvalidValue;                          \
        }                                                                   \
    }
    KLA_DECODE_DK(16)
    KLA_DECODE_DK(32)
    KLA_DECODE_DK(64)
    KLA_DECODE_DK(128)
#undef KLA_DECODE_DK
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.dtype == KLA_BF16) return launch_dtype<__nv_bfloat16>(a, stream);
    return launch_dtype<float>(a, stream);
}

}  // namespace kla
