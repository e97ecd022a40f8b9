// Chunkwise KLA forward pass on CUDA cores, all arithmetic in fp32.
//
// This is the general path: every supported (dk, dv, C) and both I/O types,
// and the only path for fp32 inputs (whose tolerance tensor-core operand
// rounding cannot meet).  One CTA owns one (batch, head, dv tile) and walks
// the chunks of its sequence in order, keeping its dk x dvt slice of the
// state in shared memory.
//
// Per chunk (rows r, i = 0..C-1; g = in-chunk cumulative log decay,
// gamma_r = exp(g_r), Gamma_ri = exp(g_r - g_i) for r >= i):
//   beta_r = eta_r / (||k_r||^2 + eps)                    Kaczmarz step
//   A  = I + strict_lower(Diag(beta) (Gamma o K K^T)),    T = A^{-1}
//   U~ = T Diag(beta) (V - Diag(gamma) K S)               chunk residuals
//   O  = Diag(gamma) Q S + lower_incl(Gamma o Q K^T) U~
//   S  = gamma_C S + (Diag(Gamma_{C,.}) K)^T U~
// This is the gated-DeltaNet block solver with B = Diag(beta) as the only
// change (gist.science/es/paper/2605.08587, section "Implementacion"), with
// U - W S (U = T B V, W = T B Diag(gamma) K) regrouped as T B times the
// residual.  Only exponents g_r - g_i with r >= i (and g_r, g_C - g_i) are
// ever exponentiated, so no factor exceeds 1.  T comes from a blocked
// inverse (16 x 16 tiles); every product is register-tiled.  With separate
// write keys kw (the diagonal-preconditioned variant) K K^T and Q K^T become
// K Kw^T and Q Kw^T, ||k||^2 becomes k . kw and the state is written along
// Kw; the residual is still read along K.
//
// A ragged last chunk is padded in-kernel with k = q = v = 0, eta = 0,
// log_alpha = 0: such a step has beta = 0 and alpha = 1, an exact identity.
#include "kla_internal.cuh"
#include "simt_blocks.cuh"

namespace kla {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtMaxC = 64;

template <int DK, int DVT>
struct SimtSmem {
    static constexpr int LDK = DK + 1;     // padded rows: conflict-free dots
    static constexpr int LDV = DVT + 1;
    static constexpr int LDC = kSimtMaxC + 1;
    static constexpr int Q = 0;
    static constexpr int K = Q + kSimtMaxC * LDK;
    static constexpr int KW = K + kSimtMaxC * LDK;     // write keys, if any
    static constexpr int S = KW + kSimtMaxC * LDK;     // DK x DVT state slice
    static constexpr int X = S + DK * LDV;             // V, then the residual
    static constexpr int F = X + kSimtMaxC * LDV;      // Diag(beta) X
    static constexpr int U = F + kSimtMaxC * LDV;      // U~
    static constexpr int QS = U + kSimtMaxC * LDV;     // Q S
    static constexpr int A = QS + kSimtMaxC * LDV;
    static constexpr int P = A + kSimtMaxC * LDC;
    static constexpr int TM = P + kSimtMaxC * LDC;     // A^{-1}
    static constexpr int G = TM + kSimtMaxC * LDC;     // cumulative log decay
    static constexpr int BETA = G + kSimtMaxC;
    static constexpr int GAM = BETA + kSimtMaxC;       // exp(g_r)
    static constexpr int KDEC = GAM + kSimtMaxC;       // exp(g_last - g_r)
    static constexpr int TOTAL = KDEC + kSimtMaxC;
    static constexpr size_t BYTES = sizeof(float) * (size_t)TOTAL;
};

template <int DK, int DVT, typename IO>
__global__ void __launch_bounds__(kSimtThreads)
kla_chunk_simt_kernel(FwdArgs a) {
    using L = SimtSmem<DK, DVT>;
    constexpr int LDK = L::LDK, LDV = L::LDV, LDC = L::LDC;
    constexpr int NCQ = DVT / 4;
    extern __shared__ float sm[];
    float* Qs = sm + L::Q;
    float* Ks = sm + L::K;
    // write keys: a separate tensor when given, else the keys themselves
    float* KWs = a.kw ? sm + L::KW : Ks;
    float* Ss = sm + L::S;
    float* Xs = sm + L::X;
    float* Fs = sm + L::F;
    float* Us = sm + L::U;
    float* QSs = sm + L::QS;
    float* As = sm + L::A;
    float* Ps = sm + L::P;
    float* Tm = sm + L::TM;
    float* gs = sm + L::G;
    float* bs = sm + L::BETA;
    float* gam = sm + L::GAM;
    float* kd = sm + L::KDEC;

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int j0 = blockIdx.y * DVT;
    const int tid = threadIdx.x;
    const int C = a.C, T = a.T, H = a.H, dv = a.dv;
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    const IO* kwp = static_cast<const IO*>(a.kw);
    IO* o = static_cast<IO*>(a.o);

    // initial state slice
    for (int idx = tid; idx < DK * DVT; idx += kSimtThreads) {
        const int c = idx / DVT, j = idx % DVT;
        Ss[c * LDV + j] =
            a.h0 ? a.h0[((size_t)bh * DK + c) * dv + j0 + j] : 0.f;
    }

    for (int t0 = 0; t0 < T; t0 += C) {
        // ---- load the chunk (zero-padded past T) ----
        for (int idx = tid; idx < C * DK; idx += kSimtThreads) {
            const int r = idx / DK, c = idx % DK;
            const int t = t0 + r;
            float qv = 0.f, kv = 0.f, wv = 0.f;
            if (t < T) {
                const size_t off = (((size_t)b * T + t) * H + h) * DK + c;
                qv = to_f32(q[off]);
                kv = to_f32(k[off]);
                if (kwp) wv = to_f32(kwp[off]);
            }
            Qs[r * LDK + c] = qv;
            Ks[r * LDK + c] = kv;
            if (kwp) KWs[r * LDK + c] = wv;
        }
        for (int idx = tid; idx < C * DVT; idx += kSimtThreads) {
            const int r = idx / DVT, j = idx % DVT;
            const int t = t0 + r;
            Xs[r * LDV + j] =
                t < T ? to_f32(v[(((size_t)b * T + t) * H + h) * dv + j0 + j])
                      : 0.f;
        }
        if (tid < C) {
            const int t = t0 + tid;
            const size_t off = ((size_t)b * T + t) * H + h;
            gs[tid] = t < T ? a.log_alpha[off] : 0.f;
            bs[tid] = t < T ? a.eta[off] : 0.f;
        }
        __syncthreads();

        // ---- beta_r and the in-chunk cumulative log decay ----
        if (tid < C) {   // n = k . (write key), ||k||^2 without write keys
            float n = 0.f;
            for (int c = 0; c < DK; ++c)
                n = fmaf(Ks[tid * LDK + c], KWs[tid * LDK + c], n);
            const float denom = n + a.eps;
            if (!a.gdn) bs[tid] = denom == 0.f ? 0.f : bs[tid] / denom;
        }
        if (tid == 32) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) {
                acc += gs[r];
                gs[r] = acc;
            }
        }
        __syncthreads();
        if (tid < C) {
            gam[tid] = expf(gs[tid]);
            kd[tid] = expf(gs[C - 1] - gs[tid]);
        }
        if (a.ckpt) {   // the state this chunk starts from
            float* ck = a.ckpt + ((size_t)bh * ((T + C - 1) / C) + t0 / C) *
                                     DK * dv + j0;
            for (int idx = tid; idx < DK * DVT; idx += kSimtThreads) {
                const int c = idx / DVT, j = idx % DVT;
                ck[(size_t)c * dv + j] = Ss[c * LDV + j];
            }
        }

        // ---- A, P, T = A^{-1} ----
        build_a_p<DK, kSimtThreads>(C, Qs, Ks, KWs, LDK, gs, bs, As, Ps, LDC);
        __syncthreads();
        invert_unit_lower<kSimtThreads>(As, Tm, C, LDC);

        // ---- K S and Q S (2 x 4 tiles): X = V - Diag(gamma) K S,
        // F = Diag(beta) X ----
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kSimtThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float ks[2][4] = {}, qs[2][4] = {};
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                const float k0 = Ks[r0 * LDK + c], k1 = Ks[(r0 + 1) * LDK + c];
                const float x0 = Qs[r0 * LDK + c], x1 = Qs[(r0 + 1) * LDK + c];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float sv = Ss[c * LDV + q0 + jj];
                    ks[0][jj] = fmaf(k0, sv, ks[0][jj]);
                    ks[1][jj] = fmaf(k1, sv, ks[1][jj]);
                    qs[0][jj] = fmaf(x0, sv, qs[0][jj]);
                    qs[1][jj] = fmaf(x1, sv, qs[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = r0 + rr;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = q0 + jj;
                    const float x = fmaf(-gam[r], ks[rr][jj], Xs[r * LDV + j]);
                    Fs[r * LDV + j] = bs[r] * x;
                    QSs[r * LDV + j] = qs[rr][jj];
                }
            }
        }
        __syncthreads();

        // ---- U~ = T F ----
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kSimtThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float u[2][4] = {};
            for (int i = 0; i <= r0 + 1; ++i) {
                const float t0v = i <= r0 ? Tm[r0 * LDC + i] : 0.f;
                const float t1v = Tm[(r0 + 1) * LDC + i];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float f = Fs[i * LDV + q0 + jj];
                    u[0][jj] = fmaf(t0v, f, u[0][jj]);
                    u[1][jj] = fmaf(t1v, f, u[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    Us[(r0 + rr) * LDV + q0 + jj] = u[rr][jj];
        }
        __syncthreads();

        // ---- O = Diag(gamma) Q S + P U~ (skipped when only the states are
        // wanted) ----
        for (int tile = tid; o && tile < (C / 2) * NCQ; tile += kSimtThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float acc[2][4];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    acc[rr][jj] = gam[r0 + rr] * QSs[(r0 + rr) * LDV + q0 + jj];
            for (int i = 0; i <= r0 + 1; ++i) {
                const float p0 = i <= r0 ? Ps[r0 * LDC + i] : 0.f;
                const float p1 = Ps[(r0 + 1) * LDC + i];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float u = Us[i * LDV + q0 + jj];
                    acc[0][jj] = fmaf(p0, u, acc[0][jj]);
                    acc[1][jj] = fmaf(p1, u, acc[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int t = t0 + r0 + rr;
                if (t >= T) continue;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    o[(((size_t)b * T + t) * H + h) * dv + j0 + q0 + jj] =
                        from_f32<IO>(acc[rr][jj]);
            }
        }

        // ---- S = gamma_C S + (Diag(Gamma_C) Kw)^T U~ (4 x 4 tiles) ----
        const float gC = gam[C - 1];
        for (int tile = tid; tile < (DK / 4) * NCQ; tile += kSimtThreads) {
            const int c0 = (tile / NCQ) * 4, q0 = (tile % NCQ) * 4;
            float acc[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    acc[x][jj] = gC * Ss[(c0 + x) * LDV + q0 + jj];
            for (int r = 0; r < C; ++r) {
                float kv[4], u[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    kv[x] = kd[r] * KWs[r * LDK + c0 + x];
                    u[x] = Us[r * LDV + q0 + x];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        acc[x][jj] = fmaf(kv[x], u[jj], acc[x][jj]);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    Ss[(c0 + x) * LDV + q0 + jj] = acc[x][jj];
        }
        __syncthreads();
    }

    if (a.hT) {
        for (int idx = tid; idx < DK * DVT; idx += kSimtThreads) {
            const int c = idx / DVT, j = idx % DVT;
            a.hT[((size_t)bh * DK + c) * dv + j0 + j] = Ss[c * LDV + j];
        }
    }
}

template <int DK, int DVT, typename T>
cudaError_t launch_shape(const FwdArgs& a, cudaStream_t stream) {
    using L = SimtSmem<DK, DVT>;
    auto kern = kla_chunk_simt_kernel<DK, DVT, T>;
    cudaError_t err = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
    if (err != cudaSuccess) return err;
    dim3 grid((unsigned)((long)a.B * a.H), (unsigned)(a.dv / DVT));
    kern<<<grid, kSimtThreads, L::BYTES, stream>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const FwdArgs& a, cudaStream_t stream) {
    // dv tile: all of dv when dv == 16, else 32 columns.
#define KLA_SIMT_DK(DKV)                                                    \
    if (a.dk == DKV) {                                                      \
        if (a.dv == 16) return launch_shape<DKV, 16, T>(a, stream);         \
        return launch_shape<DKV, 32, T>(a, stream);                         \
    }
    KLA_SIMT_DK(16)
    KLA_SIMT_DK(32)
    KLA_SIMT_DK(64)
    KLA_SIMT_DK(128)
#undef KLA_SIMT_DK
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk_simt(const FwdArgs& a, cudaStream_t stream) {
    if ((long)a.B * a.H == 0 || a.T == 0) return cudaSuccess;
    if (a.C > kSimtMaxC) return cudaErrorInvalidValue;
    if (a.dtype == KLA_BF16) return launch_dtype<__nv_bfloat16>(a, stream);
    return launch_dtype<float>(a, stream);
}

}  // namespace kla
