// Chunkwise KLA backward pass on CUDA cores, all arithmetic in fp32, for every
// supported (dk, dv, C) and both I/O types.
//
// Per chunk (rows r, i = 0..C-1; g = in-chunk cumulative log decay,
// gamma_r = exp(g_r), Gamma_ri = exp(g_r - g_i), lambda_t = exp(g_C - g_t),
// beta, A = I + strict_lower(Diag(beta)(Gamma o K K^T)), T = A^{-1},
// P = lower_incl(Gamma o Q K^T) as in the forward; S = the state the chunk
// starts from, dS' = dL/dS at its end):
//   X   = V - Diag(gamma) K S,   F = Diag(beta) X,   U~ = T F
//   dU~ = P^T dO + Diag(lambda) K dS'
//   dF  = T^T dU~,   dX = Diag(beta) dF = dV
//   dS  = gamma_C dS' + Q^T Diag(gamma) dO - K^T Diag(gamma) dX
//   dP  = dO U~^T (lower incl.),   dA = -dF U~^T (strictly lower)
//   dQ  = Diag(gamma) dO S^T + (Gamma o dP) K
//   dK  = Diag(lambda) U~ dS'^T - Diag(gamma) dX S^T + (Gamma o dP)^T Q
//         + (D + D^T) K + 2 Diag(dn) K,      D = Diag(beta) (Gamma o dA)
//   dbeta_r = sum_j dF_rj X_rj + sum_{i<r} dA_ri Gamma_ri k_r.k_i
//   deta = dbeta / (||k||^2 + eps),  dn = -dbeta beta / (||k||^2 + eps)
//          (learned-step rule: deta = dbeta, dn = 0)
//   dg_r = dgamma_r gamma_r + sum_i dGamma_ri Gamma_ri
//          - sum_r' dGamma_r'r Gamma_r'r - dlambda_r lambda_r
//          (+ sum_t dlambda_t lambda_t + <dS', S> gamma_C on the last row),
//   dlog_alpha_j = sum_{r >= j} dg_r.
// This differentiates the chunkwise form of the forward pass (the gated
// DeltaNet block solver with B = Diag(beta); gist.science/es/paper/2605.08587,
// section "Implementacion").
//
// Three launches: a forward pass writes the state at every chunk start
// (ckpt; the tensor-core kernel where it applies, else the CUDA-core one);
// the reverse recurrence walks the chunks backwards (one CTA per (batch,
// head, dv tile): the recurrence for dS is column-separable) and writes dS'
// of every chunk (dsck) and dh0; the gradient kernel then forms every
// gradient of one chunk's tokens per CTA, all chunks in parallel.  For bf16
// with dk = 128 and C = 64 the last two run on the tensor cores
// (kla_bwd_state_lm_kernel, kla_bwd_grad_lm_kernel), else on the CUDA cores
// in fp32 (kla_bwd_state_kernel, kla_bwd_grad_kernel).
#include <type_traits>

#include "kla_internal.cuh"
#include "simt_blocks.cuh"
#include "tc_primitives.cuh"

namespace kla {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdMaxC = 64;

__device__ __forceinline__ void load_chunk_qk(const BwdArgs& a, int b, int h,
                                              int t0, int DK, int LDK,
                                              float* Qs, float* Ks,
                                              float* gs, float* bs) {
    const int C = a.C, T = a.T, H = a.H;
    for (int idx = threadIdx.x; idx < C * DK; idx += kBwdThreads) {
        const int r = idx / DK, c = idx % DK;
        const int t = t0 + r;
        float qv = 0.f, kv = 0.f;
        if (t < T) {
            const size_t off = (((size_t)b * T + t) * H + h) * DK + c;
            if (a.dtype == KLA_BF16) {
                qv = to_f32(static_cast<const __nv_bfloat16*>(a.q)[off]);
                kv = to_f32(static_cast<const __nv_bfloat16*>(a.k)[off]);
            } else {
                qv = static_cast<const float*>(a.q)[off];
                kv = static_cast<const float*>(a.k)[off];
            }
        }
        Qs[r * LDK + c] = qv;
        Ks[r * LDK + c] = kv;
    }
    if (threadIdx.x < C) {
        const int t = t0 + threadIdx.x;
        const size_t off = ((size_t)b * T + t) * H + h;
        gs[threadIdx.x] = t < T ? a.log_alpha[off] : 0.f;
        bs[threadIdx.x] = t < T ? a.eta[off] : 0.f;
    }
}

// beta (raw eta in bs on entry), ||k||^2 (nrm, may be null), the cumulative
// log decay in gs, gamma and lambda.  Ends with a barrier.
template <int DK>
__device__ __forceinline__ void chunk_gates(const BwdArgs& a, const float* Ks,
                                            int LDK, float* gs, float* bs,
                                            float* gam, float* lam,
                                            float* nrm) {
    const int C = a.C, tid = threadIdx.x;
    if (tid < C) {
        float n = 0.f;
        for (int c = 0; c < DK; ++c) {
            const float x = Ks[tid * LDK + c];
            n = fmaf(x, x, n);
        }
        if (nrm) nrm[tid] = n;
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
        lam[tid] = expf(gs[C - 1] - gs[tid]);
    }
}

template <typename IO>
__device__ __forceinline__ float ld_io(const void* p, size_t off) {
    return to_f32(static_cast<const IO*>(p)[off]);
}

// ------------------------------------------------------------------ dS
template <int DK, int DVT>
struct StateSmem {
    static constexpr int LDK = DK + 1;
    static constexpr int LDV = DVT + 1;
    static constexpr int LDC = kBwdMaxC + 1;
    static constexpr int Q = 0;
    static constexpr int K = Q + kBwdMaxC * LDK;
    static constexpr int DO = K + kBwdMaxC * LDK;
    static constexpr int W = DO + kBwdMaxC * LDV;
    static constexpr int DS = W + kBwdMaxC * LDV;
    static constexpr int A = DS + DK * LDV;
    static constexpr int P = A + kBwdMaxC * LDC;
    static constexpr int G = P + kBwdMaxC * LDC;
    static constexpr int BETA = G + kBwdMaxC;
    static constexpr int GAM = BETA + kBwdMaxC;
    static constexpr int LAM = GAM + kBwdMaxC;
    static constexpr int TM = LAM + kBwdMaxC;           // A^{-1}
    static constexpr int W2 = TM + kBwdMaxC * LDC;      // dF
    static constexpr int TOTAL = W2 + kBwdMaxC * LDV;
    static constexpr size_t BYTES = sizeof(float) * (size_t)TOTAL;
};

template <int DK, int DVT, typename IO>
__global__ void __launch_bounds__(kBwdThreads)
kla_bwd_state_kernel(BwdArgs a) {
    using L = StateSmem<DK, DVT>;
    extern __shared__ float sm[];
    float* Qs = sm + L::Q;
    float* Ks = sm + L::K;
    float* Ds = sm + L::DO;
    float* Ws = sm + L::W;
    float* dS = sm + L::DS;
    float* As = sm + L::A;
    float* Ps = sm + L::P;
    float* gs = sm + L::G;
    float* bs = sm + L::BETA;
    float* gam = sm + L::GAM;
    float* lam = sm + L::LAM;
    float* Tm = sm + L::TM;
    float* W2 = sm + L::W2;

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int j0 = blockIdx.y * DVT;
    const int tid = threadIdx.x;
    const int C = a.C, T = a.T, H = a.H, dv = a.dv;
    const int nch = (T + C - 1) / C;

    for (int idx = tid; idx < DK * DVT; idx += kBwdThreads) {
        const int c = idx / DVT, j = idx % DVT;
        dS[c * L::LDV + j] =
            a.dhT ? a.dhT[((size_t)bh * DK + c) * dv + j0 + j] : 0.f;
    }

    for (int ch = nch - 1; ch >= 0; --ch) {
        const int t0 = ch * C;
        load_chunk_qk(a, b, h, t0, DK, L::LDK, Qs, Ks, gs, bs);
        for (int idx = tid; idx < C * DVT; idx += kBwdThreads) {
            const int r = idx / DVT, j = idx % DVT;
            const int t = t0 + r;
            Ds[r * L::LDV + j] =
                t < T ? ld_io<IO>(a.dout, (((size_t)b * T + t) * H + h) * dv +
                                              j0 + j)
                      : 0.f;
        }
        __syncthreads();
        chunk_gates<DK>(a, Ks, L::LDK, gs, bs, gam, lam, nullptr);
        build_a_p<DK, kBwdThreads>(C, Qs, Ks, Ks, L::LDK, gs, bs, As, Ps,
                                  L::LDC);
        {   // dL/dS at the end of this chunk
            float* out = a.dsck + ((size_t)bh * nch + ch) * DK * dv + j0;
            for (int idx = tid; idx < DK * DVT; idx += kBwdThreads) {
                const int c = idx / DVT, j = idx % DVT;
                out[(size_t)c * dv + j] = dS[c * L::LDV + j];
            }
        }
        __syncthreads();
        invert_unit_lower<kBwdThreads>(As, Tm, C, L::LDC);

        constexpr int NCQ = DVT / 4;
        constexpr int LDK = L::LDK, LDV = L::LDV, LDC = L::LDC;
        // dU~ = P^T dO + Diag(lambda) K dS' (2 x 4 tiles)
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kBwdThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float kd[2][4] = {}, pd[2][4] = {};
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                const float k0 = Ks[r0 * LDK + c], k1 = Ks[(r0 + 1) * LDK + c];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float dsv = dS[c * LDV + q0 + jj];
                    kd[0][jj] = fmaf(k0, dsv, kd[0][jj]);
                    kd[1][jj] = fmaf(k1, dsv, kd[1][jj]);
                }
            }
            for (int i = r0; i < C; ++i) {
                const float p0 = Ps[i * LDC + r0];
                const float p1 = i > r0 ? Ps[i * LDC + r0 + 1] : 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float d = Ds[i * LDV + q0 + jj];
                    pd[0][jj] = fmaf(p0, d, pd[0][jj]);
                    pd[1][jj] = fmaf(p1, d, pd[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    Ws[(r0 + rr) * LDV + q0 + jj] =
                        fmaf(lam[r0 + rr], kd[rr][jj], pd[rr][jj]);
        }
        __syncthreads();

        // dF = T^T dU~ (2 x 4 tiles)
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kBwdThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float df[2][4] = {};
            for (int i = r0; i < C; ++i) {
                const float t0v = Tm[i * LDC + r0];
                const float t1v = i > r0 ? Tm[i * LDC + r0 + 1] : 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float w = Ws[i * LDV + q0 + jj];
                    df[0][jj] = fmaf(t0v, w, df[0][jj]);
                    df[1][jj] = fmaf(t1v, w, df[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    W2[(r0 + rr) * LDV + q0 + jj] = df[rr][jj];
        }
        __syncthreads();

        // dS = gamma_C dS' + Q^T Diag(gamma) dO - K^T Diag(gamma beta) dF
        // (4 x 4 tiles of the DK x DVT slice)
        const float gC = gam[C - 1];
        for (int tile = tid; tile < (DK / 4) * NCQ; tile += kBwdThreads) {
            const int c0 = (tile / NCQ) * 4, q0 = (tile % NCQ) * 4;
            float acc[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    acc[x][jj] = gC * dS[(c0 + x) * LDV + q0 + jj];
            for (int r = 0; r < C; ++r) {
                const float gr = gam[r], gbr = gam[r] * bs[r];
                float qv[4], kv[4], d[4], w[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    qv[x] = gr * Qs[r * LDK + c0 + x];
                    kv[x] = gbr * Ks[r * LDK + c0 + x];
                    d[x] = Ds[r * LDV + q0 + x];
                    w[x] = W2[r * LDV + q0 + x];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        acc[x][jj] = fmaf(qv[x], d[jj],
                                          fmaf(-kv[x], w[jj], acc[x][jj]));
            }
            // all reads of dS happen in this tile's own entries
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    dS[(c0 + x) * LDV + q0 + jj] = acc[x][jj];
        }
        __syncthreads();
    }

    if (a.dh0) {
        for (int idx = tid; idx < DK * DVT; idx += kBwdThreads) {
            const int c = idx / DVT, j = idx % DVT;
            a.dh0[((size_t)bh * DK + c) * dv + j0 + j] = dS[c * L::LDV + j];
        }
    }
}

// ------------------------------------- reverse state recurrence, tensor cores
// The bf16 case with dk = 128, 64-column dv slices and C = 64 runs on the
// tensor cores (kla_bwd_state_lm_kernel, below the gradient kernels).
constexpr int kTcDK = 128, kTcDV = 64, kTcC = 64;

// The tensor-core recurrence applies: bf16, dk = 128, C = 64, dv a multiple
// of 64, and q, k, dO 16-byte aligned (its tile loads are 16 bytes wide).
__host__ __forceinline__ bool state_tc_ok(const BwdArgs& a) {
    auto al16 = [](const void* p) {
        return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    };
    return a.dtype == KLA_BF16 && a.dk == kTcDK && a.C == kTcC &&
           a.dv % kTcDV == 0 && al16(a.q) && al16(a.k) && al16(a.dout);
}

// ------------------------------------------------------------- gradients
template <int DK, int DVT>
struct GradSmem {
    static constexpr int LDK = DK + 1;
    static constexpr int LDV = DVT + 1;
    static constexpr int LDC = kBwdMaxC + 1;
    static constexpr int Q = 0;
    static constexpr int K = Q + kBwdMaxC * LDK;
    static constexpr int A = K + kBwdMaxC * LDK;       // later dGamma Gamma
    static constexpr int P = A + kBwdMaxC * LDC;
    static constexpr int DP = P + kBwdMaxC * LDC;      // later Gamma o dP
    static constexpr int DA = DP + kBwdMaxC * LDC;     // later D
    static constexpr int ST = DA + kBwdMaxC * LDC;     // S tile
    static constexpr int DST = ST + DK * LDV;          // dS' tile
    static constexpr int X = DST + DK * LDV;           // V, then X
    static constexpr int DO = X + kBwdMaxC * LDV;
    static constexpr int U = DO + kBwdMaxC * LDV;      // F, then U~
    static constexpr int W = U + kBwdMaxC * LDV;       // dU~, then dF
    static constexpr int KS = W + kBwdMaxC * LDV;
    static constexpr int G = KS + kBwdMaxC * LDV;
    static constexpr int BETA = G + kBwdMaxC;
    static constexpr int GAM = BETA + kBwdMaxC;
    static constexpr int LAM = GAM + kBwdMaxC;
    static constexpr int NRM = LAM + kBwdMaxC;
    static constexpr int DB = NRM + kBwdMaxC;          // dbeta, later dn
    static constexpr int DGAM = DB + kBwdMaxC;
    static constexpr int DLAM = DGAM + kBwdMaxC;
    static constexpr int DG = DLAM + kBwdMaxC;
    static constexpr int DGC = DG + kBwdMaxC;          // <dS', S>
    static constexpr int TM = DGC + 4;                 // A^{-1}
    static constexpr int TOTAL = TM + kBwdMaxC * LDC;
    static constexpr size_t BYTES = sizeof(float) * (size_t)TOTAL;
};

template <int DK, int DVT, typename IO>
__global__ void __launch_bounds__(kBwdThreads)
kla_bwd_grad_kernel(BwdArgs a) {
    using L = GradSmem<DK, DVT>;
    constexpr int LDK = L::LDK, LDV = L::LDV, LDC = L::LDC;
    constexpr int NCC = DK / 16;      // owned columns of a C x DK tile
    constexpr int NCQ = DVT / 4;      // column quads of a C x DVT matrix
    extern __shared__ float sm[];
    float* Qs = sm + L::Q;
    float* Ks = sm + L::K;
    float* As = sm + L::A;
    float* Ps = sm + L::P;
    float* dP = sm + L::DP;
    float* dA = sm + L::DA;
    float* St = sm + L::ST;
    float* dSt = sm + L::DST;
    float* Xs = sm + L::X;
    float* Ds = sm + L::DO;
    float* Us = sm + L::U;
    float* Ws = sm + L::W;
    float* KS = sm + L::KS;
    float* gs = sm + L::G;
    float* bs = sm + L::BETA;
    float* gam = sm + L::GAM;
    float* lam = sm + L::LAM;
    float* nrm = sm + L::NRM;
    float* db = sm + L::DB;
    float* dgam = sm + L::DGAM;
    float* dlam = sm + L::DLAM;
    float* dg = sm + L::DG;
    float* dgc = sm + L::DGC;
    float* Tm = sm + L::TM;

    const int C = a.C, T = a.T, H = a.H, dv = a.dv;
    const int nch = (T + C - 1) / C;
    const long blk = blockIdx.x;
    const int bh = (int)(blk / nch), ch = (int)(blk % nch);
    const int b = bh / H, h = bh % H;
    const int t0 = ch * C;
    const int tid = threadIdx.x;
    const float* Sg = a.ckpt + ((size_t)bh * nch + ch) * DK * dv;
    const float* dSg = a.dsck + ((size_t)bh * nch + ch) * DK * dv;

    load_chunk_qk(a, b, h, t0, DK, LDK, Qs, Ks, gs, bs);
    for (int idx = tid; idx < C * LDC; idx += kBwdThreads) {
        dP[idx] = 0.f;
        dA[idx] = 0.f;
    }
    if (tid < kBwdMaxC) {
        db[tid] = 0.f;
        dgam[tid] = 0.f;
        dlam[tid] = 0.f;
    }
    if (tid == 0) dgc[0] = 0.f;
    __syncthreads();
    chunk_gates<DK>(a, Ks, LDK, gs, bs, gam, lam, nrm);
    build_a_p<DK, kBwdThreads>(C, Qs, Ks, Ks, LDK, gs, bs, As, Ps, LDC);
    __syncthreads();
    invert_unit_lower<kBwdThreads>(As, Tm, C, LDC);

    // owned 4 x NCC tile of the C x DK gradients dQ, dK: rows 4 rg + rr,
    // columns cg + 16 cc
    const int cg = tid % 16, rg = tid / 16;
    float dq_acc[4][NCC], dk_acc[4][NCC];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int cc = 0; cc < NCC; ++cc) dq_acc[rr][cc] = dk_acc[rr][cc] = 0.f;

    for (int j0 = 0; j0 < dv; j0 += DVT) {
        float sdot = 0.f;
        for (int idx = tid; idx < DK * DVT; idx += kBwdThreads) {
            const int c = idx / DVT, j = idx % DVT;
            const float sv = Sg[(size_t)c * dv + j0 + j];
            const float dsv = dSg[(size_t)c * dv + j0 + j];
            St[c * LDV + j] = sv;
            dSt[c * LDV + j] = dsv;
            sdot = fmaf(sv, dsv, sdot);
        }
        atomicAdd(dgc, sdot);
        for (int idx = tid; idx < C * DVT; idx += kBwdThreads) {
            const int r = idx / DVT, j = idx % DVT;
            const int t = t0 + r;
            const size_t off = (((size_t)b * T + t) * H + h) * dv + j0 + j;
            Xs[r * LDV + j] = t < T ? ld_io<IO>(a.v, off) : 0.f;
            Ds[r * LDV + j] = t < T ? ld_io<IO>(a.dout, off) : 0.f;
        }
        __syncthreads();

        // K S, Q S (2 x 4 tiles): X = V - Diag(gamma) K S, F = Diag(beta) X
        // (into W), dgamma += dO . Q S
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kBwdThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float ks[2][4] = {}, qs[2][4] = {};
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                const float k0 = Ks[r0 * LDK + c], k1 = Ks[(r0 + 1) * LDK + c];
                const float x0 = Qs[r0 * LDK + c], x1 = Qs[(r0 + 1) * LDK + c];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float sv = St[c * LDV + q0 + jj];
                    ks[0][jj] = fmaf(k0, sv, ks[0][jj]);
                    ks[1][jj] = fmaf(k1, sv, ks[1][jj]);
                    qs[0][jj] = fmaf(x0, sv, qs[0][jj]);
                    qs[1][jj] = fmaf(x1, sv, qs[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = r0 + rr;
                float dgp = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = q0 + jj;
                    KS[r * LDV + j] = ks[rr][jj];
                    const float x = fmaf(-gam[r], ks[rr][jj], Xs[r * LDV + j]);
                    Xs[r * LDV + j] = x;
                    Ws[r * LDV + j] = bs[r] * x;
                    dgp = fmaf(Ds[r * LDV + j], qs[rr][jj], dgp);
                }
                atomicAdd(&dgam[r], dgp);
            }
        }
        __syncthreads();

        // U~ = T F
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kBwdThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float u[2][4] = {};
            for (int i = 0; i <= r0 + 1; ++i) {
                const float t0v = i <= r0 ? Tm[r0 * LDC + i] : 0.f;
                const float t1v = Tm[(r0 + 1) * LDC + i];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float f = Ws[i * LDV + q0 + jj];
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

        // dU~ = P^T dO + Diag(lambda) K dS' (into W); dlambda_r = (K dS')_r.U~_r
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kBwdThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float kd[2][4] = {}, pd[2][4] = {};
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                const float k0 = Ks[r0 * LDK + c], k1 = Ks[(r0 + 1) * LDK + c];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float dsv = dSt[c * LDV + q0 + jj];
                    kd[0][jj] = fmaf(k0, dsv, kd[0][jj]);
                    kd[1][jj] = fmaf(k1, dsv, kd[1][jj]);
                }
            }
            for (int i = r0; i < C; ++i) {
                const float p0 = Ps[i * LDC + r0];
                const float p1 = i > r0 ? Ps[i * LDC + r0 + 1] : 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float d = Ds[i * LDV + q0 + jj];
                    pd[0][jj] = fmaf(p0, d, pd[0][jj]);
                    pd[1][jj] = fmaf(p1, d, pd[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = r0 + rr;
                float dlp = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = q0 + jj;
                    Ws[r * LDV + j] = fmaf(lam[r], kd[rr][jj], pd[rr][jj]);
                    dlp = fmaf(kd[rr][jj], Us[r * LDV + j], dlp);
                }
                atomicAdd(&dlam[r], dlp);
            }
        }
        __syncthreads();

        // dF = T^T dU~ (into the K S slots, once read); dV = dX =
        // Diag(beta) dF; dbeta from F = Diag(beta) X; dgamma from X
        for (int tile = tid; tile < (C / 2) * NCQ; tile += kBwdThreads) {
            const int r0 = (tile / NCQ) * 2, q0 = (tile % NCQ) * 4;
            float df[2][4] = {};
            for (int i = r0; i < C; ++i) {
                const float t0v = Tm[i * LDC + r0];
                const float t1v = i > r0 ? Tm[i * LDC + r0 + 1] : 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float w = Ws[i * LDV + q0 + jj];
                    df[0][jj] = fmaf(t0v, w, df[0][jj]);
                    df[1][jj] = fmaf(t1v, w, df[1][jj]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = r0 + rr;
                const int t = t0 + r;
                float dbp = 0.f, dgp = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = q0 + jj;
                    const float dx = bs[r] * df[rr][jj];
                    if (t < T)
                        static_cast<IO*>(a.dv_)[(((size_t)b * T + t) * H + h) *
                                                    dv + j0 + j] =
                            from_f32<IO>(dx);
                    dbp = fmaf(df[rr][jj], Xs[r * LDV + j], dbp);
                    dgp = fmaf(-dx, KS[r * LDV + j], dgp);
                    KS[r * LDV + j] = df[rr][jj];
                }
                atomicAdd(&db[r], dbp);
                atomicAdd(&dgam[r], dgp);
            }
        }
        __syncthreads();

        // dP = dO U~^T (i <= r), dA = -dF U~^T (i < r): 4 x 4 tiles
        {
            const int nrt = C / 4;
            for (int tile = tid; tile < nrt * nrt; tile += kBwdThreads) {
                const int r0 = (tile / nrt) * 4, i0 = (tile % nrt) * 4;
                if (i0 > r0 + 3) continue;
                float ap[4][4] = {}, aa[4][4] = {};
#pragma unroll 4
                for (int j = 0; j < DVT; ++j) {
                    float d[4], f[4], u[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        d[x] = Ds[(r0 + x) * LDV + j];
                        f[x] = KS[(r0 + x) * LDV + j];
                        u[x] = Us[(i0 + x) * LDV + j];
                    }
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                        for (int ii = 0; ii < 4; ++ii) {
                            ap[rr][ii] = fmaf(d[rr], u[ii], ap[rr][ii]);
                            aa[rr][ii] = fmaf(f[rr], u[ii], aa[rr][ii]);
                        }
                }
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const int r = r0 + rr, i = i0 + ii;
                        if (i <= r) dP[r * LDC + i] += ap[rr][ii];
                        if (i < r) dA[r * LDC + i] -= aa[rr][ii];
                    }
            }
        }
        // owned (r, c): dQ += gamma_r dO S^T;
        // dK += lambda_r U~ dS'^T - gamma_r beta_r dF S^T
#pragma unroll 2
        for (int j = 0; j < DVT; ++j) {
            float d[4], u[4], f[4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int r = 4 * rg + rr;
                const bool in = r < C;
                d[rr] = in ? gam[r] * Ds[r * LDV + j] : 0.f;
                u[rr] = in ? lam[r] * Us[r * LDV + j] : 0.f;
                f[rr] = in ? gam[r] * bs[r] * KS[r * LDV + j] : 0.f;
            }
#pragma unroll
            for (int cc = 0; cc < NCC; ++cc) {
                const int c = cg + 16 * cc;
                const float sv = St[c * LDV + j], dsv = dSt[c * LDV + j];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    dq_acc[rr][cc] = fmaf(d[rr], sv, dq_acc[rr][cc]);
                    dk_acc[rr][cc] =
                        fmaf(u[rr], dsv, fmaf(-f[rr], sv, dk_acc[rr][cc]));
                }
            }
        }
        __syncthreads();
    }

    // dGamma o Gamma (into A), Gamma o dP (into dP), D (into dA), and the
    // A-part of dbeta: 4 x 4 tiles of the lower triangle
    {
        const int nrt = C / 4;
        for (int tile = tid; tile < nrt * nrt; tile += kBwdThreads) {
            const int r0 = (tile / nrt) * 4, i0 = (tile % nrt) * 4;
            if (i0 > r0 + 3) continue;
            float qk[4][4] = {}, kk[4][4] = {};
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                float qr[4], kr[4], ki[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    qr[x] = Qs[(r0 + x) * LDK + c];
                    kr[x] = Ks[(r0 + x) * LDK + c];
                    ki[x] = Ks[(i0 + x) * LDK + c];
                }
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        qk[rr][ii] = fmaf(qr[rr], ki[ii], qk[rr][ii]);
                        kk[rr][ii] = fmaf(kr[rr], ki[ii], kk[rr][ii]);
                    }
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int r = r0 + rr;
                float dbp = 0.f;
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const int i = i0 + ii;
                    float dgg = 0.f, dpt = 0.f, dd = 0.f;
                    if (i <= r) {
                        const float gmm = expf(gs[r] - gs[i]);
                        const float dpv = dP[r * LDC + i];
                        float dgm = dpv * qk[rr][ii];
                        dpt = gmm * dpv;
                        if (i < r) {
                            const float dav = dA[r * LDC + i];
                            dgm = fmaf(dav * bs[r], kk[rr][ii], dgm);
                            dd = bs[r] * gmm * dav;
                            dbp = fmaf(dav * gmm, kk[rr][ii], dbp);
                        }
                        dgg = dgm * gmm;
                    }
                    As[r * LDC + i] = dgg;
                    dP[r * LDC + i] = dpt;
                    dA[r * LDC + i] = dd;
                }
                atomicAdd(&db[r], dbp);
            }
        }
    }
    __syncthreads();

    // per row: dg, deta, dn (dn replaces dbeta in db)
    if (tid < C) {
        const int r = tid;
        float g = dgam[r] * gam[r] - dlam[r] * lam[r];
        for (int i = 0; i <= r; ++i) g += As[r * LDC + i];
        for (int rr = r; rr < C; ++rr) g -= As[rr * LDC + r];
        if (r == C - 1) {
            for (int t = 0; t < C; ++t) g = fmaf(dlam[t], lam[t], g);
            g = fmaf(dgc[0], gam[C - 1], g);
        }
        dg[r] = g;
        const float dbeta = db[r];
        float deta, dn = 0.f;
        if (a.gdn) {
            deta = dbeta;
        } else {
            const float denom = nrm[r] + a.eps;
            deta = denom == 0.f ? 0.f : dbeta / denom;
            if (denom != 0.f) dn = -dbeta * bs[r] / denom;
        }
        const int t = t0 + r;
        if (t < T) a.deta[((size_t)b * T + t) * H + h] = deta;
        db[r] = dn;
    }
    __syncthreads();
    if (tid < C) {   // dlog_alpha_j = sum_{r >= j} dg_r
        float acc = 0.f;
        for (int r = tid; r < C; ++r) acc += dg[r];
        const int t = t0 + tid;
        if (t < T) a.dlog_alpha[((size_t)b * T + t) * H + h] = acc;
    }

    // dQ += (Gamma o dP) K;  dK += (Gamma o dP)^T Q + (D + D^T) K + 2 dn k
    for (int i = 0; i < C; ++i) {
        float kv[NCC], qv[NCC];
#pragma unroll
        for (int cc = 0; cc < NCC; ++cc) {
            kv[cc] = Ks[i * LDK + cg + 16 * cc];
            qv[cc] = Qs[i * LDK + cg + 16 * cc];
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = 4 * rg + rr;
            if (r >= C) continue;
            const float dp = i <= r ? dP[r * LDC + i] : 0.f;
            const float dd = i < r ? dA[r * LDC + i] : 0.f;
            const float dpT = i >= r ? dP[i * LDC + r] : 0.f;
            const float ddT = i > r ? dA[i * LDC + r] : 0.f;
#pragma unroll
            for (int cc = 0; cc < NCC; ++cc) {
                dq_acc[rr][cc] = fmaf(dp, kv[cc], dq_acc[rr][cc]);
                dk_acc[rr][cc] = fmaf(dd + ddT, kv[cc],
                                      fmaf(dpT, qv[cc], dk_acc[rr][cc]));
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int r = 4 * rg + rr;
        const int t = t0 + r;
        if (r >= C || t >= T) continue;
#pragma unroll
        for (int cc = 0; cc < NCC; ++cc) {
            const int c = cg + 16 * cc;
            const size_t off = (((size_t)b * T + t) * H + h) * DK + c;
            static_cast<IO*>(a.dq)[off] = from_f32<IO>(dq_acc[rr][cc]);
            static_cast<IO*>(a.dk_)[off] = from_f32<IO>(
                fmaf(2.f * db[r], Ks[r * LDK + c], dk_acc[rr][cc]));
        }
    }
}

// Lower 16 x 8 tiles (mt, nt) of a 64 x 64 matrix (8 nt <= 16 mt + 15):
// tile index 0 .. 19 -> (mt, nt).
__device__ __forceinline__ void lower_tile(int idx, int& mt, int& nt) {
    mt = idx < 2 ? 0 : idx < 6 ? 1 : idx < 12 ? 2 : 3;
    const int first = mt == 0 ? 0 : mt == 1 ? 2 : mt == 2 ? 6 : 12;
    nt = idx - first;
}

// ------------------------------ gradients, tensor cores, bf16 operand tiles
// The per-chunk gradients of kla_bwd_grad_kernel for bf16 inputs with
// dk = 128, C = 64, every product on the tensor cores (warp-level m16n8k16
// MMAs, bf16 operands, fp32 accumulation), every MMA operand kept once in
// shared memory as a bf16 tile whose rows are 16-byte
// aligned and 16 bytes apart modulo 128 (row strides of 136, 72 and 40
// elements), read by ldmatrix: one instruction per 16 x 16 (or two 16 x 8)
// fragment, transposed on the fly where the product needs the other
// orientation, and no bank conflict.  fp32 tiles stay only where an
// elementwise step needs them (X, K S, U~) and for the inverse; dP and dA
// accumulate in registers over the dv steps.  Inputs are bf16, so q and k
// go to shared memory unconverted, and K K^T, Q K^T (for A, P and the
// decay and beta terms at the end) are tensor-core products of the exact
// inputs.
using bf16 = __nv_bfloat16;

namespace lm {
constexpr int C = 64, DK = 128, DVT = 32;
constexpr int LQ = DK + 8;    // q, k rows (bf16)
constexpr int LC = C + 8;     // C x C bf16 tiles
constexpr int LV = DVT + 8;   // C x DVT and DK x DVT bf16 tiles
constexpr int LF = C + 1;     // C x C fp32 (inverse, final phase)
constexpr int LX = DVT + 1;   // C x DVT fp32
// byte offsets
constexpr int QB = 0;
constexpr int KB = QB + C * LQ * 2;
constexpr int TB = KB + C * LQ * 2;          // T = A^{-1}, lower
constexpr int PB = TB + C * LC * 2;          // P, lower incl.
constexpr int F0 = PB + C * LC * 2;          // fp32: A, later dP
constexpr int F1 = F0 + C * LF * 4;          // fp32: T, later D
constexpr int F2 = F1 + C * LF * 4;          // fp32: dGamma o Gamma
constexpr int SB = F2 + C * LF * 4;          // S (DK x DVT), later Gamma o dP
constexpr int DSB = SB + DK * LV * 2;        // dS', later D + D^T
constexpr int XF = DSB + DK * LV * 2;        // V, then X (fp32)
constexpr int KSF = XF + C * LX * 4;         // K S (fp32)
constexpr int UF = KSF + C * LX * 4;         // U~ (fp32)
constexpr int FB = UF + C * LX * 4;          // F = Diag(beta) X
constexpr int UB = FB + C * LV * 2;          // U~
constexpr int ULB = UB + C * LV * 2;         // Diag(lambda) U~
constexpr int DUB = ULB + C * LV * 2;        // dU~
constexpr int DOB = DUB + C * LV * 2;        // dO
constexpr int DOG = DOB + C * LV * 2;        // Diag(gamma) dO
constexpr int DFB = DOG + C * LV * 2;        // dF
constexpr int DFS = DFB + C * LV * 2;        // -Diag(gamma beta) dF
constexpr int SMALL = DFS + C * LV * 2;      // fp32 vectors of C
constexpr int NVEC = 11;   // gs bs gam lam nrm db dgam dlam dg gb dgc
constexpr int BYTES = SMALL + NVEC * C * 4;
static_assert(C * LC * 2 * 2 <= 2 * DK * LV * 2, "final tiles fit");
static_assert(BYTES <= 232448, "shared memory");
static_assert(QB % 16 == 0 && KB % 16 == 0 && TB % 16 == 0 && PB % 16 == 0 &&
                  SB % 16 == 0 && DSB % 16 == 0 && FB % 16 == 0 &&
                  UB % 16 == 0 && ULB % 16 == 0 && DUB % 16 == 0 &&
                  DOB % 16 == 0 && DOG % 16 == 0 && DFB % 16 == 0 &&
                  DFS % 16 == 0,
              "ldmatrix rows are 16-byte aligned");

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
    asm volatile(
        "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(tc::smem_u32(p)));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const void* p) {
    asm volatile(
        "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, "
        "[%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(tc::smem_u32(p)));
}

// A fragment (16 x 16) of the row-major tile at p (row stride ld elements):
// A(m, k) = p[m ld + k].
__device__ __forceinline__ void a_row(uint32_t (&a)[4], const bf16* p, int ld,
                                      int lane) {
    ldsm4(a, p + (lane & 15) * ld + (lane >> 4) * 8);
}
// A fragment of the transpose: A(m, k) = p[k ld + m].
__device__ __forceinline__ void a_trn(uint32_t (&a)[4], const bf16* p, int ld,
                                      int lane) {
    const int i = lane >> 3;
    ldsm4t(a, p + ((i >> 1) * 8 + (lane & 7)) * ld + (i & 1) * 8);
}
// B fragments of two adjacent 16 x 8 tiles (columns n .. n + 15) of the
// row-major tile at p: B(k, n) = p[k ld + n]; b[0..1] the first, b[2..3]
// the second.
__device__ __forceinline__ void b_row2(uint32_t (&b)[4], const bf16* p, int ld,
                                       int lane) {
    const int i = lane >> 3;
    ldsm4t(b, p + ((i & 1) * 8 + (lane & 7)) * ld + (i >> 1) * 8);
}
// The same for B(k, n) = p[n ld + k] (the tile holds B's columns as rows).
__device__ __forceinline__ void b_col2(uint32_t (&b)[4], const bf16* p, int ld,
                                       int lane) {
    const int i = lane >> 3;
    ldsm4(b, p + ((i >> 1) * 8 + (lane & 7)) * ld + (i & 1) * 8);
}
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4],
                                    uint32_t b0, uint32_t b1) {
    tc::mma_m16n8k16(d, a, b0, b1);
}
__device__ __forceinline__ float bf(const bf16* p, int i) {
    return __bfloat162float(p[i]);
}
// 16-byte asynchronous copy global -> shared (zeros when !valid; src must
// still point into the tensor).
__device__ __forceinline__ void cp_async16(void* dst, const void* src,
                                           bool valid) {
    asm volatile(
        "cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
            tc::smem_u32(dst)),
        "l"(src), "r"(valid ? 16 : 0)
        : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// staging of one dv step in the fp32 scratch (S | dS' fp32, V | dO bf16)
constexpr int STG_DS = DK * DVT * 4, STG_V = 2 * DK * DVT * 4,
              STG_DO = STG_V + C * DVT * 2, STG_END = STG_DO + C * DVT * 2;
static_assert(F0 + STG_END <= SB, "staging fits in the fp32 scratch");

// acc (16 x 8) += A (16 x 16 fp32 block, row stride la) x B[:, 0..7] (16 x 8
// of an fp32 block, row stride lb): two tf32 m16n8k8 MMAs.
__device__ __forceinline__ void mm16x8_tf32(float (&acc)[4], const float* A,
                                            int la, const float* B, int lb,
                                            int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[4];
        a[0] = tc::to_tf32(A[g * la + 8 * kk + t]);
        a[1] = tc::to_tf32(A[(g + 8) * la + 8 * kk + t]);
        a[2] = tc::to_tf32(A[g * la + 8 * kk + t + 4]);
        a[3] = tc::to_tf32(A[(g + 8) * la + 8 * kk + t + 4]);
        tc::mma_m16n8k8_tf32(acc, a, tc::to_tf32(B[(8 * kk + t) * lb + g]),
                             tc::to_tf32(B[(8 * kk + t + 4) * lb + g]));
    }
}

// T = A^{-1} for the unit lower-triangular 64 x 64 A (fp32, row stride la;
// only its strict lower part is read), into the lower part of Tm (row
// stride lt; the 16 x 16 blocks above the diagonal are left as they were).
// The diagonal blocks by fp32 column substitution (threads 0..63), the
// blocks below them in three levels, T_IJ = -T_II (sum_{m=J}^{I-1} A_Im
// T_mJ) for 8-column slabs on the tensor cores (tf32 operands, fp32
// accumulation), the sum passed through Y (16 x 8 floats per warp).  All 256
// threads take part; ends with a barrier.
__device__ __forceinline__ void invert_lower64(const float* A, int la,
                                               float* Tm, int lt, float* Y) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    if (tid < 64) {
        const int bb = tid >> 4, cl = tid & 15;
        const float* Ab = A + 16 * bb * la + 16 * bb;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == cl ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < r; i += 2) {
                a0 = fmaf(Ab[r * la + i], x[i], a0);
                if (i + 1 < r) a1 = fmaf(Ab[r * la + i + 1], x[i + 1], a1);
            }
            if (r > cl) x[r] = -(a0 + a1);
        }
        float* Tb = Tm + 16 * bb * lt + 16 * bb + cl;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * lt] = x[r];
    }
    __syncthreads();
    float* Yw = Y + warp * 128;
    auto slab = [&](int I, int J, int n0) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int m = J; m < I; ++m)
            mm16x8_tf32(acc, A + 16 * I * la + 16 * m, la,
                        Tm + 16 * m * lt + 16 * J + n0, lt, lane);
        Yw[g * 8 + 2 * t] = acc[0];
        Yw[g * 8 + 2 * t + 1] = acc[1];
        Yw[(g + 8) * 8 + 2 * t] = acc[2];
        Yw[(g + 8) * 8 + 2 * t + 1] = acc[3];
        __syncwarp();
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mm16x8_tf32(d, Tm + 16 * I * lt + 16 * I, lt, Yw, 8, lane);
        __syncwarp();
        float* dst = Tm + 16 * I * lt + 16 * J + n0;
        dst[g * lt + 2 * t] = -d[0];
        dst[g * lt + 2 * t + 1] = -d[1];
        dst[(g + 8) * lt + 2 * t] = -d[2];
        dst[(g + 8) * lt + 2 * t + 1] = -d[3];
    };
    // level 1: (1,0), (2,1), (3,2) -- two 8-column slabs each
    if (warp < 6) slab((warp >> 1) + 1, warp >> 1, 8 * (warp & 1));
    __syncthreads();
    // level 2: (2,0), (3,1)
    if (warp < 4) slab(2 + (warp >> 1), warp >> 1, 8 * (warp & 1));
    __syncthreads();
    // level 3: (3,0)
    if (warp < 2) slab(3, 0, 8 * warp);
    __syncthreads();
}

// Sum over the four lanes that share a fragment row (lane >> 2).
__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}

// ||k_r||^2 from a bf16 row (row stride LQ), four threads per row, 32
// dimensions each (16-byte loads); the sum ends in all four.
__device__ __forceinline__ float row_norm2(const bf16* Kb, int r, int q4) {
    float n = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(Kb + r * LQ + 32 * q4 +
                                                        8 * u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16);
            const float hi = __uint_as_float(w[e] & 0xffff0000u);
            n = fmaf(lo, lo, n);
            n = fmaf(hi, hi, n);
        }
    }
    return quad_sum(n);
}

// Q K^T and K K^T on this warp's lower 16 x 8 tiles of the C x C products
// (tile indices warp + NW x below 20, for NW warps), the tiles' MMA chains
// interleaved.
template <int NW = 8>
__device__ __forceinline__ void qk_kk_tiles(
    float (&qk)[(20 + NW - 1) / NW][4], float (&kk)[(20 + NW - 1) / NW][4],
    int (&mt)[(20 + NW - 1) / NW], int (&nt)[(20 + NW - 1) / NW],
    const bf16* Qb, const bf16* Kb, int warp, int lane) {
    constexpr int XT = (20 + NW - 1) / NW;
#pragma unroll
    for (int x = 0; x < XT; ++x) {
        const int idx = warp + NW * x;
        lower_tile(idx < 20 ? idx : warp, mt[x], nt[x]);
#pragma unroll
        for (int e = 0; e < 4; ++e) qk[x][e] = kk[x][e] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < DK / 16; ++ks) {
#pragma unroll
        for (int x = 0; x < XT; ++x) {
            if (warp + NW * x < 20) {
                uint32_t aq[4], ak[4], bk[4];
                a_row(aq, Qb + 16 * mt[x] * LQ + 16 * ks, LQ, lane);
                a_row(ak, Kb + 16 * mt[x] * LQ + 16 * ks, LQ, lane);
                // K^T columns 8 nt .. 8 nt + 7 (and the next 8, unused)
                b_col2(bk, Kb + 8 * nt[x] * LQ + 16 * ks, LQ, lane);
                mma(qk[x], aq, bk[0], bk[1]);
                mma(kk[x], ak, bk[0], bk[1]);
            }
        }
    }
}
}  // namespace lm

// ------------------------------------ per-chunk records of the backward
// What the two tensor-core backward kernels need of a chunk and that does
// not depend on the state or on dO (layout bwdrec): written by the
// two-kernel forward's pre-pass when the checkpoints come from that path,
// else by kla_bwd_prep_kernel.
namespace brec = bwdrec;

template <typename IO, int NW>
__global__ void __launch_bounds__(32 * NW, 1)
kla_bwd_grad_lm_kernel(BwdArgs a) {
    using namespace lm;
    // NW warps: the C x DVT products' 16 x 8 tiles (TPW per warp, WPR warps
    // per 16-row block), the 20 lower 16 x 8 tiles of the C x C products
    // (XT at most per warp) and the dq / dk fragments (rows 16 (w & 3),
    // CQ columns) are dealt out to them
    constexpr int NT = 32 * NW, WPR = NW / 4, TPW = 4 / WPR;
    constexpr int XT = (20 + NW - 1) / NW, CQ = 128 / WPR, NQ = CQ / 8;
    static_assert(NW == 8 || NW == 16, "8 or 16 warps");
    extern __shared__ __align__(16) uint8_t smraw[];
    bf16* Qb = reinterpret_cast<bf16*>(smraw + QB);
    bf16* Kb = reinterpret_cast<bf16*>(smraw + KB);
    bf16* Tb = reinterpret_cast<bf16*>(smraw + TB);
    bf16* Pb = reinterpret_cast<bf16*>(smraw + PB);
    float* F0f = reinterpret_cast<float*>(smraw + F0);
    float* F1f = reinterpret_cast<float*>(smraw + F1);
    float* F2f = reinterpret_cast<float*>(smraw + F2);
    bf16* Sb = reinterpret_cast<bf16*>(smraw + SB);
    bf16* dSb = reinterpret_cast<bf16*>(smraw + DSB);
    float* Xf = reinterpret_cast<float*>(smraw + XF);
    float* KSf = reinterpret_cast<float*>(smraw + KSF);
    float* Uf = reinterpret_cast<float*>(smraw + UF);
    bf16* Fb = reinterpret_cast<bf16*>(smraw + FB);
    bf16* Ub = reinterpret_cast<bf16*>(smraw + UB);
    bf16* Ulb = reinterpret_cast<bf16*>(smraw + ULB);
    bf16* dUb = reinterpret_cast<bf16*>(smraw + DUB);
    bf16* dOb = reinterpret_cast<bf16*>(smraw + DOB);
    bf16* dOg = reinterpret_cast<bf16*>(smraw + DOG);
    bf16* dFb = reinterpret_cast<bf16*>(smraw + DFB);
    bf16* dFs = reinterpret_cast<bf16*>(smraw + DFS);
    float* vec = reinterpret_cast<float*>(smraw + SMALL);
    float* gs = vec;             // cumulative log decay
    float* bs = vec + C;         // beta (eta on entry)
    float* gam = vec + 2 * C;
    float* lam = vec + 3 * C;
    float* nrm = vec + 4 * C;
    float* db = vec + 5 * C;     // dbeta, later dn
    float* dgam = vec + 6 * C;
    float* dlam = vec + 7 * C;
    float* dg = vec + 8 * C;
    float* gb = vec + 9 * C;     // -gamma beta
    float* dgc = vec + 10 * C;   // <dS', S>
    // the final phase's bf16 tiles over S and dS'
    bf16* Gdp = Sb;              // Gamma o dP (C x C)
    bf16* Ddt = dSb;             // D + D^T

    const int T = a.T, H = a.H, dv = a.dv;
    const int nch = (T + C - 1) / C;
    const long blk = blockIdx.x;
    const int bh = (int)(blk / nch), ch = (int)(blk % nch);
    const int b = bh / H, h = bh % H;
    const int t0 = ch * C;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const float* Sg = a.ckpt + ((size_t)bh * nch + ch) * DK * dv;
    const float* dSg = a.dsck + ((size_t)bh * nch + ch) * DK * dv;

    {   // q, k rows (bf16, 16-byte loads straight to shared memory); T, P
        // (bf16), g, beta and ||k||^2 from the chunk's record
#pragma unroll
        for (int u = 0; u < 1024 / NT; ++u) {
            const int idx = tid + u * NT;   // 64 rows x 16 chunks
            const int r = idx >> 4, c8 = idx & 15;
            const int t = t0 + r;
            uint4 qv = make_uint4(0, 0, 0, 0), kv = make_uint4(0, 0, 0, 0);
            if (t < T) {
                const size_t off = (((size_t)b * T + t) * H + h) * DK + 8 * c8;
                qv = *reinterpret_cast<const uint4*>(
                    static_cast<const IO*>(a.q) + off);
                kv = *reinterpret_cast<const uint4*>(
                    static_cast<const IO*>(a.k) + off);
            }
            *reinterpret_cast<uint4*>(Qb + r * LQ + 8 * c8) = qv;
            *reinterpret_cast<uint4*>(Kb + r * LQ + 8 * c8) = kv;
        }
        const uint8_t* rec = a.rec + ((size_t)bh * nch + ch) * brec::BYTES;
#pragma unroll
        for (int m = 0; m < 512 / NT; ++m) {   // 512 pieces of 16 bytes
            const int u = tid + m * NT, r = u >> 3, c8 = u & 7;
            *reinterpret_cast<uint4*>(Tb + r * LC + 8 * c8) =
                reinterpret_cast<const uint4*>(rec + brec::T_OFF)[u];
            *reinterpret_cast<uint4*>(Pb + r * LC + 8 * c8) =
                reinterpret_cast<const uint4*>(rec + brec::P_OFF)[u];
        }
        if (tid < C) {
            gs[tid] = reinterpret_cast<const float*>(rec + brec::G_OFF)[tid];
            bs[tid] = reinterpret_cast<const float*>(rec + brec::B_OFF)[tid];
            nrm[tid] = reinterpret_cast<const float*>(rec + brec::N_OFF)[tid];
            db[tid] = dgam[tid] = dlam[tid] = 0.f;
        }
        if (tid == 0) dgc[0] = 0.f;
    }
    __syncthreads();
    if (tid < C) {
        gam[tid] = expf(gs[tid]);
        lam[tid] = expf(gs[C - 1] - gs[tid]);
        gb[tid] = -gam[tid] * bs[tid];
    }

    // dq, dk of this warp's rows 16 mo .. and columns CQ co .. (fragments)
    const int mo = warp & 3, co = CQ * (warp >> 2);
    float dq[NQ][4], dk[NQ][4];
#pragma unroll
    for (int nt = 0; nt < NQ; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dq[nt][e] = dk[nt][e] = 0.f;
    // dP, dA of this warp's lower tiles (idx = warp + NW x)
    float dPa[XT][4], dAa[XT][4];
#pragma unroll
    for (int x = 0; x < XT; ++x)
#pragma unroll
        for (int e = 0; e < 4; ++e) dPa[x][e] = dAa[x][e] = 0.f;
    // this warp's TPW 16 x 8 tiles of the C x DVT products: rows 16 pm,
    // columns pn .. pn + 8 TPW - 1 (the B fragments are loaded two tiles
    // at a time; with one tile per warp the second is not used)
    const int pm = warp / WPR, pn = 8 * TPW * (warp % WPR);
    float sdot = 0.f;
    __syncthreads();

    // Steps after the first are staged one step ahead by cp.async in the
    // fp32 scratch, which the dv steps leave free; each thread copies and
    // later reads back the same 16-byte pieces, so no barrier guards the
    // staging area.
    uint8_t* stage = smraw + F0;
    auto stage_issue = [&](int jn) {
#pragma unroll
        for (int u = 0; u < 1024 / NT; ++u) {
            const int idx = tid + u * NT;   // 128 rows x 8
            const int c = idx >> 3, j4 = idx & 7;
            cp_async16(stage + (c * DVT + 4 * j4) * 4,
                       Sg + (size_t)c * dv + jn + 4 * j4, true);
            cp_async16(stage + STG_DS + (c * DVT + 4 * j4) * 4,
                       dSg + (size_t)c * dv + jn + 4 * j4, true);
        }
        if (tid < 256) {
            const int r = tid >> 2, j8 = tid & 3;   // 64 rows x 4
            const int t = t0 + r;
            const size_t off = (((size_t)b * T + (t < T ? t : t0)) * H + h) *
                                   dv + jn + 8 * j8;
            cp_async16(stage + STG_V + (r * DVT + 8 * j8) * 2,
                       static_cast<const IO*>(a.v) + off, t < T);
            cp_async16(stage + STG_DO + (r * DVT + 8 * j8) * 2,
                       static_cast<const IO*>(a.dout) + off, t < T);
        }
        cp_async_commit();
    };

    for (int j0 = 0; j0 < dv; j0 += DVT) {
        {   // S, dS' (DK x DVT fp32 -> bf16), V (fp32), dO (bf16, and
            // Diag(gamma) dO): from global memory for the first step (every
            // load issued before the stores), from the staging area after
            constexpr int U = 1024 / NT;
            float4 sv[U], dsv[U];
            const bool vt = tid < 256;   // V and dO: 64 rows x 4 pieces
            const int r = (tid & 255) >> 2, j8 = tid & 3;
            const int t = t0 + r;
            uint4 vv = make_uint4(0, 0, 0, 0), dov = make_uint4(0, 0, 0, 0);
            if (j0 == 0) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int idx = tid + u * NT;   // 128 rows x 8
                    const int c = idx >> 3, j4 = idx & 7;
                    sv[u] = *reinterpret_cast<const float4*>(
                        Sg + (size_t)c * dv + j0 + 4 * j4);
                    dsv[u] = *reinterpret_cast<const float4*>(
                        dSg + (size_t)c * dv + j0 + 4 * j4);
                }
                if (vt && t < T) {
                    const size_t off =
                        (((size_t)b * T + t) * H + h) * dv + j0 + 8 * j8;
                    vv = *reinterpret_cast<const uint4*>(
                        static_cast<const IO*>(a.v) + off);
                    dov = *reinterpret_cast<const uint4*>(
                        static_cast<const IO*>(a.dout) + off);
                }
            } else {
                cp_async_wait_all();
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int idx = tid + u * NT;
                    const int c = idx >> 3, j4 = idx & 7;
                    sv[u] = *reinterpret_cast<const float4*>(
                        stage + (c * DVT + 4 * j4) * 4);
                    dsv[u] = *reinterpret_cast<const float4*>(
                        stage + STG_DS + (c * DVT + 4 * j4) * 4);
                }
                if (vt) {
                    vv = *reinterpret_cast<const uint4*>(
                        stage + STG_V + (r * DVT + 8 * j8) * 2);
                    dov = *reinterpret_cast<const uint4*>(
                        stage + STG_DO + (r * DVT + 8 * j8) * 2);
                }
            }
            if (j0 + DVT < dv) stage_issue(j0 + DVT);   // next step in flight
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int idx = tid + u * NT;
                const int c = idx >> 3, j = 4 * (idx & 7);
                sdot = fmaf(sv[u].x, dsv[u].x, sdot);
                sdot = fmaf(sv[u].y, dsv[u].y, sdot);
                sdot = fmaf(sv[u].z, dsv[u].z, sdot);
                sdot = fmaf(sv[u].w, dsv[u].w, sdot);
                uint2 s2, d2;
                s2.x = tc::pack_bf16x2(sv[u].x, sv[u].y);
                s2.y = tc::pack_bf16x2(sv[u].z, sv[u].w);
                d2.x = tc::pack_bf16x2(dsv[u].x, dsv[u].y);
                d2.y = tc::pack_bf16x2(dsv[u].z, dsv[u].w);
                *reinterpret_cast<uint2*>(Sb + c * LV + j) = s2;
                *reinterpret_cast<uint2*>(dSb + c * LV + j) = d2;
            }
            if (vt) {
            *reinterpret_cast<uint4*>(dOb + r * LV + 8 * j8) = dov;
            const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
            const uint32_t dw[4] = {dov.x, dov.y, dov.z, dov.w};
            const float gr = gam[r];
            uint4 dg4;
            uint32_t* dgw = &dg4.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                Xf[r * LX + 8 * j8 + 2 * e] = __uint_as_float(vw[e] << 16);
                Xf[r * LX + 8 * j8 + 2 * e + 1] =
                    __uint_as_float(vw[e] & 0xffff0000u);
                dgw[e] = tc::pack_bf16x2(gr * __uint_as_float(dw[e] << 16),
                                         gr * __uint_as_float(dw[e] & 0xffff0000u));
            }
            *reinterpret_cast<uint4*>(dOg + r * LV + 8 * j8) = dg4;
            }
        }
        __syncthreads();

        // K S, Q S: X = V - Diag(gamma) K S, F = Diag(beta) X,
        // dgamma += dO . Q S
        {
            float ks[TPW][4] = {}, qs[TPW][4] = {};
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t ak[4], aq[4], bs4[4];
                a_row(ak, Kb + 16 * pm * LQ + 16 * kk, LQ, lane);
                a_row(aq, Qb + 16 * pm * LQ + 16 * kk, LQ, lane);
                b_row2(bs4, Sb + 16 * kk * LV + pn, LV, lane);
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt) {
                    mma(ks[nt], ak, bs4[2 * nt], bs4[2 * nt + 1]);
                    mma(qs[nt], aq, bs4[2 * nt], bs4[2 * nt + 1]);
                }
            }
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * pm + g8 + 8 * hm;
                float dgp = 0.f;
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt) {
                    const int j = pn + 8 * nt + 2 * t4;
                    float xs[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float v = ks[nt][2 * hm + e];
                        KSf[r * LX + j + e] = v;
                        const float x = fmaf(-gam[r], v, Xf[r * LX + j + e]);
                        Xf[r * LX + j + e] = x;
                        xs[e] = bs[r] * x;
                        dgp = fmaf(bf(dOb, r * LV + j + e), qs[nt][2 * hm + e],
                                   dgp);
                    }
                    *reinterpret_cast<uint32_t*>(Fb + r * LV + j) =
                        tc::pack_bf16x2(xs[0], xs[1]);
                }
                dgp = quad_sum(dgp);
                if (t4 == 0) atomicAdd(&dgam[r], dgp);
            }
        }
        __syncthreads();

        // U~ = T F (T lower triangular)
        {
            float u[TPW][4] = {};
            for (int kk = 0; kk <= pm; ++kk) {
                uint32_t at[4], bf4[4];
                a_row(at, Tb + 16 * pm * LC + 16 * kk, LC, lane);
                b_row2(bf4, Fb + 16 * kk * LV + pn, LV, lane);
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt)
                    mma(u[nt], at, bf4[2 * nt], bf4[2 * nt + 1]);
            }
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * pm + g8 + 8 * hm;
                const float lr = lam[r];
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt) {
                    const int j = pn + 8 * nt + 2 * t4;
                    const float u0 = u[nt][2 * hm], u1 = u[nt][2 * hm + 1];
                    Uf[r * LX + j] = u0;
                    Uf[r * LX + j + 1] = u1;
                    *reinterpret_cast<uint32_t*>(Ub + r * LV + j) =
                        tc::pack_bf16x2(u0, u1);
                    *reinterpret_cast<uint32_t*>(Ulb + r * LV + j) =
                        tc::pack_bf16x2(lr * u0, lr * u1);
                }
            }
        }
        __syncthreads();

        // dU~ = P^T dO + Diag(lambda) K dS';  dlambda_r += (K dS')_r . U~_r
        {
            float kd[TPW][4] = {}, pd[TPW][4] = {};
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t ak[4], bd4[4];
                a_row(ak, Kb + 16 * pm * LQ + 16 * kk, LQ, lane);
                b_row2(bd4, dSb + 16 * kk * LV + pn, LV, lane);
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt)
                    mma(kd[nt], ak, bd4[2 * nt], bd4[2 * nt + 1]);
            }
            for (int kk = pm; kk < C / 16; ++kk) {   // P^T(r, i) = P(i, r)
                uint32_t ap[4], bo4[4];
                a_trn(ap, Pb + 16 * kk * LC + 16 * pm, LC, lane);
                b_row2(bo4, dOb + 16 * kk * LV + pn, LV, lane);
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt)
                    mma(pd[nt], ap, bo4[2 * nt], bo4[2 * nt + 1]);
            }
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * pm + g8 + 8 * hm;
                const float lr = lam[r];
                float dlp = 0.f;
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt) {
                    const int j = pn + 8 * nt + 2 * t4;
                    const float k0 = kd[nt][2 * hm], k1 = kd[nt][2 * hm + 1];
                    *reinterpret_cast<uint32_t*>(dUb + r * LV + j) =
                        tc::pack_bf16x2(fmaf(lr, k0, pd[nt][2 * hm]),
                                        fmaf(lr, k1, pd[nt][2 * hm + 1]));
                    dlp = fmaf(k0, Uf[r * LX + j], dlp);
                    dlp = fmaf(k1, Uf[r * LX + j + 1], dlp);
                }
                dlp = quad_sum(dlp);
                if (t4 == 0) atomicAdd(&dlam[r], dlp);
            }
        }
        __syncthreads();

        // dF = T^T dU~; dV = Diag(beta) dF; dbeta += dF . X;
        // dgamma -= dX . K S
        {
            float df[TPW][4] = {};
            for (int kk = pm; kk < C / 16; ++kk) {   // T^T(r, i) = T(i, r)
                uint32_t at[4], bu4[4];
                a_trn(at, Tb + 16 * kk * LC + 16 * pm, LC, lane);
                b_row2(bu4, dUb + 16 * kk * LV + pn, LV, lane);
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt)
                    mma(df[nt], at, bu4[2 * nt], bu4[2 * nt + 1]);
            }
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * pm + g8 + 8 * hm;
                const int t = t0 + r;
                const float br = bs[r], gbr = gb[r];
                float dbp = 0.f, dgp = 0.f;
#pragma unroll
                for (int nt = 0; nt < TPW; ++nt) {
                    const int j = pn + 8 * nt + 2 * t4;
                    const float f0 = df[nt][2 * hm], f1 = df[nt][2 * hm + 1];
                    const float x0 = br * f0, x1 = br * f1;
                    dbp = fmaf(f0, Xf[r * LX + j], dbp);
                    dbp = fmaf(f1, Xf[r * LX + j + 1], dbp);
                    dgp = fmaf(-x0, KSf[r * LX + j], dgp);
                    dgp = fmaf(-x1, KSf[r * LX + j + 1], dgp);
                    *reinterpret_cast<uint32_t*>(dFb + r * LV + j) =
                        tc::pack_bf16x2(f0, f1);
                    *reinterpret_cast<uint32_t*>(dFs + r * LV + j) =
                        tc::pack_bf16x2(gbr * f0, gbr * f1);
                    if (t < T) {
                        const size_t off =
                            (((size_t)b * T + t) * H + h) * dv + j0 + j;
                        *reinterpret_cast<uint32_t*>(
                            static_cast<IO*>(a.dv_) + off) =
                            tc::pack_bf16x2(x0, x1);
                    }
                }
                dbp = quad_sum(dbp);
                dgp = quad_sum(dgp);
                if (t4 == 0) {
                    atomicAdd(&db[r], dbp);
                    atomicAdd(&dgam[r], dgp);
                }
            }
        }
        __syncthreads();

        // dP += dO U~^T, dA -= dF U~^T (this warp's lower tiles, registers)
#pragma unroll
        for (int x = 0; x < XT; ++x) {
            const int idx = warp + NW * x;
            if (idx >= 20) break;
            int mt, nt;
            lower_tile(idx, mt, nt);
#pragma unroll
            for (int kk = 0; kk < DVT / 16; ++kk) {
                uint32_t ad[4], af[4], bu[4];
                a_row(ad, dOb + 16 * mt * LV + 16 * kk, LV, lane);
                a_row(af, dFb + 16 * mt * LV + 16 * kk, LV, lane);
                // B(j, i) = U~(i, j): U~ rows 8 nt .. (and the next 8, unused)
                b_col2(bu, Ub + 8 * nt * LV + 16 * kk, LV, lane);
                mma(dPa[x], ad, bu[0], bu[1]);
                mma(dAa[x], af, bu[0], bu[1]);
            }
        }
        // dq += Diag(gamma) dO S^T;
        // dk += Diag(lambda) U~ dS'^T - Diag(gamma beta) dF S^T
#pragma unroll
        for (int kk = 0; kk < DVT / 16; ++kk) {
            uint32_t ad[4], au[4], af[4];
            a_row(ad, dOg + 16 * mo * LV + 16 * kk, LV, lane);
            a_row(au, Ulb + 16 * mo * LV + 16 * kk, LV, lane);
            a_row(af, dFs + 16 * mo * LV + 16 * kk, LV, lane);
#pragma unroll
            for (int np = 0; np < NQ / 2; ++np) {   // pairs of 8-column tiles
                const int c0 = co + 16 * np;
                uint32_t bs4[4], bd4[4];
                // B(j, c) = S(c, j)
                b_col2(bs4, Sb + c0 * LV + 16 * kk, LV, lane);
                b_col2(bd4, dSb + c0 * LV + 16 * kk, LV, lane);
#pragma unroll
                for (int hn = 0; hn < 2; ++hn) {
                    mma(dq[2 * np + hn], ad, bs4[2 * hn], bs4[2 * hn + 1]);
                    mma(dk[2 * np + hn], au, bd4[2 * hn], bd4[2 * hn + 1]);
                    mma(dk[2 * np + hn], af, bs4[2 * hn], bs4[2 * hn + 1]);
                }
            }
        }
        __syncthreads();
    }
    {   // <dS', S> over the whole state
        float s = sdot;
#pragma unroll
        for (int off = 16; off; off >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) atomicAdd(dgc, s);
    }
    // dP (lower incl.) into F0, dA (strictly lower) into F1 (only these
    // entries are read below; the final tiles of Gamma o dP are written in
    // full, zeros above the diagonal included)
#pragma unroll
    for (int x = 0; x < XT; ++x) {
        const int idx = warp + NW * x;
        if (idx >= 20) break;
        int mt, nt;
        lower_tile(idx, mt, nt);
#pragma unroll
        for (int hm = 0; hm < 2; ++hm)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 16 * mt + g8 + 8 * hm;
                const int i = 8 * nt + 2 * t4 + e;
                if (i <= r) F0f[r * LF + i] = dPa[x][2 * hm + e];
                if (i < r) F1f[r * LF + i] = -dAa[x][2 * hm + e];
            }
    }
    __syncthreads();

    // dGamma o Gamma (F2), Gamma o dP (bf16), D (over dA in F1) and the
    // A-part of dbeta, from Q K^T and K K^T of the lower tiles
    {
        float qk[XT][4], kk4[XT][4];
        int mt[XT], nt[XT];
        qk_kk_tiles<NW>(qk, kk4, mt, nt, Qb, Kb, warp, lane);
#pragma unroll
        for (int x = 0; x < XT; ++x) {
            if (warp + NW * x >= 20) break;
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * mt[x] + g8 + 8 * hm;
                float dbp = 0.f;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = 8 * nt[x] + 2 * t4 + e;
                    float dgg = 0.f, dpt = 0.f, dd = 0.f;
                    if (i <= r) {
                        const float gmm = expf(gs[r] - gs[i]);
                        const float dpv = F0f[r * LF + i];
                        float dgm = dpv * qk[x][2 * hm + e];
                        dpt = gmm * dpv;
                        if (i < r) {
                            const float dav = F1f[r * LF + i];
                            dgm = fmaf(dav * bs[r], kk4[x][2 * hm + e], dgm);
                            dd = bs[r] * gmm * dav;
                            dbp = fmaf(dav * gmm, kk4[x][2 * hm + e], dbp);
                        }
                        dgg = dgm * gmm;
                    }
                    F2f[r * LF + i] = dgg;
                    Gdp[r * LC + i] = __float2bfloat16_rn(dpt);
                    F1f[r * LF + i] = dd;
                }
                dbp = quad_sum(dbp);
                if (t4 == 0) atomicAdd(&db[r], dbp);
            }
        }
    }
    __syncthreads();

    // per row (four threads each): dg, deta, dn (dn replaces dbeta in db);
    // D + D^T (bf16) from D's strictly lower part
    if (tid < 256) {
        const int r = tid >> 2, q4 = tid & 3;
        float sp = 0.f;
        for (int i = q4; i <= r; i += 4) sp += F2f[r * LF + i];
        for (int rr = r + q4; rr < C; rr += 4) sp -= F2f[rr * LF + r];
        if (r == C - 1)
            for (int t = q4; t < C; t += 4) sp = fmaf(dlam[t], lam[t], sp);
        sp = quad_sum(sp);
        if (q4 == 0) {
            float gsum = sp + dgam[r] * gam[r] - dlam[r] * lam[r];
            if (r == C - 1) gsum = fmaf(dgc[0], gam[C - 1], gsum);
            dg[r] = gsum;
            const float dbeta = db[r];
            float deta, dn = 0.f;
            if (a.gdn) {
                deta = dbeta;
            } else {
                const float denom = nrm[r] + a.eps;
                deta = denom == 0.f ? 0.f : dbeta / denom;
                if (denom != 0.f) dn = -dbeta * bs[r] / denom;
            }
            const int t = t0 + r;
            if (t < T) a.deta[((size_t)b * T + t) * H + h] = deta;
            db[r] = dn;
        }
    }
    for (int i = tid; i < C * C; i += NT) {
        const int r = i >> 6, c = i & 63;
        const float d =
            c < r ? F1f[r * LF + c] : c > r ? F1f[c * LF + r] : 0.f;
        Ddt[r * LC + c] = __float2bfloat16_rn(d);
    }
    __syncthreads();
    if (warp == 0) {   // dlog_alpha_j = sum_{r >= j} dg_r (a suffix scan)
        const float x0 = dg[2 * lane], x1 = dg[2 * lane + 1];
        float sc = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, sc, off);
            if (lane + off < 32) sc += y;
        }
        const int t = t0 + 2 * lane;
        const size_t off = ((size_t)b * T + t) * H + h;
        if (t < T) a.dlog_alpha[off] = sc;
        if (t + 1 < T) a.dlog_alpha[off + H] = sc - x0;
    }

    // dq += (Gamma o dP) K;  dk += (Gamma o dP)^T Q + (D + D^T) K
    for (int kk = 0; kk < C / 16; ++kk) {
        uint32_t ap[4], apt[4], ad[4];
        const bool low = kk <= mo, up = kk >= mo;
        if (low) a_row(ap, Gdp + 16 * mo * LC + 16 * kk, LC, lane);
        if (up) a_trn(apt, Gdp + 16 * kk * LC + 16 * mo, LC, lane);
        a_row(ad, Ddt + 16 * mo * LC + 16 * kk, LC, lane);
#pragma unroll
        for (int np = 0; np < NQ / 2; ++np) {
            const int c0 = co + 16 * np;
            uint32_t bk4[4], bq4[4];
            b_row2(bk4, Kb + 16 * kk * LQ + c0, LQ, lane);
            b_row2(bq4, Qb + 16 * kk * LQ + c0, LQ, lane);
#pragma unroll
            for (int hn = 0; hn < 2; ++hn) {
                if (low) mma(dq[2 * np + hn], ap, bk4[2 * hn], bk4[2 * hn + 1]);
                if (up) mma(dk[2 * np + hn], apt, bq4[2 * hn], bq4[2 * hn + 1]);
                mma(dk[2 * np + hn], ad, bk4[2 * hn], bk4[2 * hn + 1]);
            }
        }
    }
#pragma unroll
    for (int hm = 0; hm < 2; ++hm) {
        const int r = 16 * mo + g8 + 8 * hm;
        const int t = t0 + r;
        if (t >= T) continue;
        const float dn2 = 2.f * db[r];
#pragma unroll
        for (int nt = 0; nt < NQ; ++nt) {
            const int c = co + 8 * nt + 2 * t4;
            const size_t off = (((size_t)b * T + t) * H + h) * DK + c;
            IO* q2 = static_cast<IO*>(a.dq) + off;
            IO* k2 = static_cast<IO*>(a.dk_) + off;
            q2[0] = from_f32<IO>(dq[nt][2 * hm]);
            q2[1] = from_f32<IO>(dq[nt][2 * hm + 1]);
            k2[0] = from_f32<IO>(fmaf(dn2, bf(Kb, r * LQ + c), dk[nt][2 * hm]));
            k2[1] = from_f32<IO>(
                fmaf(dn2, bf(Kb, r * LQ + c + 1), dk[nt][2 * hm + 1]));
        }
    }
}

// One CTA per (batch, head, chunk), all chunks in parallel: q, k and the
// gates of the chunk, beta from ||k||^2, the cumulative decay, A and P from
// K K^T and Q K^T on the tensor cores, T = A^{-1}; the record.
namespace bp {
constexpr int QB = 0;
constexpr int KB = QB + lm::C * lm::LQ * 2;
constexpr int PB = KB + lm::C * lm::LQ * 2;
constexpr int AF = PB + lm::C * lm::LC * 2;
constexpr int TF = AF + lm::C * lm::LF * 4;
constexpr int YS = TF + lm::C * lm::LF * 4;   // 8 warps x 16 x 8 fp32
constexpr int VEC = YS + 8 * 128 * 4;         // gs, bs, nrm
constexpr int BYTES = VEC + 3 * lm::C * 4;
static_assert(2 * (BYTES + 1024) <= 233472, "two CTAs per SM");
}  // namespace bp

template <typename IO>
__global__ void __launch_bounds__(kBwdThreads, 2)
kla_bwd_prep_kernel(BwdArgs a) {
    using namespace lm;
    extern __shared__ __align__(16) uint8_t smraw[];
    bf16* Qb = reinterpret_cast<bf16*>(smraw + bp::QB);
    bf16* Kb = reinterpret_cast<bf16*>(smraw + bp::KB);
    bf16* Pb = reinterpret_cast<bf16*>(smraw + bp::PB);
    float* Af = reinterpret_cast<float*>(smraw + bp::AF);
    float* Tf = reinterpret_cast<float*>(smraw + bp::TF);
    float* Ys = reinterpret_cast<float*>(smraw + bp::YS);
    float* gs = reinterpret_cast<float*>(smraw + bp::VEC);
    float* bs = gs + C;
    float* nrm = gs + 2 * C;

    const int T = a.T, H = a.H;
    const int nch = (T + C - 1) / C;
    const long blk = blockIdx.x;
    const int bh = (int)(blk / nch), ch = (int)(blk % nch);
    const int b = bh / H, h = bh % H;
    const int t0 = ch * C;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int u = 0; u < 4; ++u) {   // q, k: 64 rows x 16 pieces of 16 bytes
        const int idx = tid + u * kBwdThreads;
        const int r = idx >> 4, c8 = idx & 15;
        const int t = t0 + r;
        uint4 qv = make_uint4(0, 0, 0, 0), kv = make_uint4(0, 0, 0, 0);
        if (t < T) {
            const size_t off = (((size_t)b * T + t) * H + h) * DK + 8 * c8;
            qv = *reinterpret_cast<const uint4*>(
                static_cast<const IO*>(a.q) + off);
            kv = *reinterpret_cast<const uint4*>(
                static_cast<const IO*>(a.k) + off);
        }
        *reinterpret_cast<uint4*>(Qb + r * LQ + 8 * c8) = qv;
        *reinterpret_cast<uint4*>(Kb + r * LQ + 8 * c8) = kv;
    }
    if (tid < C) {
        const int t = t0 + tid;
        const size_t off = ((size_t)b * T + t) * H + h;
        gs[tid] = t < T ? a.log_alpha[off] : 0.f;
        bs[tid] = t < T ? a.eta[off] : 0.f;
    }
    for (int i = tid; i < C * LC / 2; i += kBwdThreads)   // P's upper part
        reinterpret_cast<uint32_t*>(Pb)[i] = 0u;
    __syncthreads();
    {   // ||k||^2 (four threads per row), beta, cumulative decay
        const int r = tid >> 2, q4 = tid & 3;
        const float n = row_norm2(Kb, r, q4);
        if (q4 == 0) {
            nrm[r] = n;
            const float denom = n + a.eps;
            if (!a.gdn) bs[r] = denom == 0.f ? 0.f : bs[r] / denom;
        }
        if (warp == 0) {   // inclusive scan of the 64 log decays
            const float x0 = gs[2 * lane], x1 = gs[2 * lane + 1];
            float sc = x0 + x1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, sc, off);
                if (lane >= off) sc += y;
            }
            gs[2 * lane] = sc - x1;
            gs[2 * lane + 1] = sc;
        }
    }
    __syncthreads();
    {   // A (unit lower, fp32) and P (bf16) from K K^T and Q K^T
        float qk[3][4], kk[3][4];
        int mt[3], nt[3];
        qk_kk_tiles(qk, kk, mt, nt, Qb, Kb, warp, lane);
#pragma unroll
        for (int x = 0; x < 3; ++x) {
            if (x == 2 && warp >= 4) break;
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * mt[x] + g8 + 8 * hm;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = 8 * nt[x] + 2 * t4 + e;
                    float av = i == r ? 1.f : 0.f, pv = 0.f;
                    if (i <= r) {
                        const float dec = expf(gs[r] - gs[i]);
                        pv = dec * qk[x][2 * hm + e];
                        if (i < r) av = bs[r] * dec * kk[x][2 * hm + e];
                    }
                    Af[r * LF + i] = av;
                    Pb[r * LC + i] = __float2bfloat16_rn(pv);
                }
            }
        }
    }
    __syncthreads();
    invert_lower64(Af, LF, Tf, LF, Ys);   // ends with a barrier
    uint8_t* rec = a.rec + ((size_t)bh * nch + ch) * brec::BYTES;
#pragma unroll
    for (int m = 0; m < 2; ++m) {   // T and P rows, 8 bf16 per 16 bytes
        const int u = tid + m * kBwdThreads;   // 512 pieces each
        const int r = u >> 3, c8 = u & 7;
        float tv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = 8 * c8 + e;
            tv[e] = c <= r ? Tf[r * LF + c] : 0.f;
        }
        uint4 tw;
        tw.x = tc::pack_bf16x2(tv[0], tv[1]);
        tw.y = tc::pack_bf16x2(tv[2], tv[3]);
        tw.z = tc::pack_bf16x2(tv[4], tv[5]);
        tw.w = tc::pack_bf16x2(tv[6], tv[7]);
        *reinterpret_cast<uint4*>(rec + brec::T_OFF + (r * C + 8 * c8) * 2) =
            tw;
        *reinterpret_cast<uint4*>(rec + brec::P_OFF + (r * C + 8 * c8) * 2) =
            *reinterpret_cast<const uint4*>(Pb + r * LC + 8 * c8);
    }
    if (tid < C) {
        reinterpret_cast<float*>(rec + brec::G_OFF)[tid] = gs[tid];
        reinterpret_cast<float*>(rec + brec::B_OFF)[tid] = bs[tid];
        reinterpret_cast<float*>(rec + brec::N_OFF)[tid] = nrm[tid];
    }
}

// ------------------------- reverse state recurrence, bf16 operand tiles
// kla_bwd_state_kernel's per-chunk algebra for bf16, dk = 128, C = 64 and
// 64-column dv slices, every product on the tensor cores: dU~ = P^T dO +
// Diag(lambda) K dS', dF = T^T dU~ and dS = gamma_C dS' + Q^T Diag(gamma) dO
// - K^T Diag(gamma beta) dF as m16n8k16 MMAs (bf16 operands, fp32
// accumulation) whose operands are bf16 tiles read by ldmatrix, in the
// layout of kla_bwd_grad_lm_kernel; T, P and the gates come from the
// chunk's record (kla_bwd_prep_kernel).  dS itself stays in fp32 registers
// for the whole walk (warp w owns key rows 16 w .. 16 w + 15, all 64
// columns of the slice) and is copied to shared memory in bf16, as the
// operand of K dS', once per chunk.
namespace sm2 {
constexpr int C = 64, DK = 128, DV = 64;
constexpr int LQ = DK + 8, LC = C + 8, LV = DV + 8;
constexpr int QB = 0;
constexpr int KB = QB + C * LQ * 2;
constexpr int DOB = KB + C * LQ * 2;   // dO
constexpr int DOG = DOB + C * LV * 2;  // Diag(gamma) dO
constexpr int PB = DOG + C * LV * 2;
constexpr int TB = PB + C * LC * 2;
constexpr int DSB = TB + C * LC * 2;   // dS' (DK x DV)
constexpr int DUB = DSB + DK * LV * 2;
constexpr int DFS = DUB + C * LV * 2;  // -Diag(gamma beta) dF
constexpr int VEC = DFS + C * LV * 2;  // gs, bs, gam, lam
constexpr int BYTES = VEC + 4 * C * 4;
static_assert(BYTES <= 232448, "shared memory");
static_assert(KB % 16 == 0 && DOB % 16 == 0 && DOG % 16 == 0 &&
                  PB % 16 == 0 && TB % 16 == 0 && DSB % 16 == 0 &&
                  DUB % 16 == 0 && DFS % 16 == 0 && VEC % 16 == 0,
              "16-byte aligned rows");
}  // namespace sm2

template <typename IO>
__global__ void __launch_bounds__(kBwdThreads, 1)
kla_bwd_state_lm_kernel(BwdArgs a) {
    using namespace sm2;
    using lm::a_row;
    using lm::a_trn;
    using lm::b_row2;
    using lm::mma;
    extern __shared__ __align__(16) uint8_t smraw[];
    bf16* Qb = reinterpret_cast<bf16*>(smraw + QB);
    bf16* Kb = reinterpret_cast<bf16*>(smraw + KB);
    bf16* dOb = reinterpret_cast<bf16*>(smraw + DOB);
    bf16* dOg = reinterpret_cast<bf16*>(smraw + DOG);
    bf16* Pb = reinterpret_cast<bf16*>(smraw + PB);
    bf16* Tb = reinterpret_cast<bf16*>(smraw + TB);
    bf16* dSb = reinterpret_cast<bf16*>(smraw + DSB);
    bf16* dUb = reinterpret_cast<bf16*>(smraw + DUB);
    bf16* dFs = reinterpret_cast<bf16*>(smraw + DFS);
    float* gs = reinterpret_cast<float*>(smraw + VEC);
    float* bs = gs + C;
    float* gam = gs + 2 * C;
    float* lam = gs + 3 * C;

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int j0 = blockIdx.y * DV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int T = a.T, H = a.H, dv = a.dv;
    const int nch = (T + C - 1) / C;

    // dS of this warp's key rows 16 warp + g8 (+ 8), columns 8 nt + 2 t4
    // (+ 1): fragment layout, 8 column tiles
    float dS[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 16 * warp + g8 + 8 * (e >> 1);
            const int j = 8 * nt + 2 * t4 + (e & 1);
            dS[nt][e] =
                a.dhT ? a.dhT[((size_t)bh * DK + c) * dv + j0 + j] : 0.f;
        }

    // A chunk's tiles (q, k: 64 x 128, dO: 64 x 64, bf16) and its record (T,
    // P, g, beta) are loaded into registers, 16 bytes a load, while the
    // previous chunk computes, and stored to shared memory (unconverted)
    // when it is done.
    const uint4* q4 = static_cast<const uint4*>(a.q);
    const uint4* k4 = static_cast<const uint4*>(a.k);
    const uint4* d4 = static_cast<const uint4*>(a.dout);
    uint4 pq[4], pk[4], pd[2], pt[2], pp[2], pg;
    auto fetch = [&](int c) {
        const int t0c = c * C;
#pragma unroll
        for (int m = 0; m < 4; ++m) {   // row tid / 16 + 16 m, dims 8 (tid % 16)
            const int r = tid / 16 + 16 * m, t = t0c + r;
            const size_t e =
                ((((size_t)b * T + t) * H + h) * DK) / 8 + tid % 16;
            pq[m] = t < T ? q4[e] : make_uint4(0, 0, 0, 0);
            pk[m] = t < T ? k4[e] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {   // row tid / 8 + 32 m, dv 8 (tid % 8)
            const int r = tid / 8 + 32 * m, t = t0c + r;
            const size_t e =
                ((((size_t)b * T + t) * H + h) * dv + j0) / 8 + tid % 8;
            pd[m] = t < T ? d4[e] : make_uint4(0, 0, 0, 0);
        }
        const uint4* rc = reinterpret_cast<const uint4*>(
            a.rec + ((size_t)bh * nch + c) * brec::BYTES);
#pragma unroll
        for (int m = 0; m < 2; ++m) {   // piece tid + 256 m of T and of P
            pt[m] = rc[brec::T_OFF / 16 + tid + 256 * m];
            pp[m] = rc[brec::P_OFF / 16 + tid + 256 * m];
        }
        if (tid < 32) pg = rc[brec::G_OFF / 16 + tid];   // g, then beta
    };
    fetch(nch - 1);
    // this warp's tiles of the C x DV products: rows 16 (w >> 1), columns
    // 32 (w & 1) .. + 31 (four 16 x 8 tiles)
    const int pm = warp >> 1, pn = 32 * (warp & 1);

    for (int ch = nch - 1; ch >= 0; --ch) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int r = tid / 16 + 16 * m, c8 = tid % 16;
            *reinterpret_cast<uint4*>(Qb + r * LQ + 8 * c8) = pq[m];
            *reinterpret_cast<uint4*>(Kb + r * LQ + 8 * c8) = pk[m];
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            *reinterpret_cast<uint4*>(dOb + (tid / 8 + 32 * m) * LV +
                                      8 * (tid % 8)) = pd[m];
            const int u = tid + 256 * m, r = u >> 3, c8 = u & 7;
            *reinterpret_cast<uint4*>(Tb + r * LC + 8 * c8) = pt[m];
            *reinterpret_cast<uint4*>(Pb + r * LC + 8 * c8) = pp[m];
        }
        if (tid < 32) reinterpret_cast<uint4*>(gs)[tid] = pg;
        {   // dL/dS at the end of this chunk: to the workspace (fp32) and,
            // in bf16, to shared memory as an operand
            float* out = a.dsck + ((size_t)bh * nch + ch) * DK * dv + j0;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int hm = 0; hm < 2; ++hm) {
                    const int c = 16 * warp + g8 + 8 * hm;
                    const int j = 8 * nt + 2 * t4;
                    *reinterpret_cast<float2*>(out + (size_t)c * dv + j) =
                        make_float2(dS[nt][2 * hm], dS[nt][2 * hm + 1]);
                    *reinterpret_cast<uint32_t*>(dSb + c * LV + j) =
                        tc::pack_bf16x2(dS[nt][2 * hm], dS[nt][2 * hm + 1]);
                }
        }
        __syncthreads();
        if (ch > 0) fetch(ch - 1);   // in flight during this chunk
        if (tid < C) {
            gam[tid] = expf(gs[tid]);
            lam[tid] = expf(gs[C - 1] - gs[tid]);
        }
        __syncthreads();

        // Diag(gamma) dO (bf16) and dU~ = P^T dO + Diag(lambda) K dS'
        {
            const int r = tid >> 2, c16 = 16 * (tid & 3);
            const float gr = gam[r];
#pragma unroll
            for (int u = 0; u < 16; u += 2) {
                const float x0 = lm::bf(dOb, r * LV + c16 + u);
                const float x1 = lm::bf(dOb, r * LV + c16 + u + 1);
                *reinterpret_cast<uint32_t*>(dOg + r * LV + c16 + u) =
                    tc::pack_bf16x2(gr * x0, gr * x1);
            }
        }
        {
            float kd[4][4] = {}, pd4[4][4] = {};
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t ak[4], b0[4], b1[4];
                a_row(ak, Kb + 16 * pm * LQ + 16 * kk, LQ, lane);
                b_row2(b0, dSb + 16 * kk * LV + pn, LV, lane);
                b_row2(b1, dSb + 16 * kk * LV + pn + 16, LV, lane);
                mma(kd[0], ak, b0[0], b0[1]);
                mma(kd[1], ak, b0[2], b0[3]);
                mma(kd[2], ak, b1[0], b1[1]);
                mma(kd[3], ak, b1[2], b1[3]);
            }
            for (int kk = pm; kk < C / 16; ++kk) {   // P^T(r, i) = P(i, r)
                uint32_t ap[4], b0[4], b1[4];
                a_trn(ap, Pb + 16 * kk * LC + 16 * pm, LC, lane);
                b_row2(b0, dOb + 16 * kk * LV + pn, LV, lane);
                b_row2(b1, dOb + 16 * kk * LV + pn + 16, LV, lane);
                mma(pd4[0], ap, b0[0], b0[1]);
                mma(pd4[1], ap, b0[2], b0[3]);
                mma(pd4[2], ap, b1[0], b1[1]);
                mma(pd4[3], ap, b1[2], b1[3]);
            }
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * pm + g8 + 8 * hm;
                const float lr = lam[r];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int j = pn + 8 * nt + 2 * t4;
                    *reinterpret_cast<uint32_t*>(dUb + r * LV + j) =
                        tc::pack_bf16x2(
                            fmaf(lr, kd[nt][2 * hm], pd4[nt][2 * hm]),
                            fmaf(lr, kd[nt][2 * hm + 1], pd4[nt][2 * hm + 1]));
                }
            }
        }
        __syncthreads();

        // dF = T^T dU~, stored as -Diag(gamma beta) dF
        {
            float df[4][4] = {};
            for (int kk = pm; kk < C / 16; ++kk) {   // T^T(r, i) = T(i, r)
                uint32_t at[4], b0[4], b1[4];
                a_trn(at, Tb + 16 * kk * LC + 16 * pm, LC, lane);
                b_row2(b0, dUb + 16 * kk * LV + pn, LV, lane);
                b_row2(b1, dUb + 16 * kk * LV + pn + 16, LV, lane);
                mma(df[0], at, b0[0], b0[1]);
                mma(df[1], at, b0[2], b0[3]);
                mma(df[2], at, b1[0], b1[1]);
                mma(df[3], at, b1[2], b1[3]);
            }
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int r = 16 * pm + g8 + 8 * hm;
                const float sc = -gam[r] * bs[r];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int j = pn + 8 * nt + 2 * t4;
                    *reinterpret_cast<uint32_t*>(dFs + r * LV + j) =
                        tc::pack_bf16x2(sc * df[nt][2 * hm],
                                        sc * df[nt][2 * hm + 1]);
                }
            }
        }
        __syncthreads();

        // dS = gamma_C dS' + Q^T Diag(gamma) dO - K^T Diag(gamma beta) dF
        {
            const float gC = gam[C - 1];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) dS[nt][e] *= gC;
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk) {
                uint32_t aq[4], ak[4];
                a_trn(aq, Qb + 16 * kk * LQ + 16 * warp, LQ, lane);   // Q^T
                a_trn(ak, Kb + 16 * kk * LQ + 16 * warp, LQ, lane);   // K^T
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t bo[4], bf4[4];
                    b_row2(bo, dOg + 16 * kk * LV + 16 * np, LV, lane);
                    b_row2(bf4, dFs + 16 * kk * LV + 16 * np, LV, lane);
                    mma(dS[2 * np], aq, bo[0], bo[1]);
                    mma(dS[2 * np + 1], aq, bo[2], bo[3]);
                    mma(dS[2 * np], ak, bf4[0], bf4[1]);
                    mma(dS[2 * np + 1], ak, bf4[2], bf4[3]);
                }
            }
        }
        __syncthreads();
    }

    if (a.dh0) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hm = 0; hm < 2; ++hm) {
                const int c = 16 * warp + g8 + 8 * hm;
                const int j = 8 * nt + 2 * t4;
                *reinterpret_cast<float2*>(a.dh0 +
                                           ((size_t)bh * DK + c) * dv + j0 +
                                           j) =
                    make_float2(dS[nt][2 * hm], dS[nt][2 * hm + 1]);
            }
    }
}

// DVS: dv columns per CTA of the reverse state recurrence; DVT: dv columns
// per step of the gradient kernel.
template <int DK, int DVS, int DVT, typename IO>
cudaError_t launch_shape(const BwdArgs& a, cudaStream_t stream) {
    using LS = StateSmem<DK, DVS>;
    using LG = GradSmem<DK, DVT>;
    auto ks = kla_bwd_state_kernel<DK, DVS, IO>;
    auto kg = kla_bwd_grad_kernel<DK, DVT, IO>;
    cudaError_t e = cudaFuncSetAttribute(
        ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LS::BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)LG::BYTES);
    if (e != cudaSuccess) return e;
    const long bhs = (long)a.B * a.H;
    const long nch = (a.T + a.C - 1) / a.C;
    auto a16 = [](const void* p) {
        return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    };
    // the gradient step on the tensor cores (16-byte loads of q, k, v,
    // o_grad)
    const bool grad_tc = DK == kTcDK && DVT == 32 &&
                         std::is_same<IO, __nv_bfloat16>::value &&
                         a.C == kTcC && a16(a.q) && a16(a.k) && a16(a.v) &&
                         a16(a.dout);
    const bool state_tc = DK == kTcDK && DVS == kTcDV &&
                          std::is_same<IO, __nv_bfloat16>::value &&
                          state_tc_ok(a);
    if constexpr (DK == kTcDK && std::is_same<IO, __nv_bfloat16>::value) {
        if ((grad_tc || state_tc) && !a.rec_ready) {   // their records
            if (!a.rec) return cudaErrorInvalidValue;
            auto kp = kla_bwd_prep_kernel<IO>;
            e = cudaFuncSetAttribute(
                kp, cudaFuncAttributeMaxDynamicSharedMemorySize, bp::BYTES);
            if (e != cudaSuccess) return e;
            kp<<<(unsigned)(bhs * nch), kBwdThreads, bp::BYTES, stream>>>(a);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    if constexpr (DK == kTcDK && DVS == kTcDV &&
                  std::is_same<IO, __nv_bfloat16>::value) {
        if (state_tc) {   // the reverse recurrence on the tensor cores
            auto kt = kla_bwd_state_lm_kernel<IO>;
            e = cudaFuncSetAttribute(
                kt, cudaFuncAttributeMaxDynamicSharedMemorySize, sm2::BYTES);
            if (e != cudaSuccess) return e;
            kt<<<dim3((unsigned)bhs, (unsigned)(a.dv / DVS)), kBwdThreads,
                 sm2::BYTES, stream>>>(a);
        } else {
            ks<<<dim3((unsigned)bhs, (unsigned)(a.dv / DVS)), kBwdThreads,
                 LS::BYTES, stream>>>(a);
        }
    } else {
        ks<<<dim3((unsigned)bhs, (unsigned)(a.dv / DVS)), kBwdThreads,
             LS::BYTES, stream>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if constexpr (DK == kTcDK && DVT == 32 &&
                  std::is_same<IO, __nv_bfloat16>::value) {
        if (grad_tc) {
            constexpr int kGradWarps = 8;   // 16 warps (128 registers) measured slower
            auto km = kla_bwd_grad_lm_kernel<IO, kGradWarps>;
            e = cudaFuncSetAttribute(
                km, cudaFuncAttributeMaxDynamicSharedMemorySize, lm::BYTES);
            if (e != cudaSuccess) return e;
            km<<<(unsigned)(bhs * nch), 32 * kGradWarps, lm::BYTES, stream>>>(
                a);
            return cudaGetLastError();
        }
    }
    kg<<<(unsigned)(bhs * nch), kBwdThreads, LG::BYTES, stream>>>(a);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_dtype(const BwdArgs& a, cudaStream_t stream) {
    // The reverse state recurrence is one CTA per (batch, head, dv slice),
    // sequential over the chunks: 64-column slices when 32-column ones
    // would need more than one wave of CTAs (one CTA per SM).
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // where the tensor-core reverse recurrence applies: 64-column slices
    // always
    const bool tc = std::is_same<IO, __nv_bfloat16>::value && state_tc_ok(a);
    const bool wide =
        tc || (a.dv >= 64 && (long)a.B * a.H * (a.dv / 32) > sms);
#define KLA_BWD_DK(DKV)                                                     \
    if (a.dk == DKV) {                                                      \
        if (a.dv == 16) return launch_shape<DKV, 16, 16, IO>(a, stream);    \
        if (wide) return launch_shape<DKV, 64, 32, IO>(a, stream);          \
        return launch_shape<DKV, 32, 32, IO>(a, stream);                    \
    }
    KLA_BWD_DK(16)
    KLA_BWD_DK(32)
    KLA_BWD_DK(64)
    KLA_BWD_DK(128)
#undef KLA_BWD_DK
    return cudaErrorInvalidValue;
}

}  // namespace

size_t chunk_bwd_state_floats(int B, int T, int H, int dk, int dv, int C) {
    if (C <= 0) return 0;
    const size_t nch = (size_t)(T + C - 1) / C;
    return (size_t)B * H * nch * dk * dv;
}

size_t chunk_bwd_workspace_bytes(int B, int T, int H, int dk, int dv, int C) {
    if (C <= 0) return 0;
    const size_t nch = (size_t)(T + C - 1) / C;
    const size_t rec = (dk == kTcDK && C == kTcC)
                           ? (size_t)B * H * nch * brec::BYTES
                           : 0;
    const size_t fwd = (dk == kTcDK && dv == kTcDK && C == kTcC)
                           ? chunk_tc2_workspace_bytes(B, T, H)
                           : 0;
    return 2 * sizeof(float) * chunk_bwd_state_floats(B, T, H, dk, dv, C) +
           rec + fwd;
}

cudaError_t launch_chunk_bwd(const BwdArgs& a_in, cudaStream_t stream) {
    if ((long)a_in.B * a_in.H == 0 || a_in.T == 0) return cudaSuccess;
    if (a_in.C > kBwdMaxC) return cudaErrorInvalidValue;
    BwdArgs a = a_in;
    // 1. states at every chunk start (a forward pass, o not written): the
    // two-kernel tensor-core path, whose pre-pass also writes the
    // backward's per-chunk records, where it applies; else the fused
    // tensor-core kernel or the CUDA-core one
    FwdArgs f{a.q, a.k, a.v, a.log_alpha, a.eta, a.eps, a.gdn, a.h0,
              nullptr, nullptr, a.B, a.T, a.H, a.dk, a.dv, a.C, a.dtype};
    f.ckpt = a.ckpt;
    cudaError_t e;
    if (a.rec && a.fwd_rec && chunk_tc2_eligible(f)) {
        f.bwd_rec = a.rec;
        e = launch_chunk_tc2(f, a.fwd_rec, stream);
        a.rec_ready = true;
    } else {
        e = chunk_tc_eligible(f) ? launch_chunk_tc(f, stream)
                                 : launch_chunk_simt(f, stream);
    }
    if (e != cudaSuccess) return e;
    // 2 and 3. dS' per chunk and dh0, then the gradients
    if (a.dtype == KLA_BF16) return launch_dtype<__nv_bfloat16>(a, stream);
    return launch_dtype<float>(a, stream);
}

}  // namespace kla
