// Tensor-core (tcgen05) chunkwise KLA forward pass for bf16 q/k/v/o,
// dk = dv = 128, chunk C = 64, fp32 state.
//
// Algorithm (per (batch, head); rows r, i of a chunk; g = in-chunk cumulative
// log decay, gamma_r = exp(g_r), Gamma_ri = exp(g_r - g_i), r >= i):
//   beta_r = eta_r / (||k_r||^2 + eps)           (||k_r||^2 = diag of K K^T)
//   A  = I + strict_lower(Diag(beta) (Gamma o K K^T)),   T = A^{-1}
//   W  = T Diag(beta gamma) K,   U = T Diag(beta) V
//   U~ = U - W S
//   O  = Diag(gamma) Q S + lower_incl(Gamma o Q K^T) U~
//   S <- gamma_C S + K^T Diag(Gamma_{C,.}) U~
// i.e. the gated-DeltaNet block solver with B = Diag(beta) as the only
// change (gist.science/es/paper/2605.08587, section "Implementacion").
//
// Work decomposition: one CTA per (batch, head, half of dv); the CTA walks
// the chunks of its sequence in order with its 128 x 64 slice of S resident
// in registers (fp32, one key row per thread) and a bf16 copy in shared
// memory as the MMA operand.  Per chunk, five tcgen05 MMAs (bf16 operands,
// fp32 accumulation in TMEM):
//   (1) G  = [K; Q] K^T                  -> K K^T, Q K^T          (128x64x128)
//   (2) [W; U] = blockdiag(TW, TU) [K; V] -> W, U                 (128x128x128)
//   (3) X  = [Q; W] S                    -> Q S, W S              (128x64x128)
//   (4) dS = K^T Diag(Gamma_C) U~                                 (128x64x64)
//   (5) OI = [P; -] U~,  P = Gamma o Q K^T (lower incl.)          (128x64x64)
// CUDA cores do the elementwise work, the gates, and T = A^{-1} (fp32 column
// substitution).  q, k, v tiles arrive by TMA (128-byte swizzle, double
// buffered one chunk ahead); o and hT are written with vector stores.
//
// Every mbarrier wait is bounded (2 s): on time-out the CTA records a fault
// in the library's fault word, drains its outstanding copies and MMAs (again
// bounded), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kla_internal.cuh"
#include "tc_primitives.cuh"

namespace kla {

namespace {

__device__ unsigned int g_fault_word = 0;

constexpr int kC = 64;        // chunk length
constexpr int kD = 128;       // dk = dv
constexpr int kNV = 64;       // dv columns per CTA
constexpr int kThreads = 128;

// ---- shared memory map (bytes from a 1024-aligned base) -------------------
// stage s (s = 0, 1) at s * kStage:  per key half h in {0, 1}:
//   K_h at h*24K, Q_h at h*24K + 8K, W_h at h*24K + 16K   (each 64 x 64 bf16)
//   V   at 48K                                           (64 x 64 bf16)
// [K_h; Q_h] and [Q_h; W_h] are therefore contiguous 128-row K-major operands.
constexpr int kHalfStride = 24576;
constexpr int kOffQ = 8192;
constexpr int kOffW = 16384;
constexpr int kOffV = 49152;
constexpr int kStage = 57344;
constexpr int kSBuf = 2 * kStage;            // bf16 S, 128 x 64, MN-major B
constexpr int kBD = kSBuf + 16384;           // blockdiag(TW, TU), 2 x 16 KB
constexpr int kPBuf = kBD + 32768;           // P, 64 x 64 K-major
constexpr int kUtBuf = kPBuf + 8192;         // U~ (bf16), MN-major B
constexpr int kUtsBuf = kUtBuf + 8192;       // Gamma_C U~ (bf16), MN-major B
constexpr int kAStride = 68;                 // fp32 A / T row stride (floats)
constexpr int kAF32 = kUtsBuf + 8192;        // fp32 strictly-lower A
constexpr int kTF32 = kAF32 + kC * kAStride * 4;   // fp32 T = A^{-1}
constexpr int kYStride = 17;
constexpr int kYF32 = kTF32 + kC * kAStride * 4;   // 6 blocks T_ii A_im
constexpr int kGF32 = kYF32 + 6 * 16 * kYStride * 4;
constexpr int kBeta = kGF32 + 256;
constexpr int kWTot = kBeta + 256;
constexpr int kBars = kWTot + 16;
constexpr int kSmemUsed = kBars + 64;
constexpr int kSmemBytes = kSmemUsed + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmaBytes = 2 * 16384 + 8192;

// ---- TMEM columns ----------------------------------------------------------
constexpr uint32_t kColG = 0;      // 64
constexpr uint32_t kColWU = 64;    // 128
constexpr uint32_t kColX = 192;    // 64
constexpr uint32_t kColDS = 256;   // 64
constexpr uint32_t kColOI = 320;   // 64
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdG = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdWU = tc::idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdX = tc::idesc_bf16(128, 64, false, true);
constexpr uint32_t kIdDS = tc::idesc_bf16(128, 64, true, true);
constexpr uint32_t kIdOI = tc::idesc_bf16(128, 64, false, true);

struct TcParams {
    const float* log_alpha;
    const float* eta;
    const float* h0;
    __nv_bfloat16* o;
    float* hT;
    float eps;
    int T, H;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Write 64 fp32 values as one 128-byte swizzled bf16 row.
__device__ __forceinline__ void st_row_sw128(uint8_t* base, int row,
                                             const float* x) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 v;
        v.x = pack_bf16(x[8 * j + 0], x[8 * j + 1]);
        v.y = pack_bf16(x[8 * j + 2], x[8 * j + 3]);
        v.z = pack_bf16(x[8 * j + 4], x[8 * j + 5]);
        v.w = pack_bf16(x[8 * j + 6], x[8 * j + 7]);
        const int chunk = j ^ (row & 7);
        *reinterpret_cast<uint4*>(base + row * 128 + chunk * 16) = v;
    }
}

// 64 consecutive TMEM columns of this thread's lane -> x[0..63].
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* x) {
    tc::tmem_ld16(taddr + 0, *reinterpret_cast<float(*)[16]>(x + 0));
    tc::tmem_ld16(taddr + 16, *reinterpret_cast<float(*)[16]>(x + 16));
    tc::tmem_ld16(taddr + 32, *reinterpret_cast<float(*)[16]>(x + 32));
    tc::tmem_ld16(taddr + 48, *reinterpret_cast<float(*)[16]>(x + 48));
    tc::tmem_ld_wait();
}

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
    const bool ok = tc::mbar_wait(bar, parity);
    return __syncthreads_or(ok ? 0 : 1) == 0;
}

// K-major SW128 descriptor (rows 128 B apart, 8-row atoms 1024 B apart).
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) {
    return tc::sdesc_sw128(addr, 16, 1024);
}
// MN-major SW128 descriptor: `lbo` = bytes between 64-wide MN atoms.
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr, uint32_t lbo) {
    return tc::sdesc_sw128(addr, lbo, 1024);
}

// T = A^{-1} for the 64 x 64 unit lower-triangular A (strictly lower part in
// Af, zeros elsewhere), blocked in 16 x 16 tiles and computed in fp32 by all
// 128 threads:
//   T_ii = A_ii^{-1}                       (column substitution, 64 threads)
//   Y_im = T_ii A_im                       (i > m, six tiles in parallel)
//   T_ij = -sum_{m=j}^{i-1} Y_im T_mj      (by distance i - j = 1, 2, 3)
// Tiles of T above the diagonal are never read.
__device__ __forceinline__ void invert_unit_lower64(const float* Af, float* Tf,
                                                    float* Yf, int tid) {
    if (tid < kC) {
        const int bb = tid >> 4, cl = tid & 15;
        const float* Ab = Af + (16 * bb) * kAStride + 16 * bb;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) t[r] = (r == cl) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < r; i += 2) {
                a0 = fmaf(Ab[r * kAStride + i], t[i], a0);
                if (i + 1 < r) a1 = fmaf(Ab[r * kAStride + i + 1], t[i + 1], a1);
            }
            if (r > cl) t[r] = -(a0 + a1);
        }
        float* Tb = Tf + (16 * bb) * kAStride + 16 * bb + cl;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * kAStride] = t[r];
    }
    __syncthreads();
    // Y_im = T_ii A_im, tile yb = i(i-1)/2 + m
#pragma unroll
    for (int j = 0; j < 12; ++j) {
        const int e = tid + kThreads * j;
        const int yb = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int i = yb < 1 ? 1 : (yb < 3 ? 2 : 3);
        const int m = yb - i * (i - 1) / 2;
        const float* Tr = Tf + (16 * i + r) * kAStride + 16 * i;
        const float* Ac = Af + (16 * i) * kAStride + 16 * m + c;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            a0 = fmaf(Tr[k], Ac[k * kAStride], a0);
            a1 = fmaf(Tr[k + 1], Ac[(k + 1) * kAStride], a1);
        }
        Yf[(yb * 16 + r) * kYStride + c] = a0 + a1;
    }
    __syncthreads();
    // distance 1: T_{i,i-1} = -Y_{i,i-1} T_{i-1,i-1}
#pragma unroll
    for (int j = 0; j < 6; ++j) {
        const int e = tid + kThreads * j;
        const int i = 1 + (e >> 8), r = (e >> 4) & 15, c = e & 15;
        const float* Y = Yf + ((i * (i - 1) / 2 + i - 1) * 16 + r) * kYStride;
        const float* Tc = Tf + (16 * (i - 1)) * kAStride + 16 * (i - 1) + c;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            a0 = fmaf(Y[k], Tc[k * kAStride], a0);
            a1 = fmaf(Y[k + 1], Tc[(k + 1) * kAStride], a1);
        }
        Tf[(16 * i + r) * kAStride + 16 * (i - 1) + c] = -(a0 + a1);
    }
    __syncthreads();
    // distance 2: T_{i,i-2} = -(Y_{i,i-2} T_{i-2,i-2} + Y_{i,i-1} T_{i-1,i-2})
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int e = tid + kThreads * j;
        const int i = 2 + (e >> 8), r = (e >> 4) & 15, c = e & 15;
        const int jj = i - 2;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            const int m = jj + mm;
            const float* Y = Yf + ((i * (i - 1) / 2 + m) * 16 + r) * kYStride;
            const float* Tc = Tf + (16 * m) * kAStride + 16 * jj + c;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                a0 = fmaf(Y[k], Tc[k * kAStride], a0);
                a1 = fmaf(Y[k + 1], Tc[(k + 1) * kAStride], a1);
            }
        }
        Tf[(16 * i + r) * kAStride + 16 * jj + c] = -(a0 + a1);
    }
    __syncthreads();
    // distance 3: T_30 = -(Y_30 T_00 + Y_31 T_10 + Y_32 T_20)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = tid + kThreads * j;
        const int r = (e >> 4) & 15, c = e & 15;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            const float* Y = Yf + ((3 + m) * 16 + r) * kYStride;
            const float* Tc = Tf + (16 * m) * kAStride + c;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                a0 = fmaf(Y[k], Tc[k * kAStride], a0);
                a1 = fmaf(Y[k + 1], Tc[(k + 1) * kAStride], a1);
            }
        }
        Tf[(48 + r) * kAStride + c] = -(a0 + a1);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
kla_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_u32(sm);
    float* Af = reinterpret_cast<float*>(sm + kAF32);
    float* Tf = reinterpret_cast<float*>(sm + kTF32);
    float* Yf = reinterpret_cast<float*>(sm + kYF32);
    float* gS = reinterpret_cast<float*>(sm + kGF32);
    float* betaS = reinterpret_cast<float*>(sm + kBeta);
    float* wtot = reinterpret_cast<float*>(sm + kWTot);
    uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + kBars);
    uint64_t* bar_mma = bar_tma + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_tma + 3);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int j0 = blockIdx.y * kNV;
    const int T = p.T;
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
        tc::mbar_init(&bar_tma[0], 1);
        tc::mbar_init(&bar_tma[1], 1);
        tc::mbar_init(bar_mma, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // blockdiag(TW, TU) starts all zero; per chunk only the lower 16x16
    // tiles of TW (box0 rows 0..63) and TU (box1 rows 64..127) are written.
    {
        uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = tid; i < 2048; i += kThreads)
            *reinterpret_cast<uint4*>(sm + kBD + 16 * i) = z;
    }
    // initial state: row tid of S (64 columns of this CTA's half)
    float S[kNV];
    {
        const float* src = p.h0 ? p.h0 + ((size_t)bh * kD + tid) * kD + j0
                                : nullptr;
#pragma unroll
        for (int j = 0; j < kNV; j += 4) {
            float4 v = src ? *reinterpret_cast<const float4*>(src + j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
        }
        st_row_sw128(sm + kSBuf, tid, S);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);

    if (tid == 0 && nchunks > 0) {
        tc::mbar_arrive_expect_tx(&bar_tma[0], kTmaBytes);
        uint8_t* st = sm;
        tc::tma_load_4d(st, &tm_k, &bar_tma[0], 0, h, 0, b);
        tc::tma_load_4d(st + kHalfStride, &tm_k, &bar_tma[0], 64, h, 0, b);
        tc::tma_load_4d(st + kOffQ, &tm_q, &bar_tma[0], 0, h, 0, b);
        tc::tma_load_4d(st + kHalfStride + kOffQ, &tm_q, &bar_tma[0], 64, h,
                        0, b);
        tc::tma_load_4d(st + kOffV, &tm_v, &bar_tma[0], j0, h, 0, b);
    }

    // gates of the next chunk, prefetched into registers (rows 0..63)
    auto load_gates = [&](int c, float& la, float& et) {
        const int t = c * kC + tid;
        if (tid < kC && t < T) {
            const size_t off = ((size_t)b * T + t) * p.H + h;
            la = p.log_alpha[off];
            et = p.eta[off];
        } else {
            la = 0.f;
            et = 0.f;
        }
    };
    float la_cur, eta_cur;
    load_gates(0, la_cur, eta_cur);

    uint32_t ph_tma[2] = {0, 0};
    uint32_t ph_mma = 0;
    bool failed = false;
    bool tma_pending[2] = {nchunks > 0, false};
    bool mma_pending = false;

    for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        uint8_t* st = sm + s * kStage;
        const uint32_t sst = sbase + s * kStage;
        const int t0 = c * kC;

        if (!wait_all(&bar_tma[s], ph_tma[s])) { failed = true; break; }
        ph_tma[s] ^= 1;
        tma_pending[s] = false;
        if (c + 1 < nchunks) {
            if (tid == 0) {
                uint8_t* nx = sm + (s ^ 1) * kStage;
                const int tn = t0 + kC;
                tc::mbar_arrive_expect_tx(&bar_tma[s ^ 1], kTmaBytes);
                tc::tma_load_4d(nx, &tm_k, &bar_tma[s ^ 1], 0, h, tn, b);
                tc::tma_load_4d(nx + kHalfStride, &tm_k, &bar_tma[s ^ 1], 64, h,
                                tn, b);
                tc::tma_load_4d(nx + kOffQ, &tm_q, &bar_tma[s ^ 1], 0, h, tn,
                                b);
                tc::tma_load_4d(nx + kHalfStride + kOffQ, &tm_q,
                                &bar_tma[s ^ 1], 64, h, tn, b);
                tc::tma_load_4d(nx + kOffV, &tm_v, &bar_tma[s ^ 1], j0, h, tn,
                                b);
            }
            tma_pending[s ^ 1] = true;
        }
        float la_nxt, eta_nxt;
        load_gates(c + 1, la_nxt, eta_nxt);

        // ---- (1) G = [K; Q] K^T ----
        tc::tc_fence_after();
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * kHalfStride + (ks & 3) * 32;
                tc::mma_bf16(tmem + kColG, desc_k(sst + off), desc_k(sst + off),
                             kIdG, ks > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        // in-chunk cumulative log decay (rows 0..63: warps 0 and 1)
        float gpart = la_cur;
        if (warp < 2) {
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, gpart, off);
                if ((tid & 31) >= off) gpart += y;
            }
            if ((tid & 31) == 31) wtot[warp] = gpart;
        }
        if (!wait_all(bar_mma, ph_mma)) { failed = true; break; }
        ph_mma ^= 1;
        mma_pending = false;
        tc::tc_fence_after();

        float x[kC];
        tmem_ld64(tlane + kColG, x);        // KK^T row (tid<64) / QK^T row
        if (tid < kC) {
            const float g = gpart + (tid >= 32 ? wtot[0] : 0.f);
            gS[tid] = g;
            float diag = 0.f;
#pragma unroll
            for (int j = 0; j < kC; ++j) diag = (j == tid) ? x[j] : diag;
            const float denom = diag + p.eps;
            betaS[tid] = denom == 0.f ? 0.f : eta_cur / denom;
        }
        __syncthreads();
        if (tid < kC) {
            const int r = tid;
            const float gr = gS[r];
            const float br = betaS[r];
            float* Ar = Af + r * kAStride;
#pragma unroll
            for (int i = 0; i < kC; i += 4) {
                float4 v;
                v.x = (i + 0 < r) ? br * __expf(gr - gS[i + 0]) * x[i + 0] : 0.f;
                v.y = (i + 1 < r) ? br * __expf(gr - gS[i + 1]) * x[i + 1] : 0.f;
                v.z = (i + 2 < r) ? br * __expf(gr - gS[i + 2]) * x[i + 2] : 0.f;
                v.w = (i + 3 < r) ? br * __expf(gr - gS[i + 3]) * x[i + 3] : 0.f;
                *reinterpret_cast<float4*>(Ar + i) = v;
            }
        } else {
            const int r = tid - kC;
            const float gr = gS[r];
#pragma unroll
            for (int i = 0; i < kC; ++i)
                x[i] = (i <= r) ? __expf(gr - gS[i]) * x[i] : 0.f;
            st_row_sw128(sm + kPBuf, r, x);
        }
        __syncthreads();

        // ---- T = A^{-1} (blocked, fp32) ----
        invert_unit_lower64(Af, Tf, Yf, tid);
        // TW = T Diag(beta gamma) -> box0 rows 0..63, TU = T Diag(beta) ->
        // box1 rows 64..127, lower 16x16 tiles only (the rest stays zero).
        // Item = (row r, 8-column chunk q): 64 rows x 8 chunks.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = tid + kThreads * j;
            const int r = e >> 3, q = e & 7;
            if ((q >> 1) <= (r >> 4)) {
                const float* Tr = Tf + r * kAStride + 8 * q;
                float vw[8], vu[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float tv = (8 * q + k <= r) ? Tr[k] : 0.f;
                    const float bc = betaS[8 * q + k];
                    vu[k] = tv * bc;
                    vw[k] = vu[k] * __expf(gS[8 * q + k]);
                }
                uint4 w4, u4;
                w4.x = pack_bf16(vw[0], vw[1]); w4.y = pack_bf16(vw[2], vw[3]);
                w4.z = pack_bf16(vw[4], vw[5]); w4.w = pack_bf16(vw[6], vw[7]);
                u4.x = pack_bf16(vu[0], vu[1]); u4.y = pack_bf16(vu[2], vu[3]);
                u4.z = pack_bf16(vu[4], vu[5]); u4.w = pack_bf16(vu[6], vu[7]);
                *reinterpret_cast<uint4*>(sm + kBD + r * 128 +
                                          ((q ^ (r & 7)) << 4)) = w4;
                *reinterpret_cast<uint4*>(sm + kBD + 16384 + (64 + r) * 128 +
                                          ((q ^ (r & 7)) << 4)) = u4;
            }
        }
        tc::fence_proxy_async_smem();
        __syncthreads();
        tc::tc_fence_after();

        // ---- (2) [W; U] = blockdiag(TW, TU) [K; V] ----
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t a = sbase + kBD + (ks >> 2) * 16384 + (ks & 3) * 32;
                uint64_t bdesc;
                if (ks < 4)
                    bdesc = desc_mn(sst + (ks & 3) * 2048, kHalfStride);
                else
                    bdesc = desc_mn(sst + kOffV + (ks & 3) * 2048, 0);
                tc::mma_bf16(tmem + kColWU, desc_k(a), bdesc, kIdWU, ks > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma)) { failed = true; break; }
        ph_mma ^= 1;
        mma_pending = false;
        tc::tc_fence_after();

        if (tid < kC) {
            // W row tid -> bf16 into W_0 (cols 0..63) and W_1 (cols 64..127);
            // U (lanes 64..127) stays in TMEM until U~ is formed.
            tmem_ld64(tlane + kColWU, x);
            st_row_sw128(st + kOffW, tid, x);
            tmem_ld64(tlane + kColWU + 64, x);
            st_row_sw128(st + kHalfStride + kOffW, tid, x);
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();

        // ---- (3) X = [Q; W] S ----
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t a = sst + (ks >> 2) * kHalfStride + kOffQ + (ks & 3) * 32;
                tc::mma_bf16(tmem + kColX, desc_k(a),
                             desc_mn(sbase + kSBuf + ks * 2048, 0), kIdX, ks > 0);
            }
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma)) { failed = true; break; }
        ph_mma ^= 1;
        mma_pending = false;
        tc::tc_fence_after();

        const float g_last = gS[kC - 1];
        if (tid >= kC) {                           // Q S stays in TMEM
            const int r = tid - kC;
            float u[kNV];
            tmem_ld64(tlane + kColWU, u);          // U row
            tmem_ld64(tlane + kColX, x);           // W S row
#pragma unroll
            for (int j = 0; j < kNV; ++j) u[j] -= x[j];   // U~ row
            st_row_sw128(sm + kUtBuf, r, u);
            const float dec = __expf(g_last - gS[r]);
#pragma unroll
            for (int j = 0; j < kNV; ++j) u[j] *= dec;
            st_row_sw128(sm + kUtsBuf, r, u);
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();

        // ---- (4) dS = K^T Diag(Gamma_C) U~ ; (5) OI = [P; -] U~ ----
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16(tmem + kColDS, desc_mn(sst + ks * 2048, kHalfStride),
                             desc_mn(sbase + kUtsBuf + ks * 2048, 0), kIdDS,
                             ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16(tmem + kColOI, desc_k(sbase + kPBuf + ks * 32),
                             desc_mn(sbase + kUtBuf + ks * 2048, 0), kIdOI,
                             ks > 0);
            tc::mma_commit(bar_mma);
        }
        mma_pending = true;
        if (!wait_all(bar_mma, ph_mma)) { failed = true; break; }
        ph_mma ^= 1;
        mma_pending = false;
        tc::tc_fence_after();

        {
            const float gC = __expf(g_last);
            tmem_ld64(tlane + kColDS, x);          // dS row tid
#pragma unroll
            for (int j = 0; j < kNV; ++j) S[j] = fmaf(gC, S[j], x[j]);
            st_row_sw128(sm + kSBuf, tid, S);
        }
        if (tid < kC) {
            float qs[kNV];
            tmem_ld64(tlane + kColX, qs);          // Q S row
            tmem_ld64(tlane + kColOI, x);          // P U~ row
            const float gam = __expf(gS[tid]);
#pragma unroll
            for (int j = 0; j < kNV; ++j) qs[j] *= gam;
            const int t = t0 + tid;
            if (t < T) {
                __nv_bfloat16* dst =
                    p.o + (((size_t)b * T + t) * p.H + h) * kD + j0;
#pragma unroll
                for (int j = 0; j < kNV; j += 8) {
                    uint4 v;
                    v.x = pack_bf16(qs[j + 0] + x[j + 0], qs[j + 1] + x[j + 1]);
                    v.y = pack_bf16(qs[j + 2] + x[j + 2], qs[j + 3] + x[j + 3]);
                    v.z = pack_bf16(qs[j + 4] + x[j + 4], qs[j + 5] + x[j + 5]);
                    v.w = pack_bf16(qs[j + 6] + x[j + 6], qs[j + 7] + x[j + 7]);
                    *reinterpret_cast<uint4*>(dst + j) = v;
                }
            }
        }
        la_cur = la_nxt;
        eta_cur = eta_nxt;
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    }

    if (failed) {
        if (tid == 0) {
            atomicOr(&g_fault_word, 1u);
            // drain what may still be in flight, each wait bounded
            if (mma_pending) tc::mbar_wait(bar_mma, ph_mma, 100000000ull);
            for (int i = 0; i < 2; ++i)
                if (tma_pending[i])
                    tc::mbar_wait(&bar_tma[i], ph_tma[i], 100000000ull);
        }
        __syncthreads();
    } else if (p.hT) {
        float* dst = p.hT + ((size_t)bh * kD + tid) * kD + j0;
#pragma unroll
        for (int j = 0; j < kNV; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn,
                                             12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// [B, T, H, 128] bf16, box = 64 features x 1 head x 64 tokens x 1 batch.
bool make_map(CUtensorMap* m, const void* base, int B, int T, int H) {
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T,
                          (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2,
                             (cuuint64_t)T * H * kD * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kC, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* ptr) {
    return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
}

}  // namespace

bool chunk_tc_eligible(const FwdArgs& a) {
    return a.dtype == KLA_BF16 && a.dk == kD && a.dv == kD && a.C == kC &&
           aligned16(a.q) && aligned16(a.k) && aligned16(a.v) &&
           aligned16(a.o) && (!a.h0 || aligned16(a.h0)) &&
           (!a.hT || aligned16(a.hT)) && get_encoder();
}

cudaError_t launch_chunk_tc(const FwdArgs& a, cudaStream_t stream) {
    if ((long)a.B * a.H == 0 || a.T == 0) return cudaSuccess;
    if (!get_encoder()) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.B, a.T, a.H) ||
        !make_map(&mk, a.k, a.B, a.T, a.H) ||
        !make_map(&mv, a.v, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(
            kla_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
            kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    TcParams p{a.log_alpha, a.eta, a.h0,
               static_cast<__nv_bfloat16*>(a.o), a.hT, a.eps, a.T, a.H};
    dim3 grid((unsigned)((long)a.B * a.H), kD / kNV);
    kla_chunk_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_fault(cudaStream_t stream, unsigned int* word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_fault_word, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned int));
}

}  // namespace kla
