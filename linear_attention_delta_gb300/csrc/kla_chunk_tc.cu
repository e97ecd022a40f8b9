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
// Work decomposition: one CTA per (batch, head, half of dv), 256 threads in
// two specialised warpgroups that run one chunk apart:
//   * intra warpgroup (warps 0-3), chunk c+1:  G = [K;Q] K^T on the tensor
//     cores, beta and the cumulative decay, the Gamma-masked A, T = A^{-1}
//     (fp32 substitution on the 16x16 diagonal tiles, warp-level mma for the
//     off-diagonal tiles) written straight out as TW = T Diag(beta gamma) and
//     TU = T Diag(beta), then W = TW K and U = TU V issued on the tensor
//     cores;
//   * state warpgroup (warps 4-7), chunk c:  W to a bf16 operand,
//     P = Gamma o Q K^T (warps 6, 7, off the critical path), U~ = U - W S
//     accumulated in TMEM by a negated-operand MMA onto U, Q S,
//     dS = K^T Diag(Gamma_C) U~ and P U~ on the tensor cores;
//     the 128 x 64 fp32 state slice lives in registers (one key row per
//     thread), its bf16 copy in shared memory is the MMA operand; o is
//     written from registers.
// The warpgroups hand over through mbarriers (chunk handed over / chunk
// done); G, W and U have two TMEM buffers each, so the intra side never waits
// for the state side to finish reading them.  q, k, v tiles arrive by TMA (128-byte swizzle) in a three-deep
// ring, refilled by the state warpgroup as it frees each stage.
//
// Every mbarrier wait is bounded (2 s) and also gives up when the other
// warpgroup has failed: the CTA then records a fault in the library's fault
// word, drains what it issued (bounded), frees TMEM and returns.
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
constexpr int kThreads = 256;
constexpr int kNS = 3;        // TMA stages

// ---- shared memory map (bytes from a 1024-aligned base) -------------------
// stage (40 KB): K_0 | Q_0 | K_1 | Q_1 | V   (each 64 rows x 128 B, swizzled;
// K_h / Q_h hold key dims 64h..64h+63).  [K_h; Q_h] is a 128-row K-major
// operand; the 64 rows after Q_h, W_h, TU and P are don't-care rows of padded
// M=128 MMAs whose TMEM lanes 64..127 are never read.
constexpr int kOffQ = 8192;
constexpr int kHalf = 16384;
constexpr int kOffV = 32768;
constexpr int kStage = 40960;
constexpr int kWBuf = kNS * kStage;          // W_0 | W_1   (K-major, 64 rows)
constexpr int kSBuf = kWBuf + 16384;         // bf16 S, 128 x 64, MN-major
constexpr int kTWU = kSBuf + 16384;          // TW (rows 0..63) | TU
constexpr int kPBuf = kTWU + 16384;          // P, 64 x 64 K-major
constexpr int kUtBuf = kPBuf + 8192;         // U~ bf16, MN-major
constexpr int kUtsBuf = kUtBuf + 8192;       // Diag(Gamma_C) U~ bf16
constexpr int kTileF = 16 * 17;              // fp32 16x16 tile, row stride 17
constexpr int kADiag = kUtsBuf + 8192;       // 4 fp32 diagonal tiles of A
constexpr int kAOff = kADiag + 4 * kTileF * 4;   // 6 bf16 tiles A_im, i > m
constexpr int kTF = kAOff + 6 * 256 * 2;     // 10 fp32 tiles T_ij, i >= j
constexpr int kGBuf = kTF + 10 * kTileF * 4; // 2 x {g2, beta, beta*gamma}
constexpr int kGBufStride = 3 * 64;          // floats per buffer
constexpr int kBars = kGBuf + 2 * kGBufStride * 4;
constexpr int kNumBars = 10;
constexpr int kMisc = kBars + 8 * kNumBars;  // abort flag, warp total, TMEM
constexpr int kSmemUsed = kMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kBars % 8 == 0, "mbarrier alignment");
constexpr uint32_t kTmaBytes = 2 * 16384 + 8192;

// mbarrier slots
constexpr int kBarTma = 0;     // kNS: stage full (TMA)
constexpr int kBarG = 3;       // G MMA done
constexpr int kBarWU = 4;      // W, U MMAs done
constexpr int kBarX = 5;       // U~ = U - W S formed in TMEM
constexpr int kBarDS = 6;      // Q S, dS, P U~ done
constexpr int kBarWReady = 7;  // intra -> state: gates and TW | TU written
constexpr int kBarSDone = 9;   // state -> intra: chunk finished

// ---- TMEM columns (two buffers, by chunk parity b) -------------------------
// G[b]: lanes 0..63 K K^T, lanes 64..127 Q K^T; then P U~ (lanes 0..63).
// W[b]: lanes 0..63 W (128 cols); then Q S in its first 64 columns.
// U[b]: lanes 0..63 U, then U~ = U - W S; then dS (lane = key row).
constexpr uint32_t kColG = 0;      // + 64 b
constexpr uint32_t kColW = 128;    // + 128 b
constexpr uint32_t kColU = 384;    // + 64 b
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdG = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdW = tc::idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdN64 = tc::idesc_bf16(128, 64, false, true);
constexpr uint32_t kIdDS = tc::idesc_bf16(128, 64, true, true);
constexpr uint32_t kIdNegW = tc::idesc_bf16(128, 64, false, true, true);

constexpr int kBarIntra = 1;   // named barrier ids
constexpr int kBarState = 2;
constexpr int kBarW13 = 3;     // intra warps 1..3
constexpr int kBarW23 = 4;     // intra warps 2..3
constexpr int kBarState01 = 5; // state warps 4, 5

constexpr float kLog2e = 1.4426950408889634f;

struct TcParams {
    const float* log_alpha;
    const float* eta;
    const float* h0;
    __nv_bfloat16* o;
    float* hT;
    float eps;
    int gdn;
    int T, H;
};

// Write 64 fp32 values as one 128-byte swizzled bf16 row.
__device__ __forceinline__ void st_row_sw128(uint8_t* base, int row,
                                             const float* x) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 v;
        v.x = tc::pack_bf16x2(x[8 * j + 0], x[8 * j + 1]);
        v.y = tc::pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
        v.z = tc::pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
        v.w = tc::pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
        *reinterpret_cast<uint4*>(base + row * 128 + ((j ^ (row & 7)) << 4)) = v;
    }
}

// 64 consecutive TMEM columns of this thread's lane -> x[0..63].
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* x) {
    tc::tmem_ld32(taddr + 0, x);
    tc::tmem_ld32(taddr + 32, x + 32);
    tc::tmem_ld_wait();
}

__device__ __forceinline__ uint64_t desc_k(uint32_t addr) {
    return tc::sdesc_sw128(addr, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr, uint32_t lbo) {
    return tc::sdesc_sw128(addr, lbo, 1024);
}

// Every thread of a warpgroup waits on the mbarrier, then the warpgroup
// agrees on the outcome (true = all saw the phase complete).  On failure the
// CTA-wide abort flag is raised so that the other warpgroup stops too.
__device__ __forceinline__ bool wg_wait(uint64_t* bar, uint32_t parity,
                                        int* abort_flag, int bar_id) {
    const bool ok = tc::mbar_wait_or_abort(bar, parity, abort_flag);
    const bool any_fail = tc::named_bar_or(bar_id, 128, !ok);
    if (any_fail) *reinterpret_cast<volatile int*>(abort_flag) = 1;
    return !any_fail;
}

__device__ __forceinline__ uint32_t ld_bf16_pair(const __nv_bfloat16* p0,
                                                 const __nv_bfloat16* p1) {
    const uint32_t lo = *reinterpret_cast<const unsigned short*>(p0);
    const uint32_t hi = *reinterpret_cast<const unsigned short*>(p1);
    return lo | (hi << 16);
}

// packed index of lower tile (i, j), i >= j
__host__ __device__ constexpr int tri(int i) { return i * (i + 1) / 2; }

// A fragment (16x16, row-major) of an fp32 tile with row stride 17.
__device__ __forceinline__ void afrag_f32(const float* t, int g, int q,
                                          uint32_t (&a)[4]) {
    a[0] = tc::pack_bf16x2(t[g * 17 + 2 * q], t[g * 17 + 2 * q + 1]);
    a[1] = tc::pack_bf16x2(t[(g + 8) * 17 + 2 * q],
                           t[(g + 8) * 17 + 2 * q + 1]);
    a[2] = tc::pack_bf16x2(t[g * 17 + 2 * q + 8], t[g * 17 + 2 * q + 9]);
    a[3] = tc::pack_bf16x2(t[(g + 8) * 17 + 2 * q + 8],
                           t[(g + 8) * 17 + 2 * q + 9]);
}

// acc[nt] += X * Z for the two 8-column halves nt; X an A fragment, Z a
// 16x16 fp32 tile (row stride 17).
__device__ __forceinline__ void mm_tile_f32(float (&acc)[2][4],
                                            const uint32_t (&x)[4],
                                            const float* z, int g, int q) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = nt * 8 + g;
        const uint32_t b0 = tc::pack_bf16x2(z[(2 * q) * 17 + n],
                                            z[(2 * q + 1) * 17 + n]);
        const uint32_t b1 = tc::pack_bf16x2(z[(2 * q + 8) * 17 + n],
                                            z[(2 * q + 9) * 17 + n]);
        tc::mma_m16n8k16(acc[nt], x, b0, b1);
    }
}

// Same with Z a bf16 16x16 tile (row stride 16).
__device__ __forceinline__ void mm_tile_bf16(float (&acc)[2][4],
                                             const uint32_t (&x)[4],
                                             const __nv_bfloat16* z, int g,
                                             int q) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int n = nt * 8 + g;
        const uint32_t b0 = ld_bf16_pair(z + (2 * q) * 16 + n,
                                         z + (2 * q + 1) * 16 + n);
        const uint32_t b1 = ld_bf16_pair(z + (2 * q + 8) * 16 + n,
                                         z + (2 * q + 9) * 16 + n);
        tc::mma_m16n8k16(acc[nt], x, b0, b1);
    }
}

// Byte offset of element (row, col) in a K-major bf16 operand with 128-byte
// swizzled rows (64 columns per row).
__device__ __forceinline__ int sw_off(int row, int col) {
    return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

// Tile (I, J) of T, given as -acc in accumulator-fragment layout: keep the
// fp32 copy when later tiles need it (tf != nullptr) and write the bf16
// operands TW = T Diag(beta gamma) (rows 0..63 of twu) and TU = T Diag(beta)
// (rows 64..127).  gb = {g2[64], beta[64], beta*gamma[64]} of this chunk.
__device__ __forceinline__ void store_t_tile(float* tf, uint8_t* twu,
                                             const float* gb, int I, int J,
                                             const float (&acc)[2][4], int g,
                                             int q) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int c = nt * 8 + 2 * q;
        const int col = 16 * J + c;
        const float t00 = -acc[nt][0], t01 = -acc[nt][1];
        const float t10 = -acc[nt][2], t11 = -acc[nt][3];
        if (tf) {
            tf[g * 17 + c] = t00;
            tf[g * 17 + c + 1] = t01;
            tf[(g + 8) * 17 + c] = t10;
            tf[(g + 8) * 17 + c + 1] = t11;
        }
        const float b0 = gb[64 + col], b1 = gb[64 + col + 1];
        const float w0 = gb[128 + col], w1 = gb[128 + col + 1];
        const int r0 = 16 * I + g, r1 = r0 + 8;
        *reinterpret_cast<uint32_t*>(twu + sw_off(r0, col)) =
            tc::pack_bf16x2(t00 * w0, t01 * w1);
        *reinterpret_cast<uint32_t*>(twu + sw_off(r1, col)) =
            tc::pack_bf16x2(t10 * w0, t11 * w1);
        *reinterpret_cast<uint32_t*>(twu + 8192 + sw_off(r0, col)) =
            tc::pack_bf16x2(t00 * b0, t01 * b1);
        *reinterpret_cast<uint32_t*>(twu + 8192 + sw_off(r1, col)) =
            tc::pack_bf16x2(t10 * b0, t11 * b1);
    }
}

__device__ __forceinline__ void zero_acc(float (&acc)[2][4]) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[nt][k] = 0.f;
}

// Off-diagonal tiles of block row I of T = A^{-1}, by warp I (I = 1..3):
//   Y_Im = T_II A_Im (m < I), kept in registers as A fragments;
//   T_Ij = -sum_{m=j}^{I-1} Y_Im T_mj, for j = I-1, I-2, I-3 in turn, with
//   barriers between the distances because T_mj comes from other warps.
// Tiles of block row 3 are never read again, so only TW/TU receive them.
template <int I>
__device__ __forceinline__ void offdiag_row(const __nv_bfloat16* Ao, float* Tt,
                                            uint8_t* twu, const float* gb,
                                            int lane) {
    const int g = lane >> 2, q = lane & 3;
    uint32_t ta[4];
    afrag_f32(Tt + (tri(I) + I) * kTileF, g, q, ta);
    uint32_t ya[I][4];
#pragma unroll
    for (int m = 0; m < I; ++m) {
        float acc[2][4];
        zero_acc(acc);
        mm_tile_bf16(acc, ta, Ao + (tri(I - 1) + m) * 256, g, q);
        ya[m][0] = tc::pack_bf16x2(acc[0][0], acc[0][1]);
        ya[m][1] = tc::pack_bf16x2(acc[0][2], acc[0][3]);
        ya[m][2] = tc::pack_bf16x2(acc[1][0], acc[1][1]);
        ya[m][3] = tc::pack_bf16x2(acc[1][2], acc[1][3]);
    }
    float* keep = I < 3 ? Tt : nullptr;
    {   // distance 1
        float acc[2][4];
        zero_acc(acc);
        mm_tile_f32(acc, ya[I - 1], Tt + (tri(I - 1) + I - 1) * kTileF, g, q);
        store_t_tile(keep ? keep + (tri(I) + I - 1) * kTileF : nullptr, twu,
                     gb, I, I - 1, acc, g, q);
    }
    tc::named_bar_sync(kBarW13, 96);
    if constexpr (I >= 2) {   // distance 2
        float acc[2][4];
        zero_acc(acc);
        mm_tile_f32(acc, ya[I - 2], Tt + (tri(I - 2) + I - 2) * kTileF, g, q);
        mm_tile_f32(acc, ya[I - 1], Tt + (tri(I - 1) + I - 2) * kTileF, g, q);
        store_t_tile(keep ? keep + (tri(I) + I - 2) * kTileF : nullptr, twu,
                     gb, I, I - 2, acc, g, q);
        tc::named_bar_sync(kBarW23, 64);
    }
    if constexpr (I == 3) {   // distance 3
        float acc[2][4];
        zero_acc(acc);
        mm_tile_f32(acc, ya[0], Tt + tri(0) * kTileF, g, q);
        mm_tile_f32(acc, ya[1], Tt + tri(1) * kTileF, g, q);
        mm_tile_f32(acc, ya[2], Tt + tri(2) * kTileF, g, q);
        store_t_tile(nullptr, twu, gb, 3, 0, acc, g, q);
    }
}

// T = A^{-1} (64x64 unit lower triangular), written out as TW | TU.
// A: fp32 diagonal tiles (strictly lower part, zero above) and bf16 tiles
// A_im (i > m) at tri(i-1) + m.  T: fp32 tiles (i >= j) at tri(i) + j, kept
// for the tiles that later tiles are built from.
//
// Diagonal tiles T_ii = A_ii^{-1} (fp32 column substitution): thread
// (bb = tid / 16, cl = tid % 16) of intra warps 0 and 1, i.e. each of those
// warps inverts the two diagonal tiles of the rows it has just built.
__device__ __forceinline__ void invert_diag_tiles(const float* Ad, float* Tt,
                                                  uint8_t* twu,
                                                  const float* gb, int tid) {
    {
        const int bb = tid >> 4, cl = tid & 15;
        const float* Ab = Ad + bb * kTileF;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) t[r] = (r == cl) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int i = 0; i < r; i += 2) {
                a0 = fmaf(Ab[r * 17 + i], t[i], a0);
                if (i + 1 < r) a1 = fmaf(Ab[r * 17 + i + 1], t[i + 1], a1);
            }
            if (r > cl) t[r] = -(a0 + a1);
        }
        float* Tb = Tt + (tri(bb) + bb) * kTileF + cl;
        const int col = 16 * bb + cl;
        const float bc = gb[64 + col], wc = gb[128 + col];
        __nv_bfloat16* tw = reinterpret_cast<__nv_bfloat16*>(twu);
        __nv_bfloat16* tu = reinterpret_cast<__nv_bfloat16*>(twu + 8192);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            Tb[r * 17] = t[r];
            const int off = sw_off(16 * bb + r, col) >> 1;
            tw[off] = __float2bfloat16_rn(t[r] * wc);
            tu[off] = __float2bfloat16_rn(t[r] * bc);
        }
    }
}

// Off-diagonal tiles, after every diagonal tile is in place (warps 1..3).
__device__ __forceinline__ void invert_offdiag_tiles(const __nv_bfloat16* Ao,
                                                     float* Tt, uint8_t* twu,
                                                     const float* gb,
                                                     int tid) {
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (warp == 1) offdiag_row<1>(Ao, Tt, twu, gb, lane);
    else if (warp == 2) offdiag_row<2>(Ao, Tt, twu, gb, lane);
    else if (warp == 3) offdiag_row<3>(Ao, Tt, twu, gb, lane);
}

__device__ __forceinline__ uint32_t col_g(int c) { return kColG + 64 * (c & 1); }
__device__ __forceinline__ uint32_t col_w(int c) { return kColW + 128 * (c & 1); }
__device__ __forceinline__ uint32_t col_u(int c) { return kColU + 64 * (c & 1); }

__global__ void __launch_bounds__(kThreads, 1)
kla_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_u32(sm);
    float* Ad = reinterpret_cast<float*>(sm + kADiag);
    __nv_bfloat16* Ao = reinterpret_cast<__nv_bfloat16*>(sm + kAOff);
    float* Tt = reinterpret_cast<float*>(sm + kTF);
    float* gbuf = reinterpret_cast<float*>(sm + kGBuf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
    int* abort_flag = reinterpret_cast<int*>(sm + kMisc);
    float* wtot = reinterpret_cast<float*>(sm + kMisc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc + 8);

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
        for (int i = 0; i < kNumBars; ++i) tc::mbar_init(&bars[i], 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // TW | TU start all zero; per chunk only their lower 16x16 tiles change.
    for (int i = tid; i < 1024; i += kThreads)
        *reinterpret_cast<uint4*>(sm + kTWU + 16 * i) = make_uint4(0, 0, 0, 0);

    float S[kNV];   // state rows (state warpgroup)
    if (tid >= 128) {
        const int row = tid - 128;
        const float* src = p.h0 ? p.h0 + ((size_t)bh * kD + row) * kD + j0
                                : nullptr;
#pragma unroll
        for (int j = 0; j < kNV; j += 4) {
            float4 v = src ? *reinterpret_cast<const float4*>(src + j)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
        }
        st_row_sw128(sm + kSBuf, row, S);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto issue_tma = [&](int c) {
        const int s = c % kNS;
        uint8_t* st = sm + s * kStage;
        const int t0 = c * kC;
        uint64_t* bar = &bars[kBarTma + s];
        tc::mbar_arrive_expect_tx(bar, kTmaBytes);
        tc::tma_load_4d(st, &tm_k, bar, 0, h, t0, b);
        tc::tma_load_4d(st + kOffQ, &tm_q, bar, 0, h, t0, b);
        tc::tma_load_4d(st + kHalf, &tm_k, bar, 64, h, t0, b);
        tc::tma_load_4d(st + kHalf + kOffQ, &tm_q, bar, 64, h, t0, b);
        tc::tma_load_4d(st + kOffV, &tm_v, bar, j0, h, t0, b);
    };
    if (tid == 0)
        for (int c = 0; c < kNS && c < nchunks; ++c) issue_tma(c);

    if (tid < 128) {
        // ==================================================== intra warpgroup
        const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
        bool failed = false, g_pending = false;
        auto load_gates = [&](int c, float& la, float& et) {
            const int t = c * kC + tid;
            la = 0.f;
            et = 0.f;
            if (tid < kC && t < T) {
                const size_t off = ((size_t)b * T + t) * p.H + h;
                la = p.log_alpha[off];
                et = p.eta[off];
            }
        };
        auto issue_g = [&](int c) {
            const uint32_t sst = sbase + (c % kNS) * kStage;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
                tc::mma_bf16(tmem + col_g(c), desc_k(sst + off),
                             desc_k(sst + off), kIdG, ks > 0);
            }
            tc::mma_commit(&bars[kBarG]);
        };
        float la_cur, eta_cur;
        load_gates(0, la_cur, eta_cur);
        if (nchunks > 0) {
            if (wg_wait(&bars[kBarTma], 0, abort_flag, kBarIntra)) {
                tc::tc_fence_after();
                if (tid == 0) issue_g(0);
                g_pending = true;
            } else {
                failed = true;
            }
        }
        for (int c = 0; c < nchunks && !failed; ++c) {
            float la_nxt, eta_nxt;
            load_gates(c + 1, la_nxt, eta_nxt);
            // gate buffer of chunk c-2: released (state side waited for it
            // before G(c) was issued, see the end of the previous iteration)
            float* gb = gbuf + (c & 1) * kGBufStride;   // g2 | beta | bg

            // cumulative log2-decay: warp scans on rows 0..31 and 32..63
            float g2 = la_cur * kLog2e;
            if (warp < 2) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, g2, off);
                    if ((tid & 31) >= off) g2 += y;
                }
                if (tid == 31) *wtot = g2;
            }
            if (!wg_wait(&bars[kBarG], c & 1, abort_flag, kBarIntra)) {
                failed = true; break;
            }
            g_pending = false;
            tc::tc_fence_after();
            float x[kC];
            if (warp < 2) {
                tmem_ld64(tlane + col_g(c), x);     // K K^T row tid
                if (tid >= 32) g2 += *wtot;
                float diag = 0.f;
#pragma unroll
                for (int j = 0; j < kC; ++j) diag = (j == tid) ? x[j] : diag;
                const float denom = diag + p.eps;
                const float beta =
                    p.gdn ? eta_cur : (denom == 0.f ? 0.f : eta_cur / denom);
                gb[tid] = g2;
                gb[kC + tid] = beta;
                gb[2 * kC + tid] = beta * tc::ex2(g2);
            }
            // TW | TU are still read by the W, U MMAs of chunk c-1
            if (c >= 1) {
                if (!wg_wait(&bars[kBarWU], (c - 1) & 1, abort_flag,
                             kBarIntra)) { failed = true; break; }
            } else {
                tc::named_bar_sync(kBarIntra, 128);
            }
            // ---- A (warps 0, 1), then each warp inverts its diagonal tiles
            if (warp < 2) {
                const int r = tid, ti = r >> 4, rr = r & 15;
                const float gr = gb[r], br = gb[kC + r];
                const int mmax = warp == 0 ? 1 : 3;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (m > mmax) break;
                    float v[16];
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        const int i = 16 * m + cc;
                        v[cc] = (i < r) ? br * tc::ex2(gr - gb[i]) * x[i] : 0.f;
                    }
                    if (m < ti) {
                        __nv_bfloat16* dst =
                            Ao + (tri(ti - 1) + m) * 256 + rr * 16;
#pragma unroll
                        for (int cc = 0; cc < 16; cc += 8) {
                            uint4 u;
                            u.x = tc::pack_bf16x2(v[cc + 0], v[cc + 1]);
                            u.y = tc::pack_bf16x2(v[cc + 2], v[cc + 3]);
                            u.z = tc::pack_bf16x2(v[cc + 4], v[cc + 5]);
                            u.w = tc::pack_bf16x2(v[cc + 6], v[cc + 7]);
                            *reinterpret_cast<uint4*>(dst + cc) = u;
                        }
                    } else if (m == ti) {
                        float* dst = Ad + ti * kTileF + rr * 17;
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) dst[cc] = v[cc];
                    }
                }
                __syncwarp();
                invert_diag_tiles(Ad, Tt, sm + kTWU, gb, tid);
                tc::fence_proxy_async_smem();
            }
            tc::named_bar_sync(kBarIntra, 128);

            if (warp == 0) {
                // Warp 0 has no off-diagonal tile: it issues the next chunk's
                // G once its tiles have landed and chunk c-1 (last user of
                // that G buffer and of the gate buffer) is done.
                if (c + 1 < nchunks) {
                    const int s1 = (c + 1) % kNS;
                    bool ok = tc::mbar_wait_or_abort(&bars[kBarTma + s1],
                                                     ((c + 1) / kNS) & 1,
                                                     abort_flag);
                    if (ok && c >= 1)
                        ok = tc::mbar_wait_or_abort(&bars[kBarSDone],
                                                    (c - 1) & 1, abort_flag);
                    if (__all_sync(0xffffffffu, ok)) {
                        tc::tc_fence_after();
                        if (tid == 0) issue_g(c + 1);
                        g_pending = true;
                    } else {
                        *reinterpret_cast<volatile int*>(abort_flag) = 1;
                    }
                }
            } else {
                // ---- off-diagonal tiles of T = A^{-1}, as TW | TU ----
                invert_offdiag_tiles(Ao, Tt, sm + kTWU, gb, tid);
                tc::fence_proxy_async_smem();
                tc::named_bar_sync(kBarW13, 96);
                // chunk handed over: the state side issues W, U itself
                if (tid == 32) tc::mbar_arrive(&bars[kBarWReady]);
            }
            la_cur = la_nxt;
            eta_cur = eta_nxt;
        }
        if (failed && tid == 0) {   // let issued MMAs finish (bounded)
            if (g_pending) tc::mbar_wait(&bars[kBarG], 0, 100000000ull);
        }
    } else {
        // ==================================================== state warpgroup
        const int sw = warp - 4;                 // TMEM lane quarter
        const uint32_t tlane = tmem + ((uint32_t)(sw * 32) << 16);
        const int row = tid - 128;               // TMEM lane = key row
        bool failed = false, x_pending = false, ds_pending = false;
        bool wu_pending = false;
        for (int c = 0; c < nchunks && !failed; ++c) {
            const int s = c % kNS;
            const uint32_t sst = sbase + s * kStage;
            const float* gb = gbuf + (c & 1) * kGBufStride;
            if (!wg_wait(&bars[kBarWReady], c & 1, abort_flag, kBarState)) {
                failed = true; break;
            }
            tc::tc_fence_after();
            if (tid == 224) {
                // W = [TW; -] K (B: K, MN-major, key halves kHalf apart) and
                // U = [TU; -] V
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + col_w(c), desc_k(sbase + kTWU + ks * 32),
                                 desc_mn(sst + ks * 2048, kHalf), kIdW, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + col_u(c),
                                 desc_k(sbase + kTWU + 8192 + ks * 32),
                                 desc_mn(sst + kOffV + ks * 2048, 0), kIdN64,
                                 ks > 0);
                tc::mma_commit(&bars[kBarWU]);
            }
            wu_pending = true;
            bool wu_ok = true;
            if (sw < 2) {   // warps 4, 5 agree before their pair barrier
                const bool ok =
                    tc::mbar_wait_or_abort(&bars[kBarWU], c & 1, abort_flag);
                wu_ok = !tc::named_bar_or(kBarState01, 64, !ok);
                if (!wu_ok) *reinterpret_cast<volatile int*>(abort_flag) = 1;
                tc::tc_fence_after();
            }
            if (sw < 2 && wu_ok) {   // W row -> bf16 K-major operand
                float x[kNV];
                tmem_ld64(tlane + col_w(c), x);
                st_row_sw128(sm + kWBuf, row, x);
                tmem_ld64(tlane + col_w(c) + 64, x);
                st_row_sw128(sm + kWBuf + 8192, row, x);
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                tc::named_bar_sync(kBarState01, 64);
                tc::tc_fence_after();
                if (tid == 128) {
                    // U~ = U - W S into U's columns (critical path), then Q S
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_bf16(tmem + col_u(c),
                                     desc_k(sbase + kWBuf + (ks >> 2) * 8192 +
                                            (ks & 3) * 32),
                                     desc_mn(sbase + kSBuf + ks * 2048, 0),
                                     kIdNegW, true);
                    tc::mma_commit(&bars[kBarX]);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_bf16(tmem + col_w(c),
                                     desc_k(sst + (ks >> 2) * kHalf + kOffQ +
                                            (ks & 3) * 32),
                                     desc_mn(sbase + kSBuf + ks * 2048, 0),
                                     kIdN64, ks > 0);
                }
            } else {        // P row = Gamma o Q K^T, lower incl.
                const int r = row - kC;
                const float gr = gb[r];
                uint8_t* prow = sm + kPBuf + r * 128;
                const int jmax = (r >> 3) + 1;   // 8-column groups needed
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (__any_sync(0xffffffffu, j < jmax)) {
                        float x[8];
                        tc::tmem_ld8(tlane + col_g(c) + 8 * j, x);
                        const float4 g0 = *reinterpret_cast<const float4*>(gb + 8 * j);
                        const float4 g1 = *reinterpret_cast<const float4*>(gb + 8 * j + 4);
                        tc::tmem_ld_wait();
                        const float gi[8] = {g0.x, g0.y, g0.z, g0.w,
                                             g1.x, g1.y, g1.z, g1.w};
                        float e[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            e[k] = (8 * j + k <= r) ? tc::ex2(gr - gi[k]) * x[k]
                                                    : 0.f;
                        v.x = tc::pack_bf16x2(e[0], e[1]);
                        v.y = tc::pack_bf16x2(e[2], e[3]);
                        v.z = tc::pack_bf16x2(e[4], e[5]);
                        v.w = tc::pack_bf16x2(e[6], e[7]);
                    }
                    *reinterpret_cast<uint4*>(prow + ((j ^ (r & 7)) << 4)) = v;
                }
            }
            x_pending = true;
            if (!wg_wait(&bars[kBarX], c & 1, abort_flag, kBarState)) {
                failed = true; break;
            }
            x_pending = false;
            tc::tc_fence_after();
            const float g_last = gb[kC - 1];
            if (sw < 2) {   // rows 0..63: U~ and Diag(Gamma_C) U~ as operands
                float u[kNV];
                tmem_ld64(tlane + col_u(c), u);
                st_row_sw128(sm + kUtBuf, row, u);
                const float dec = tc::ex2(g_last - gb[row]);
#pragma unroll
                for (int j = 0; j < kNV; ++j) u[j] *= dec;
                st_row_sw128(sm + kUtsBuf, row, u);
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::named_bar_sync(kBarState, 128);
            tc::tc_fence_after();
            if (tid == 128) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + col_u(c), desc_mn(sst + ks * 2048, kHalf),
                                 desc_mn(sbase + kUtsBuf + ks * 2048, 0), kIdDS,
                                 ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + col_g(c),
                                 desc_k(sbase + kPBuf + ks * 32),
                                 desc_mn(sbase + kUtBuf + ks * 2048, 0), kIdN64,
                                 ks > 0);
                tc::mma_commit(&bars[kBarDS]);
            }
            ds_pending = true;
            if (!wg_wait(&bars[kBarDS], c & 1, abort_flag, kBarState)) {
                failed = true; break;
            }
            ds_pending = false;
            tc::tc_fence_after();
            {
                float x[kNV];
                const float gC = tc::ex2(g_last);
                tmem_ld64(tlane + col_u(c), x);
#pragma unroll
                for (int j = 0; j < kNV; ++j) S[j] = fmaf(gC, S[j], x[j]);
                st_row_sw128(sm + kSBuf, row, S);
            }
            if (sw < 2) {   // rows 0..63: o = gamma Q S + P U~
                float qs[kNV], x[kNV];
                tmem_ld64(tlane + col_w(c), qs);
                tmem_ld64(tlane + col_g(c), x);
                const float gam = tc::ex2(gb[row]);
                const int t = c * kC + row;
                if (t < T) {
                    __nv_bfloat16* dst =
                        p.o + (((size_t)b * T + t) * p.H + h) * kD + j0;
#pragma unroll
                    for (int j = 0; j < kNV; j += 8) {
                        uint4 v;
                        v.x = tc::pack_bf16x2(fmaf(gam, qs[j + 0], x[j + 0]),
                                              fmaf(gam, qs[j + 1], x[j + 1]));
                        v.y = tc::pack_bf16x2(fmaf(gam, qs[j + 2], x[j + 2]),
                                              fmaf(gam, qs[j + 3], x[j + 3]));
                        v.z = tc::pack_bf16x2(fmaf(gam, qs[j + 4], x[j + 4]),
                                              fmaf(gam, qs[j + 5], x[j + 5]));
                        v.w = tc::pack_bf16x2(fmaf(gam, qs[j + 6], x[j + 6]),
                                              fmaf(gam, qs[j + 7], x[j + 7]));
                        *reinterpret_cast<uint4*>(dst + j) = v;
                    }
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::named_bar_sync(kBarState, 128);
            if (tid == 128) {
                tc::mbar_arrive(&bars[kBarSDone]);
                if (c + kNS < nchunks) issue_tma(c + kNS);
            }
        }
        if (failed && tid == 224 && wu_pending)
            tc::mbar_wait(&bars[kBarWU], 0, 100000000ull);
        if (failed && tid == 128) {   // let issued MMAs finish (bounded)
            if (x_pending) tc::mbar_wait(&bars[kBarX], 0, 100000000ull);
            if (ds_pending) tc::mbar_wait(&bars[kBarDS], 0, 100000000ull);
        }
    }

    __syncthreads();
    const bool any_failed = *reinterpret_cast<volatile int*>(abort_flag) != 0;
    if (any_failed) {
        if (tid == 0) {
            atomicOr(&g_fault_word, 1u);
            for (int s = 0; s < kNS; ++s)   // copies possibly in flight
                tc::mbar_wait(&bars[kBarTma + s], 0, 100000000ull);
        }
    } else if (tid >= 128 && p.hT) {
        const int row = tid - 128;
        float* dst = p.hT + ((size_t)bh * kD + row) * kD + j0;
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
               static_cast<__nv_bfloat16*>(a.o), a.hT, a.eps, a.gdn, a.T, a.H};
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
