// Tensor-core (tcgen05) chunkwise KLA forward pass for bf16 q/k/v/o,
// dk = dv = 128, chunk C = 64, fp32 state.
//
// Algorithm (per (batch, head); rows r, i of a chunk; g = in-chunk cumulative
// log decay, gamma_r = exp(g_r), Gamma_ri = exp(g_r - g_i), r >= i):
//   beta_r = eta_r / (||k_r||^2 + eps)           (||k_r||^2 = diag of K K^T)
//   A  = I + strict_lower(Diag(beta) (Gamma o K K^T)),   T = A^{-1}
//   U~ = T Diag(beta) (V - Diag(gamma) K S)
//   O  = Diag(gamma) Q S + lower_incl(Gamma o Q K^T) U~
//   S <- gamma_C S + K^T Diag(Gamma_{C,.}) U~
// i.e. the gated-DeltaNet block solver with B = Diag(beta) as the only
// change (gist.science/es/paper/2605.08587, section "Implementacion"), with
// U - W S (U = T Diag(beta) V, W = T Diag(beta gamma) K) regrouped as one
// product of T Diag(beta) with the residual V - Diag(gamma) K S.
//
// Work decomposition: one CTA per (batch, head, half of dv), 256 threads in
// three specialised groups:
//   * A team (warps 0, 1), chunk c+2 or so: beta and the cumulative decay
//     from G = [K;Q] K^T, the Gamma-masked A and the fp32 inverses of its
//     16x16 diagonal tiles;
//   * T team (warps 2, 3), one chunk behind the A team: the off-diagonal
//     tiles of T = A^{-1} (warp-level mma), written with the diagonal ones as
//     the bf16 operand TU = T Diag(beta);
//   * state warpgroup (warps 4-7), chunk c: [K;Q] S on the tensor cores
//     (K S and Q S in one MMA), the residual X = V - Diag(gamma) K S written
//     over V, U~ = TU X, P = Gamma o Q K^T, dS = K^T Diag(Gamma_C) U~ and
//     P U~; the 128 x 64 fp32 state slice lives in registers (one key row per
//     thread), its bf16 copy in shared memory is the MMA operand; o is
//     written from registers.
// Only U~ = TU X waits for the intra-chunk side; [K;Q] S and the residual of
// chunk c start as soon as the state of chunk c-1 is in place.  The groups
// hand over through mbarriers; q, k, v tiles arrive by TMA (128-byte swizzle)
// in a three-deep ring.
//
// Every mbarrier wait is bounded (2 s) and also gives up when another group
// has failed: the CTA then records a fault in the library's fault word,
// drains what it issued (bounded), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include <atomic>

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
constexpr int kPrefetch = 2;  // chunks beyond the ring prefetched into L2

// ---- shared memory map (bytes from a 1024-aligned base) -------------------
// stage (40 KB): K_0 | Q_0 | K_1 | Q_1 | V   (each 64 rows x 128 B, swizzled;
// K_h / Q_h hold key dims 64h..64h+63).  [K_h; Q_h] is a 128-row K-major
// operand.  The residual X overwrites V in place.
constexpr int kOffQ = 8192;
constexpr int kHalf = 16384;
constexpr int kOffV = 32768;
constexpr int kStage = 40960;
// With separate write keys (the preconditioned variant) a stage also holds
// KW_0 | KW_1 (64 rows x 128 B each, like K_h) and the ring is two deep, in
// the same 120 KB.
constexpr int kOffKW = 40960;
constexpr int kStageKW = 57344;
constexpr int kNSKW = 2;
static_assert(kNSKW * kStageKW <= kNS * kStage, "write-key ring");
constexpr int kSBuf = kNS * kStage;          // bf16 S, 128 x 64, MN-major
constexpr int kTU = kSBuf + 16384;           // 2 x {TU | P}, by chunk parity
constexpr int kTUStride = 16384;             // TU, P: 64 x 64 K-major each
constexpr int kOffP = 8192;
// [TU; P] is one 128-row K-major operand: U~ = TU X reads rows 0..63 (lanes
// 64..127 of its result are never read), P U~ reads rows 64..127 (lanes
// 0..63 of its result are never read).
constexpr int kUtBuf = kTU + 2 * kTUStride;  // U~ bf16, MN-major
constexpr int kUtsBuf = kUtBuf + 8192;       // Diag(Gamma_C) U~ bf16
constexpr int kTileF = 16 * 17;              // fp32 16x16 tile, row stride 17
constexpr int kADiag = kUtsBuf + 8192;       // 4 fp32 diagonal tiles of A
constexpr int kAOff = kADiag + 4 * kTileF * 4;   // 2 x 6 bf16 tiles A_im
constexpr int kAOffStride = 6 * 256 * 2;
constexpr int kTD = kAOff + 2 * kAOffStride; // 2 x 4 fp32 tiles T_ii
constexpr int kTDStride = 4 * kTileF * 4;
constexpr int kTO = kTD + 2 * kTDStride;     // fp32 T_21, T_20 (T team)
constexpr int kT10 = kTO + 2 * kTileF * 4;   // 2 x fp32 T_10 (A team)
constexpr int kYBuf = kT10 + 2 * kTileF * 4; // 2 x {Y_20, Y_21, Y_30, Y_31,
constexpr int kYStride = 5 * 512;            //   Y_32} as mma A fragments
constexpr int kP30 = kYBuf + 2 * kYStride;   // partial sum of T_30 (fp32)
constexpr int kGBuf = kP30 + 32 * 8 * 4;     // 4 x {g2, beta, e, gamma}
constexpr int kGBufStride = 4 * 64;          // floats per buffer
constexpr int kNumGBufs = 4;                 // by chunk index mod 4
constexpr int kBars = kGBuf + kNumGBufs * kGBufStride * 4;
constexpr int kNumBars = 21;
constexpr int kMisc = kBars + 8 * kNumBars;  // abort flag, warp total, TMEM,
                                             // last TMA chunk issued
constexpr int kSmemUsed = kMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kBars % 8 == 0, "mbarrier alignment");
static_assert(kTU % 1024 == 0 && kUtBuf % 1024 == 0 &&
              kUtsBuf % 1024 == 0 && kSBuf % 1024 == 0, "operand alignment");
constexpr uint32_t kTmaBytes = 2 * 16384 + 8192;
constexpr uint32_t kTmaBytesKW = kTmaBytes + 16384;

// mbarrier slots (all with one arrival per phase)
constexpr int kBarTma = 0;       // kNS: stage full (TMA)
constexpr int kBarG = 3;         // 2: G of chunk c done, by c & 1
constexpr int kBarKS = 5;        // [K;Q] S done
constexpr int kBarUT = 6;        // 2: U~ = TU X done (TU free), by c & 1
constexpr int kBarDS = 8;        // dS done
constexpr int kBarOI = 9;        // 2: P U~ done (P free), by c & 1
constexpr int kBarWReady = 11;   // 2: TU, P of chunk c written, by c & 1
constexpr int kBarAReady = 13;   // 4: A team done with chunk c, by c & 3
constexpr int kBarTDone = 17;    // 2: T team done with chunk c, by c & 1
constexpr int kBarPDone = 19;    // 2: P of chunk c built (G free), by c & 1

// ---- TMEM columns -----------------------------------------------------------
// G[c & 1]: lanes 0..63 K K^T, lanes 64..127 Q K^T (free once P is built).
// KS[c & 1]: lanes 0..63 K S, lanes 64..127 Q S.
// UT: lanes 0..63 U~.   DS: dS (lane = key row).   OI: lanes 64..127 P U~.
constexpr uint32_t kColG = 0;      // + 64 (c & 1)
constexpr uint32_t kColKS = 128;   // + 64 (c & 1)
constexpr uint32_t kColUT = 256;
constexpr uint32_t kColDS = 320;
constexpr uint32_t kColOI = 384;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdG = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdN64 = tc::idesc_bf16(128, 64, false, true);
constexpr uint32_t kIdDS = tc::idesc_bf16(128, 64, true, true);

constexpr int kBarATeam = 1;     // named barrier ids
constexpr int kBarTTeam = 2;
constexpr int kBarState = 3;
constexpr int kBarState01 = 4;   // state warps 4, 5
constexpr int kBarState23 = 5;   // state warps 6, 7

constexpr float kLog2e = 1.4426950408889634f;
// Decay spread (log2) within a 16-row tile up to which the factorised form
// 2^(g_r - g_ref) 2^(g_ref - g_i) stays far from fp32 overflow.
constexpr float kMaxTileSpread = 96.f;

struct TcParams {
    const float* log_alpha;
    const float* eta;
    const float* h0;
    __nv_bfloat16* o;      // null in checkpoint mode
    float* hT;
    float* ckpt;           // checkpoint mode: the state at every chunk start
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

// 16 fp32 values times `scale` as 16-byte chunks j, j+1 (8 bf16 each) of a
// 128-byte swizzled bf16 row.
__device__ __forceinline__ void st_chunks_sw128(uint8_t* base, int row, int j,
                                                const float (&x)[16],
                                                float scale) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 v;
        v.x = tc::pack_bf16x2(x[8 * h + 0] * scale, x[8 * h + 1] * scale);
        v.y = tc::pack_bf16x2(x[8 * h + 2] * scale, x[8 * h + 3] * scale);
        v.z = tc::pack_bf16x2(x[8 * h + 4] * scale, x[8 * h + 5] * scale);
        v.w = tc::pack_bf16x2(x[8 * h + 6] * scale, x[8 * h + 7] * scale);
        *reinterpret_cast<uint4*>(base + row * 128 +
                                  (((j + h) ^ (row & 7)) << 4)) = v;
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

// Every thread of a group waits on the mbarrier, then the group agrees on
// the outcome (true = all saw the phase complete).  On failure the CTA-wide
// abort flag is raised so that the other groups stop too.
__device__ __forceinline__ bool team_wait(uint64_t* bar, uint32_t parity,
                                          int* abort_flag, int bar_id,
                                          int nthreads, bool ok = true) {
    ok = ok && tc::mbar_wait_or_abort(bar, parity, abort_flag);
    const bool any_fail = tc::named_bar_or(bar_id, nthreads, !ok);
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
// operand TU = T Diag(beta) (64 x 64, K-major, swizzled rows).
__device__ __forceinline__ void store_tu_tile(float* tf, uint8_t* tu,
                                              const float* beta, int I, int J,
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
        const float b0 = beta[col], b1 = beta[col + 1];
        const int r0 = 16 * I + g, r1 = r0 + 8;
        *reinterpret_cast<uint32_t*>(tu + sw_off(r0, col)) =
            tc::pack_bf16x2(t00 * b0, t01 * b1);
        *reinterpret_cast<uint32_t*>(tu + sw_off(r1, col)) =
            tc::pack_bf16x2(t10 * b0, t11 * b1);
    }
}

__device__ __forceinline__ void zero_acc(float (&acc)[2][4]) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[nt][k] = 0.f;
}

// Y = T_II A_Im as a bf16 A fragment (T_II fp32, A_Im bf16).
__device__ __forceinline__ void y_frag(const uint32_t (&ta)[4],
                                       const __nv_bfloat16* aim, int g, int q,
                                       uint32_t (&y)[4]) {
    float acc[2][4];
    zero_acc(acc);
    mm_tile_bf16(acc, ta, aim, g, q);
    y[0] = tc::pack_bf16x2(acc[0][0], acc[0][1]);
    y[1] = tc::pack_bf16x2(acc[0][2], acc[0][3]);
    y[2] = tc::pack_bf16x2(acc[1][0], acc[1][1]);
    y[3] = tc::pack_bf16x2(acc[1][2], acc[1][3]);
}

// Diagonal tiles T_ii = A_ii^{-1} (A_ii unit lower triangular, fp32 column
// substitution): thread (bb = t / 16, cl = t % 16) of the A team computes
// column cl of T_bb, kept in fp32 (Td) and written to the bf16 operand
// TU = T Diag(beta) (zero upper half included).  Ad: strictly lower parts of
// A_ii (row stride 17).
__device__ __forceinline__ void invert_diag_tiles(const float* Ad, float* Td,
                                                  uint8_t* tu,
                                                  const float* beta, int t) {
    const int bb = t >> 4, cl = t & 15;
    const float* Ab = Ad + bb * kTileF;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) x[r] = (r == cl) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 16; ++r) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < r; i += 2) {
            a0 = fmaf(Ab[r * 17 + i], x[i], a0);
            if (i + 1 < r) a1 = fmaf(Ab[r * 17 + i + 1], x[i + 1], a1);
        }
        if (r > cl) x[r] = -(a0 + a1);
    }
    float* Tb = Td + bb * kTileF + cl;
    const int col = 16 * bb + cl;
    const float bc = beta[col];
    __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(tu);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        Tb[r * 17] = x[r];
        d[sw_off(16 * bb + r, col) >> 1] = __float2bfloat16_rn(x[r] * bc);
    }
}

// A team, after the diagonal inverses: warp 0 forms T_10 = -T_11 A_10 T_00
// (kept in fp32 for the T team, and written to TU) and Y_20, Y_21; warp 1
// forms Y_30, Y_31, Y_32 (Y_Im = T_II A_Im, left as mma A fragments in Yb,
// per lane, in the order Y_20, Y_21, Y_30, Y_31, Y_32).
__device__ __forceinline__ void a_team_products(const __nv_bfloat16* Ao,
                                                const float* Td, float* T10,
                                                uint4* Yb, uint8_t* tu,
                                                const float* beta, int warp,
                                                int lane) {
    const int g = lane >> 2, q = lane & 3;
    uint32_t ta[4], y[4];
    if (warp == 0) {
        afrag_f32(Td + kTileF, g, q, ta);
        y_frag(ta, Ao + 0 * 256, g, q, y);
        float acc[2][4];
        zero_acc(acc);
        mm_tile_f32(acc, y, Td, g, q);
        store_tu_tile(T10, tu, beta, 1, 0, acc, g, q);
        afrag_f32(Td + 2 * kTileF, g, q, ta);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            y_frag(ta, Ao + (1 + k) * 256, g, q, y);
            Yb[k * 32 + lane] = make_uint4(y[0], y[1], y[2], y[3]);
        }
    } else {
        afrag_f32(Td + 3 * kTileF, g, q, ta);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            y_frag(ta, Ao + (3 + k) * 256, g, q, y);
            Yb[(2 + k) * 32 + lane] = make_uint4(y[0], y[1], y[2], y[3]);
        }
    }
}

// T team: the remaining off-diagonal tiles of T = A^{-1},
//   T_Ij = -sum_{m=j}^{I-1} Y_Im T_mj,
// warp 2: T_21, T_20 and the part Y_30 T_00 + Y_31 T_10 of T_30; warp 3:
// T_32, T_31, T_30.  What warp 3 needs from warp 2 (T_21; T_20 and the part
// of T_30) is handed over through two team barriers.  Td: fp32 T_ii; T10:
// fp32 T_10; To: fp32 T_21 | T_20; P30: the T_30 part, fragment layout.
__device__ __forceinline__ void t_team_offdiag(const uint4* Yb,
                                               const float* Td,
                                               const float* T10, float* To,
                                               float* P30, uint8_t* tu,
                                               const float* beta, int warp,
                                               int lane) {
    const int g = lane >> 2, q = lane & 3;
    const float* T00 = Td;
    const float* T11 = Td + kTileF;
    const float* T22 = Td + 2 * kTileF;
    float* T21 = To;
    float* T20 = To + kTileF;
    auto ld_y = [&](int k, uint32_t (&y)[4]) {
        const uint4 v = Yb[k * 32 + lane];
        y[0] = v.x; y[1] = v.y; y[2] = v.z; y[3] = v.w;
    };
    float acc[2][4];
    if (warp == 2) {
        uint32_t y20[4], y21[4], y30[4], y31[4];
        ld_y(0, y20); ld_y(1, y21); ld_y(2, y30); ld_y(3, y31);
        zero_acc(acc);
        mm_tile_f32(acc, y21, T11, g, q);
        store_tu_tile(T21, tu, beta, 2, 1, acc, g, q);
        tc::named_bar_sync(kBarTTeam, 64);          // T_21 out
        zero_acc(acc);
        mm_tile_f32(acc, y20, T00, g, q);
        mm_tile_f32(acc, y21, T10, g, q);
        store_tu_tile(T20, tu, beta, 2, 0, acc, g, q);
        zero_acc(acc);
        mm_tile_f32(acc, y30, T00, g, q);
        mm_tile_f32(acc, y31, T10, g, q);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) P30[(nt * 4 + k) * 32 + lane] = acc[nt][k];
        tc::named_bar_sync(kBarTTeam, 64);          // T_20, T_30 part out
    } else {
        uint32_t y31[4], y32[4];
        ld_y(3, y31); ld_y(4, y32);
        zero_acc(acc);
        mm_tile_f32(acc, y32, T22, g, q);
        store_tu_tile(nullptr, tu, beta, 3, 2, acc, g, q);
        zero_acc(acc);
        mm_tile_f32(acc, y31, T11, g, q);
        tc::named_bar_sync(kBarTTeam, 64);          // T_21 in
        mm_tile_f32(acc, y32, T21, g, q);
        store_tu_tile(nullptr, tu, beta, 3, 1, acc, g, q);
        tc::named_bar_sync(kBarTTeam, 64);          // T_20, T_30 part in
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[nt][k] = P30[(nt * 4 + k) * 32 + lane];
        mm_tile_f32(acc, y32, T20, g, q);
        store_tu_tile(nullptr, tu, beta, 3, 0, acc, g, q);
    }
}

__device__ __forceinline__ uint32_t col_g(int c) { return kColG + 64 * (c & 1); }
__device__ __forceinline__ uint32_t col_ks(int c) { return kColKS + 64 * (c & 1); }

__device__ __forceinline__ void unpack_bf16x2(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
}

// kCkpt: write the state at every chunk start (p.ckpt) instead of o.
// kKW: separate write keys (tm_kw): G = [K;Q] Kw^T (so beta's denominator is
// k . kw, A uses K Kw^T and P uses Q Kw^T) and dS = Kw^T Diag(Gamma_C) U~;
// the residual still reads K S.  The modes are separate instantiations so
// that none carries another's code.
template <bool kCkpt, bool kKW>
__global__ void __launch_bounds__(kThreads, 1)
kla_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_kw, TcParams p) {
    constexpr int NS = kKW ? kNSKW : kNS;            // ring depth
    constexpr int STAGE = kKW ? kStageKW : kStage;   // bytes per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_u32(sm);
    float* gbuf = reinterpret_cast<float*>(sm + kGBuf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
    int* abort_flag = reinterpret_cast<int*>(sm + kMisc);
    float* wtot = reinterpret_cast<float*>(sm + kMisc + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc + 8);
    int* tma_issued = reinterpret_cast<int*>(sm + kMisc + 12);

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
        if constexpr (kKW) tc::prefetch_tmap(&tm_kw);
        for (int i = 0; i < kNumBars; ++i) tc::mbar_init(&bars[i], 1);
        *abort_flag = 0;
        *tma_issued = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    // both TU buffers start all zero; per chunk only their lower 16x16 tiles
    // change
    for (int i = tid; i < 1024; i += kThreads)
        *reinterpret_cast<uint4*>(sm + kTU + (i >> 9) * kTUStride +
                                  16 * (i & 511)) = make_uint4(0, 0, 0, 0);

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
        const int s = c % NS;
        uint8_t* st = sm + s * STAGE;
        const int t0 = c * kC;
        uint64_t* bar = &bars[kBarTma + s];
        tc::mbar_arrive_expect_tx(bar, kKW ? kTmaBytesKW : kTmaBytes);
        if constexpr (kKW) {
            tc::tma_load_4d(st + kOffKW, &tm_kw, bar, 0, h, t0, b);
            tc::tma_load_4d(st + kOffKW + 8192, &tm_kw, bar, 64, h, t0, b);
        }
        tc::tma_load_4d(st, &tm_k, bar, 0, h, t0, b);
        tc::tma_load_4d(st + kOffQ, &tm_q, bar, 0, h, t0, b);
        tc::tma_load_4d(st + kHalf, &tm_k, bar, 64, h, t0, b);
        tc::tma_load_4d(st + kHalf + kOffQ, &tm_q, bar, 64, h, t0, b);
        tc::tma_load_4d(st + kOffV, &tm_v, bar, j0, h, t0, b);
    };
    // L2 prefetch of chunk c's tiles, so that its ring load later hits L2
    auto prefetch_l2 = [&](int c) {
        const int t0 = c * kC;
        tc::tma_prefetch_4d(&tm_k, 0, h, t0, b);
        tc::tma_prefetch_4d(&tm_q, 0, h, t0, b);
        tc::tma_prefetch_4d(&tm_k, 64, h, t0, b);
        tc::tma_prefetch_4d(&tm_q, 64, h, t0, b);
        tc::tma_prefetch_4d(&tm_v, j0, h, t0, b);
        if constexpr (kKW) {
            tc::tma_prefetch_4d(&tm_kw, 0, h, t0, b);
            tc::tma_prefetch_4d(&tm_kw, 64, h, t0, b);
        }
    };
    // G = [K; Q] K^T (or [K; Q] Kw^T) of chunk c into G[c & 1]
    auto issue_g = [&](int c) {
        const uint32_t sst = sbase + (c % NS) * STAGE;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
            const uint32_t offb =
                kKW ? kOffKW + (ks >> 2) * 8192 + (ks & 3) * 32 : off;
            tc::mma_bf16(tmem + col_g(c), desc_k(sst + off),
                         desc_k(sst + offb), kIdG, ks > 0);
        }
        tc::mma_commit(&bars[kBarG + (c & 1)]);
    };
    if (tid == 0) {
        for (int c = 0; c < NS && c < nchunks; ++c) issue_tma(c);
        *tma_issued = nchunks < NS ? nchunks : NS;
        for (int c = NS; c < NS + kPrefetch && c < nchunks; ++c)
            prefetch_l2(c);
    }

    if (tid < 64) {
        // =========================================================== A team
        const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
        bool failed = false;
        int g_last_c = -1;   // last chunk whose G this thread issued
        auto load_gates = [&](int c, float& la, float& et) {
            const int t = c * kC + tid;
            la = 0.f;
            et = 0.f;
            if (t < T) {
                const size_t off = ((size_t)b * T + t) * p.H + h;
                la = p.log_alpha[off];
                et = p.eta[off];
            }
        };
        // G of chunks 0 and 1; the state side issues G(c + 2) once chunk c
        // has built P (the last read of that G buffer)
        for (int c = 0; c < 2 && c < nchunks && !failed; ++c) {
            if (team_wait(&bars[kBarTma + c], 0, abort_flag, kBarATeam, 64)) {
                tc::tc_fence_after();
                if (tid == 0) issue_g(c);
                g_last_c = c;
            } else {
                failed = true;
            }
        }
        float la_cur, eta_cur;
        load_gates(0, la_cur, eta_cur);
        for (int c = 0; c < nchunks && !failed; ++c) {
            float la_nxt, eta_nxt;
            load_gates(c + 1, la_nxt, eta_nxt);
            // gate buffer c & 3: chunk c-4 is finished on every side (the
            // T team finished chunk c-2, which needed U~ of chunk c-3)
            float* gb = gbuf + (c & 3) * kGBufStride;    // g2|beta|e|gamma
            float* Ad = reinterpret_cast<float*>(sm + kADiag);
            __nv_bfloat16* Ao =
                reinterpret_cast<__nv_bfloat16*>(sm + kAOff + (c & 1) * kAOffStride);
            float* Td = reinterpret_cast<float*>(sm + kTD + (c & 1) * kTDStride);
            uint8_t* tu = sm + kTU + (c & 1) * kTUStride;
            float* T10 = reinterpret_cast<float*>(sm + kT10 + (c & 1) * kTileF * 4);
            uint4* Yb = reinterpret_cast<uint4*>(sm + kYBuf + (c & 1) * kYStride);

            // cumulative log2-decay: warp scans on rows 0..31 and 32..63
            float g2 = la_cur * kLog2e;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, g2, off);
                if ((tid & 31) >= off) g2 += y;
            }
            if (tid == 31) *wtot = g2;
            // buffers of chunk c-2 must have been consumed: A_im, T_ii, Y by
            // the T team; TU, P by U~ = TU X and P U~
            bool ok = true;
            if (c >= 2) {
                const uint32_t ph = ((c - 2) >> 1) & 1;
                ok = tc::mbar_wait_or_abort(&bars[kBarTDone + (c & 1)], ph,
                                            abort_flag) &&
                     tc::mbar_wait_or_abort(&bars[kBarUT + (c & 1)], ph,
                                            abort_flag) &&
                     tc::mbar_wait_or_abort(&bars[kBarOI + (c & 1)], ph,
                                            abort_flag);
            }
            if (!team_wait(&bars[kBarG + (c & 1)], (c >> 1) & 1, abort_flag,
                           kBarATeam, 64, ok)) {
                failed = true; break;
            }
            tc::tc_fence_after();
            // K K^T row tid, columns of this warp's own 32 rows: the diagonal
            float xd[32];
            tc::tmem_ld32(tlane + col_g(c) + 32 * warp, xd);
            tc::tmem_ld_wait();
            if (tid >= 32) g2 += *wtot;
            // xd[lane] by halving on the lane bits (stays in registers)
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j)
                    xd[j] = (tid & w) ? xd[j + w] : xd[j];
            const float diag = xd[0];
            const float denom = diag + p.eps;
            const float beta =
                p.gdn ? eta_cur : (denom == 0.f ? 0.f : eta_cur / denom);
            // e_i = 2^(g_ref - g_i), g_ref = g at the last column of i's
            // 16-column tile: Gamma_ri = 2^(g_r - g_ref) e_i
            const float gref = __shfl_sync(0xffffffffu, g2, (tid & 16) | 15);
            gb[tid] = g2;
            gb[kC + tid] = beta;
            gb[2 * kC + tid] = tc::ex2(gref - g2);
            gb[3 * kC + tid] = tc::ex2(g2);
            tc::named_bar_sync(kBarATeam, 64);

            // ---- A: row r = tid, tiles m <= r / 16 (a rolled loop, each
            // tile reloaded from TMEM); the diagonal tile in fp32 (Ad), those
            // below it in bf16 (Ao)
            {
                const int r = tid, ti = r >> 4, rr = r & 15;
                const int mmax = warp == 0 ? 1 : 3;
#pragma unroll 1
                for (int m = 0; m <= mmax; ++m) {
                    float xm[16];
                    tc::tmem_ld16(tlane + col_g(c) + 16 * m, xm);
                    const float gref_m = gb[16 * m + 15];
                    const bool fact =
                        m < ti || fabsf(gb[16 * m] - gref_m) <= kMaxTileSpread;
                    const float bm = beta * tc::ex2(g2 - gref_m);
                    tc::tmem_ld_wait();
                    float v[16];
                    if (fact) {
                        const float* e = gb + 2 * kC + 16 * m;
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc)
                            v[cc] = (16 * m + cc < r) ? bm * e[cc] * xm[cc] : 0.f;
                    } else {   // wide decay spread inside the tile
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) {
                            const int i = 16 * m + cc;
                            v[cc] = (i < r) ? beta * tc::ex2(g2 - gb[i]) * xm[cc]
                                            : 0.f;
                        }
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
            }
            tc::tc_fence_before();   // K K^T reads done before G is reused
            // G of chunk c+1 into G[(c+1) & 1], once chunk c-1 has built P
            // from it and chunk c+1's tiles have landed (chunks 0 and 1 are
            // issued before the loop)
            if (tid == 0 && c >= 1 && c + 1 < nchunks) {
                const bool gok =
                    tc::mbar_wait_or_abort(&bars[kBarPDone + ((c + 1) & 1)],
                                           ((c - 1) >> 1) & 1, abort_flag) &&
                    tc::mbar_wait_or_abort(&bars[kBarTma + (c + 1) % NS],
                                           ((c + 1) / NS) & 1, abort_flag);
                if (gok) {
                    tc::tc_fence_after();
                    issue_g(c + 1);
                    g_last_c = c + 1;
                } else {
                    *reinterpret_cast<volatile int*>(abort_flag) = 1;
                }
            }
            __syncwarp();
            invert_diag_tiles(Ad, Td, tu, gb + kC, tid);   // warp w: 2w, 2w+1
            tc::named_bar_sync(kBarATeam, 64);             // all T_ii in place
            a_team_products(Ao, Td, T10, Yb, tu, gb + kC, warp, tid & 31);
            tc::fence_proxy_async_smem();                  // TU tiles written
            tc::named_bar_sync(kBarATeam, 64);
            if (tid == 0) tc::mbar_arrive(&bars[kBarAReady + (c & 3)]);
            la_cur = la_nxt;
            eta_cur = eta_nxt;
        }
        if (failed && tid == 0 && g_last_c >= 0)   // drain (bounded)
            tc::mbar_wait(&bars[kBarG + (g_last_c & 1)], (g_last_c >> 1) & 1,
                          100000000ull);
    } else if (tid < 128) {
        // =========================================================== T team
        const int t = tid - 64;
        const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c = 0; c < nchunks; ++c) {
            // the A team waited for the release of this chunk's TU and P
            // buffers before handing the chunk over
            bool ok = tc::mbar_wait_or_abort(&bars[kBarG + (c & 1)],
                                             (c >> 1) & 1, abort_flag);
            if (!team_wait(&bars[kBarAReady + (c & 3)], (c >> 2) & 1,
                           abort_flag, kBarTTeam, 64, ok))
                break;
            tc::tc_fence_after();
            const float* gb = gbuf + (c & 3) * kGBufStride;
            uint8_t* tu = sm + kTU + (c & 1) * kTUStride;
            {   // ---- P row t = Gamma o Q K^T, lower incl. (lanes 64..127)
                const int r = t;
                const float gr = gb[r];
                uint8_t* prow = tu + kOffP + r * 128;
                const int jmax = (r >> 3) + 1;   // 8-column groups needed
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (__any_sync(0xffffffffu, j < jmax)) {
                        float x[8];
                        tc::tmem_ld8(tlane + col_g(c) + 8 * j, x);
                        const float4 g0 =
                            *reinterpret_cast<const float4*>(gb + 8 * j);
                        const float4 g1 =
                            *reinterpret_cast<const float4*>(gb + 8 * j + 4);
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
            tc::tc_fence_before();
            tc::named_bar_sync(kBarTTeam, 64);   // Q K^T of G[c & 1] read
            if (t == 0) tc::mbar_arrive(&bars[kBarPDone + (c & 1)]);
            const float* Td =
                reinterpret_cast<const float*>(sm + kTD + (c & 1) * kTDStride);
            const float* T10 =
                reinterpret_cast<const float*>(sm + kT10 + (c & 1) * kTileF * 4);
            const uint4* Yb =
                reinterpret_cast<const uint4*>(sm + kYBuf + (c & 1) * kYStride);
            t_team_offdiag(Yb, Td, T10, reinterpret_cast<float*>(sm + kTO),
                           reinterpret_cast<float*>(sm + kP30), tu, gb + kC,
                           warp, tid & 31);
            tc::fence_proxy_async_smem();
            tc::named_bar_sync(kBarTTeam, 64);
            if (t == 0) {
                tc::mbar_arrive(&bars[kBarWReady + (c & 1)]);
                tc::mbar_arrive(&bars[kBarTDone + (c & 1)]);
            }
        }
    } else {
        // ==================================================== state warpgroup
        const int sw = warp - 4;                 // TMEM lane quarter
        const uint32_t tlane = tmem + ((uint32_t)(sw * 32) << 16);
        const int row = tid - 128;               // TMEM lane
        bool failed = false;
        int last_bar = -1;                       // last commit of this thread
        uint32_t last_par = 0;
        // o of chunk cc = gamma Q S + P U~ (warps 6, 7: lanes 64..127)
        auto write_o = [&](int cc) {
            if constexpr (kCkpt) return;   // only the states are wanted
            const int r = row - kC;
            const float gam = gbuf[(cc & 3) * kGBufStride + 3 * kC + r];
            const int t = cc * kC + r;
            __nv_bfloat16* dst = p.o + (((size_t)b * T + t) * p.H + h) * kD + j0;
            const bool store = t < T;
#pragma unroll 1
            for (int jj = 0; jj < 4; ++jj) {   // 16 columns a step
                float qs[16], x[16];
                tc::tmem_ld16(tlane + col_ks(cc) + 16 * jj, qs);
                tc::tmem_ld16(tlane + kColOI + 16 * jj, x);
                tc::tmem_ld_wait();
                if (!store) continue;
#pragma unroll
                for (int j = 0; j < 16; j += 8) {
                    uint4 v;
                    v.x = tc::pack_bf16x2(fmaf(gam, qs[j + 0], x[j + 0]),
                                          fmaf(gam, qs[j + 1], x[j + 1]));
                    v.y = tc::pack_bf16x2(fmaf(gam, qs[j + 2], x[j + 2]),
                                          fmaf(gam, qs[j + 3], x[j + 3]));
                    v.z = tc::pack_bf16x2(fmaf(gam, qs[j + 4], x[j + 4]),
                                          fmaf(gam, qs[j + 5], x[j + 5]));
                    v.w = tc::pack_bf16x2(fmaf(gam, qs[j + 6], x[j + 6]),
                                          fmaf(gam, qs[j + 7], x[j + 7]));
                    *reinterpret_cast<uint4*>(dst + 16 * jj + j) = v;
                }
            }
        };
        for (int c = 0; c < nchunks && !failed; ++c) {
            const int s = c % NS;
            const uint32_t sst = sbase + s * STAGE;
            const float* gb = gbuf + (c & 3) * kGBufStride;
            const uint32_t tu = sbase + kTU + (c & 1) * kTUStride;
            if constexpr (kCkpt) {   // the state chunk c starts from (fp32)
                float* dst = p.ckpt + (((size_t)bh * nchunks + c) * kD + row) *
                                          kD + j0;
#pragma unroll
                for (int j = 0; j < kNV; j += 4)
                    *reinterpret_cast<float4*>(dst + j) =
                        make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
            }
            bool ok = true;
            if (sw < 2)   // the stage of chunk c (warps 6, 7 do not read it)
                ok = team_wait(&bars[kBarTma + s], (c / NS) & 1, abort_flag,
                               kBarState01, 64);
            tc::tc_fence_after();
            if (ok && tid == 128) {   // [K; Q] S: K S lanes 0..63, Q S 64..127
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(tmem + col_ks(c),
                                 desc_k(sst + (ks >> 2) * kHalf + (ks & 3) * 32),
                                 desc_mn(sbase + kSBuf + ks * 2048, 0), kIdN64,
                                 ks > 0);
                tc::mma_commit(&bars[kBarKS]);
                last_bar = kBarKS; last_par = c & 1;
            }
            __syncwarp();   // the issuing lane rejoins before the waits
            if (sw < 2) {
                // ---- residual X = V - Diag(gamma) K S, over V in the stage
                ok = ok && tc::mbar_wait_or_abort(&bars[kBarAReady + (c & 3)],
                                                  (c >> 2) & 1, abort_flag);
                ok = team_wait(&bars[kBarKS], c & 1, abort_flag, kBarState01,
                               64, ok);
                if (ok) {
                    tc::tc_fence_after();
                    const float gam = gb[3 * kC + row];
                    uint8_t* vrow = sm + s * STAGE + kOffV + row * 128;
#pragma unroll 1
                    for (int jj = 0; jj < 4; ++jj) {   // 16 columns a step
                        float x[16];
                        tc::tmem_ld16(tlane + col_ks(c) + 16 * jj, x);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint4* pv = reinterpret_cast<uint4*>(
                                vrow + (((2 * jj + h) ^ (row & 7)) << 4));
                            uint4 u = *pv;
                            const float* xh = x + 8 * h;
                            float v0, v1;
                            unpack_bf16x2(u.x, v0, v1);
                            u.x = tc::pack_bf16x2(fmaf(-gam, xh[0], v0),
                                                  fmaf(-gam, xh[1], v1));
                            unpack_bf16x2(u.y, v0, v1);
                            u.y = tc::pack_bf16x2(fmaf(-gam, xh[2], v0),
                                                  fmaf(-gam, xh[3], v1));
                            unpack_bf16x2(u.z, v0, v1);
                            u.z = tc::pack_bf16x2(fmaf(-gam, xh[4], v0),
                                                  fmaf(-gam, xh[5], v1));
                            unpack_bf16x2(u.w, v0, v1);
                            u.w = tc::pack_bf16x2(fmaf(-gam, xh[6], v0),
                                                  fmaf(-gam, xh[7], v1));
                            *pv = u;
                        }
                    }
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_before();
                }
                // TU of chunk c written by the T team
                ok = team_wait(&bars[kBarWReady + (c & 1)], (c >> 1) & 1,
                               abort_flag, kBarState01, 64, ok);
                if (ok && tid == 128) {   // U~ = TU X
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_bf16(tmem + kColUT, desc_k(tu + ks * 32),
                                     desc_mn(sst + kOffV + ks * 2048, 0),
                                     kIdN64, ks > 0);
                    tc::mma_commit(&bars[kBarUT + (c & 1)]);
                    last_bar = kBarUT + (c & 1); last_par = (c >> 1) & 1;
                }
                __syncwarp();
                ok = team_wait(&bars[kBarUT + (c & 1)], (c >> 1) & 1,
                               abort_flag, kBarState01, 64, ok);
                if (ok) {   // rows 0..63: U~ and Diag(Gamma_C) U~ as operands
                    tc::tc_fence_after();
                    const float dec = tc::ex2(gb[kC - 1] - gb[row]);
#pragma unroll 1
                    for (int jj = 0; jj < 4; ++jj) {   // 16 columns a step
                        float u[16];
                        tc::tmem_ld16(tlane + kColUT + 16 * jj, u);
                        tc::tmem_ld_wait();
                        st_chunks_sw128(sm + kUtBuf, row, 2 * jj, u, 1.f);
                        st_chunks_sw128(sm + kUtsBuf, row, 2 * jj, u, dec);
                    }
                    tc::fence_proxy_async_smem();
                }
            } else if (c >= 1) {
                // ---- o of the previous chunk (its P U~ was issued last)
                ok = team_wait(&bars[kBarOI + ((c - 1) & 1)],
                               ((c - 1) >> 1) & 1, abort_flag, kBarState23, 64);
                if (ok) {
                    tc::tc_fence_after();
                    write_o(c - 1);
                }
            }
            tc::tc_fence_before();
            if (tc::named_bar_or(kBarState, 128, !ok)) {
                *reinterpret_cast<volatile int*>(abort_flag) = 1;
                failed = true; break;
            }
            tc::tc_fence_after();
            if (tid == 128) {   // dS = K^T Diag(Gamma_C) U~, then P U~
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + kColDS,
                                 kKW ? desc_mn(sst + kOffKW + ks * 2048, 8192)
                                     : desc_mn(sst + ks * 2048, kHalf),
                                 desc_mn(sbase + kUtsBuf + ks * 2048, 0), kIdDS,
                                 ks > 0);
                tc::mma_commit(&bars[kBarDS]);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + kColOI, desc_k(tu + ks * 32),
                                 desc_mn(sbase + kUtBuf + ks * 2048, 0), kIdN64,
                                 ks > 0);
                tc::mma_commit(&bars[kBarOI + (c & 1)]);
                last_bar = kBarOI + (c & 1); last_par = (c >> 1) & 1;
            }
            __syncwarp();
            if (!team_wait(&bars[kBarDS], c & 1, abort_flag, kBarState, 128)) {
                failed = true; break;
            }
            tc::tc_fence_after();
            {   // S <- gamma_C S + dS (row = key dim)
                float x[kNV];
                const float gC = gb[3 * kC + kC - 1];
                tmem_ld64(tlane + kColDS, x);
#pragma unroll
                for (int j = 0; j < kNV; ++j) S[j] = fmaf(gC, S[j], x[j]);
                st_row_sw128(sm + kSBuf, row, S);
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::named_bar_sync(kBarState, 128);
            if (tid == 224 && c + NS < nchunks) {
                issue_tma(c + NS);
                *reinterpret_cast<volatile int*>(tma_issued) = c + NS + 1;
                if (c + NS + kPrefetch < nchunks)
                    prefetch_l2(c + NS + kPrefetch);
            }
        }
        if (!failed && sw >= 2 && nchunks > 0) {   // o of the last chunk
            const int cl = nchunks - 1;
            if (team_wait(&bars[kBarOI + (cl & 1)], (cl >> 1) & 1, abort_flag,
                          kBarState23, 64)) {
                tc::tc_fence_after();
                write_o(cl);
            }
        }
        // let this thread's MMAs finish before TMEM and shared memory go
        if (failed && last_bar >= 0)
            tc::mbar_wait(&bars[last_bar], last_par, 100000000ull);
    }

    __syncthreads();
    const bool any_failed = *reinterpret_cast<volatile int*>(abort_flag) != 0;
    if (any_failed) {
        if (tid == 0) {
            atomicOr(&g_fault_word, 1u);
            // copies possibly in flight: the last NS chunks issued
            const int n = *reinterpret_cast<volatile int*>(tma_issued);
            for (int c = n - NS < 0 ? 0 : n - NS; c < n; ++c)
                tc::mbar_wait(&bars[kBarTma + c % NS], (c / NS) & 1,
                              100000000ull);
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

}  // namespace

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

namespace {

bool aligned16(const void* ptr) {
    return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
}

}  // namespace

bool chunk_tc_eligible(const FwdArgs& a) {
    return a.dtype == KLA_BF16 && a.dk == kD && a.dv == kD && a.C == kC &&
           aligned16(a.q) && aligned16(a.k) && aligned16(a.v) &&
           aligned16(a.o) && (!a.h0 || aligned16(a.h0)) &&
           (!a.hT || aligned16(a.hT)) && aligned16(a.kw) && get_encoder();
}

cudaError_t launch_chunk_tc(const FwdArgs& a, cudaStream_t stream) {
    if ((long)a.B * a.H == 0 || a.T == 0) return cudaSuccess;
    if (!get_encoder()) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv, mkw;
    if (!make_map(&mq, a.q, a.B, a.T, a.H) ||
        !make_map(&mk, a.k, a.B, a.T, a.H) ||
        !(a.v_zero ? make_map(&mv, a.v, 1, kC, a.H)
                   : make_map(&mv, a.v, a.B, a.T, a.H)) ||
        !make_map(&mkw, a.kw ? a.kw : a.k, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    // exactly one of o (the forward) and ckpt (the backward's checkpoints);
    // write keys only in the forward
    if ((a.o == nullptr) == (a.ckpt == nullptr)) return cudaErrorInvalidValue;
    if (a.kw && a.ckpt) return cudaErrorInvalidValue;
    const int mode = a.ckpt ? 1 : a.kw ? 2 : 0;
    auto kern = mode == 1   ? kla_chunk_tc_kernel<true, false>
                : mode == 2 ? kla_chunk_tc_kernel<false, true>
                            : kla_chunk_tc_kernel<false, false>;
    // the shared-memory opt-in, once per (instantiation, device)
    static std::atomic<unsigned long long> attr_done[3];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (!bit || !(attr_done[mode].load() & bit)) {
        e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[mode].fetch_or(bit);
    }
    TcParams p{a.log_alpha, a.eta, a.h0,
               static_cast<__nv_bfloat16*>(a.o), a.hT, a.ckpt, a.eps, a.gdn,
               a.T, a.H};
    dim3 grid((unsigned)((long)a.B * a.H), kD / kNV);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mkw, p);
    return cudaGetLastError();
}

cudaError_t read_and_clear_fault(cudaStream_t stream, unsigned int* word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_fault_word, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    unsigned int w2 = 0;
    e = read_and_clear_fault2(&w2);
    *word |= w2;
    return e;
}

}  // namespace kla
