// Two-kernel tensor-core forward pass for bf16 q/k/v/o, dk = dv = 128,
// chunk C = 64, fp32 state: a chunk-parallel pre-pass and a sequential
// state pass.
//
// Per (batch, head) and chunk (rows r, i; g = in-chunk cumulative log decay,
// gamma_r = exp(g_r), Gamma_ri = exp(g_r - g_i), Gamma_C,r = exp(g_C - g_r)),
// the gated-DeltaNet block solver with B = Diag(beta) as the only change
// (gist.science/es/paper/2605.08587, section "Implementacion"):
//   beta_r = eta_r / (||k_r||^2 + eps)
//   A   = I + strict_lower(Diag(beta) (Gamma o K K^T)),   T = A^{-1}
//   TU  = T Diag(beta),     P = lower_incl(Gamma o Q K^T),   PTU = P TU
//   W   = TU Diag(gamma) K,           U = TU V
//   Q'  = Diag(gamma) Q - PTU Diag(gamma) K
//   U~  = U - W S                     (the new values of the chunk)
//   O   = Diag(gamma) Q S + P U~ = Q' S + PTU V
//   S  <- gamma_C S + K^T Diag(Gamma_C) U~
// Only the last three lines involve the state; everything else depends on
// the chunk's own inputs.
//
// Pre-pass (kla_prep_kernel): a persistent grid whose CTAs take
// chunk-heads in chunk-major order, all independent.  G = [K; Q] K^T on the
// tensor cores (tcgen05, TMEM accumulator); beta from its diagonal; A in
// fp32 and P in bf16; T = A^{-1} by blocks (fp32 substitution on the 16x16
// diagonal blocks, tf32 warp-level MMAs for the rest); PTU = P TU on the
// tensor cores; TU and PTU written to global memory (one bulk copy) as the
// exact shared-memory image of a 128-row K-major bf16 tensor-core operand
// [TU; PTU], followed by g, and the record's ready flag raised.  Past a
// release point only the CTAs of a few reserved TPCs keep working, so that
// the state pass, launched as a programmatic dependent, runs on the other
// SMs beside the pre-pass's last chunks and reads each record once its flag
// is up.
//
// With separate write keys Kw (the preconditioned variant) G = [K; Q] Kw^T
// (so beta's denominator is k . kw, A uses K Kw^T and P uses Q Kw^T) and the
// state takes Kw^T Diag(Gamma_C) U~; W, Q' and the residual keep K.
//
// State pass (kla_state_kernel): one CTA per (batch, head, 64 columns of
// dv), walking the chunks in order.  Two helper warpgroups prepare the next
// chunks (in turns) while the chain warpgroup runs chunk c:
//   helper: K_gamma = Diag(gamma) K (in place of K); [-W; -PTU K_gamma] =
//           -[TU; PTU] K_gamma and [U; PTU V] = [TU; PTU] V on the tensor
//           cores; -W and Q' written over K_gamma and Q in the stage,
//           Diag(Gamma_C) K over TU and PTU;
//   chain:  [U~; O] = [U; PTU V] + [-W; Q'] S   (one MMA group of 8),
//           U~ to shared memory, dS = (Diag(Gamma_C) K)^T U~  (4 MMAs),
//           S <- gamma_C S + dS in registers (fp32, one key row per thread),
//           o from the lower half of the first accumulator, written through
//           shared memory by a TMA store.
// So only two dependent tensor-core round trips remain per chunk.
//
// Every wait on an mbarrier is bounded; a CTA that gives up raises its abort
// flag, records the fault in the library's fault word, lets its own copies
// and MMAs finish (bounded), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "kla_internal.cuh"
#include "tc_primitives.cuh"

namespace kla {

namespace {

__device__ unsigned int g_fault_word2 = 0;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr float kLog2e = 1.4426950408889634f;

// Record of one chunk-head written by the pre-pass (bytes): the 128-row
// K-major operand [TU; PTU] (128-byte swizzled rows) and g (log2 units).
constexpr int kRecTU = 0;
constexpr int kRecPTU = 8192;
constexpr int kRecG = 16384;
constexpr int kRecBytes = 16640;

// Byte offset of element (row, col) of a 64-column bf16 tile stored as
// 128-byte swizzled rows (the layout TMA writes with 128-byte swizzle and the
// tensor cores read from a 1024-byte-aligned base).
__host__ __device__ constexpr int swz(int row, int col) {
    return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ uint64_t desc_k(uint32_t addr) {
    return tc::sdesc_sw128(addr, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr, uint32_t lbo) {
    return tc::sdesc_sw128(addr, lbo, 1024);
}

// ===================================================================
// Pre-pass
// ===================================================================

constexpr int kPrepThreads = 128;
// L and T are lower triangular in 16 x 16 blocks: only the 10 blocks (I, J)
// with J <= I of L are stored, block bidx(I, J) = I (I + 1) / 2 + J, as 16
// rows of 20 floats (rows 80 bytes apart: the 8 rows a quarter warp reads
// or writes at once fall in 8 different 4-bank groups).  The diagonal
// blocks T_II replace L_II once solved; the 6 blocks of T below them are
// stored apart, block oidx(I, J) = I (I - 1) / 2 + J.
constexpr int kBs = 20;                       // packed block row stride
constexpr int kBlk = 16 * kBs;                // floats per packed block
constexpr int kPackBytes = 10 * kBlk * 4;     // 12800
__host__ __device__ constexpr int bidx(int I, int J) {
    return I * (I + 1) / 2 + J;
}
__host__ __device__ constexpr int oidx(int I, int J) {
    return I * (I - 1) / 2 + J;
}
// shared memory map (from a 1024-aligned base)
constexpr int kPKQ = 0;          // K_0 | Q_0 | K_1 | Q_1 (TMA), 32 KB; after G
                                 // the record image [TU | P, then PTU | g],
constexpr int kPL = kRecBytes;   // L (strictly lower part of A), packed, and
constexpr int kPY = kPL + kPackBytes;   // 4 warps x 16 x 8 fp32 scratch
constexpr int kPT = 32768;       // T below its diagonal blocks, packed
constexpr int kPKW = 32768;      // write keys Kw_0 | Kw_1 (TMA, write-key
                                 // mode), read by G only: T goes over them
// the rest of the map, after T (or after the write keys)
template <bool kKw>
struct PrepMap {
    static constexpr int G = kKw ? kPKW + 16384 : kPT + 6 * kBlk * 4;  // g2
    static constexpr int Beta = G + 256;          // beta[64]
    static constexpr int E = Beta + 256;          // column factors e_i[64]
    static constexpr int Bars = E + 256;          // 3 mbarriers
    static constexpr int Misc = Bars + 24;        // TMEM slot, words
    static constexpr int Smem = Misc + 32 + 1024;
    static constexpr int PerSm = kKw ? 4 : 5;     // CTAs resident per SM
};
static_assert(kPY + 4 * 16 * 8 * 4 <= kPT, "pre-pass map");
static_assert(kPL % 16 == 0 && kPT % 16 == 0, "float4 rows");
static_assert(kPT + 6 * kBlk * 4 <= PrepMap<true>::G, "T within the keys");
// five (four with write keys) CTAs per SM (the driver keeps 1 KB of each
// CTA's shared memory)
static_assert(5 * (PrepMap<false>::Smem + 1024) <= 233472, "pre-pass smem");
static_assert(4 * (PrepMap<true>::Smem + 1024) <= 233472, "pre-pass smem");

// Work distribution of the pre-pass.  Its grid is persistent (as many CTAs
// as fit at once); each CTA takes chunk-heads from a counter in chunk-major
// order (every head's chunk 0, then chunk 1, ...) and raises the record's
// ready flag once the record is in memory.  Past item `release`, only the
// CTAs of the first reserved_sms / 2 TPCs (SM ids 2t and 2t + 1) to
// register keep taking work; the others exit, and their SMs take the state
// pass, which starts on chunk 0 while the reserved SMs finish the last
// chunks.  Roles go by TPC because a state-pass CTA whose TPC mate kept
// pre-pass CTAs ran its chain up to 20 % slower.  Control words (zeroed
// before each launch): next item below `release`, next item from
// `release`, TPCs registered as reserved, then one role per TPC (0 unset,
// 1 reserved, 2 released, 3 being decided).
constexpr int kMaxSmId = 256;
constexpr int kCtrlWords = 4 + kMaxSmId / 2;

struct PrepParams {
    const float* log_alpha;
    const float* eta;
    uint8_t* rec;        // [B, H, nchunks, kRecBytes]
    float eps;
    int gdn;
    int T, H, nchunks;
    uint8_t* brec;       // null, or the backward's records [B, H, nchunks]
    unsigned int* ready; // [B, H, nchunks] record flags (1: in memory)
    unsigned int* ctrl;  // kCtrlWords control words
    int items;           // B H nchunks
    int release;         // items taken by every SM; the rest by reserved SMs
    int reserved_sms;
};

// acc (16 x 8, fragment layout) += A (16 x 16 packed fp32 block) x
// B[:, n0 .. n0 + 7] (16 x 8 of a packed fp32 block), tf32 MMAs.
__device__ __forceinline__ void mm16x8(float (&acc)[4], const float* A,
                                       const float* B, int n0, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[4];
        a[0] = tc::to_tf32(A[g * kBs + 8 * kk + t]);
        a[1] = tc::to_tf32(A[(g + 8) * kBs + 8 * kk + t]);
        a[2] = tc::to_tf32(A[g * kBs + 8 * kk + t + 4]);
        a[3] = tc::to_tf32(A[(g + 8) * kBs + 8 * kk + t + 4]);
        const uint32_t b0 = tc::to_tf32(B[(8 * kk + t) * kBs + n0 + g]);
        const uint32_t b1 = tc::to_tf32(B[(8 * kk + t + 4) * kBs + n0 + g]);
        tc::mma_m16n8k8_tf32(acc, a, b0, b1);
    }
}

// One 16 x 8 slab of an off-diagonal block of T = A^{-1} (A = I + L):
//   T_IJ[:, n0..n0+7] = -T_II sum_{m=J}^{I-1} L_Im T_mJ[:, n0..n0+7].
// The sum is formed in registers, passed through this warp's scratch Y
// (16 x 8, row stride 8) and multiplied by T_II.
// Block (I, J) of T: the diagonal ones sit in L's storage, the others in To.
__device__ __forceinline__ float* tblock(float* L, float* To, int I, int J) {
    return I == J ? L + bidx(I, I) * kBlk : To + oidx(I, J) * kBlk;
}

__device__ void offdiag_slab(float* L, float* T, float* Y, int I, int J,
                             int n0, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int m = J; m < I; ++m)
        mm16x8(acc, L + bidx(I, m) * kBlk, tblock(L, T, m, J), n0,
               lane);
    Y[g * 8 + 2 * t] = acc[0];
    Y[g * 8 + 2 * t + 1] = acc[1];
    Y[(g + 8) * 8 + 2 * t] = acc[2];
    Y[(g + 8) * 8 + 2 * t + 1] = acc[3];
    __syncwarp();
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const float* Tii = L + bidx(I, I) * kBlk;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t a[4];
        a[0] = tc::to_tf32(Tii[g * kBs + 8 * kk + t]);
        a[1] = tc::to_tf32(Tii[(g + 8) * kBs + 8 * kk + t]);
        a[2] = tc::to_tf32(Tii[g * kBs + 8 * kk + t + 4]);
        a[3] = tc::to_tf32(Tii[(g + 8) * kBs + 8 * kk + t + 4]);
        const uint32_t b0 = tc::to_tf32(Y[(8 * kk + t) * 8 + g]);
        const uint32_t b1 = tc::to_tf32(Y[(8 * kk + t + 4) * 8 + g]);
        tc::mma_m16n8k8_tf32(d, a, b0, b1);
    }
    __syncwarp();
    float* dst = T + oidx(I, J) * kBlk + n0;
    dst[g * kBs + 2 * t] = -d[0];
    dst[g * kBs + 2 * t + 1] = -d[1];
    dst[(g + 8) * kBs + 2 * t] = -d[2];
    dst[(g + 8) * kBs + 2 * t + 1] = -d[3];
}

// kKw: separate write keys (tm_kw): G = [K; Q] Kw^T, so that beta's
// denominator is k . kw, A uses K Kw^T and P uses Q Kw^T.
template <bool kKw>
__global__ void __launch_bounds__(kPrepThreads, PrepMap<kKw>::PerSm)
kla_prep_kernel(const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_kw, PrepParams p) {
    using PM = PrepMap<kKw>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_u32(sm);
    float* Lt = reinterpret_cast<float*>(sm + kPL);
    float* Tt = reinterpret_cast<float*>(sm + kPT);
    float* g2s = reinterpret_cast<float*>(sm + PM::G);
    float* betas = reinterpret_cast<float*>(sm + PM::Beta);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PM::Bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PM::Misc);
    float* wtot = reinterpret_cast<float*>(sm + PM::Misc + 4);
    int* failed_flag = reinterpret_cast<int*>(sm + PM::Misc + 8);
    int* item_slot = reinterpret_cast<int*>(sm + PM::Misc + 12);
    uint8_t* out = sm + kPKQ;   // record image, over the consumed K / Q

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the state pass may be scheduled once every pre-pass CTA has started;
    // it reads a record only after its ready flag is up
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr uint64_t kLimit = 2000000000ull;
    const int nbh = p.items / p.nchunks;

    // thread 0's work state: whether this SM keeps working past `release`,
    // whether items below it remain, and the item whose record store is in
    // flight (its flag goes up once the store has completed)
    bool reserved = true, below = true;
    int pending = -1, next = -1;
    // the next item: chunk-major, below `release` from every SM, past it from
    // the reserved SMs only (-1: none left for this CTA)
    auto claim = [&]() -> int {
        if (below) {
            const unsigned int i = atomicAdd(p.ctrl + 0, 1u);
            if (i < (unsigned)p.release) return (int)i;
            below = false;
        }
        if (!reserved) return -1;
        const unsigned int i = (unsigned)p.release + atomicAdd(p.ctrl + 1, 1u);
        return i < (unsigned)p.items ? (int)i : -1;
    };
    // the record of item i is in memory: its flag goes up (thread 0, which
    // issued the record's bulk store)
    auto publish = [&](int i) {
        tc::tma_store_wait_all<0>();
        tc::fence_proxy_async_global();
        tc::st_release_gpu(p.ready + i, 1u);
    };
    if (tid == 0) {
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        if constexpr (kKw) tc::prefetch_tmap(&tm_kw);
        for (int i = 0; i < 3; ++i) tc::mbar_init(&bars[i], 1);
        *failed_flag = 0;
        tc::fence_mbar_init();
        const unsigned int sid = tc::smid();
        if (p.release < p.items && sid < (unsigned)kMaxSmId) {
            // the first CTA of a TPC decides its role for all of them
            unsigned int* role = p.ctrl + 4 + (sid >> 1);
            unsigned int r = atomicCAS(role, 0u, 3u);
            if (r == 0u) {
                r = atomicAdd(p.ctrl + 2, 1u) < (unsigned)p.reserved_sms / 2
                        ? 1u
                        : 2u;
                atomicExch(role, r);
            } else if (r == 3u) {
                const uint64_t w0 = tc::globaltimer_ns();
                while (r == 3u && tc::globaltimer_ns() - w0 < kLimit) {
                    __nanosleep(32);
                    r = tc::ld_acquire_gpu(role);
                }
            }
            reserved = r != 2u;   // undecided after the limit: keep working
        }
        next = claim();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, 64);   // five CTAs per SM fit in TMEM
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool failed = false;

    for (uint32_t it = 0;; ++it) {
        const uint32_t ph = it & 1u;
        if (tid == 0) {
            const int item = next;   // claimed while the previous tiles landed
            *item_slot = item;
            if (item >= 0) {
                const int cc = item / nbh, bb = item % nbh;
                const int hh = bb % p.H, b0 = bb / p.H;
                tc::mbar_arrive_expect_tx(&bars[0], kKw ? 32768 + 16384 : 32768);
                tc::tma_load_4d(sm + kPKQ, &tm_k, &bars[0], 0, hh, cc * kC, b0);
                tc::tma_load_4d(sm + kPKQ + 8192, &tm_q, &bars[0], 0, hh, cc * kC, b0);
                tc::tma_load_4d(sm + kPKQ + 16384, &tm_k, &bars[0], 64, hh, cc * kC, b0);
                tc::tma_load_4d(sm + kPKQ + 24576, &tm_q, &bars[0], 64, hh, cc * kC, b0);
                if constexpr (kKw) {
                    tc::tma_load_4d(sm + kPKW, &tm_kw, &bars[0], 0, hh, cc * kC, b0);
                    tc::tma_load_4d(sm + kPKW + 8192, &tm_kw, &bars[0], 64, hh, cc * kC, b0);
                }
            } else if (pending >= 0) {
                publish(pending);
                pending = -1;
            }
        }
        __syncthreads();
        const int item = *item_slot;
        if (item < 0) break;
        const int c = item / nbh;
        const int bh = item % nbh;
        const int b = bh / p.H, h = bh % p.H;
        const int t0 = c * kC;
        uint8_t* brec = p.brec ? p.brec + ((size_t)bh * p.nchunks + c) *
                                              bwdrec::BYTES
                               : nullptr;
        // gates of this chunk: cumulative log2 decay (two warp scans)
        float la = 0.f, et = 0.f;
        if (tid < kC && t0 + tid < p.T) {
            const size_t off = ((size_t)b * p.T + t0 + tid) * p.H + h;
            la = p.log_alpha[off];
            et = p.eta[off];
        }
        float g2 = la * kLog2e;
        if (tid < kC) {
    #pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, g2, off);
                if (lane >= off) g2 += y;
            }
            if (tid == 31) *wtot = g2;
        }
        __syncthreads();
        if (tid >= 32 && tid < kC) g2 += *wtot;
        if (tid < kC) g2s[tid] = g2;
        // Gamma_ri = 2^(g_r - g_m) e_i with g_m the g of the last column m of
        // i's 16-column tile and e_i = 2^(g_m - g_i) <= 1: one ex2 per row and
        // tile instead of one per element (a tile whose g spans more than 2^96
        // takes the direct form, so that neither factor can overflow)
        float* ecol = reinterpret_cast<float*>(sm + PM::E);
        if (tid < kC)
            ecol[tid] = tc::ex2(__shfl_sync(0xffffffffu, g2, (lane & 16) | 15) -
                                g2);

        // G = [K; Q] K^T: lanes 0..63 K K^T, lanes 64..127 Q K^T (columns 0..63)
        if (tid == 0) {
            next = claim();   // while this item's tiles land
            if (tc::mbar_wait(&bars[0], ph, kLimit)) {
                tc::tc_fence_after();
                constexpr uint32_t idG = tc::idesc_bf16(128, 64, false, false);
    #pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    // A: [K; Q]; B: the keys' rows of the same tiles, or the
                    // write keys
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    const uint32_t offw =
                        kKw ? kPKW + (ks >> 2) * 8192 + (ks & 3) * 32
                            : kPKQ + off;
                    tc::mma_bf16(tmem, desc_k(sbase + kPKQ + off),
                                 desc_k(sbase + offw), idG, ks > 0);
                }
                tc::mma_commit(&bars[1]);
                if (pending >= 0) {   // the previous item's record (long done)
                    publish(pending);
                    pending = -1;
                }
            } else {
                *reinterpret_cast<volatile int*>(failed_flag) = 1;
            }
        }
        __syncthreads();   // g2s complete; the issuing lane rejoined
        bool ok = *reinterpret_cast<volatile int*>(failed_flag) == 0;
        ok = ok && tc::mbar_wait(&bars[1], ph, kLimit);
        ok = !__syncthreads_or(!ok);
        if (!ok) {
            if (tid == 0) {
                atomicOr(&g_fault_word2, 1u);
                tc::mbar_wait(&bars[0], ph, 100000000ull);   // copies in flight
                tc::mbar_wait(&bars[1], ph, 100000000ull);   // the MMAs, if issued
            }
            failed = true;
            break;
        }
        tc::tc_fence_after();
        {
            float x[64];
            const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
            tc::tmem_ld32(ta, x);
            tc::tmem_ld32(ta + 32, x + 32);
            tc::tmem_ld_wait();
            if (tid < kC) {
                // A row r = tid: beta_r Gamma_ri (K K^T)_ri for i < r (fp32),
                // into the packed blocks (I, m), m <= I, of its block row I
                const int r = tid, I = r >> 4;
                float kk = 0.f;   // ||k_r||^2, the diagonal of K K^T
    #pragma unroll
                for (int i = 0; i < 64; ++i) kk = i == r ? x[i] : kk;
                const float denom = kk + p.eps;
                const float br = p.gdn ? et : (denom == 0.f ? 0.f : et / denom);
                betas[r] = br;
                if (brec) {   // gates of the backward's record (g in natural log)
                    reinterpret_cast<float*>(brec + bwdrec::G_OFF)[r] =
                        g2 * 0.6931471805599453f;
                    reinterpret_cast<float*>(brec + bwdrec::B_OFF)[r] = br;
                    reinterpret_cast<float*>(brec + bwdrec::N_OFF)[r] = kk;
                }
    #pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (m > I) break;
                    float* Lr = Lt + bidx(I, m) * kBlk + (r & 15) * kBs - 16 * m;
                    const float gm = g2s[16 * m + 15];
                    const bool fact = fabsf(g2s[16 * m] - gm) <= 96.f;
                    const float bf = br * tc::ex2(g2 - gm);
    #pragma unroll
                    for (int i = 16 * m; i < 16 * m + 16; i += 4) {
                        const float4 e = *reinterpret_cast<const float4*>(ecol + i);
                        const float4 gi = *reinterpret_cast<const float4*>(g2s + i);
                        float4 a;
                        a.x = fact ? bf * e.x : br * tc::ex2(g2 - gi.x);
                        a.y = fact ? bf * e.y : br * tc::ex2(g2 - gi.y);
                        a.z = fact ? bf * e.z : br * tc::ex2(g2 - gi.z);
                        a.w = fact ? bf * e.w : br * tc::ex2(g2 - gi.w);
                        a.x = i + 0 < r ? a.x * x[i + 0] : 0.f;
                        a.y = i + 1 < r ? a.y * x[i + 1] : 0.f;
                        a.z = i + 2 < r ? a.z * x[i + 2] : 0.f;
                        a.w = i + 3 < r ? a.w * x[i + 3] : 0.f;
                        *reinterpret_cast<float4*>(Lr + i) = a;
                    }
                }
            } else {
                // P row r = tid - 64: Gamma_ri (Q K^T)_ri for i <= r, as bf16
                // operand rows behind TU in the record image
                const int r = tid - kC;
                const float gr = g2s[r];
    #pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float gm = g2s[16 * m + 15];
                    const bool fact = fabsf(g2s[16 * m] - gm) <= 96.f;
                    const float f = tc::ex2(gr - gm);
    #pragma unroll
                    for (int i = 16 * m; i < 16 * m + 16; i += 8) {
                        float e[8];
    #pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float gam =
                                fact ? f * ecol[i + k] : tc::ex2(gr - g2s[i + k]);
                            e[k] = i + k <= r ? gam * x[i + k] : 0.f;
                        }
                        uint4 v;
                        v.x = tc::pack_bf16x2(e[0], e[1]);
                        v.y = tc::pack_bf16x2(e[2], e[3]);
                        v.z = tc::pack_bf16x2(e[4], e[5]);
                        v.w = tc::pack_bf16x2(e[6], e[7]);
                        *reinterpret_cast<uint4*>(out + kRecPTU + swz(r, i)) = v;
                        if (brec)   // P, rows of 64, for the backward
                            *reinterpret_cast<uint4*>(brec + bwdrec::P_OFF +
                                                      (r * kC + i) * 2) = v;
                    }
                }
            }
        }
        __syncthreads();
        // diagonal blocks T_bb = (I + L_bb)^{-1}: thread (bb, cl) solves column
        // cl by substitution (threads 0..63)
        if (tid < kC) {
            const int bb = tid >> 4, cl = tid & 15;
            const float* Lb = Lt + bidx(bb, bb) * kBlk;
            float xv[16];
    #pragma unroll
            for (int r = 0; r < 16; ++r) xv[r] = (r == cl) ? 1.f : 0.f;
    #pragma unroll
            for (int r = 1; r < 16; ++r) {
                float a0 = 0.f, a1 = 0.f;
    #pragma unroll
                for (int i = 0; i < r; i += 2) {
                    a0 = fmaf(Lb[r * kBs + i], xv[i], a0);
                    if (i + 1 < r) a1 = fmaf(Lb[r * kBs + i + 1], xv[i + 1], a1);
                }
                if (r > cl) xv[r] = -(a0 + a1);
            }
            __syncwarp();   // this warp's two blocks of L are read: T over them
            float* Tb = Lt + bidx(bb, bb) * kBlk + cl;
    #pragma unroll
            for (int r = 0; r < 16; ++r) Tb[r * kBs] = xv[r];
        }
        __syncthreads();
        float* Y = reinterpret_cast<float*>(sm + kPY) + warp * 128;
        // level 1: (1,0), (2,1), (3,2); 6 slabs of 8 columns on 4 warps
        for (int job = warp; job < 6; job += 4) {
            const int I = (job >> 1) + 1;
            offdiag_slab(Lt, Tt, Y, I, I - 1, 8 * (job & 1), lane);
            __syncwarp();
        }
        __syncthreads();
        // level 2: (2,0), (3,1)
        offdiag_slab(Lt, Tt, Y, 2 + (warp >> 1), warp >> 1, 8 * (warp & 1), lane);
        __syncthreads();
        // level 3: (3,0)
        if (warp < 2) offdiag_slab(Lt, Tt, Y, 3, 0, 8 * warp, lane);
        __syncthreads();

        // TU = T Diag(beta) as bf16 operand rows: thread -> (row, 32 columns)
        {
            const int r = tid >> 1, c0 = 32 * (tid & 1);
    #pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint4 v;
                const int col = c0 + j, I = r >> 4, J = col >> 4;
                const float* tr =
                    tblock(Lt, Tt, I, J < I ? J : I) + (r & 15) * kBs + (col & 15);
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);   // J > I
                const float4 ta =
                    J <= I ? *reinterpret_cast<const float4*>(tr) : z;
                const float4 tb =
                    J <= I ? *reinterpret_cast<const float4*>(tr + 4) : z;
                const float4 ba = *reinterpret_cast<const float4*>(betas + c0 + j);
                const float4 bb =
                    *reinterpret_cast<const float4*>(betas + c0 + j + 4);
                v.x = tc::pack_bf16x2(ta.x * ba.x, ta.y * ba.y);
                v.y = tc::pack_bf16x2(ta.z * ba.z, ta.w * ba.w);
                v.z = tc::pack_bf16x2(tb.x * bb.x, tb.y * bb.y);
                v.w = tc::pack_bf16x2(tb.z * bb.z, tb.w * bb.w);
                *reinterpret_cast<uint4*>(out + kRecTU + swz(r, c0 + j)) = v;
                if (brec) {   // T itself, rows of 64, for the backward
                    uint4 w;
                    w.x = tc::pack_bf16x2(ta.x, ta.y);
                    w.y = tc::pack_bf16x2(ta.z, ta.w);
                    w.z = tc::pack_bf16x2(tb.x, tb.y);
                    w.w = tc::pack_bf16x2(tb.z, tb.w);
                    *reinterpret_cast<uint4*>(brec + bwdrec::T_OFF +
                                              (r * kC + col) * 2) = w;
                }
            }
        }
        if (tid < kC) reinterpret_cast<float*>(out + kRecG)[tid] = g2s[tid];
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        // PTU = P TU on the tensor cores: [TU; P] TU, lanes 64..127, over G's
        // columns (G was read out before the barriers above); TU is K-major as
        // the A rows and MN-major as B
        if (tid == 0) {
            tc::tc_fence_after();
            constexpr uint32_t idP = tc::idesc_bf16(128, 64, false, true);
    #pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_bf16(tmem, desc_k(sbase + kPKQ + kRecTU + ks * 32),
                             desc_mn(sbase + kPKQ + kRecTU + ks * 2048, 0), idP,
                             ks > 0);
            tc::mma_commit(&bars[2]);
        }
        __syncwarp();
        ok = tc::mbar_wait(&bars[2], ph, kLimit);
        if (!__syncthreads_or(!ok)) {
            tc::tc_fence_after();
            if (tid >= kC) {   // PTU rows over P
                const int r = tid - kC;
                float x[64];
                const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
                tc::tmem_ld32(ta, x);
                tc::tmem_ld32(ta + 32, x + 32);
                tc::tmem_ld_wait();
    #pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 v;
                    v.x = tc::pack_bf16x2(x[8 * j + 0], x[8 * j + 1]);
                    v.y = tc::pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
                    v.z = tc::pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
                    v.w = tc::pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
                    *reinterpret_cast<uint4*>(out + kRecPTU + swz(r, 8 * j)) = v;
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncthreads();
            if (tid == 0) {   // the record, one bulk copy
                tc::bulk_store(p.rec + ((size_t)bh * p.nchunks + c) * kRecBytes,
                               out, kRecBytes);
                tc::tma_store_commit();
                tc::tma_store_wait_read<0>();   // the image may be overwritten
                pending = bh * p.nchunks + c;
            }
        } else {
            if (tid == 0) {
                atomicOr(&g_fault_word2, 1u);
                tc::mbar_wait(&bars[2], ph, 100000000ull);
            }
            failed = true;
        }
        __syncthreads();
        if (failed) break;
    }   // items
    if (tid == 0 && pending >= 0) publish(pending);
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

// ===================================================================
// State pass
// ===================================================================

constexpr int kNV = 64;              // dv columns per CTA
constexpr int kNS = 3;               // stages of the TMA ring
// stage map (bytes from the stage base, 1024-aligned)
constexpr int kSK0 = 0;              // K_0, later -W_0     } [-W_0; Q'_0]
constexpr int kSQ0 = 8192;           // Q_0, later Q'_0     }
constexpr int kSK1 = 16384;          // K_1, later -W_1     } [-W_1; Q'_1]
constexpr int kSQ1 = 24576;          // Q_1, later Q'_1     }
constexpr int kSV = 32768;           // V (64 tokens x 64 columns)
constexpr int kSTU = 40960;          // [TU; PTU], later [KG_0 | KG_1] with
                                     // KG = Diag(Gamma_C) K
constexpr int kSG = kSTU + kRecG;    // g (log2), 64 floats
constexpr int kStage = 58368;
constexpr int kSS = kNS * kStage;    // S bf16, 128 x 64, MN-major
constexpr int kSUt = kSS + 16384;    // U~ bf16, 64 x 64, MN-major
constexpr int kSO = kSUt + 8192;     // o of a chunk, bf16 (TMA store image)
constexpr int kSBars = kSO + 8192;
// mbarriers: full[3] (TMA), ready[3] (helper done with the stage), hmma[2]
// (helper MMAs, by helper group), c1 (chain MMA group 1), c2 (dS),
// accfree[3] (accumulator c mod 3 read out), empty[3] (the chain is done
// with a stage)
constexpr int kBFull = 0, kBReady = 3, kBHmma = 6, kBC1 = 8, kBC2 = 9,
              kBAccFree = 10, kBEmpty = 13, kNumBars = 16;
constexpr int kSMisc = kSBars + 8 * kNumBars;   // abort, TMEM slot, issued
constexpr int kSSmem = kSMisc + 16 + 1024;
static_assert(kSG + 256 <= kStage && kStage % 1024 == 0, "stage map");
static_assert(kSSmem <= 232448, "state-pass shared memory");
constexpr uint32_t kStageTx = 4 * 8192 + 8192 + kRecBytes;

// TMEM columns
constexpr uint32_t kColH = 0;        // helper group 0: [-W; -PTU Kg] (128)
constexpr uint32_t kColAcc = 128;    // + 64 (c mod 3 < 2): [U; PTU V], then
constexpr uint32_t kColAcc2 = 448;   // [U~; O]; c mod 3 = 2 here
constexpr uint32_t kColDS = 256;     // dS
constexpr uint32_t kColH1 = 320;     // helper group 1: [-W; -PTU Kg] (128)
constexpr uint32_t kTmemCols = 512;

// Three accumulators [U; PTU V] in turn: the helper of chunk c writes one
// while the chain still reads those of chunks c - 1 and c - 2, so a helper
// waits only for the chain of chunk c - 3.
__device__ __forceinline__ uint32_t acc_col(int c) {
    const int r = c % 3;
    return r == 2 ? kColAcc2 : kColAcc + 64 * r;
}

// Two helper warpgroups take the chunks in turns (group c & 1), so each has
// two chain periods for one chunk.
constexpr int kChainThreads = 128, kHelperThreads = 128, kHelperGroups = 2;
constexpr int kStateThreads = kChainThreads + kHelperGroups * kHelperThreads;
constexpr int kBarChain = 2, kBarChainLo = 3, kBarChainHi = 4,
              kBarHelper0 = 5;   // + helper group

struct StateParams {
    const float* h0;
    __nv_bfloat16* o;     // null in checkpoint mode
    float* hT;
    float* ckpt;          // checkpoint mode: the state at every chunk start
    const uint8_t* rec;   // records of the pre-pass
    int T, H, nchunks;
    uint64_t wait_ns;     // limit of every mbarrier wait
    int no_issue;         // self-test: the producer issues nothing
    const unsigned int* ready;   // record flags of a running pre-pass, or
                                 // null (the records are in memory)
    const __nv_bfloat16* kw;     // write keys [B, T, H, 128] (write-key mode)
};

// Write 64 fp32 values as one 128-byte swizzled bf16 row.
__device__ __forceinline__ void st_row(uint8_t* base, int row,
                                       const float* x) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint4 v;
        v.x = tc::pack_bf16x2(x[8 * j + 0], x[8 * j + 1]);
        v.y = tc::pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
        v.z = tc::pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
        v.w = tc::pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
        *reinterpret_cast<uint4*>(base + row * 128 + ((j ^ (row & 7)) << 4)) =
            v;
    }
}

// Write 32 fp32 values as 16-byte chunks 4 hf .. 4 hf + 3 (the columns
// 32 hf .. 32 hf + 31) of a 128-byte swizzled bf16 row.
__device__ __forceinline__ void st_half_row(uint8_t* base, int row, int hf,
                                            const float* x) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 v;
        v.x = tc::pack_bf16x2(x[8 * j + 0], x[8 * j + 1]);
        v.y = tc::pack_bf16x2(x[8 * j + 2], x[8 * j + 3]);
        v.z = tc::pack_bf16x2(x[8 * j + 4], x[8 * j + 5]);
        v.w = tc::pack_bf16x2(x[8 * j + 6], x[8 * j + 7]);
        *reinterpret_cast<uint4*>(base + row * 128 +
                                  (((4 * hf + j) ^ (row & 7)) << 4)) = v;
    }
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) {
    return *reinterpret_cast<__nv_bfloat162*>(&u);
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) {
    return *reinterpret_cast<uint32_t*>(&v);
}

// 8 bf16 times s (packed bf16 multiplies; s is rounded to bf16 first)
__device__ __forceinline__ uint4 scale8(uint4 u, __nv_bfloat162 s) {
    uint4 r;
    r.x = as_u32(__hmul2(as_bf2(u.x), s));
    r.y = as_u32(__hmul2(as_bf2(u.y), s));
    r.z = as_u32(__hmul2(as_bf2(u.z), s));
    r.w = as_u32(__hmul2(as_bf2(u.w), s));
    return r;
}

// kKw: separate write keys: the state takes Kw^T Diag(Gamma_C) U~ (the
// residual and W keep the keys).
template <bool kCkpt, bool kKw>
__global__ void __launch_bounds__(kStateThreads, 1)
kla_state_kernel(const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_o, StateParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = tc::smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kSBars);
    int* abort_flag = reinterpret_cast<int*>(sm + kSMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSMisc + 4);
    int* issued = reinterpret_cast<int*>(sm + kSMisc + 8);
    volatile int* vabort = abort_flag;

    // a second state pass sharing the pre-pass (launched right after this
    // one as its programmatic dependent) may start once every CTA of this
    // grid is resident; it too reads records by their flags
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int j0 = blockIdx.y * kNV;
    const int nchunks = p.nchunks;

    // Loads of chunk c into its stage (TMA tiles of K, Q, V and the record
    // of the pre-pass): the first kNS by thread 0 at the start, then chunk
    // c >= kNS by lane 0 of the helper group that prepares it, as soon as
    // the chain has released the stage (chunk c - kNS done).  With flags,
    // the record's flag is awaited first (while the chain still holds the
    // stage).  Chunks two rings ahead are prefetched into L2 (a record not
    // yet written is fetched again when it is loaded: L2 is coherent).
    const uint8_t* rec0 = p.rec + (size_t)bh * nchunks * kRecBytes;
    const unsigned int* ready0 = p.ready ? p.ready + (size_t)bh * nchunks
                                         : nullptr;
    auto prefetch = [&](int c) {
        const int t0 = c * kC;
        tc::tma_prefetch_4d(&tm_k, 0, h, t0, b);
        tc::tma_prefetch_4d(&tm_q, 0, h, t0, b);
        tc::tma_prefetch_4d(&tm_k, 64, h, t0, b);
        tc::tma_prefetch_4d(&tm_q, 64, h, t0, b);
        tc::tma_prefetch_4d(&tm_v, j0, h, t0, b);
        tc::bulk_prefetch_l2(rec0 + (size_t)c * kRecBytes, kRecBytes);
    };
    // false when the record's flag did not come up in time (the caller
    // raises the abort flag and issues no copy of the chunk).  A helper's
    // issuing lane reads the flag of its next chunk while its current
    // copies land (peek_record), so that the issue, which is on the path of
    // every chunk, seldom waits for a flag.
    int peeked = -1;   // a chunk whose flag this thread has seen up
    auto await_record = [&](int c) {
        if (!ready0 || c == peeked) return true;
        if (!tc::flag_wait(ready0 + c, 1u, vabort, p.wait_ns)) return false;
        tc::fence_proxy_async_global();   // before the bulk load that follows
        return true;
    };
    auto peek_record = [&](int c) {
        if (!ready0 || c >= nchunks) return;
        if (tc::ld_acquire_gpu(ready0 + c) == 1u) {
            tc::fence_proxy_async_global();
            peeked = c;
        }
    };
    auto issue_tiles = [&](int c) {
        const int s = c % kNS;
        uint8_t* st = sm + s * kStage;
        uint64_t* bar = &bars[kBFull + s];
        const int t0 = c * kC;
        tc::mbar_arrive_expect_tx(bar, kStageTx);
        tc::tma_load_4d(st + kSK0, &tm_k, bar, 0, h, t0, b);
        tc::tma_load_4d(st + kSQ0, &tm_q, bar, 0, h, t0, b);
        tc::tma_load_4d(st + kSK1, &tm_k, bar, 64, h, t0, b);
        tc::tma_load_4d(st + kSQ1, &tm_q, bar, 64, h, t0, b);
        tc::tma_load_4d(st + kSV, &tm_v, bar, j0, h, t0, b);
        atomicMax(issued, c + 1);
    };
    auto issue_record = [&](int c) {
        tc::bulk_load(sm + (c % kNS) * kStage + kSTU,
                      rec0 + (size_t)c * kRecBytes, kRecBytes,
                      &bars[kBFull + c % kNS]);
        if (c + 2 * kNS < nchunks) prefetch(c + 2 * kNS);
    };
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) tc::mbar_init(&bars[i], 1);
        *abort_flag = 0;
        *issued = 0;
        tc::fence_mbar_init();
        if (!p.no_issue) {   // the first tiles: inputs, ready at launch
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            for (int c = 0; c < kNS && c < nchunks; ++c) issue_tiles(c);
        }
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    float S[kNV];
    if (tid < kChainThreads) {   // S rows (key dims) of this column slice
        const float* src =
            p.h0 ? p.h0 + ((size_t)bh * kD + tid) * kD + j0 : nullptr;
#pragma unroll
        for (int j = 0; j < kNV; j += 4) {
            const float4 v = src ? *reinterpret_cast<const float4*>(src + j)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
        }
        st_row(sm + kSS, tid, S);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Without ready flags this is a programmatic dependent that reads the
    // records once the pre-pass grid has completed (a no-op when launched
    // normally); with them it reads each record once its flag is up, while
    // the pre-pass may still be running.
    if (!p.ready) asm volatile("griddepcontrol.wait;" ::: "memory");

    if (tid == 0 && !p.no_issue) {   // the first records, once flagged
        for (int c = 0; c < kNS && c < nchunks; ++c) {
            if (!await_record(c)) {
                *vabort = 1;
                break;
            }
            issue_record(c);
        }
        for (int c = kNS; c < 2 * kNS && c < nchunks; ++c) prefetch(c);
    }

    if (tid >= kChainThreads) {
        // ========================================================== helpers
        const int grp = (tid - kChainThreads) / kHelperThreads;
        const int hl = (tid - kChainThreads) % kHelperThreads;  // TMEM lane
        const int bar_id = kBarHelper0 + grp;
        const uint32_t colH = grp ? kColH1 : kColH;
        uint64_t* hbar = &bars[kBHmma + grp];
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        // [-W; -PTU Kg]: the negation rides on the instruction (negate A)
        constexpr uint32_t idA = tc::idesc_bf16(128, 128, false, true, true);
        constexpr uint32_t idB = tc::idesc_bf16(128, kNV, false, true);
        int committed = -1, nmma = 0;
        for (int c = grp; c < nchunks; c += kHelperGroups) {
            const int s = c % kNS;
            uint8_t* st = sm + s * kStage;
            const uint32_t sst = sbase + s * kStage;
            bool ok = true;
            if (c >= kNS && hl == 0 && !p.no_issue) {
                // this group's lane 0 loads the chunk once the chain is done
                // with chunk c - kNS (the helpers wait for the data anyway;
                // the chain's own thread would pay the issue on its path)
                ok = await_record(c) &&
                     tc::mbar_wait_or_abort(&bars[kBEmpty + s],
                                            ((c - kNS) / kNS) & 1, vabort,
                                            p.wait_ns);
                if (ok) {
                    issue_tiles(c);
                    issue_record(c);
                } else {
                    *vabort = 1;
                }
            }
            if (hl == 0 && !p.no_issue && c + kHelperGroups >= kNS)
                peek_record(c + kHelperGroups);
            __syncwarp();
            ok = ok && tc::mbar_wait_or_abort(&bars[kBFull + s],
                                              (c / kNS) & 1, vabort, p.wait_ns);
            if (ok && c >= 3)   // accumulator of chunk c - 3 read out
                ok = tc::mbar_wait_or_abort(&bars[kBAccFree + c % 3],
                                            ((c - 3) / 3) & 1, vabort,
                                            p.wait_ns);
            if (tc::named_bar_or(bar_id, kHelperThreads, !ok)) {
                *vabort = 1;
                break;
            }
            // Diag(gamma) K in place of K (the operand of the next MMAs);
            // Diag(Gamma_C) K kept in registers until TU, PTU are read.
            // (16-byte chunk (j + r) mod 8 at step j: the 8 rows a quarter
            // warp touches at once sit in 8 different bank groups; a chunk
            // keeps its swizzled position, the scaling is per row)
            const float* g2 = reinterpret_cast<const float*>(st + kSG);
            const int r = hl & 63, hh = hl >> 6;
            const __nv_bfloat162 gam = __float2bfloat162_rn(tc::ex2(g2[r]));
            const __nv_bfloat162 gamC =
                __float2bfloat162_rn(tc::ex2(g2[kC - 1] - g2[r]));
            uint4 kG[8];
            {
                uint8_t* krow = st + (hh ? kSK1 : kSK0) + r * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int cj = ((j + r) & 7) << 4;
                    const uint4 u = *reinterpret_cast<const uint4*>(krow + cj);
                    *reinterpret_cast<uint4*>(krow + cj) = scale8(u, gam);
                    if constexpr (!kKw) kG[j] = scale8(u, gamC);
                }
                if constexpr (kKw) {
                    // this row's write keys straight from global memory (in
                    // flight during the MMAs below), 16-byte piece
                    // ((j + r) mod 8) xor (r mod 8) at step j, so that it
                    // lands where the swizzled tile keeps it
                    const int t = c * kC + r;
                    const __nv_bfloat16* kwrow =
                        p.kw + (((size_t)b * p.T + (t < p.T ? t : 0)) * p.H +
                                h) * kD + hh * 64;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        kG[j] = t < p.T
                                    ? __ldg(reinterpret_cast<const uint4*>(
                                          kwrow + 8 * (((j + r) & 7) ^ (r & 7))))
                                    : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tc::fence_proxy_async_smem();
            tc::named_bar_sync(bar_id, kHelperThreads);
            if (hl == 0) {
                tc::tc_fence_after();
                // [-W; -PTU Kg] = -[TU; PTU] Kg    (M 128, N 128, K 64; the
                // two 64-feature halves of Kg are 16 KB apart)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + colH, desc_k(sst + kSTU + ks * 32),
                                 desc_mn(sst + kSK0 + ks * 2048, kSK1 - kSK0),
                                 idA, ks > 0);
                // [U; PTU V] = [TU; PTU] V       (M 128, N 64, K 64)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + acc_col(c),
                                 desc_k(sst + kSTU + ks * 32),
                                 desc_mn(sst + kSV + ks * 2048, 0), idB,
                                 ks > 0);
                tc::mma_commit(hbar);
            }
            __syncwarp();   // the issuing lane rejoins before the waits
            committed = nmma++;
            if (tc::named_bar_or(bar_id, kHelperThreads,
                                 !tc::mbar_wait_or_abort(hbar, committed & 1,
                                                         vabort, p.wait_ns))) {
                *vabort = 1;
                break;
            }
            tc::tc_fence_after();
            {   // Diag(Gamma_C) K (or Kw) over [TU; PTU] (read by the
                // finished MMAs)
                uint8_t* grow = st + kSTU + hh * 8192 + r * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(grow + (((j + r) & 7) << 4)) =
                        kKw ? scale8(kG[j], gamC) : kG[j];
            }
            // the four 32-column blocks of this row, handed to put(q4, x):
            // block q + 1 comes in from TMEM while block q is written out
            // (in the write-key instantiation one at a time: its register
            // budget has no room for the second block)
            auto four_blocks = [&](auto&& put) {
                if constexpr (kKw) {
#pragma unroll 1
                    for (int q4 = 0; q4 < 4; ++q4) {
                        float x[32];
                        tc::tmem_ld32(tl + colH + 32 * q4, x);
                        tc::tmem_ld_wait();
                        put(q4, x);
                    }
                } else {
                    float xa[32], xb[32];
                    tc::tmem_ld32(tl + colH, xa);
                    tc::tmem_ld_wait();
                    tc::tmem_ld32(tl + colH + 32, xb);
                    put(0, xa);
                    tc::tmem_ld_wait();
                    tc::tmem_ld32(tl + colH + 64, xa);
                    put(1, xb);
                    tc::tmem_ld_wait();
                    tc::tmem_ld32(tl + colH + 96, xb);
                    put(2, xa);
                    tc::tmem_ld_wait();
                    put(3, xb);
                }
            };
            if (hl < kC) {
                // -W row hl over Kg (both halves; read by the finished MMA)
                four_blocks([&](int q4, const float* x) {
                    st_half_row(st + ((q4 >> 1) ? kSK1 : kSK0), hl, q4 & 1, x);
                });
            } else {
                // Q' row = gamma_r Q_r + (-PTU Kg)_r over Q (in place; packed
                // bf16 fma, the TMEM values rounded to bf16 first)
                const int rq = hl - kC;
                const __nv_bfloat162 gq =
                    __float2bfloat162_rn(tc::ex2(g2[rq]));
                four_blocks([&](int q4, const float* x) {
                    uint8_t* qrow = st + ((q4 >> 1) ? kSQ1 : kSQ0) + rq * 128;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4* pq = reinterpret_cast<uint4*>(
                            qrow + (((4 * (q4 & 1) + j) ^ (rq & 7)) << 4));
                        uint4 u = *pq;
                        const float* xj = x + 8 * j;
                        u.x = as_u32(__hfma2(gq, as_bf2(u.x), as_bf2(
                            tc::pack_bf16x2(xj[0], xj[1]))));
                        u.y = as_u32(__hfma2(gq, as_bf2(u.y), as_bf2(
                            tc::pack_bf16x2(xj[2], xj[3]))));
                        u.z = as_u32(__hfma2(gq, as_bf2(u.z), as_bf2(
                            tc::pack_bf16x2(xj[4], xj[5]))));
                        u.w = as_u32(__hfma2(gq, as_bf2(u.w), as_bf2(
                            tc::pack_bf16x2(xj[6], xj[7]))));
                        *pq = u;
                    }
                });
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::named_bar_sync(bar_id, kHelperThreads);
            if (hl == 0) tc::mbar_arrive(&bars[kBReady + s]);
        }
        if (*vabort && hl == 0 && committed >= 0)   // drain own MMAs
            tc::mbar_wait(hbar, committed & 1, 100000000ull);
    } else {
        // ============================================================ chain
        const int row = tid;                      // TMEM lane
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        constexpr uint32_t idN = tc::idesc_bf16(128, kNV, false, true);
        constexpr uint32_t idDS = tc::idesc_bf16(128, kNV, true, true);
        int last_c1 = -1, last_c2 = -1;
        bool failed = false;
        for (int c = 0; c < nchunks && !failed; ++c) {
            const int s = c % kNS;
            const uint8_t* st = sm + s * kStage;
            const uint32_t sst = sbase + s * kStage;
            const uint32_t acc = tmem + acc_col(c);
            if constexpr (kCkpt) {   // the state chunk c starts from (fp32)
                float* dst = p.ckpt +
                             (((size_t)bh * nchunks + c) * kD + row) * kD + j0;
#pragma unroll
                for (int j = 0; j < kNV; j += 4)
                    *reinterpret_cast<float4*>(dst + j) =
                        make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
            }
            if (tc::named_bar_or(kBarChain, kChainThreads,
                                 !tc::mbar_wait_or_abort(&bars[kBReady + s],
                                                         (c / kNS) & 1,
                                                         vabort, p.wait_ns))) {
                failed = true;
                break;
            }
            tc::tc_fence_after();
            if (tid == 0) {   // [U~; O] = [U; PTU V] + [-W; Q'] S
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(acc,
                                 desc_k(sst + (ks >> 2) * 16384 +
                                        (ks & 3) * 32),
                                 desc_mn(sbase + kSS + ks * 2048, 0), idN,
                                 true);
                tc::mma_commit(&bars[kBC1]);
                last_c1 = c;
            }
            __syncwarp();
            const float* g2 = reinterpret_cast<const float*>(st + kSG);
            bool ok = tc::mbar_wait_or_abort(&bars[kBC1], c & 1, vabort, p.wait_ns);
            if (warp < 2) {
                // U~ row (token) to shared memory, then dS = KG^T U~
                if (ok) {
                    tc::tc_fence_after();
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float x[32];
                        tc::tmem_ld32(tl + (acc - tmem) + 32 * hf, x);
                        tc::tmem_ld_wait();
                        st_half_row(sm + kSUt, row, hf, x);
                    }
                    tc::fence_proxy_async_smem();
                }
                tc::tc_fence_before();
                ok = !tc::named_bar_or(kBarChainLo, 64, !ok);
                if (ok && tid == 0) {
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_bf16(tmem + kColDS,
                                     desc_mn(sst + kSTU + ks * 2048, 8192),
                                     desc_mn(sbase + kSUt + ks * 2048, 0),
                                     idDS, ks > 0);
                    tc::mma_commit(&bars[kBC2]);
                    last_c2 = c;
                }
                __syncwarp();
            } else if (ok && !kCkpt) {
                // o of the chunk (row - 64 = token) through shared memory
                // and one TMA store (rows past T are clipped by the copy);
                // the image is free once the previous store has read it
                if (tid == kC) tc::tma_store_wait_read<0>();
                tc::tc_fence_after();
                tc::named_bar_sync(kBarChainHi, 64);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float x[32];
                    tc::tmem_ld32(tl + (acc - tmem) + 32 * hf, x);
                    tc::tmem_ld_wait();
                    st_half_row(sm + kSO, row - kC, hf, x);
                }
                tc::fence_proxy_async_smem();
                tc::named_bar_sync(kBarChainHi, 64);
                if (tid == kC) {
                    tc::tma_store_4d(&tm_o, sm + kSO, j0, h, c * kC, b);
                    tc::tma_store_commit();
                }
            }
            ok = ok && tc::mbar_wait_or_abort(&bars[kBC2], c & 1, vabort, p.wait_ns);
            if (tc::named_bar_or(kBarChain, kChainThreads, !ok)) {
                failed = true;
                break;
            }
            tc::tc_fence_after();
            {   // S <- gamma_C S + dS
                const float gC = tc::ex2(g2[kC - 1]);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float x[32];
                    tc::tmem_ld32(tl + kColDS + 32 * hf, x);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        S[32 * hf + j] = fmaf(gC, S[32 * hf + j], x[j]);
                    st_half_row(sm + kSS, row, hf, S + 32 * hf);
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            tc::named_bar_sync(kBarChain, kChainThreads);
            if (tid == 0) {
                tc::mbar_arrive(&bars[kBAccFree + c % 3]);
                if (c + kNS < nchunks)   // stage free
                    tc::mbar_arrive(&bars[kBEmpty + s]);
            }
        }
        if (failed) {
            *vabort = 1;
            if (tid == 0) {   // drain own MMAs
                if (last_c1 >= 0)
                    tc::mbar_wait(&bars[kBC1], last_c1 & 1, 100000000ull);
                if (last_c2 >= 0)
                    tc::mbar_wait(&bars[kBC2], last_c2 & 1, 100000000ull);
            }
        }
    }

    if (tid == kC && !kCkpt) tc::tma_store_wait_all<0>();   // o written
    __syncthreads();
    if (*vabort) {
        if (tid == 0) {
            atomicOr(&g_fault_word2, 1u);
            const int n = *reinterpret_cast<volatile int*>(issued);
            for (int c = n - kNS < 0 ? 0 : n - kNS; c < n; ++c)
                tc::mbar_wait(&bars[kBFull + c % kNS], (c / kNS) & 1,
                              100000000ull);
        }
    } else if (tid < kChainThreads && p.hT) {
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

bool aligned16(const void* ptr) {
    return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0;
}

// [1, 64, H, 128] map standing for an all-zero V: every load of the kernel
// falls outside it (and reads zeros) except the first chunk of sequence 0,
// which reads the zero tile itself.
bool make_v_map(CUtensorMap* m, const FwdArgs& a) {
    return a.v_zero ? make_map(m, a.v, 1, kC, a.H)
                    : make_map(m, a.v, a.B, a.T, a.H);
}

cudaError_t set_smem(const void* kern, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load() & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit);
    return e;
}

std::atomic<unsigned long long> g_prep_attr[2], g_state_attr[3];

}  // namespace

size_t chunk_tc2_record_bytes(int B, int T, int H) {
    const size_t nch = ((size_t)T + kC - 1) / kC;
    return (size_t)B * H * nch * kRecBytes;
}

namespace {
size_t flag_bytes(int B, int T, int H) {
    const size_t nch = ((size_t)T + kC - 1) / kC;
    return ((size_t)B * H * nch * 4 + 15) / 16 * 16;
}
}  // namespace

size_t chunk_tc2_workspace_bytes(int B, int T, int H) {
    return chunk_tc2_record_bytes(B, T, H) + flag_bytes(B, T, H) +
           kCtrlWords * 4;
}

bool chunk_tc2_eligible(const FwdArgs& a) {
    return a.dtype == KLA_BF16 && a.dk == kD && a.dv == kD && a.C == kC &&
           (!a.kw || (aligned16(a.kw) && !a.ckpt)) && aligned16(a.q) &&
           aligned16(a.k) && aligned16(a.v) &&
           (!a.o || aligned16(a.o)) && (!a.h0 || aligned16(a.h0)) &&
           (!a.hT || aligned16(a.hT)) && get_encoder();
}

namespace {

// Chunk indices (of every head) the whole GPU prepares before SMs go to the
// state pass: the fewest such that the reserved SMs, producing the rest in
// order, stay ahead of the state pass.  The rates are GB300 measurements on
// the 1B and 340M layers (a pre-pass item takes ~9.5 us with five per SM;
// the state pass starts its chain ~6 us after its SMs are free and takes
// ~1.6 us per chunk); a sweep of the release point put the best times at
// 42 of 64 and 22 of 32 chunk indices, where this gives 43 and 22.  With
// write keys (four per SM) the same rates give 48 of 64 on the 1B layer,
// where a sweep put the best at 42-44 and 48 costs 2%: an item time of
// 7.1 us, fitted to that sweep rather than timed, gives 42.  A wrong
// estimate costs time, never correctness: the state pass waits for each
// flag.
int release_chunks(int nbh, int nchunks, int reserved_sms, int per_sm,
                   double item_us) {
    const double start_us = 6.0, chunk_us = 1.6;
    const double rate = reserved_sms * per_sm / item_us;   // items per us
    for (int kc = 0; kc < nchunks; ++kc) {
        bool ok = true;
        for (int j = kc; j < nchunks && ok; ++j)
            ok = (j - kc + 1) * nbh / rate <= start_us + chunk_us * j;
        if (ok) return kc;
    }
    return nchunks;
}

struct DeviceShape {
    int sms = 0, prep_per_sm = 0;
};

// SM count and resident pre-pass CTAs per SM of instantiation kKw.
template <bool kKw>
cudaError_t device_shape(DeviceShape* d) {
    static std::atomic<unsigned long long> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) {
        const unsigned long long v = cached[dev].load();
        if (v) {
            d->sms = (int)(v >> 32);
            d->prep_per_sm = (int)(v & 0xffffffffu);
            return cudaSuccess;
        }
    }
    e = cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // CTAs of the pre-pass resident per SM: five (four with write keys) by
    // construction (launch bounds, shared memory, TMEM), fewer if this
    // device's shared memory or register file holds fewer
    int smem_sm = 0;
    e = cudaDeviceGetAttribute(&smem_sm,
                               cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kla_prep_kernel<kKw>);
    if (e != cudaSuccess) return e;
    const int by_smem = smem_sm / (PrepMap<kKw>::Smem + 1024);
    const int by_regs = 65536 / (std::max(fa.numRegs, 1) * kPrepThreads);
    d->prep_per_sm =
        std::min(PrepMap<kKw>::PerSm, std::min(by_smem, by_regs));
    if (d->sms <= 0 || d->prep_per_sm <= 0) return cudaErrorInvalidValue;
    if (dev < 64)
        cached[dev].store(((unsigned long long)d->sms << 32) |
                          (unsigned)d->prep_per_sm);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_prep_tc2(const FwdArgs& a, void* ws, cudaStream_t stream,
                            int state_ctas) {
    if ((long)a.B * a.H == 0 || a.T == 0) return cudaSuccess;
    if (!get_encoder()) return cudaErrorNotSupported;
    if (!ws || !aligned16(ws)) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mkw;
    if (!make_map(&mq, a.q, a.B, a.T, a.H) ||
        !make_map(&mk, a.k, a.B, a.T, a.H) ||
        !make_map(&mkw, a.kw ? a.kw : a.k, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    if (a.kw && a.bwd_rec) return cudaErrorInvalidValue;   // forward only
    const int nchunks = (a.T + kC - 1) / kC;
    const long nbh = (long)a.B * a.H;
    const long items = nbh * nchunks;
    if (items > 0x7fffffffL) return cudaErrorInvalidValue;
    const bool kw = a.kw != nullptr;
    const void* kern = kw ? (const void*)kla_prep_kernel<true>
                          : (const void*)kla_prep_kernel<false>;
    cudaError_t e = set_smem(
        kern, kw ? PrepMap<true>::Smem : PrepMap<false>::Smem,
        g_prep_attr[kw ? 1 : 0]);
    if (e != cudaSuccess) return e;
    DeviceShape d;
    e = kw ? device_shape<true>(&d) : device_shape<false>(&d);
    if (e != cudaSuccess) return e;
    uint8_t* rec = static_cast<uint8_t*>(ws);
    unsigned int* ready = reinterpret_cast<unsigned int*>(
        rec + chunk_tc2_record_bytes(a.B, a.T, a.H));
    unsigned int* ctrl = reinterpret_cast<unsigned int*>(
        reinterpret_cast<uint8_t*>(ready) + flag_bytes(a.B, a.T, a.H));
    e = cudaMemsetAsync(ready, 0, flag_bytes(a.B, a.T, a.H) + kCtrlWords * 4,
                        stream);
    if (e != cudaSuccess) return e;
    // SMs left to the pre-pass once the state pass runs (when it leaves some)
    const int reserved = state_ctas > 0 && state_ctas < d.sms
                             ? d.sms - state_ctas
                             : 0;
    const long release =
        reserved ? nbh * release_chunks((int)nbh, nchunks, reserved,
                                        d.prep_per_sm, kw ? 7.1 : 9.5)
                 : items;
    const long grid = std::min(items, (long)d.sms * d.prep_per_sm);
    PrepParams pp{a.log_alpha, a.eta, rec, a.eps, a.gdn, a.T, a.H, nchunks,
                  a.bwd_rec, ready, ctrl, (int)items, (int)release,
                  reserved};
    if (kw)
        kla_prep_kernel<true><<<(unsigned)grid, kPrepThreads,
                                PrepMap<true>::Smem, stream>>>(mq, mk, mkw, pp);
    else
        kla_prep_kernel<false><<<(unsigned)grid, kPrepThreads,
                                 PrepMap<false>::Smem, stream>>>(mq, mk, mkw,
                                                                 pp);
    return cudaGetLastError();
}

const unsigned int* chunk_tc2_ready(const void* ws, int B, int T, int H) {
    return reinterpret_cast<const unsigned int*>(
        static_cast<const uint8_t*>(ws) + chunk_tc2_record_bytes(B, T, H));
}

int chunk_tc2_state_ctas(int B, int H) { return B * H * (kD / kNV); }

cudaError_t launch_state_tc2(const FwdArgs& a, const void* rec,
                             const unsigned int* ready, cudaStream_t stream) {
    if ((long)a.B * a.H == 0 || a.T == 0) return cudaSuccess;
    if (!get_encoder()) return cudaErrorNotSupported;
    if ((a.o == nullptr) == (a.ckpt == nullptr)) return cudaErrorInvalidValue;
    if (!rec || !aligned16(rec)) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, a.B, a.T, a.H) ||
        !make_map(&mk, a.k, a.B, a.T, a.H) || !make_v_map(&mv, a) ||
        !make_map(&mo, a.o ? a.o : a.q, a.B, a.T, a.H))
        return cudaErrorInvalidValue;
    if (a.kw && a.ckpt) return cudaErrorInvalidValue;   // forward only
    const int nchunks = (a.T + kC - 1) / kC;
    const int which = a.ckpt ? 1 : a.kw ? 2 : 0;
    auto kern = which == 1   ? kla_state_kernel<true, false>
                : which == 2 ? kla_state_kernel<false, true>
                             : kla_state_kernel<false, false>;
    cudaError_t e = set_smem((const void*)kern, kSSmem, g_state_attr[which]);
    if (e != cudaSuccess) return e;
    StateParams sp{a.h0, static_cast<__nv_bfloat16*>(a.o), a.hT, a.ckpt,
                   static_cast<const uint8_t*>(rec), a.T, a.H, nchunks,
                   2000000000ull, 0, ready,
                   static_cast<const __nv_bfloat16*>(a.kw)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long)a.B * a.H), kD / kNV);
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = kSSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ready ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, sp);
}

cudaError_t launch_chunk_tc2(const FwdArgs& a, void* workspace,
                             cudaStream_t stream) {
    if ((a.o == nullptr) == (a.ckpt == nullptr)) return cudaErrorInvalidValue;
    cudaError_t e = launch_prep_tc2(a, workspace, stream,
                                    chunk_tc2_state_ctas(a.B, a.H));
    if (e != cudaSuccess) return e;
    return launch_state_tc2(a, workspace,
                            chunk_tc2_ready(workspace, a.B, a.T, a.H), stream);
}

namespace {
// Device memory the self-test's tensor maps point at; never read (the
// self-test's producer issues no copy).
__device__ __align__(1024) uint8_t g_selftest_tile[64 * kD * 2];
}  // namespace

cudaError_t launch_state_selftest(cudaStream_t stream) {
    if (!get_encoder()) return cudaErrorNotSupported;
    void* base = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&base, g_selftest_tile);
    if (e != cudaSuccess) return e;
    CUtensorMap m;
    if (!make_map(&m, base, 1, kC, 1)) return cudaErrorInvalidValue;
    e = set_smem((const void*)kla_state_kernel<false, false>, kSSmem,
                 g_state_attr[0]);
    if (e != cudaSuccess) return e;
    // one CTA, one chunk; its waits give up after 1 ms
    StateParams sp{nullptr, static_cast<__nv_bfloat16*>(base), nullptr,
                   nullptr, static_cast<const uint8_t*>(base), kC, 1, 1,
                   1000000ull, 1, nullptr, nullptr};
    kla_state_kernel<false, false><<<dim3(1, 1), kStateThreads, kSSmem,
                                     stream>>>(
        m, m, m, m, sp);
    return cudaGetLastError();
}

cudaError_t read_and_clear_fault2(unsigned int* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_fault_word2,
                                         sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_fault_word2, &zero, sizeof(unsigned int));
}

}  // namespace kla
