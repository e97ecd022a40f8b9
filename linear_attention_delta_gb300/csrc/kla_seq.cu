// kla_chunk_fwd_seq: the forward pass of a few long sequences, split along
// the sequence so that more SMs work on each one.
//
// The recurrence is linear in the state, so a segment of a sequence maps its
// start state S_s to its end state Phi_s S_s + B_s and gives the outputs
// O0_s + O_hom,s S_s (one row per token), where B_s and O0_s come from the
// segment run from a zero state, and Phi_s and O_hom,s from the segment run
// from the identity with V = 0 (then S_t = Phi_t and o_t = Phi_t^T q_t).
// Both runs are the forward kernel itself, with the P segments of every
// sequence taken as P sequences of one batch ([B, T, H, d] is
// [B P, T / P, H, d]); on the two-kernel path they share one pre-pass and
// run at the same time as programmatic dependents on the caller's stream
// (on the fused kernel, on two streams).  A small
// kernel then chains the start states, S_{s+1} = Phi_s S_s + B_s, and a
// tensor-core kernel adds O_hom,s S_s to the outputs of every segment after
// the first (whose run started from the true initial state).  With one
// sequence the homogeneous run skips the first segment, whose Phi and O_hom
// are never used.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kla_internal.cuh"

namespace kla {

int device_sm_count() {
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev] &&
        cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount,
                               dev) != cudaSuccess)
        cached[dev] = 0;
    return cached[dev];
}

}  // namespace kla

namespace {

constexpr int kD = 128;            // dk = dv (tensor-core kernel)
constexpr int kC = 64;
constexpr int kMaxSegments = 8;
constexpr size_t kAlign = 256;

size_t round_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

// Byte layout of the workspace.
struct Layout {
    size_t h0s, hts, eye, phi, ohom, sst, zero, rec, total;
};

Layout layout(int B, int T, int H, int P) {
    Layout L;
    const size_t st = (size_t)B * P * H * kD * kD * sizeof(float);
    size_t off = 0;
    L.h0s = off; off += round_up(st);   // start states, zero-state run
    L.hts = off; off += round_up(st);   // end states, zero-state run
    L.eye = off; off += round_up(st);   // identity, homogeneous run
    L.phi = off; off += round_up(st);   // end states, homogeneous run
    L.ohom = off; off += round_up((size_t)B * T * H * kD * 2);
    L.sst = off; off += round_up((size_t)B * P * H * kD * kD * 2);
    L.zero = off; off += round_up((size_t)kC * H * kD * 2);
    // pre-pass records of the two-kernel tensor-core path, shared by the
    // two runs
    L.rec = off; off += round_up(kla::chunk_tc2_workspace_bytes(B * P, T / P, H));
    L.total = off;
    return L;
}

// Segments per sequence: as asked, or (0) the most, up to 8, for which the
// two concurrent runs (2 B H P CTAs each) still fit on the SMs at once.
int choose_segments(int B, int T, int H, int asked) {
    if (asked > 0) return asked;
    const int sms = kla::device_sm_count();
    int P = 1;
    while (2 * P <= kMaxSegments && 4L * B * H * (2 * P) <= sms &&
           T % (2 * P * kC) == 0)
        P *= 2;
    return P;
}

__global__ void set_identity(float* S, long n_mat) {
    const long total = n_mat * kD * kD;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
         i += (long)gridDim.x * blockDim.x) {
        const int e = (int)(i % (kD * kD));
        S[i] = (e / kD == e % kD) ? 1.f : 0.f;
    }
}

// Start states of the segments, one CTA per (b, h, 32 columns of dv):
// S_1 = end state of segment 0, S_{s+1} = Phi_s S_s + B_s.  Writes S_s
// (s >= 1) as a bf16 [dv][dk] operand and the final state.
constexpr int kCombCols = 32;
__global__ void __launch_bounds__(256)
chain_states(const float* __restrict__ hts, const float* __restrict__ phi,
             __nv_bfloat16* __restrict__ sst, float* __restrict__ hT, int P,
             int H) {
    __shared__ float S[kD][kCombCols + 1];
    __shared__ float Sn[kD][kCombCols + 1];
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int j0 = blockIdx.y * kCombCols;
    const int tid = threadIdx.x;
    auto mat = [&](const float* base, int s) {
        return base + (((size_t)(b * P + s) * H + h) * kD) * kD;
    };
    for (int i = tid; i < kD * kCombCols; i += 256) {
        const int r = i / kCombCols, c = i % kCombCols;
        S[r][c] = mat(hts, 0)[r * kD + j0 + c];
    }
    __syncthreads();
    for (int s = 1; s < P; ++s) {
        __nv_bfloat16* out = sst + (((size_t)(b * P + s) * H + h) * kD) * kD;
        for (int i = tid; i < kD * kCombCols; i += 256) {
            const int n = i / kD, kk = i % kD;   // [dv][dk]
            out[(size_t)(j0 + n) * kD + kk] = __float2bfloat16_rn(S[kk][n]);
        }
        const float* F = mat(phi, s);
        const float* Bs = mat(hts, s);
        // 4 rows x 4 columns per thread
        const int r0 = (tid / 8) * 4, c0 = (tid % 8) * 4;
        float acc[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y)
                acc[x][y] = Bs[(size_t)(r0 + x) * kD + j0 + c0 + y];
        for (int kk = 0; kk < kD; ++kk) {
            float f[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) f[x] = F[(size_t)(r0 + x) * kD + kk];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    acc[x][y] = fmaf(f[x], S[kk][c0 + y], acc[x][y]);
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) Sn[r0 + x][c0 + y] = acc[x][y];
        __syncthreads();
        for (int i = tid; i < kD * kCombCols; i += 256) {
            const int r = i / kCombCols, c = i % kCombCols;
            S[r][c] = Sn[r][c];
        }
        __syncthreads();
    }
    if (hT) {
        for (int i = tid; i < kD * kCombCols; i += 256) {
            const int r = i / kCombCols, c = i % kCombCols;
            hT[(((size_t)b * H + h) * kD + r) * kD + j0 + c] = S[r][c];
        }
    }
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4],
                                               const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// o[rows of segment s] += O_hom,s S_s.  One CTA takes a run of 128-row
// tiles of one (b, s >= 1, h): S_s is loaded once, and the next tiles of
// O_hom and o come in (cp.async, double-buffered) while the current ones
// are used; warp w forms rows 16 w .. 16 w + 15 of a tile, all 128 columns
// (m16n8k16, bf16 operands, fp32 accumulation), added to o in fp32 and
// rounded once in shared memory, and the tile goes back to o in 16-byte
// row pieces.
constexpr int kRows = 128;
constexpr int kLd = kD + 8;        // bf16 row stride: conflict-free fragments

__device__ __forceinline__ void cp_async16(void* dst, const void* src,
                                           bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(256, 1)
add_segment_start(__nv_bfloat16* __restrict__ o,
                  const __nv_bfloat16* __restrict__ ohom,
                  const __nv_bfloat16* __restrict__ sst, int T, int H, int P,
                  int tseg, int tiles_per_cta) {
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(smem);
    __nv_bfloat16* As0 = Bs + kD * kLd;                 // two O_hom tiles
    __nv_bfloat16* Os0 = As0 + 2 * kRows * kLd;         // two o tiles
    const int h = blockIdx.y;
    const int b = blockIdx.z / (P - 1), s = blockIdx.z % (P - 1) + 1;
    const int ntiles = (tseg + kRows - 1) / kRows;
    const int t_begin = blockIdx.x * tiles_per_cta;
    const int t_end = min(t_begin + tiles_per_cta, ntiles);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t row_stride = (size_t)H * kD;
    auto tok = [&](int r) { return (size_t)b * T + (size_t)s * tseg + r; };
    const int g = lane >> 2, q = lane & 3;
    const int ra = warp * 16 + g;

    auto load_tile = [&](int t, int buf) {
        for (int i = tid; i < kRows * (kD / 8); i += 256) {
            const int r = i / (kD / 8), c8 = i % (kD / 8);
            const int row = t * kRows + r;
            const bool valid = row < tseg;
            const size_t off =
                tok(valid ? row : 0) * row_stride + (size_t)h * kD + 8 * c8;
            cp_async16(As0 + (buf * kRows + r) * kLd + 8 * c8, ohom + off,
                       valid);
            cp_async16(Os0 + (buf * kRows + r) * kLd + 8 * c8, o + off, valid);
        }
    };
    const __nv_bfloat16* S =
        sst + (((size_t)(b * P + s) * H + h) * kD) * kD;   // [dv][dk]
    for (int i = tid; i < kD * (kD / 8); i += 256) {
        const int n = i / (kD / 8), c8 = i % (kD / 8);
        cp_async16(Bs + n * kLd + 8 * c8, S + (size_t)n * kD + 8 * c8, true);
    }
    if (t_begin < t_end) load_tile(t_begin, 0);
    cp_async_commit();

    for (int t = t_begin; t < t_end; ++t) {
        const int buf = (t - t_begin) & 1;
        const __nv_bfloat16* As = As0 + buf * kRows * kLd;
        __nv_bfloat16* Os = Os0 + buf * kRows * kLd;
        if (t + 1 < t_end)   // the next tiles into the other buffers
            load_tile(t + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();   // all but the group just committed
        __syncthreads();

        float acc[kD / 8][4];
#pragma unroll
        for (int nt = 0; nt < kD / 8; ++nt)
            acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            const int k0 = 16 * ks + 2 * q;
            uint32_t a[4];
            a[0] = *reinterpret_cast<const uint32_t*>(As + ra * kLd + k0);
            a[1] = *reinterpret_cast<const uint32_t*>(As + (ra + 8) * kLd + k0);
            a[2] = *reinterpret_cast<const uint32_t*>(As + ra * kLd + k0 + 8);
            a[3] =
                *reinterpret_cast<const uint32_t*>(As + (ra + 8) * kLd + k0 + 8);
#pragma unroll
            for (int nt = 0; nt < kD / 8; ++nt) {
                const __nv_bfloat16* bn = Bs + (8 * nt + g) * kLd + k0;
                mma_bf16_16816(acc[nt], a,
                               *reinterpret_cast<const uint32_t*>(bn),
                               *reinterpret_cast<const uint32_t*>(bn + 8));
            }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            __nv_bfloat162* orow = reinterpret_cast<__nv_bfloat162*>(
                Os + (ra + 8 * half) * kLd + 2 * q);
#pragma unroll
            for (int nt = 0; nt < kD / 8; ++nt) {
                const float2 o0 = __bfloat1622float2(orow[4 * nt]);
                orow[4 * nt] = __floats2bfloat162_rn(
                    o0.x + acc[nt][2 * half], o0.y + acc[nt][2 * half + 1]);
            }
        }
        __syncthreads();
        for (int i = tid; i < kRows * (kD / 8); i += 256) {
            const int r = i / (kD / 8), c8 = i % (kD / 8);
            const int row = t * kRows + r;
            if (row < tseg)
                *reinterpret_cast<uint4*>(o + tok(row) * row_stride +
                                          (size_t)h * kD + 8 * c8) =
                    *reinterpret_cast<const uint4*>(Os + r * kLd + 8 * c8);
        }
        __syncthreads();   // these buffers are refilled next iteration
    }
    cp_async_wait<0>();
}

constexpr size_t kAddSmem = 5 * (size_t)kRows * kLd * sizeof(__nv_bfloat16);

// Second stream and events of one device, created on first use.
struct Aux {
    bool ready = false;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_aux_mu;   // also serialises the enqueue of whole calls
Aux g_aux[64];

cudaError_t init_aux(Aux& a) {
    cudaError_t e = cudaStreamCreateWithFlags(&a.s, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(add_segment_start,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kAddSmem);
    if (e != cudaSuccess) {   // release what was made, so a retry starts clean
        if (a.join) cudaEventDestroy(a.join);
        if (a.fork) cudaEventDestroy(a.fork);
        if (a.s) cudaStreamDestroy(a.s);
        a = Aux{};
        return e;
    }
    a.ready = true;
    return cudaSuccess;
}

bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

extern "C" kla_status kla_chunk_fwd_seq_workspace_size(
    int B, int T, int H, int dk, int dv, int C, kla_dtype dtype,
    int segments, size_t* bytes) {
    if (!bytes || B < 0 || T < 0 || H < 0 || segments < 0)
        return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_BF16 || dk != kD || dv != kD || C != kC)
        return KLA_ERR_UNSUPPORTED_SHAPE;
    const int P = choose_segments(B, T, H, segments);
    if (P > kMaxSegments || T % (P * kC) != 0)
        return KLA_ERR_UNSUPPORTED_SHAPE;
    *bytes = ((long long)B * H == 0 || T == 0 || P == 1)
                 ? 0
                 : layout(B, T, H, P).total;
    return KLA_OK;
}

extern "C" kla_status kla_chunk_fwd_seq(
    const void* q, const void* k, const void* v, const float* log_alpha,
    const float* eta, float eps, const float* h0, void* o, float* hT, int B,
    int T, int H, int dk, int dv, int C, kla_dtype dtype, kla_step_rule rule,
    int segments, void* workspace, size_t workspace_bytes,
    kla_stream_t stream) {
    size_t need = 0;
    kla_status st = kla_chunk_fwd_seq_workspace_size(B, T, H, dk, dv, C,
                                                     dtype, segments, &need);
    if (st != KLA_OK) return st;
    if (rule != KLA_STEP_KACZMARZ && rule != KLA_STEP_GIVEN)
        return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return KLA_ERR_INVALID_ARG;
    const int P = choose_segments(B, T, H, segments);
    if ((long long)B * H == 0 || T == 0 || P == 1)   // nothing to split
        return kla_chunk_fwd_ex(q, k, v, log_alpha, eta, eps, h0, o, hT, B, T,
                                H, dk, dv, C, dtype, KLA_ALGO_TC_FUSED, rule,
                                stream);
    if (!q || !k || !v || !log_alpha || !eta || !o) return KLA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        !aligned16(log_alpha) || !aligned16(eta) || (h0 && !aligned16(h0)) ||
        (hT && !aligned16(hT)))
        return KLA_ERR_INVALID_ARG;
    if (o == q || o == k || o == v || o == (const void*)log_alpha ||
        o == (const void*)eta || o == (const void*)h0 || o == (void*)hT)
        return KLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return KLA_ERR_INVALID_ARG;
    if ((long long)B * P * H * 2 > 0x7fffffffLL) return KLA_ERR_UNSUPPORTED_SHAPE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return KLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_aux_mu);
    Aux& A = g_aux[dev];
    if (!A.ready && init_aux(A) != cudaSuccess) return KLA_ERR_CUDA;

    const Layout L = layout(B, T, H, P);
    char* ws = static_cast<char*>(workspace);
    float* h0s = reinterpret_cast<float*>(ws + L.h0s);
    float* hts = reinterpret_cast<float*>(ws + L.hts);
    float* eye = reinterpret_cast<float*>(ws + L.eye);
    float* phi = reinterpret_cast<float*>(ws + L.phi);
    __nv_bfloat16* ohom = reinterpret_cast<__nv_bfloat16*>(ws + L.ohom);
    __nv_bfloat16* sst = reinterpret_cast<__nv_bfloat16*>(ws + L.sst);
    void* zero = ws + L.zero;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t mat = (size_t)H * kD * kD * sizeof(float);
    const int tseg = T / P;
    const int gdn = rule == KLA_STEP_GIVEN ? 1 : 0;

#define KLA_TRY(x)                                   \
    do {                                             \
        if ((x) != cudaSuccess) return KLA_ERR_CUDA; \
    } while (0)

    // start states: segment 0 of each sequence from h0, the others from 0;
    // the homogeneous run from the identity; the all-zero V tile
    KLA_TRY(cudaMemsetAsync(h0s, 0, (size_t)B * P * mat, s));
    if (h0)
        for (int b = 0; b < B; ++b)
            KLA_TRY(cudaMemcpyAsync(
                reinterpret_cast<char*>(h0s) + (size_t)b * P * mat,
                reinterpret_cast<const char*>(h0) + (size_t)b * mat, mat,
                cudaMemcpyDeviceToDevice, s));
    KLA_TRY(cudaMemsetAsync(zero, 0, (size_t)kC * H * kD * 2, s));
    set_identity<<<kla::device_sm_count() * 4, 256, 0, s>>>(eye,
                                                            (long)B * P * H);
    KLA_TRY(cudaGetLastError());
    KLA_TRY(cudaEventRecord(A.fork, s));
    KLA_TRY(cudaStreamWaitEvent(A.s, A.fork, 0));

    // the two runs over B P sequences of T / P tokens, at the same time
    kla::FwdArgs zs{q, k, v, log_alpha, eta, eps, gdn, h0s, o, hts,
                    B * P, tseg, H, kD, kD, kC, KLA_BF16};
    kla::FwdArgs hom{q, k, zero, log_alpha, eta, eps, gdn, eye, ohom, phi,
                     B * P, tseg, H, kD, kD, kC, KLA_BF16};
    hom.v_zero = true;
    if (B == 1) {
        // segment 0 starts from the true initial state, so its homogeneous
        // run (Phi_0, O_hom,0) is never used: run segments 1 .. P-1 only,
        // which are contiguous when there is one sequence
        const size_t tok = (size_t)tseg * H;
        hom.q = static_cast<const __nv_bfloat16*>(q) + tok * kD;
        hom.k = static_cast<const __nv_bfloat16*>(k) + tok * kD;
        hom.log_alpha = log_alpha + tok;
        hom.eta = eta + tok;
        hom.h0 = eye + (size_t)H * kD * kD;
        hom.o = ohom + tok * kD;
        hom.hT = phi + (size_t)H * kD * kD;
        hom.B = P - 1;
    }
    if (kla::chunk_tc2_eligible(zs)) {
        // one pre-pass over all B P segments, then the two state passes on
        // the same stream, each a programmatic dependent of the launch
        // before it, so that both run beside the pre-pass's last chunks and
        // read each record once its flag is up; with B = 1 the homogeneous
        // run starts at segment 1's records and flags
        char* rec = ws + L.rec;
        const unsigned int* ready = kla::chunk_tc2_ready(rec, B * P, tseg, H);
        const size_t seg1 = B == 1 ? (size_t)H * (tseg / kC) : 0;
        KLA_TRY(kla::launch_prep_tc2(
            zs, rec, s,
            kla::chunk_tc2_state_ctas(zs.B, H) +
                kla::chunk_tc2_state_ctas(hom.B, H)));
        KLA_TRY(kla::launch_state_tc2(zs, rec, ready, s));
        KLA_TRY(kla::launch_state_tc2(
            hom, rec + seg1 * kla::chunk_tc2_record_bytes(1, kC, 1),
            ready + seg1, s));
    } else {
        if (!kla::chunk_tc_eligible(zs)) return KLA_ERR_UNSUPPORTED_SHAPE;
        KLA_TRY(kla::launch_chunk_tc(zs, s));
        KLA_TRY(kla::launch_chunk_tc(hom, A.s));
    }
    KLA_TRY(cudaEventRecord(A.join, A.s));
    KLA_TRY(cudaStreamWaitEvent(s, A.join, 0));

    // chain the start states, then add O_hom S to the later segments
    chain_states<<<dim3((unsigned)(B * H), kD / kCombCols), 256, 0, s>>>(
        hts, phi, sst, hT, P, H);
    KLA_TRY(cudaGetLastError());
    // runs of tiles: about four waves of one CTA per SM
    const int ntiles = (tseg + kRows - 1) / kRows;
    const long all_tiles = (long)ntiles * H * B * (P - 1);
    const long slots = kla::device_sm_count();
    const int per_cta =
        (int)std::max(1L, std::min((long)ntiles, (all_tiles + 4 * slots - 1) /
                                                     (4 * slots)));
    add_segment_start<<<dim3((unsigned)((ntiles + per_cta - 1) / per_cta),
                             (unsigned)H, (unsigned)(B * (P - 1))),
                        256, kAddSmem, s>>>(
        static_cast<__nv_bfloat16*>(o), ohom, sst, T, H, P, tseg, per_cta);
    KLA_TRY(cudaGetLastError());
#undef KLA_TRY
    return KLA_OK;
}
