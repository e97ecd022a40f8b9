// kla_chunk_fwd_host: the forward pass from host memory to host memory, with
// the host<->device copies overlapped with the kernels.
//
// The sequence is cut into segments of whole chunks.  While the kernel runs
// segment i on the caller's stream, one copy stream brings segment i+1's
// inputs in and another takes segment i-1's output back; two device buffers
// per tensor alternate between segments.  Each segment's kernel starts from
// the fp32 state the previous one ended with, exactly as the state is
// carried from chunk to chunk inside one launch, so the result is that of
// kla_chunk_fwd_ex on the whole sequence.  The forward's own workspace (the
// pre-pass records of the two-kernel tensor-core path) is part of this
// call's workspace, so nothing is allocated.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kla_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 2;          // device buffers per tensor
constexpr int kMaxSegments = 8;
constexpr size_t kAlign = 256;

// Copy streams and events of one device, created on first use.
struct Pipe {
    bool ready = false;
    size_t max_pitch = 0;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, fin = nullptr;
    cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {},
                out_done[kSlots] = {};
};
std::mutex g_pipe_mu;   // also serialises the enqueue of whole calls
Pipe g_pipe[kMaxDevices];

// Releases whatever a failed init_pipe created (so that a retry starts
// clean).
void release_pipe(Pipe& p) {
    cudaEvent_t* ev[] = {&p.start, &p.fin, &p.in_done[0], &p.in_done[1],
                         &p.comp_done[0], &p.comp_done[1], &p.out_done[0],
                         &p.out_done[1]};
    for (cudaEvent_t* e : ev)
        if (*e) { cudaEventDestroy(*e); *e = nullptr; }
    if (p.in) { cudaStreamDestroy(p.in); p.in = nullptr; }
    if (p.out) { cudaStreamDestroy(p.out); p.out = nullptr; }
}

cudaError_t init_pipe(Pipe& p, int dev) {
    static_assert(kSlots == 2, "release_pipe lists two slots");
    int pitch = 0;
    cudaError_t e = cudaDeviceGetAttribute(&pitch, cudaDevAttrMaxPitch, dev);
    if (e != cudaSuccess) return e;
    p.max_pitch = (size_t)(unsigned)pitch;
    const unsigned sf = cudaStreamNonBlocking;
    const unsigned ef = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&p.in, sf)) == cudaSuccess &&
        (e = cudaStreamCreateWithFlags(&p.out, sf)) == cudaSuccess &&
        (e = cudaEventCreateWithFlags(&p.start, ef)) == cudaSuccess &&
        (e = cudaEventCreateWithFlags(&p.fin, ef)) == cudaSuccess) {
        for (int j = 0; j < kSlots && e == cudaSuccess; ++j) {
            if ((e = cudaEventCreateWithFlags(&p.in_done[j], ef)) ==
                    cudaSuccess &&
                (e = cudaEventCreateWithFlags(&p.comp_done[j], ef)) ==
                    cudaSuccess)
                e = cudaEventCreateWithFlags(&p.out_done[j], ef);
        }
    }
    if (e != cudaSuccess) {
        release_pipe(p);
        return e;
    }
    p.ready = true;
    return cudaSuccess;
}

size_t round_up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

// Segment length in tokens (a multiple of C) and segment count.
void segments(int T, int C, int* tseg, int* nseg) {
    const int nch = (T + C - 1) / C;
    const int per = (nch + kMaxSegments - 1) / kMaxSegments;   // chunks
    *tseg = per * C;
    *nseg = nch == 0 ? 0 : (nch + per - 1) / per;
}

// Byte layout of the workspace: per slot q | k | v | log_alpha | eta | o,
// then two fp32 states, then the forward's own workspace for one segment
// (the segments' kernels run one after another on the caller's stream).
struct Layout {
    size_t q, k, v, g, o, slot, state, fwd, total;
};

Layout layout(int B, int tseg, int H, int dk, int dv, int C,
              kla_dtype dtype) {
    Layout L;
    const size_t esz = dtype == KLA_BF16 ? 2 : 4;
    const size_t rows = (size_t)B * tseg * H;
    L.q = round_up(rows * dk * esz);
    L.k = L.q;
    L.v = round_up(rows * dv * esz);
    L.g = round_up(rows * sizeof(float));
    L.o = L.v;
    L.slot = L.q + L.k + L.v + 2 * L.g + L.o;
    L.state = round_up((size_t)B * H * dk * dv * sizeof(float));
    size_t fwd = 0;
    kla_chunk_fwd_workspace_size(B, tseg, H, dk, dv, C, dtype, KLA_ALGO_AUTO,
                                 &fwd);
    L.fwd = round_up(fwd);
    L.total = kSlots * L.slot + 2 * L.state + L.fwd;
    return L;
}

// B rows of `width` bytes, `src_pitch` apart on the source and `dst_pitch`
// apart on the destination: one 2D copy, or one copy per row when a pitch
// is beyond the device's limit.
cudaError_t copy_rows(void* dst, size_t dst_pitch, const void* src,
                      size_t src_pitch, size_t width, int rows,
                      cudaMemcpyKind kind, cudaStream_t s, size_t max_pitch) {
    if (width == 0 || rows == 0) return cudaSuccess;
    if (rows == 1)
        return cudaMemcpyAsync(dst, src, width, kind, s);
    if (dst_pitch <= max_pitch && src_pitch <= max_pitch)
        return cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, width,
                                 (size_t)rows, kind, s);
    for (int r = 0; r < rows; ++r) {
        cudaError_t e = cudaMemcpyAsync(
            static_cast<char*>(dst) + (size_t)r * dst_pitch,
            static_cast<const char*>(src) + (size_t)r * src_pitch, width,
            kind, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool supported_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool valid_sizes(int dk, int dv, int C) {
    return supported_dim(dk) && supported_dim(dv) &&
           (C == 16 || C == 32 || C == 64);
}

}  // namespace

extern "C" kla_status kla_chunk_fwd_host_workspace_size(
    int B, int T, int H, int dk, int dv, int C, kla_dtype dtype,
    size_t* bytes) {
    if (!bytes || B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || C <= 0)
        return KLA_ERR_INVALID_ARG;
    if (dtype != KLA_F32 && dtype != KLA_BF16) return KLA_ERR_INVALID_ARG;
    if (!valid_sizes(dk, dv, C)) return KLA_ERR_UNSUPPORTED_SHAPE;
    int tseg = 0, nseg = 0;
    segments(T, C, &tseg, &nseg);
    *bytes = (long long)B * H == 0 ? 0
                                   : layout(B, tseg, H, dk, dv, C, dtype).total;
    return KLA_OK;
}

extern "C" kla_status kla_chunk_fwd_host(
    const void* q, const void* k, const void* v, const float* log_alpha,
    const float* eta, float eps, const float* h0, void* o, float* hT, int B,
    int T, int H, int dk, int dv, int C, kla_dtype dtype, kla_algo algo,
    kla_step_rule rule, void* workspace, size_t workspace_bytes,
    kla_stream_t stream) {
    size_t need = 0;
    kla_status st =
        kla_chunk_fwd_host_workspace_size(B, T, H, dk, dv, C, dtype, &need);
    if (st != KLA_OK) return st;
    if (algo != KLA_ALGO_AUTO && algo != KLA_ALGO_SIMT &&
        algo != KLA_ALGO_TC && algo != KLA_ALGO_TC_FUSED)
        return KLA_ERR_INVALID_ARG;
    if (rule != KLA_STEP_KACZMARZ && rule != KLA_STEP_GIVEN)
        return KLA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return KLA_ERR_INVALID_ARG;
    if ((long long)B * H == 0) return KLA_OK;
    if (!workspace || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return KLA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !log_alpha || !eta || !o))
        return KLA_ERR_INVALID_ARG;
    if (T > 0 && (o == q || o == k || o == v ||
                  o == (const void*)log_alpha || o == (const void*)eta))
        return KLA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return KLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    Pipe& P = g_pipe[dev];
    if (!P.ready && init_pipe(P, dev) != cudaSuccess) return KLA_ERR_CUDA;

    int tseg = 0, nseg = 0;
    segments(T, C, &tseg, &nseg);
    const size_t esz = dtype == KLA_BF16 ? 2 : 4;
    const Layout L = layout(B, tseg, H, dk, dv, C, dtype);
    char* ws = static_cast<char*>(workspace);
    float* state[2] = {reinterpret_cast<float*>(ws + kSlots * L.slot),
                       reinterpret_cast<float*>(ws + kSlots * L.slot + L.state)};
    void* fwd_ws = L.fwd ? ws + kSlots * L.slot + 2 * L.state : nullptr;
    const size_t state_bytes = (size_t)B * H * dk * dv * sizeof(float);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t mp = P.max_pitch;

#define KLA_TRY(x)                                  \
    do {                                            \
        if ((x) != cudaSuccess) return KLA_ERR_CUDA; \
    } while (0)

    // the copy streams start after the caller's earlier work on `s`
    KLA_TRY(cudaEventRecord(P.start, s));
    KLA_TRY(cudaStreamWaitEvent(P.in, P.start, 0));
    KLA_TRY(cudaStreamWaitEvent(P.out, P.start, 0));

    if (T == 0) {   // hT = h0 (or zero) through the device
        if (hT) {
            if (h0)
                KLA_TRY(cudaMemcpyAsync(state[0], h0, state_bytes,
                                        cudaMemcpyHostToDevice, s));
            else
                KLA_TRY(cudaMemsetAsync(state[0], 0, state_bytes, s));
            KLA_TRY(cudaMemcpyAsync(hT, state[0], state_bytes,
                                    cudaMemcpyDeviceToHost, s));
        }
        return KLA_OK;
    }

    // segment 0 reads its initial state from state[1]
    if (h0)
        KLA_TRY(cudaMemcpyAsync(state[1], h0, state_bytes,
                                cudaMemcpyHostToDevice, P.in));

    const size_t qrow = (size_t)H * dk * esz;   // bytes per token, q and k
    const size_t vrow = (size_t)H * dv * esz;   // v and o
    const size_t grow = (size_t)H * sizeof(float);
    for (int i = 0; i < nseg; ++i) {
        const int j = i % kSlots;
        const int t0 = i * tseg;
        const int tn = T - t0 < tseg ? T - t0 : tseg;
        char* slot = ws + j * L.slot;
        char* dq = slot;
        char* dk_ = dq + L.q;
        char* dvv = dk_ + L.k;
        char* dla = dvv + L.v;
        char* det = dla + L.g;
        char* dout = det + L.g;

        // inputs of segment i (slot j free once segment i-2's kernel is done)
        if (i >= kSlots) KLA_TRY(cudaStreamWaitEvent(P.in, P.comp_done[j], 0));
        const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
        KLA_TRY(copy_rows(dq, tn * qrow, static_cast<const char*>(q) + t0 * qrow,
                          (size_t)T * qrow, tn * qrow, B, h2d, P.in, mp));
        KLA_TRY(copy_rows(dk_, tn * qrow, static_cast<const char*>(k) + t0 * qrow,
                          (size_t)T * qrow, tn * qrow, B, h2d, P.in, mp));
        KLA_TRY(copy_rows(dvv, tn * vrow, static_cast<const char*>(v) + t0 * vrow,
                          (size_t)T * vrow, tn * vrow, B, h2d, P.in, mp));
        KLA_TRY(copy_rows(dla, tn * grow,
                          reinterpret_cast<const char*>(log_alpha) + t0 * grow,
                          (size_t)T * grow, tn * grow, B, h2d, P.in, mp));
        KLA_TRY(copy_rows(det, tn * grow,
                          reinterpret_cast<const char*>(eta) + t0 * grow,
                          (size_t)T * grow, tn * grow, B, h2d, P.in, mp));
        KLA_TRY(cudaEventRecord(P.in_done[j], P.in));

        // the kernel of segment i (its o buffer free once segment i-2's
        // output has gone back)
        KLA_TRY(cudaStreamWaitEvent(s, P.in_done[j], 0));
        if (i >= kSlots) KLA_TRY(cudaStreamWaitEvent(s, P.out_done[j], 0));
        const float* sin = i == 0 ? (h0 ? state[1] : nullptr)
                                  : state[(i - 1) % 2];
        st = kla_chunk_fwd_ws(dq, dk_, dvv, reinterpret_cast<float*>(dla),
                              reinterpret_cast<float*>(det), eps, sin, dout,
                              state[i % 2], B, tn, H, dk, dv, C, dtype, algo,
                              rule, fwd_ws, L.fwd, stream);
        if (st != KLA_OK) return st;
        KLA_TRY(cudaEventRecord(P.comp_done[j], s));

        // o of segment i back to the host
        KLA_TRY(cudaStreamWaitEvent(P.out, P.comp_done[j], 0));
        KLA_TRY(copy_rows(static_cast<char*>(o) + t0 * vrow, (size_t)T * vrow,
                          dout, tn * vrow, tn * vrow, B,
                          cudaMemcpyDeviceToHost, P.out, mp));
        KLA_TRY(cudaEventRecord(P.out_done[j], P.out));
    }
    if (hT)
        KLA_TRY(cudaMemcpyAsync(hT, state[(nseg - 1) % 2], state_bytes,
                                cudaMemcpyDeviceToHost, P.out));
    // everything of this call is ordered before later work on `s`
    KLA_TRY(cudaEventRecord(P.fin, P.out));
    KLA_TRY(cudaStreamWaitEvent(s, P.fin, 0));
#undef KLA_TRY
    return KLA_OK;
}
