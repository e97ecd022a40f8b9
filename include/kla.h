/*
 * kla.h -- C ABI of libkla.so: Kaczmarz Linear Attention (KLA) on GB300
 * (sm_103a).
 *
 * The operation (gist.science/es/paper/2605.08587, "Atencion Lineal
 * Kaczmarz", sections "Derivacion Teorica" and "La Regla de Actualizacion
 * KLA"; the German and French versions carry the same formulas):
 *
 *   for every (batch b, head h), starting from S_0 = h0[b,h] (dk x dv, fp32):
 *     S~_{t-1} = alpha_t S_{t-1},          alpha_t = exp(log_alpha_t)
 *     beta_t   = eta_t / (||k_t||_2^2 + eps)   (beta_t = 0 if the denominator
 *                                                is exactly 0)
 *     e_t      = v_t - S~_{t-1}^T k_t
 *     S_t      = S~_{t-1} + beta_t k_t e_t^T
 *     o_t      = S_t^T q_t
 *
 * The page names a "decayed previous state" without a formula; this library
 * reads it as the scalar gate above, applied before the residual.  The
 * read-out o_t = S_t^T q_t (after the write, no 1/sqrt(dk) scale) is likewise
 * this library's reading; a caller wanting a scale pre-scales q.
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library keeps no pointer after a call returns.  It allocates no device
 *     memory, with two exceptions stated at the entry points: the forward
 *     pass without a workspace argument takes stream-ordered scratch for its
 *     tensor-core path (kla_chunk_fwd_ws avoids that), and
 *     kla_chunk_bwd_noalloc owns a fixed device array.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *     A status other than KLA_OK means nothing was launched (argument errors
 *     are detected on the host before any launch) or that the launch itself
 *     failed (KLA_ERR_CUDA).  Faults during execution surface at the caller's
 *     next synchronisation, as with any CUDA call; bounded device-side waits
 *     that give up are reported by kla_device_status().
 *   - No C++ exception crosses this interface.
 *   - Tensors are contiguous and row-major.  Pointers to bf16 data must be
 *     2-byte aligned and pointers to fp32 data 4-byte aligned; the tensor-core
 *     forward path additionally wants 16-byte aligned q, k, v, o (it falls
 *     back to the CUDA-core path otherwise, see kla_chunk_fwd_ex).
 */
#ifndef KLA_H
#define KLA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KLA_API __attribute__((visibility("default")))
#else
#define KLA_API
#endif

typedef enum {
    KLA_OK = 0,
    KLA_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad enum */
    KLA_ERR_UNSUPPORTED_SHAPE = -2, /* (dk, dv, C, dtype) outside the set   */
    KLA_ERR_CUDA = -3,              /* a CUDA runtime call failed            */
    KLA_ERR_TIMEOUT = -4,           /* a bounded device-side wait gave up    */
    KLA_ERR_NOT_IMPLEMENTED = -5    /* requested variant is not available    */
} kla_status;

/* Element type of q, k, v and o.  log_alpha, eta, the states h0/hT/S and all
 * internal accumulation are always fp32. */
typedef enum { KLA_F32 = 0, KLA_BF16 = 1 } kla_dtype;

/* Forward-pass kernel selection for kla_chunk_fwd_ex / kla_chunk_fwd_ws. */
typedef enum {
    KLA_ALGO_AUTO = 0,   /* tensor-core path when eligible, else CUDA cores */
    KLA_ALGO_SIMT = 1,   /* fp32 CUDA-core chunkwise kernel (any supported shape) */
    KLA_ALGO_TC = 2,     /* tcgen05 tensor cores, two kernels: a chunk-parallel
                            pre-pass and the sequential state pass, which
                            starts on the SMs the pre-pass releases and reads
                            each record once it is written (bf16, dk = dv =
                            128, C = 64; needs a workspace) */
    KLA_ALGO_TC_FUSED = 3 /* tcgen05 tensor cores, one fused kernel per
                            (batch, head, dv half) (same shapes; no workspace) */
} kla_algo;

/* How the write step beta_t is formed from eta_t.
 *   KLA_STEP_KACZMARZ: beta_t = eta_t / (||k_t||^2 + eps)  (the KLA rule)
 *   KLA_STEP_GIVEN:    beta_t = eta_t, eps ignored  (the learned scalar step of
 *                      gated DeltaNet, the rule KLA replaces -- page section
 *                      "Declaracion del Problema"; same recurrence and block
 *                      solver otherwise, section "Implementacion") */
typedef enum { KLA_STEP_KACZMARZ = 0, KLA_STEP_GIVEN = 1 } kla_step_rule;

/* Opaque stream handle; ABI-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* kla_stream_t;

/*
 * kla_chunk_fwd -- full forward pass (prefill) over T tokens, evaluated in the
 * chunkwise-parallel form (section "Implementacion" of the page: the block
 * solver of gated DeltaNet with the diagonal B = Diag(beta_1..beta_C) as the
 * only change).  The result equals the token-by-token recurrence above up to
 * floating-point rounding; C only changes how the work is blocked.
 *
 *   q, k       [B, T, H, dk]  dtype        (read)
 *   v          [B, T, H, dv]  dtype        (read)
 *   log_alpha  [B, T, H]      fp32, <= 0   (read) per-token log decay
 *   eta        [B, T, H]      fp32         (read) relaxation gate
 *   eps        scalar >= 0                 stabiliser added to ||k||^2
 *   h0         [B, H, dk, dv] fp32, row index = key dim; NULL -> zero state
 *   o          [B, T, H, dv]  dtype        (written)
 *   hT         [B, H, dk, dv] fp32 final state; NULL -> not written
 *   C          chunk length
 *
 * Supported: dk, dv in {16, 32, 64, 128}; C in {16, 32, 64}; any T >= 0
 * (a ragged last chunk is handled in-kernel); B, H >= 0.  T == 0 copies h0
 * (or zeros) to hT.  o must not overlap any input or hT, and hT must not
 * overlap any input other than h0, which it may equal exactly (byte ranges
 * from the sizes; KLA_ERR_INVALID_ARG otherwise).
 * Errors: KLA_ERR_INVALID_ARG (null required pointer, negative size,
 * eps < 0 or not finite, bad dtype), KLA_ERR_UNSUPPORTED_SHAPE, KLA_ERR_CUDA.
 */
KLA_API kla_status kla_chunk_fwd(const void* q, const void* k, const void* v,
                         const float* log_alpha, const float* eta, float eps,
                         const float* h0, void* o, float* hT,
                         int B, int T, int H, int dk, int dv, int C,
                         kla_dtype dtype, kla_stream_t stream);

/*
 * kla_chunk_fwd_ex -- kla_chunk_fwd with an explicit kernel choice and step
 * rule.  KLA_ALGO_TC and KLA_ALGO_TC_FUSED return KLA_ERR_UNSUPPORTED_SHAPE
 * unless dtype == KLA_BF16, dk == dv == 128, C == 64 and q, k, v, o, h0, hT
 * are 16-byte aligned.  An unknown algo or rule is KLA_ERR_INVALID_ARG.
 *
 * KLA_ALGO_AUTO takes the two-kernel tensor-core path (KLA_ALGO_TC) where it
 * is eligible, the faster one on GB300.  That path writes per-chunk
 * intermediates between its two kernels:
 * kla_chunk_fwd and kla_chunk_fwd_ex take that scratch
 * (kla_chunk_fwd_workspace_size bytes) with cudaMallocAsync on `stream` from
 * the device's current memory pool and release it with cudaFreeAsync after
 * the kernels, both stream-ordered; a failure there is KLA_ERR_CUDA.  A pool
 * that returns freed memory to the device at every synchronization (the
 * default release threshold) maps it anew at the next call: on GB300 that
 * cost ~0.14 ms per synchronized call of the 1B layer, more than half the
 * forward itself.  kla_chunk_fwd_ws with a caller-owned workspace avoids it.
 */
KLA_API kla_status kla_chunk_fwd_ex(const void* q, const void* k, const void* v,
                            const float* log_alpha, const float* eta,
                            float eps, const float* h0, void* o, float* hT,
                            int B, int T, int H, int dk, int dv, int C,
                            kla_dtype dtype, kla_algo algo,
                            kla_step_rule rule, kla_stream_t stream);

/*
 * kla_chunk_fwd_workspace_size -- bytes of device workspace kla_chunk_fwd_ws
 * needs with this algorithm: for bf16, dk = dv = 128, C = 64 and KLA_ALGO_TC
 * or KLA_ALGO_AUTO, the pre-pass records of the two-kernel tensor-core path
 * (16,640 bytes per (batch, head, chunk of 64 tokens)), one 4-byte ready
 * flag per record (rounded up to 16 bytes in all) and 528 bytes of the
 * pre-pass's work counters; 0 otherwise (those paths need none).  Errors:
 * KLA_ERR_INVALID_ARG (null `bytes`, negative size, bad enum),
 * KLA_ERR_UNSUPPORTED_SHAPE (dk, dv or C outside the set).
 */
KLA_API kla_status kla_chunk_fwd_workspace_size(int B, int T, int H, int dk,
                                                int dv, int C,
                                                kla_dtype dtype,
                                                kla_algo algo, size_t* bytes);

/*
 * kla_chunk_fwd_ws -- kla_chunk_fwd_ex with a caller-provided workspace, so
 * that the library allocates nothing: device memory of at least
 * kla_chunk_fwd_workspace_size(...) bytes, 16-byte aligned, overlapping no
 * argument, owned by the caller; its contents on entry do not matter.  Calls
 * that share a workspace must be ordered (the same stream does it).  When
 * the size is 0 the workspace may be NULL; when the call takes another path
 * (e.g. misaligned tensors) the workspace is not touched.  Errors: as for
 * kla_chunk_fwd_ex, plus KLA_ERR_INVALID_ARG for a missing, small,
 * misaligned or overlapping workspace.
 */
KLA_API kla_status kla_chunk_fwd_ws(const void* q, const void* k,
                                    const void* v, const float* log_alpha,
                                    const float* eta, float eps,
                                    const float* h0, void* o, float* hT,
                                    int B, int T, int H, int dk, int dv, int C,
                                    kla_dtype dtype, kla_algo algo,
                                    kla_step_rule rule, void* workspace,
                                    size_t workspace_bytes,
                                    kla_stream_t stream);

/*
 * kla_chunk_fwd_seq_workspace_size -- bytes of device workspace
 * kla_chunk_fwd_seq needs: fp32 start and end states of the 2 x B x P
 * segment runs (4 tensors [B, P, H, 128, 128]), O_hom [B, T, H, 128] bf16,
 * the bf16 start states [B, P, H, 128, 128], a [64, H, 128] bf16 zero
 * tile and the two-kernel path's pre-pass workspace over all B P segments
 * (kla_chunk_fwd_workspace_size of B P sequences of T / P tokens), each
 * rounded up to 256 bytes; 0 when
 * there is nothing to split.  segments = 0 picks P as
 * kla_chunk_fwd_seq does (for the current device).  Errors:
 * KLA_ERR_INVALID_ARG (null `bytes`, negative size or segments),
 * KLA_ERR_UNSUPPORTED_SHAPE (not bf16 with dk = dv = 128 and C = 64, P > 8,
 * or T not a multiple of 64 P).
 */
KLA_API kla_status kla_chunk_fwd_seq_workspace_size(int B, int T, int H,
                                                    int dk, int dv, int C,
                                                    kla_dtype dtype,
                                                    int segments,
                                                    size_t* bytes);

/*
 * kla_chunk_fwd_seq -- kla_chunk_fwd_ex (tensor-core kernel) for a few long
 * sequences, split into P segments per sequence so that more SMs work on
 * each.  The recurrence is linear in the state: segment s maps its start
 * state S_s to Phi_s S_s + B_s and gives the outputs O0_s + O_hom,s S_s,
 * with B_s, O0_s from the segment run from a zero state and Phi_s, O_hom,s
 * from the run from the identity with V = 0.  Both runs are the two-kernel
 * tensor-core forward over the B P segments: one pre-pass (its records
 * depend on q, k and the gates only) serves the two state passes, which
 * follow it on `stream` as programmatic dependents, so that both run at
 * once and beside the pre-pass, reading each record once it is written
 * (with B = 1 the second run skips segment 0, whose Phi and O_hom are not
 * needed); a small kernel chains S_{s+1} =
 * Phi_s S_s + B_s and a tensor-core kernel adds O_hom,s S_s to o of every
 * segment after the first.  The pages have no counterpart: it reorders the
 * sums of the chunkwise form, so o and hT equal kla_chunk_fwd_ex's up to
 * rounding (O_hom and S_s enter the last product in bf16), not bit for
 * bit.
 *
 *   q .. hT, eps, B .. C, dtype, rule: as for kla_chunk_fwd_ex (device
 *                  memory, 16-byte aligned)
 *   segments       P >= 1, or 0 to take the most segments (up to 8, T a
 *                  multiple of 64 P) for which the two runs' 4 B H P CTAs
 *                  fit on the device's SMs at once; P = 1 is
 *                  kla_chunk_fwd_ex with KLA_ALGO_TC_FUSED
 *   workspace      device memory of at least
 *                  kla_chunk_fwd_seq_workspace_size(...) bytes, 256-byte
 *                  aligned, owned by the caller; contents on entry do not
 *                  matter
 *
 * Asynchronous on `stream`; all of the call's work is ordered before later
 * work on `stream`.  The library's second stream and its two events per
 * device are created on the first call on that device and kept; calls on
 * one device are enqueued one at a time.  Errors: as for kla_chunk_fwd_ex,
 * plus KLA_ERR_UNSUPPORTED_SHAPE (as for the workspace size) and
 * KLA_ERR_INVALID_ARG for a missing, small or misaligned workspace.
 */
KLA_API kla_status kla_chunk_fwd_seq(const void* q, const void* k,
                                     const void* v, const float* log_alpha,
                                     const float* eta, float eps,
                                     const float* h0, void* o, float* hT,
                                     int B, int T, int H, int dk, int dv,
                                     int C, kla_dtype dtype,
                                     kla_step_rule rule, int segments,
                                     void* workspace, size_t workspace_bytes,
                                     kla_stream_t stream);

/*
 * kla_chunk_fwd_host_workspace_size -- bytes of device workspace
 * kla_chunk_fwd_host needs for these sizes: two buffers of every per-token
 * tensor for one segment of the sequence (at most 8 segments of whole
 * chunks), two fp32 states [B, H, dk, dv] and the forward's workspace for
 * one segment (kla_chunk_fwd_workspace_size with KLA_ALGO_AUTO).  Writes 0
 * when B * H == 0.
 * Errors: KLA_ERR_INVALID_ARG (null `bytes`, negative size, bad dtype),
 * KLA_ERR_UNSUPPORTED_SHAPE (dk, dv or C outside the supported set).
 */
KLA_API kla_status kla_chunk_fwd_host_workspace_size(int B, int T, int H,
                                                     int dk, int dv, int C,
                                                     kla_dtype dtype,
                                                     size_t* bytes);

/*
 * kla_chunk_fwd_host -- kla_chunk_fwd_ex from host memory to host memory:
 * q, k, v, log_alpha, eta, h0 are read from, and o, hT written to, host
 * buffers with the layouts of kla_chunk_fwd.  The pages have no counterpart;
 * it is the library's way of overlapping the host<->device copies with the
 * kernels.  The sequence is cut into segments of whole chunks (at most 8);
 * while the kernel runs segment i on `stream`, a copy stream of the library
 * brings segment i+1's inputs to the device and another takes segment
 * i-1's o back.  Each segment's kernel starts from the fp32 state the
 * previous one ended with, so o and hT are bit-identical to those of
 * kla_chunk_fwd_ex on device copies of the same inputs.
 *
 *   q .. hT, eps, B .. C, dtype, algo, rule: as for kla_chunk_fwd_ex, host
 *                  pointers (page-locked memory for the copies to overlap;
 *                  pageable memory works, without the overlap)
 *   workspace      device memory of at least
 *                  kla_chunk_fwd_host_workspace_size(...) bytes, 256-byte
 *                  aligned, owned by the caller; contents on entry do not
 *                  matter
 *
 * Asynchronous: returns once everything is enqueued; o and hT are valid
 * after `stream` has been synchronised (all copies are ordered before any
 * later work on `stream`), and the host inputs must stay unchanged until
 * then.  The library's two copy streams and a few events per device are
 * created on the first call on that device and kept; calls on one device are
 * enqueued one at a time.  Calls that share a workspace must be ordered by
 * the caller (the same stream does it).  Errors: as for kla_chunk_fwd_ex,
 * plus KLA_ERR_INVALID_ARG for a missing, small or misaligned workspace.
 */
KLA_API kla_status kla_chunk_fwd_host(const void* q, const void* k,
                                      const void* v, const float* log_alpha,
                                      const float* eta, float eps,
                                      const float* h0, void* o, float* hT,
                                      int B, int T, int H, int dk, int dv,
                                      int C, kla_dtype dtype, kla_algo algo,
                                      kla_step_rule rule, void* workspace,
                                      size_t workspace_bytes,
                                      kla_stream_t stream);

/*
 * kla_decode_step -- one new token for each of N sequences x H heads (the
 * recurrence above for a single t), updating the recurrent state in place.
 *
 *   q, k       [N, H, dk]      dtype   (read)
 *   v          [N, H, dv]      dtype   (read)
 *   log_alpha  [N, H]          fp32    (read)
 *   eta        [N, H]          fp32    (read)
 *   S          [N, H, dk, dv]  fp32    (read, then overwritten with S_t)
 *   o          [N, H, dv]      dtype   (written) = S_t^T q
 *
 * Supported: dk, dv in {16, 32, 64, 128}; N, H >= 0.  S must be 16-byte
 * aligned.  o and S must not overlap each other or any input (byte
 * ranges).  Errors as for kla_chunk_fwd.
 * The step is launched as a programmatic dependent of the previous kernel on
 * `stream`: its blocks may be scheduled while that kernel's last blocks run,
 * but each waits for that kernel, and its memory, before touching memory,
 * so the ordering is that of plain stream order.  It allocates, synchronises
 * and reads back nothing, so steps can be recorded in a CUDA graph.
 */
KLA_API kla_status kla_decode_step(const void* q, const void* k, const void* v,
                           const float* log_alpha, const float* eta, float eps,
                           float* S, void* o, int N, int H, int dk, int dv,
                           kla_dtype dtype, kla_stream_t stream);

/* kla_decode_step_ex -- kla_decode_step with an explicit step rule. */
KLA_API kla_status kla_decode_step_ex(const void* q, const void* k,
                              const void* v, const float* log_alpha,
                              const float* eta, float eps, float* S, void* o,
                              int N, int H, int dk, int dv, kla_dtype dtype,
                              kla_step_rule rule, kla_stream_t stream);

/*
 * Diagonal-preconditioned variant (the adjacent preconditioned-DeltaNet page,
 * section "Aproximacion Diagonal": P_t = Diag(A_t)^{-1} from the running key
 * second moments A_t = A_{t-1} + k_t (.) k_t, squashed in log space onto
 * [1/x, x], applied to the write key).  The recurrence becomes
 *     e_t = v_t - S~^T k_t,   S_t = S~ + beta_t kw_t e_t^T,   o_t = S_t^T q_t
 * with the write key kw_t = P_t (.) k_t, and with the Kaczmarz rule
 * beta_t = eta_t / (k_t . kw_t + eps) (an oblique projection: S_t^T k_t = v_t
 * at eta = 1, eps = 0); KLA_STEP_GIVEN keeps beta_t = eta_t (the page's
 * preconditioned gated DeltaNet).  A prefill is kla_precond_keys followed by
 * kla_chunk_fwd_kw; a decode step is kla_precond_keys with T = 1 followed by
 * kla_decode_step_kw, A carried from one call to the next.
 *
 * kla_precond_keys -- write keys and second moments.  Per (b, h) and key
 * dimension i:
 *     A_t,i  = A_{t-1},i + k_t,i^2                      (A_0 = A0 or 0)
 *     z_i    = mean_j log(A_t,j + delta) - log(A_t,i + delta)
 *     kw_t,i = exp(log(x) tanh(z_i / log(x))) k_t,i
 * The page fixes neither the squash nor its reference level; tanh with unit
 * slope, centred on the mean log second moment (so that P is invariant to the
 * scale of the keys), and the floor delta are this library's reading.
 *
 *   k        [B, T, H, dk]  dtype  (read)
 *   A0       [B, H, dk]     fp32   (read) or NULL (zero)
 *   k_write  [B, T, H, dk]  dtype  (written); must not overlap k, A0, AT
 *   AT       [B, H, dk]     fp32   (written: A_T) or NULL; may equal A0
 *            exactly, must not overlap it or k otherwise
 *   x > 1 (the page uses about 1.5), delta >= 0
 * Supported dk as for kla_chunk_fwd.  Errors: KLA_ERR_INVALID_ARG,
 * KLA_ERR_UNSUPPORTED_SHAPE, KLA_ERR_CUDA.
 */
KLA_API kla_status kla_precond_keys(const void* k, const float* A0,
                                    void* k_write, float* AT, int B, int T,
                                    int H, int dk, float x, float delta,
                                    kla_dtype dtype, kla_stream_t stream);

/*
 * kla_precond_keys_workspace_size -- bytes of device workspace
 * kla_precond_keys_ex takes: with dk = 128 and T > 64, two fp32 rows of dk
 * per (b, h, 64-token chunk) (B H ceil(T / 64) 1024 bytes), else 0.  Errors:
 * KLA_ERR_INVALID_ARG (NULL bytes, negative sizes, dtype),
 * KLA_ERR_UNSUPPORTED_SHAPE (dk).
 *
 * kla_precond_keys_ex -- kla_precond_keys with an optional workspace.  With
 * dk = 128 and 16-byte-aligned k and k_write the library takes its chunked
 * form: per (b, h, chunk) the sum of k^2 over the chunk, a scan of those
 * sums over the chunks of each (b, h) (A before each chunk, and A_T), then
 * the chunk's tokens in order from that A (three launches on `stream`,
 * each later one a programmatic dependent of the one before; with T <= 64,
 * a decode step for instance, the last alone, from A0).  Its
 * partial sums are grouped by chunk, so A_T and kw differ from the other
 * form's by fp32 rounding only.  Other shapes take one kernel without a
 * workspace (one cluster of CTAs per (b, h)).
 *
 *   workspace  device memory of at least
 *              kla_precond_keys_workspace_size(...) bytes, 16-byte aligned,
 *              overlapping no argument, owned by the caller, contents on
 *              entry irrelevant; or NULL (stream-ordered scratch when the
 *              chunked form needs a workspace: T > 64)
 *
 * kla_precond_keys is kla_precond_keys_ex with a NULL workspace.  Errors as
 * for kla_precond_keys, plus KLA_ERR_INVALID_ARG for a small, misaligned or
 * overlapping workspace.
 */
KLA_API kla_status kla_precond_keys_workspace_size(int B, int T, int H,
                                                   int dk, kla_dtype dtype,
                                                   size_t* bytes);
KLA_API kla_status kla_precond_keys_ex(const void* k, const float* A0,
                                       void* k_write, float* AT, int B,
                                       int T, int H, int dk, float x,
                                       float delta, kla_dtype dtype,
                                       void* workspace,
                                       size_t workspace_bytes,
                                       kla_stream_t stream);

/*
 * kla_chunk_fwd_kw -- kla_chunk_fwd_ex with separate write keys k_write
 * ([B, T, H, dk], dtype, read; e.g. from kla_precond_keys): the chunkwise
 * form with A = I + strict_lower(Diag(beta)(Gamma o K Kw^T)),
 * P = Gamma o Q Kw^T and the state written along Kw, the residual read along
 * K.  Takes the path kla_chunk_fwd_ex's KLA_ALGO_AUTO would (for bf16,
 * dk = dv = 128, C = 64 and 16-byte-aligned tensors, k_write included: the
 * two-kernel tensor-core path, G = [K; Q] Kw^T in its pre-pass and
 * Diag(Gamma_C) Kw in its state pass, with stream-ordered scratch for its
 * records), else the CUDA-core kernel.  k_write must not overlap o.  Errors
 * as for kla_chunk_fwd_ex (NULL k_write is KLA_ERR_INVALID_ARG).
 */
KLA_API kla_status kla_chunk_fwd_kw(const void* q, const void* k,
                                    const void* k_write, const void* v,
                                    const float* log_alpha, const float* eta,
                                    float eps, const float* h0, void* o,
                                    float* hT, int B, int T, int H, int dk,
                                    int dv, int C, kla_dtype dtype,
                                    kla_step_rule rule, kla_stream_t stream);

/*
 * kla_chunk_fwd_kw_ex -- kla_chunk_fwd_kw with an explicit path, as
 * kla_chunk_fwd_ex's `algo` (KLA_ALGO_TC the two-kernel path,
 * KLA_ALGO_TC_FUSED the fused tensor-core kernel's write-key mode,
 * KLA_ALGO_SIMT the CUDA-core kernel), and an optional workspace as
 * kla_chunk_fwd_ws's (kla_chunk_fwd_workspace_size(...) bytes for `algo`,
 * 16-byte aligned, overlapping no argument k_write included; NULL: the
 * library takes stream-ordered scratch when the path needs a workspace).
 * Errors as for kla_chunk_fwd_kw, plus KLA_ERR_UNSUPPORTED_SHAPE when a
 * tensor-core path is asked for a shape it does not take and
 * KLA_ERR_INVALID_ARG for a small, misaligned or overlapping workspace.
 */
KLA_API kla_status kla_chunk_fwd_kw_ex(const void* q, const void* k,
                                       const void* k_write, const void* v,
                                       const float* log_alpha,
                                       const float* eta, float eps,
                                       const float* h0, void* o, float* hT,
                                       int B, int T, int H, int dk, int dv,
                                       int C, kla_dtype dtype, kla_algo algo,
                                       kla_step_rule rule, void* workspace,
                                       size_t workspace_bytes,
                                       kla_stream_t stream);

/*
 * kla_decode_step_kw -- kla_decode_step_ex with a separate write key
 * k_write [N, H, dk] (dtype, read).  Errors as for kla_decode_step (NULL
 * k_write is KLA_ERR_INVALID_ARG).
 */
KLA_API kla_status kla_decode_step_kw(const void* q, const void* k,
                                      const void* k_write, const void* v,
                                      const float* log_alpha,
                                      const float* eta, float eps, float* S,
                                      void* o, int N, int H, int dk, int dv,
                                      kla_dtype dtype, kla_step_rule rule,
                                      kla_stream_t stream);

/*
 * kla_chunk_bwd_workspace_size -- bytes of device workspace kla_chunk_bwd
 * needs for these sizes: two fp32 tensors [B, H, ceil(T/C), dk, dv] (the
 * state at every chunk start and the gradient of the loss with respect to
 * the state at every chunk end) and, for dk = 128 and C = 64, 17,152 bytes
 * per (batch, head, chunk) of per-chunk records (the inverse, P and the
 * gates of the chunk) for the tensor-core kernels, plus, when also
 * dv = 128, the workspace of the two-kernel forward that writes the
 * checkpoints (kla_chunk_fwd_workspace_size: 16,644 bytes per (batch, head,
 * chunk), rounded up to 16 bytes, and 528 bytes).  Writes 0 for an empty
 * problem.  Errors:
 * KLA_ERR_INVALID_ARG (null `bytes`, negative size, C <= 0).
 */
KLA_API kla_status kla_chunk_bwd_workspace_size(int B, int T, int H, int dk,
                                                int dv, int C, size_t* bytes);

/*
 * kla_chunk_bwd -- backward pass of kla_chunk_fwd_ex: given the gradients of
 * a loss L with respect to o (o_grad) and to the final state (hT_grad,
 * NULL = zero), writes the gradients with respect to every input.  The
 * forward pass is recomputed (it need not have been run); the result equals
 * the reverse mode of the token-by-token recurrence above up to
 * floating-point rounding, for either step rule (with KLA_STEP_KACZMARZ, k
 * also receives the gradient through ||k||^2 in beta).  The chunkwise form
 * differentiated is that of the page's section "Implementacion"; the page
 * gives no backward pass of its own.
 *
 *   q, k, v, log_alpha, eta, eps, h0, B, T, H, dk, dv, C, dtype, rule:
 *                  as for kla_chunk_fwd_ex (read)
 *   o_grad         [B, T, H, dv]  dtype   (read)
 *   hT_grad        [B, H, dk, dv] fp32    (read) or NULL
 *   q_grad, k_grad [B, T, H, dk]  dtype   (written)
 *   v_grad         [B, T, H, dv]  dtype   (written)
 *   log_alpha_grad, eta_grad  [B, T, H] fp32 (written)
 *   h0_grad        [B, H, dk, dv] fp32    (written) or NULL
 *   workspace      device memory of at least
 *                  kla_chunk_bwd_workspace_size(...) bytes, 16-byte aligned,
 *                  owned by the caller; its contents on entry do not matter
 *                  and are garbage on return
 *
 * The forward pass writing the state at every chunk start (the two-kernel
 * tensor-core path where kla_chunk_fwd_ex's KLA_ALGO_AUTO would use it, its
 * pre-pass also writing the per-chunk records of the backward; else the
 * fused tensor-core kernel or the CUDA-core one, and for dk = 128, C = 64,
 * bf16 a pre-pass of its own for the records); the reverse recurrence of
 * dL/dS over the chunks; the per-chunk gradients.  The last two run on the
 * tensor cores (bf16 operands, fp32 accumulation) for bf16, dk = 128,
 * C = 64 and 16-byte-aligned q, k, v, o_grad (the recurrence also needs dv
 * a multiple of 64), else on the CUDA cores in fp32.  Supported shapes as
 * for kla_chunk_fwd.  No output may
 * overlap an input, another output or the workspace, and the workspace may
 * overlap no input (byte ranges from the sizes).  Errors:
 * KLA_ERR_INVALID_ARG (null required pointer, negative size, bad enum,
 * eps < 0 or not finite, overlapping buffers, workspace too small or
 * misaligned), KLA_ERR_UNSUPPORTED_SHAPE, KLA_ERR_CUDA; the argument checks
 * come before those on the workspace.
 */
KLA_API kla_status kla_chunk_bwd(const void* q, const void* k, const void* v,
                                 const float* log_alpha, const float* eta,
                                 float eps, const float* h0,
                                 const void* o_grad, const float* hT_grad,
                                 void* q_grad, void* k_grad, void* v_grad,
                                 float* log_alpha_grad, float* eta_grad,
                                 float* h0_grad, int B, int T, int H, int dk,
                                 int dv, int C, kla_dtype dtype,
                                 kla_step_rule rule, void* workspace,
                                 size_t workspace_bytes, kla_stream_t stream);

/*
 * kla_chunk_bwd_noalloc -- kla_chunk_bwd for callers that cannot allocate
 * device memory: a plain C program or plug-in that links only this library
 * and owns no device allocator, a hook running inside a framework's own
 * allocator (which must not be re-entered), or a process whose device-memory
 * budget is fixed in advance.  The paper has no counterpart; it is an
 * addition of this library.
 *
 * Arguments and results are those of kla_chunk_bwd without the workspace:
 * its scratch is a fixed 32 MiB array inside the library (every GPU that
 * loads the library holds it until the process exits).  The argument checks
 * of kla_chunk_bwd run first (KLA_ERR_INVALID_ARG, KLA_ERR_UNSUPPORTED_SHAPE);
 * then a problem whose kla_chunk_bwd_workspace_size exceeds 32 MiB (for
 * dk = dv = 128: B * H * ceil(T / C) > 203 with C = 64, > 256 with other C)
 * is rejected with KLA_ERR_UNSUPPORTED_SHAPE.  Either way nothing is
 * launched.
 *
 * Every call made outside a stream capture looks up the array's device
 * address on the current device (a failure returns KLA_ERR_CUDA), so an
 * address from before a cudaDeviceReset is never reused; a call made while
 * `stream` is being captured uses the address of the last such lookup on
 * that device, so the first call on a device must come before any capture
 * (else KLA_ERR_CUDA).  Every call shares the one array and leaves its
 * contents behind; nothing in it has to start at zero.  Calls that overlap
 * on the GPU (on different streams, or from different host threads, on the
 * same device) race on the array: serialise them.
 */
KLA_API kla_status kla_chunk_bwd_noalloc(
    const void* q, const void* k, const void* v, const float* log_alpha,
    const float* eta, float eps, const float* h0, const void* o_grad,
    const float* hT_grad, void* q_grad, void* k_grad, void* v_grad,
    float* log_alpha_grad, float* eta_grad, float* h0_grad, int B, int T,
    int H, int dk, int dv, int C, kla_dtype dtype, kla_step_rule rule,
    kla_stream_t stream);

/*
 * kla_device_status -- synchronises `stream`, then reads and clears the
 * library's device-side fault word.  Returns KLA_ERR_TIMEOUT if a bounded
 * wait inside a kernel gave up since the last call (the kernel then skipped
 * its remaining work and returned; its outputs are invalid), KLA_ERR_CUDA if
 * synchronisation failed, else KLA_OK.
 */
KLA_API kla_status kla_device_status(kla_stream_t stream);

/*
 * kla_selftest_wait_timeout -- exercises the device-side timeout path
 * without faulting anything: launches one CTA of the tensor-core state-pass
 * kernel on `stream` whose copy-issuing thread issues nothing and whose
 * waits give up after 1 ms.  Its first waits (on barriers nothing will
 * arrive on, with no copy or tensor-core operation in flight) run out, the
 * CTA takes its abort path (TMEM freed, return) and sets the fault word, so
 * that the next kla_device_status on `stream` returns KLA_ERR_TIMEOUT (and
 * the one after that KLA_OK).  The pages have no counterpart; it is a test
 * hook of this library.  Errors: KLA_ERR_CUDA (launch failed or no tensor
 * map support).
 */
KLA_API kla_status kla_selftest_wait_timeout(kla_stream_t stream);

/* Static, NUL-terminated description of a status code (never NULL). */
KLA_API const char* kla_status_string(kla_status status);

#ifdef __cplusplus
}
#endif

#endif /* KLA_H */
