// Block-level building blocks of the CUDA-core chunkwise kernels (forward
// and backward): the Gamma-masked A and P of a chunk, and the inverse of the
// unit lower-triangular A.  Shared-memory operands, fp32, every thread of
// the block participating.
#pragma once

namespace kla {

// A (unit lower, strictly lower part beta_r Gamma_ri k_r.kw_i) and
// P = Gamma o Q Kw^T (lower incl.), row stride ldc, with kw the write keys
// (the keys themselves unless given separately); 4 x 4 tiles per thread,
// NT threads.
template <int DK, int NT>
__device__ __forceinline__ void build_a_p(int C, const float* Qs,
                                          const float* Ks, const float* KWs,
                                          int LDK, const float* gs,
                                          const float* bs, float* As,
                                          float* Ps, int ldc) {
    const int nrt = C / 4;
    for (int tile = threadIdx.x; tile < nrt * nrt; tile += NT) {
        const int r0 = (tile / nrt) * 4, i0 = (tile % nrt) * 4;
        float kk[4][4] = {}, qk[4][4] = {};
        if (i0 <= r0 + 3) {
#pragma unroll 4
            for (int c = 0; c < DK; ++c) {
                float kr[4], qr[4], ki[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    kr[x] = Ks[(r0 + x) * LDK + c];
                    qr[x] = Qs[(r0 + x) * LDK + c];
                    ki[x] = KWs[(i0 + x) * LDK + c];
                }
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        kk[rr][ii] = fmaf(kr[rr], ki[ii], kk[rr][ii]);
                        qk[rr][ii] = fmaf(qr[rr], ki[ii], qk[rr][ii]);
                    }
            }
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                const int r = r0 + rr, i = i0 + ii;
                float av = (i == r) ? 1.f : 0.f;
                float pv = 0.f;
                if (i <= r) {
                    const float dec = expf(gs[r] - gs[i]);
                    pv = dec * qk[rr][ii];
                    if (i < r) av = bs[r] * dec * kk[rr][ii];
                }
                As[r * ldc + i] = av;
                Ps[r * ldc + i] = pv;
            }
    }
}

// Tm = A^{-1} for the unit lower-triangular C x C matrix A (C = 16, 32 or
// 64; row stride ldc), in 16 x 16 tiles: the diagonal tiles by column
// substitution (one thread per column), then the tiles below them by
// distance, T_IJ = -T_II (sum_{m=J}^{I-1} A_Im T_mJ), with the sum parked in
// the (otherwise unused) upper tile (J, I).  Only the lower triangle of Tm
// is meaningful on return.  Ends with a barrier.
template <int NT>
__device__ __forceinline__ void invert_unit_lower(const float* A, float* Tm,
                                                  int C, int ldc) {
    const int tid = threadIdx.x, nb = C / 16;
    if (tid < nb * 16) {
        const int bb = tid / 16, cl = tid % 16;
        const float* Ab = A + (16 * bb) * ldc + 16 * bb;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == cl) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) acc = fmaf(Ab[r * ldc + i], x[i], acc);
            if (r > cl) x[r] = -acc;
        }
        float* Tb = Tm + (16 * bb) * ldc + 16 * bb + cl;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * ldc] = x[r];
    }
    __syncthreads();
    for (int d = 1; d < nb; ++d) {
        for (int idx = tid; idx < (nb - d) * 256; idx += NT) {
            const int J = idx / 256, I = J + d, r = (idx % 256) / 16,
                      c = idx % 16;
            float acc = 0.f;
            for (int m = J; m < I; ++m)
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    acc = fmaf(A[(16 * I + r) * ldc + 16 * m + k],
                               Tm[(16 * m + k) * ldc + 16 * J + c], acc);
            Tm[(16 * J + r) * ldc + 16 * I + c] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < (nb - d) * 256; idx += NT) {
            const int J = idx / 256, I = J + d, r = (idx % 256) / 16,
                      c = idx % 16;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k)
                acc = fmaf(Tm[(16 * I + r) * ldc + 16 * I + k],
                           Tm[(16 * J + k) * ldc + 16 * I + c], acc);
            Tm[(16 * I + r) * ldc + 16 * J + c] = -acc;
        }
        __syncthreads();
    }
}

}  // namespace kla
