// chunk_update.cuh — the state-independent half of the chunk update U, as CTA-wide
// device routines called both by prefill's chunk-prep kernel and by decode's resync
// kernel.  Element sequences are those of numerics.cuh.
#pragma once

#include "numerics.cuh"

namespace cpr {

// Shared-memory scratch of one chunk's prep: keys (fp32, row stride DK + 4), A, and the
// per-token vectors.  `g_in` holds the chunk's g on entry and G on exit.
template <int DK, int C>
struct PrepSmem {
    static constexpr int KS = DK + 4;
    static constexpr size_t floats = (size_t)C * KS + (size_t)C * C + 4 * (size_t)C;
    float* kf;   // [C][KS]
    float* A;    // [C][C]
    float* G;    // [C]  g on entry, G (sequential cumulative sum) after chunk_decays_and_A
    float* be;   // [C]  beta_r * e_r
    float* bs;   // [C]  beta_r
    float* dvs;  // [C]  d_r
    __device__ explicit PrepSmem(float* base)
        : kf(base), A(base + C * KS), G(A + C * C), be(G + C), bs(be + C), dvs(bs + C) {}
};

// G, e, d, beta*e and the strictly lower-triangular A from kf, g (in G) and beta (in bs).
// Must be called by every thread of the CTA; contains __syncthreads.
template <int DK, int C>
__device__ __forceinline__ void chunk_decays_and_A(const PrepSmem<DK, C>& s)
{
    const int tid = threadIdx.x;
    __syncthreads();
    if (tid == 0) {
        float acc = s.G[0];
        for (int r = 1; r < C; ++r) {
            acc = __fadd_rn(acc, s.G[r]);
            s.G[r] = acc;
        }
    }
    __syncthreads();
    if (tid < C) {
        s.be[tid] = __fmul_rn(s.bs[tid], decay_exp(s.G[tid]));
        s.dvs[tid] = decay_exp(__fsub_rn(s.G[C - 1], s.G[tid]));
    }
    constexpr int NT = C / 4;
    for (int t = tid; t < NT * (NT + 1) / 2; t += blockDim.x) {
        int R = 0, rem = t;
        while (rem > R) {
            rem -= R + 1;
            ++R;
        }
        const int I = rem;
        float acc[4][4];
        kk_tile<DK>(s.kf, PrepSmem<DK, C>::KS, 4 * R, 4 * I, acc);
#pragma unroll
        for (int aa = 0; aa < 4; ++aa)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const int r = 4 * R + aa, i = 4 * I + bb;
                if (i < r) s.A[r * C + i] = a_entry(s.bs[r], s.G[r], s.G[i], acc[aa][bb]);
            }
    }
    __syncthreads();
}

// Column `col` of [W | U~] (col < DK: W, else U~ column col - DK) by forward
// substitution.  V element (r, n) of the chunk is vbase[r * vstride + n].
template <int DK, int DV, int C, typename T>
__device__ __forceinline__ void chunk_column(const PrepSmem<DK, C>& s, int col, const T* vbase, size_t vstride,
                                             float x[C])
{
    if (col < DK) {
#pragma unroll
        for (int r = 0; r < C; ++r) x[r] = __fmul_rn(s.be[r], s.kf[r * PrepSmem<DK, C>::KS + col]);
    } else {
#pragma unroll
        for (int r = 0; r < C; ++r) x[r] = __fmul_rn(s.bs[r], to_f32<T>(vbase[(size_t)r * vstride + (col - DK)]));
    }
    fwd_subst<C>(s.A, C, x);
}

}  // namespace cpr
