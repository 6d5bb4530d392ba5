// numerics.cuh — the numerical contract of the CPR Gated DeltaNet kernels.
//
// Every rounding-relevant operation of the layer is defined here once, as an explicit
// sequence of IEEE round-to-nearest fp32 operations (no contraction is left to the
// compiler: every product, sum and fused multiply-add is an intrinsic).  Prefill's
// intra-chunk kernel and decode's step kernel evaluate the token step with these
// definitions; prefill's chunk-update kernels and decode's resync kernel evaluate the
// chunk update with these definitions.  Thread mappings differ between kernels; the
// per-element operation sequences do not, which is what makes prefill, training
// forward and decode bit-identical ("IsoExec: Eliminating Trainer-Inference Mismatch
// in SkyRL", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": CPR is
// bitwise exact across trainer forward, rollout prefill and rollout decode).
//
// Token step (gated delta rule; S is dv x dk, row i = value index):
//   alpha = decay_exp(g)                          (e^g via 2^(g log2 e), see below)
//   x_i   = dot_dk(S_i, k)                        (canonical tree, below)
//   u_i   = beta * (v_i - alpha * x_i)            (mul, sub, mul)
//   S_ij <- fma(u_i, k_j, alpha * S_ij)           (mul, fma)
//   o_i   = dot_dk(S_i, q)
// dot_dk(a, b): eight chains over contiguous blocks of L = dk/8 entries; chain m is
//   c_m = a[mL]*b[mL], then c_m = fma(a[j], b[j], c_m) for j = mL+1 .. mL+L-1;
//   result = ((c0 + c1) + (c2 + c3)) + ((c4 + c5) + (c6 + c7)).
//
// Chunk update U(S_b, chunk of C tokens) (WY/UT form of the gated delta rule; the
// pages fix only that one fixed-order fp32 function produces every boundary state):
//   G_0 = g_0, G_r = G_{r-1} + g_r              (sequential)
//   e_r = decay_exp(G_r),  d_r = decay_exp(G_{C-1} - G_r),  gamma = e_{C-1}
//   kk_ri = sum_j k_r[j] k_i[j]: a tcgen05 product of the keys' bf16 splits, fp32
//           accumulation (exact products for bf16 keys; hi*hi + hi*lo + lo*hi for fp32)
//   A_ri  = (beta_r * decay_exp(G_r - G_i)) * kk_ri              (i < r, else 0)
//   T = (I + A)^-1 by blocks of 16 (invert_unit_lower below): each diagonal block by
//         substitution (T_rj = [r == j], then fma(-A_ri, T_ij, .) for i ascending), then the
//         blocks below the diagonal as T_ij = -T_ii sum_k A_ik T_kj, every sum in a fixed
//         ascending order
//   W0_r[c] = (beta_r * e_r) * k_r[c],  U0_r[n] = beta_r * v_r[n]   (W = T W0, U~ = T U0)
//   then, in matrix form with D = diag(d_r) (chunk_update.cuh):
//   Z^T = (D K)^T T, M^T = gamma I - Z^T W0, B = U0^T Z:  tcgen05 products (M = 128,
//         K = C) of bf16 hi/lo splits (Dekker's splitting, tc.cuh), hi*hi + hi*lo +
//         lo*hi, fp32 accumulation
//   S_new = S_b M + B:  per 64 value rows, a tcgen05 product of S_b's splits with M's
//         (M = 64, N = dk, K = dk, the same three products), then one fp32 add of B
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpr {

// exp of every decay (alpha and the chunk-update decays), written from the identity
// e^x = 2^(x log2 e): one round-to-nearest product with log2 e, then the hardware base-2
// exponential (PTX ex2.approx.f32, relative error below 2^-22 of its argument's 2^y,
// subnormal results kept).  Explicit instructions only, so every kernel computes the
// same bits; the decays here are e^x with x <= 0, results in [0, 1].
static __device__ __forceinline__ float decay_exp(float x)
{
    const float y = __fmul_rn(x, 1.4426950408889634f);  // log2(e), rounded to fp32
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// ----------------------------------------------------------------------------------
// Token step pieces.
// ----------------------------------------------------------------------------------

__device__ __forceinline__ float tree8(float c0, float c1, float c2, float c3, float c4, float c5,
                                       float c6, float c7)
{
    return __fadd_rn(__fadd_rn(__fadd_rn(c0, c1), __fadd_rn(c2, c3)),
                     __fadd_rn(__fadd_rn(c4, c5), __fadd_rn(c6, c7)));
}

// The same tree when chains are held in pairs P_m = (c_m, c_{m+4}), m = 0..3:
// (P0 + P1) + (P2 + P3) = ((c0+c1)+(c2+c3), (c4+c5)+(c6+c7)), then x + y.
__device__ __forceinline__ float tree8_pairs(float2 p0, float2 p1, float2 p2, float2 p3)
{
    const float2 r = __fadd2_rn(__fadd2_rn(p0, p1), __fadd2_rn(p2, p3));
    return __fadd_rn(r.x, r.y);
}

__device__ __forceinline__ float step_u(float alpha, float beta, float v, float x)
{
    return __fmul_rn(beta, __fsub_rn(v, __fmul_rn(alpha, x)));
}

__device__ __forceinline__ float step_s(float s, float alpha, float u, float kj)
{
    return __fmaf_rn(u, kj, __fmul_rn(alpha, s));
}

// ----------------------------------------------------------------------------------
// In-kernel L2 normalisation of queries and keys (the CPR_QK_L2NORM option): a key becomes
// k / sqrt(sum k^2 + eps), a query q / sqrt(sum q^2 + eps) * dk^-1/2.  The sum of squares
// runs in dot_dk's order (eight chains over contiguous blocks of dk/8 entries, first term a
// product, then the canonical tree); the square root and the reciprocal are correctly
// rounded; then one product per entry (two for a query, the scale last).  x(c) is entry c.
// ----------------------------------------------------------------------------------
constexpr float kL2Eps = 1e-6f;

template <int DK>
__device__ __forceinline__ constexpr float query_scale()
{
    static_assert(DK == 32 || DK == 64 || DK == 128, "dk^-1/2 for the built shapes");
    return DK == 32 ? 0x1.6a09e6p-3f : DK == 64 ? 0x1.0p-3f : 0x1.6a09e6p-4f;  // 1/sqrt(dk), rounded
}

template <int DK, typename F>
__device__ __forceinline__ float l2_inv(F x)
{
    constexpr int L = DK / 8;
    float c[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        float acc = __fmul_rn(x(m * L), x(m * L));
#pragma unroll
        for (int t = 1; t < L; ++t) acc = __fmaf_rn(x(m * L + t), x(m * L + t), acc);
        c[m] = acc;
    }
    return __frcp_rn(__fsqrt_rn(__fadd_rn(tree8(c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[7]), kL2Eps)));
}

// Normalise a row held in shared memory (entry c at row[pos(c)]), in place; `query` adds
// the dk^-1/2 scale.  One thread per row.
template <int DK, typename P>
__device__ __forceinline__ void l2_normalise_row(float* row, P pos, bool query)
{
    const float inv = l2_inv<DK>([&](int c) { return row[pos(c)]; });
#pragma unroll 8
    for (int c = 0; c < DK; ++c) {
        const float y = __fmul_rn(row[pos(c)], inv);
        row[pos(c)] = query ? __fmul_rn(y, query_scale<DK>()) : y;
    }
}

// ----------------------------------------------------------------------------------
// Chunk-update pieces.  Tile functions compute 4 x 4 blocks of one contraction; each
// element's sequence is the one stated above whatever tile or thread computes it.
// ----------------------------------------------------------------------------------

__device__ __forceinline__ float a_entry(float beta_r, float Gr, float Gi, float kk)
{
    return __fmul_rn(__fmul_rn(beta_r, decay_exp(__fsub_rn(Gr, Gi))), kk);
}

// T = (I + A)^-1 of a strictly lower-triangular C x C matrix A by blocks of 16, with all
// `nt` threads of the caller: the four (C / 16) diagonal blocks by forward substitution,
// one column per thread (x_r = [r == j] - sum_{i<r} A_ri x_i, fma in ascending i), then
// the blocks below the diagonal by distance d = 1, 2, ..: Y = sum_{k=j}^{i-1} A_ik T_kj
// (blocks k ascending, 16 terms each in ascending order), T_ij = -T_ii Y (terms in
// ascending order).  At: A transposed (At[i * C + r] = A_ri), 16-byte aligned rows.  T
// goes to Tout[r * TS + c], zero above the diagonal; Y needs 16 x 16 x (C/16 - 1) floats of
// 16-byte aligned scratch.  Every element has one fixed operation sequence, whichever
// thread computes it; a thread computes four elements of Y (rows r0..r0+3 of one column)
// or of T_ij (columns c0..c0+3 of one row) side by side, so each shared-memory load feeds
// four FMAs.  Contains __syncthreads (every thread of the block must call it); nt >= C.
template <int C, int TS>
__device__ __forceinline__ void invert_unit_lower(const float* __restrict__ At, float* __restrict__ Tout,
                                                  float* __restrict__ Y, int tid, int nt)
{
    static_assert(C % 16 == 0 && C <= 64, "blocks of 16, at most four");
    constexpr int NB = C / 16;
    constexpr int NZ = NB * (NB - 1) / 2 * 256;  // elements of the blocks above the diagonal
    for (int idx = tid; idx < NZ; idx += nt) {   // (block pairs i < j in order, 256 elements each)
        int q = idx >> 8, i = 0, j = 1;
        while (q >= NB - 1 - i) {
            q -= NB - 1 - i;
            ++i;
        }
        j = i + 1 + q;
        Tout[(16 * i + ((idx >> 4) & 15)) * TS + 16 * j + (idx & 15)] = 0.0f;
    }
    if (tid < C) {  // diagonal block k, column j (all 16 rows: zero above the diagonal)
        const int k = tid >> 4, j = tid & 15, o = 16 * k;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == j) ? 1.0f : 0.0f;
#pragma unroll
            for (int i = 0; i < r; ++i)
                if (i >= j) acc = __fmaf_rn(-At[(o + i) * C + o + r], x[i], acc);
            x[r] = r >= j ? acc : 0.0f;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tout[(o + r) * TS + o + j] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < NB; ++d) {
        const int nblk = NB - d;
        // Y of block (j + d, j): rows r0..r0+3 of column c
        for (int u = tid; u < nblk * 64; u += nt) {
            const int j = u >> 6, r0 = ((u >> 4) & 3) * 4, c = u & 15, i = j + d;
            float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
            for (int k = j; k < i; ++k) {
#pragma unroll
                for (int s = 0; s < 16; ++s) {
                    const float4 av = *reinterpret_cast<const float4*>(At + (16 * k + s) * C + 16 * i + r0);
                    const float t = Tout[(16 * k + s) * TS + 16 * j + c];
                    a0 = __fmaf_rn(av.x, t, a0);
                    a1 = __fmaf_rn(av.y, t, a1);
                    a2 = __fmaf_rn(av.z, t, a2);
                    a3 = __fmaf_rn(av.w, t, a3);
                }
            }
            float* y = Y + (j << 8) + (r0 << 4) + c;
            y[0] = a0;
            y[16] = a1;
            y[32] = a2;
            y[48] = a3;
        }
        __syncthreads();
        // T_ij = -T_ii Y: columns c0..c0+3 of row r
        for (int u = tid; u < nblk * 64; u += nt) {
            const int j = u >> 6, r = (u >> 2) & 15, c0 = (u & 3) * 4, i = j + d;
            float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
            for (int s = 0; s < 16; ++s)
                if (s <= r) {
                    const float t = Tout[(16 * i + r) * TS + 16 * i + s];
                    const float4 yv = *reinterpret_cast<const float4*>(Y + (j << 8) + (s << 4) + c0);
                    a0 = __fmaf_rn(t, yv.x, a0);
                    a1 = __fmaf_rn(t, yv.y, a1);
                    a2 = __fmaf_rn(t, yv.z, a2);
                    a3 = __fmaf_rn(t, yv.w, a3);
                }
            float* o = Tout + (16 * i + r) * TS + 16 * j + c0;
            o[0] = -a0;
            o[1] = -a1;
            o[2] = -a2;
            o[3] = -a3;
        }
        __syncthreads();
    }
}

}  // namespace cpr
