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
//   kk_ri = k_r[0]*k_i[0], then fma over j = 1 .. dk-1          (i < r)
//   A_ri  = (beta_r * decay_exp(G_r - G_i)) * kk_ri              (i < r, else 0)
//   W_r[c]  = (beta_r * e_r) * k_r[c],  then fma(-A_ri, W_i[c], .) for i = 0 .. r-1
//   U~_r[n] = beta_r * v_r[n],          then fma(-A_ri, U~_i[n], .) for i = 0 .. r-1
//   p_rn  = W_r[0]*S_b[n][0], then fma over j = 1 .. dk-1
//   dd_rn = d_r * (U~_r[n] - p_rn)
//   S_new[n][c] = gamma * S_b[n][c], then fma(dd_rn, k_r[c], .) for r = 0 .. C-1
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
// Chunk-update pieces.  Tile functions compute 4 x 4 blocks of one contraction; each
// element's sequence is the one stated above whatever tile or thread computes it.
// ----------------------------------------------------------------------------------

__device__ __forceinline__ float a_entry(float beta_r, float Gr, float Gi, float kk)
{
    return __fmul_rn(__fmul_rn(beta_r, decay_exp(__fsub_rn(Gr, Gi))), kk);
}

// kk[a][b] = k_{r0+a} . k_{i0+b} over DK entries, sequential in j.
// ks: fp32 [C][ks_stride] (rows 16-byte aligned).
template <int DK>
__device__ __forceinline__ void kk_tile(const float* ks, int ks_stride, int r0, int i0, float acc[4][4])
{
#pragma unroll
    for (int j = 0; j < DK; j += 4) {
        float4 ar[4], bi[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) ar[a] = *reinterpret_cast<const float4*>(ks + (r0 + a) * ks_stride + j);
#pragma unroll
        for (int b = 0; b < 4; ++b) bi[b] = *reinterpret_cast<const float4*>(ks + (i0 + b) * ks_stride + j);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                if (j == 0)
                    acc[a][b] = __fmul_rn(ar[a].x, bi[b].x);
                else
                    acc[a][b] = __fmaf_rn(ar[a].x, bi[b].x, acc[a][b]);
                acc[a][b] = __fmaf_rn(ar[a].y, bi[b].y, acc[a][b]);
                acc[a][b] = __fmaf_rn(ar[a].z, bi[b].z, acc[a][b]);
                acc[a][b] = __fmaf_rn(ar[a].w, bi[b].w, acc[a][b]);
            }
    }
}

// Forward substitution of one column: x[r] = init[r] - sum_{i<r} A[r][i] x[i],
// accumulated as fma(-A_ri, x_i, .) for i ascending.  A: fp32 smem [C][a_stride].
// The loops run column-outermost (x[t] is final once the terms of columns < t are in),
// so consecutive instructions are independent; every row still adds its terms in
// ascending i, which is the operation sequence above.
template <int C>
__device__ __forceinline__ void fwd_subst(const float* A, int a_stride, float x[C])
{
#pragma unroll
    for (int t = 0; t < C - 1; ++t) {
        const float xt = x[t];
#pragma unroll
        for (int r = t + 1; r < C; ++r) x[r] = __fmaf_rn(-A[r * a_stride + t], xt, x[r]);
    }
}

// dd[a][b] for r = r0+a, n = n0+b:  d_r * (U~_r[n] - W_r . S_b[n]), the dot sequential
// in j.  Wt: fp32 [DK][wt_stride] (W transposed), St: fp32 [DK][st_stride] (S_b stored
// [dk][dv], the slice's column n at offset n), Us: fp32 [C][us_stride], dvec[C].
template <int DK>
__device__ __forceinline__ void delta_tile(const float* Wt, int wt_stride, const float* St, int st_stride,
                                           const float* Us, int us_stride, const float* dvec, int r0,
                                           int n0, float out[4][4])
{
    float acc[4][4];
#pragma unroll 8
    for (int j = 0; j < DK; ++j) {
        const float4 w = *reinterpret_cast<const float4*>(Wt + j * wt_stride + r0);
        const float4 s = *reinterpret_cast<const float4*>(St + j * st_stride + n0);
        const float wv[4] = {w.x, w.y, w.z, w.w};
        const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b)
                acc[a][b] = (j == 0) ? __fmul_rn(wv[a], sv[b]) : __fmaf_rn(wv[a], sv[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const float4 u = *reinterpret_cast<const float4*>(Us + (r0 + a) * us_stride + n0);
        const float uv[4] = {u.x, u.y, u.z, u.w};
        const float d = dvec[r0 + a];
#pragma unroll
        for (int b = 0; b < 4; ++b) out[a][b] = __fmul_rn(d, __fsub_rn(uv[b], acc[a][b]));
    }
}

// S_new for value rows n0..n0+3 and key columns c0..c0+3, returned as out[c][n]
// (storage order): gamma * S_b[n][c], then fma(dd_rn, k_r[c], .) for r = 0 .. C-1.
// St: fp32 [DK][st_stride] (S_b storage slice), dd: fp32 [C][dd_stride], ks: fp32
// [C][ks_stride].
template <int C>
__device__ __forceinline__ void snew_tile(const float* St, int st_stride, const float* dd, int dd_stride,
                                          const float* ks, int ks_stride, float gamma, int n0, int c0,
                                          float out[4][4])
{
    float acc[4][4];  // [c][n]
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float4 s = *reinterpret_cast<const float4*>(St + (c0 + c) * st_stride + n0);
        acc[c][0] = __fmul_rn(gamma, s.x);
        acc[c][1] = __fmul_rn(gamma, s.y);
        acc[c][2] = __fmul_rn(gamma, s.z);
        acc[c][3] = __fmul_rn(gamma, s.w);
    }
#pragma unroll 8
    for (int r = 0; r < C; ++r) {
        const float4 d = *reinterpret_cast<const float4*>(dd + r * dd_stride + n0);
        const float4 kv = *reinterpret_cast<const float4*>(ks + r * ks_stride + c0);
        const float dv4[4] = {d.x, d.y, d.z, d.w};
        const float kv4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int n = 0; n < 4; ++n) acc[c][n] = __fmaf_rn(dv4[n], kv4[c], acc[c][n]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int n = 0; n < 4; ++n) out[c][n] = acc[c][n];
}

}  // namespace cpr
