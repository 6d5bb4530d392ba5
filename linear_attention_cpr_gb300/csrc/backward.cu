// backward.cu — the CPR backward: gradients of the Gated DeltaNet layer with respect to
// q, k, v, g, beta and the initial state, for a loss L(o, S_T).
//
// "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section "Chunkwise-Parallel
// Recurrent (CPR) Gated DeltaNet", per-layer table, row "Trainer Fwd+Bwd": the pages time a
// CPR backward but do not describe it.  This is the adjoint of the token recurrence
// (reverse time), evaluated on the forward's own chunk grid and split the way the forward
// is: a state-independent part per chunk (parallel), one sequential chain per (sequence,
// head) over the chunk boundaries, and the chunk-local work (parallel).
//
// With S dv x dk (row i = value index) and one chunk of n tokens starting from S_b, the
// chunk in WY form (Gated Delta Networks, Yang, Kautz & Hatamizadeh) is
//     G = cumsum(g), gam_r = e^{G_r}, d_r = e^{G_last - G_r}, E_ri = e^{G_r - G_i} (i <= r)
//     L = (K K^T) o E (strictly lower), T = (I + diag(beta) L)^-1
//     R = V - diag(gam) K S_b^T,  U = T diag(beta) R            (U = U~ - W S_b^T)
//     O = diag(gam) Q S_b^T + Pm U,  Pm = (Q K^T) o E (lower, with the diagonal)
//     S_end = S_b M + U^T diag(d) K,  M = gam_last I - W^T diag(d) K,  W = T diag(beta gam) K
// so the adjoint of a chunk boundary is dS_b = dS_end M^T + dO^T Qt with
// Qt = diag(gam) Q - Pm W (row t of Qt is the query carried back through the chunk's
// first t token transitions).  Three kernels:
//   kb1_chunk_maps      per (chunk, head): M^T and C_b = dO^T Qt (state-independent)
//   kb2_reverse_chain   per (sequence, head): dS at every chunk end, from the last chunk
//                       back to the first, one tensor-core product per chunk (the forward
//                       chain's routines); dS_0 is d_state_in
//   kb3_chunk_grads     per (chunk, head): the chunk's adjoint in WY form from S_b (the
//                       forward's boundary state) and dS_end (the chain's), giving dq, dk,
//                       dv, dg, dbeta of its tokens
// A final partial chunk is evaluated as a full one with zero tokens appended (k = q = v =
// dO = 0, g = 0, beta = 0): such tokens are identity maps, so the chunk's function of its
// real tokens, and hence every gradient of them, is unchanged.
// Every reduction runs in a fixed order (no atomics), so the gradients are reproducible
// from run to run and do not depend on how the batch is packed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "chunk_update.cuh"
#include "common.cuh"
#include "numerics.cuh"
#include "reverse_chain.cuh"
#include "tc.cuh"

namespace cpr {

namespace {

constexpr int kBwdThreads = 256;

template <typename T> __device__ __forceinline__ float ld_f32(const T* p) { return to_f32<T>(*p); }

// Shared-memory geometry of the chunk kernels (all strides in elements; row strides are odd
// numbers of 32-bit words so that column walks hit distinct banks).
template <int DK, int DV, int C, typename T>
struct BwdGeo {
    static_assert(C % 16 == 0 && DK % 32 == 0 && DV % 32 == 0, "16 x 16 thread grid over every tile");
    static constexpr int TK = DK + (sizeof(T) == 2 ? 2 : 1);  // q, k tile row stride
    static constexpr int TV = DV + (sizeof(T) == 2 ? 2 : 1);  // v, dO tile row stride
    static constexpr int NN = C + 1;                          // n x n fp32
    static constexpr int NDK = DK + 1, NDV = DV + 1;          // n x dk, n x dv fp32
    static constexpr int ND = NDK > NDV ? NDK : NDV;
    static constexpr size_t up16(size_t x) { return (x + 15) / 16 * 16; }
    static constexpr size_t TILE_K = up16((size_t)C * TK * sizeof(T));
    static constexpr size_t TILE_V = up16((size_t)C * TV * sizeof(T));
    static constexpr size_t NNB = up16((size_t)C * NN * 4);
    static constexpr size_t NDB = up16((size_t)C * ND * 4);
    // kb3's BIG region: half of a state's key rows (DK/2 x (DV+1)) or an n x n scratch
    // plus 16 x C column partials
    static constexpr size_t BIG_HALF = (size_t)(DK / 2) * NDV * 4;
    static constexpr size_t BIG_NN = (size_t)C * NN * 4 + (size_t)16 * C * 4;
    static constexpr size_t BIGB = up16(BIG_HALF > BIG_NN ? BIG_HALF : BIG_NN);
    static constexpr size_t VEC = up16((size_t)16 * C * 4);  // 16 per-token vectors
};

// Per-token vectors in shared memory.
struct Vecs {
    float *G, *gam, *dd, *beta, *dgam, *ddv, *dbeta, *edrow, *edcol, *dG;
    __device__ explicit Vecs(float* p, int C)
        : G(p), gam(p + C), dd(p + 2 * C), beta(p + 3 * C), dgam(p + 4 * C), ddv(p + 5 * C), dbeta(p + 6 * C),
          edrow(p + 7 * C), edcol(p + 8 * C), dG(p + 9 * C) {}
};

// acc[i][j] += sum_k A(i, k) B(k, j) over k < K, for this thread's TM rows and TN columns.
template <int TM, int TN, int K, typename FA, typename FB>
__device__ __forceinline__ void mm(float (&acc)[TM][TN], FA A, FB B)
{
#pragma unroll 2
    for (int k = 0; k < K; ++k) {
        float a[TM], b[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = A(i, k);
#pragma unroll
        for (int j = 0; j < TN; ++j) b[j] = B(k, j);
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
    }
}

template <int TM, int TN>
__device__ __forceinline__ void zero(float (&acc)[TM][TN])
{
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
}

// Thread grid: 16 row groups x 16 column groups (thread t: rg = t / 16, cg = t % 16, so
// the 16 threads of a row group are one half-warp).  A thread's rows are TM consecutive
// ones; its columns are strided by 16 (column 16 j + cg), so a half-warp reading one
// operand row touches 16 consecutive words (no bank conflicts), and a half-warp walking
// one column per thread through a row-padded buffer hits 16 distinct banks.  An n x D tile
// gives each thread TM = C/16 rows and D/16 columns, half of them in each half of the
// columns (so the columns of a half-width product are a subset of the full-width ones).
template <int C, int D>
struct NDMap {
    static constexpr int TM = C / 16, TN = D / 16, HN = TN / 2;
    static __device__ __forceinline__ int row(int t, int i) { return (t >> 4) * TM + i; }
    // column j of this thread within half h: h * D/2 + hlocal(t, j)
    static __device__ __forceinline__ int hlocal(int t, int j) { return j * 16 + (t & 15); }
    static __device__ __forceinline__ int col(int t, int j) { return (j / HN) * (D / 2) + hlocal(t, j % HN); }
    static __device__ __forceinline__ int hcol(int t, int h, int j) { return h * (D / 2) + hlocal(t, j); }
};
// An n x n tile: TM consecutive rows, TM columns strided by 16.
template <int C>
struct NNMap {
    static constexpr int TM = C / 16;
    static __device__ __forceinline__ int row(int t, int i) { return (t >> 4) * TM + i; }
    static __device__ __forceinline__ int col(int t, int j) { return j * 16 + (t & 15); }
};

// Sum of v over the 16 threads of this thread's row group (a fixed tree over the half-warp).
__device__ __forceinline__ float rowgroup_sum(float v)
{
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Load a chunk's rows [t0, t0 + len) of a [T, H, D] tensor (head h) into a tile of C rows
// (stride S), zeros beyond len.
template <int D, int S, int C, typename T>
__device__ __forceinline__ void load_tile(T* dst, const T* src, int64_t t0, int len, int H, int h)
{
    constexpr int VE = 16 / (int)sizeof(T), RV = D / VE;
    for (int idx = threadIdx.x; idx < C * RV; idx += kBwdThreads) {
        const int r = idx / RV, cv = idx % RV;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r < len) w = __ldg(reinterpret_cast<const uint4*>(src + ((t0 + r) * H + h) * D + cv * VE));
        const T* e = reinterpret_cast<const T*>(&w);
#pragma unroll
        for (int x = 0; x < VE; ++x) dst[r * S + cv * VE + x] = e[x];
    }
}

// Chunk bookkeeping shared by kb1 and kb3.
struct ChunkPos {
    int n;
    int64_t j, t0;
    int len;
};
template <int C>
__device__ __forceinline__ ChunkPos chunk_pos(const int32_t* cu, const int32_t* cu_chunks, int n_seqs, int64_t c)
{
    ChunkPos p;
    p.n = find_seq(cu_chunks, n_seqs, c);
    p.j = c - cu_chunks[p.n];
    const int64_t tb = cu[p.n], L = (int64_t)cu[p.n + 1] - tb;
    p.t0 = tb + p.j * C;
    p.len = (int)min((int64_t)C, L - p.j * C);
    return p;
}

// The state-independent phase common to kb1 and kb3: per-token vectors (G, gam, d, beta),
// L = (K K^T) o E (strict lower) into nnL, Pm = (Q K^T) o E (with diagonal) into nnP and
// T = (I + diag(beta) L)^-1 into nnT (stride NN; nnT first holds A transposed with stride
// C for the inversion, and `scratch` holds C x NN + 256 (C/16 - 1) floats meanwhile).  Tiles Kt, Qt and g, beta of the chunk's len tokens are loaded
// by the caller (zero tokens beyond len).
template <int DK, int C, int TK, int NN, typename T>
__device__ __forceinline__ void chunk_common(const T* Kt, const T* Qt, const float* g_in, Vecs v, float* nnL,
                                             float* nnP, float* nnT, float* scratch)
{
    using M = NNMap<C>;
    constexpr int TM = M::TM;
    const int t = threadIdx.x;
    if (t == 0) {
        float G = 0.0f;
        for (int r = 0; r < C; ++r) {
            G = (r == 0) ? g_in[0] : __fadd_rn(G, g_in[r]);
            v.G[r] = G;
        }
    }
    __syncthreads();
    if (t < C) {
        v.gam[t] = decay_exp(v.G[t]);
        v.dd[t] = decay_exp(__fsub_rn(v.G[C - 1], v.G[t]));
    }
    float kk[TM][TM], qk[TM][TM];
    zero(kk);
    zero(qk);
    mm<TM, TM, DK>(kk, [&](int i, int k) { return ld_f32(Kt + M::row(t, i) * TK + k); },
                   [&](int k, int j) { return ld_f32(Kt + M::col(t, j) * TK + k); });
    mm<TM, TM, DK>(qk, [&](int i, int k) { return ld_f32(Qt + M::row(t, i) * TK + k); },
                   [&](int k, int j) { return ld_f32(Kt + M::col(t, j) * TK + k); });
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int r = M::row(t, i);
#pragma unroll
        for (int j = 0; j < TM; ++j) {
            const int c = M::col(t, j);
            const float e = c <= r ? decay_exp(__fsub_rn(v.G[r], v.G[c])) : 0.0f;
            const float l = c < r ? __fmul_rn(kk[i][j], e) : 0.0f;
            nnL[r * NN + c] = l;
            nnP[r * NN + c] = __fmul_rn(qk[i][j], e);
            nnT[c * C + r] = __fmul_rn(v.beta[r], l);  // A transposed: At[i * C + r] = A_ri
        }
    }
    __syncthreads();
    // T by blocks with every thread (numerics.cuh) into the scratch, then into nnT
    invert_unit_lower<C, NN>(nnT, scratch, scratch + ((C * NN + 3) / 4) * 4, t, kBwdThreads);
    for (int idx = t; idx < C * C; idx += kBwdThreads) nnT[(idx / C) * NN + idx % C] = scratch[(idx / C) * NN + idx % C];
    __syncthreads();
}

// ------------------------------------------------------------------------------------
// kb1: per (chunk, head) the reverse chain's coefficients:
//   W   = T diag(beta gam) K                                      (n x dk)
//   Qt  = diag(gam) Q - Pm W                                       (n x dk)
//   M   = gam_last I - W^T diag(d) K     stored as the reverse chain's B operand: the
//         product dS_end M^T reads M[c][c'] at (N = c, K = c'), as bf16 hi / lo splits in
//         K-major core matrices
//   C_b = dO^T Qt                        stored [c][i] = C_b[i][c] (like a state)
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
struct Kb1Cfg {
    using Geo = BwdGeo<DK, DV, C, T>;
    static constexpr size_t K_OFF = 0, Q_OFF = Geo::TILE_K, O_OFF = 2 * Geo::TILE_K;
    static constexpr size_t L_OFF = O_OFF + Geo::TILE_V, P_OFF = L_OFF + Geo::NNB, T_OFF = P_OFF + Geo::NNB;
    static constexpr size_t W_OFF = T_OFF + Geo::NNB, QT_OFF = W_OFF + Geo::NDB;
    static constexpr size_t V_OFF = QT_OFF + Geo::NDB;
    static constexpr size_t bytes = V_OFF + Geo::VEC;
};

template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1) kb1_chunk_maps(BackwardArgs a)
{
    using Geo = BwdGeo<DK, DV, C, T>;
    using F = Kb1Cfg<DK, DV, C, T>;
    constexpr int TK = Geo::TK, TV = Geo::TV, NN = Geo::NN, ND = Geo::ND;
    extern __shared__ __align__(16) unsigned char smb[];
    T* Kt = reinterpret_cast<T*>(smb + F::K_OFF);
    T* Qt = reinterpret_cast<T*>(smb + F::Q_OFF);
    T* Ot = reinterpret_cast<T*>(smb + F::O_OFF);
    float* nnL = reinterpret_cast<float*>(smb + F::L_OFF);
    float* nnP = reinterpret_cast<float*>(smb + F::P_OFF);
    float* nnT = reinterpret_cast<float*>(smb + F::T_OFF);
    float* W = reinterpret_cast<float*>(smb + F::W_OFF);
    float* Qw = reinterpret_cast<float*>(smb + F::QT_OFF);
    Vecs v(reinterpret_cast<float*>(smb + F::V_OFF), C);
    float* g_in = v.dG;  // g of the chunk (zeros beyond len), consumed by chunk_common

    const int64_t c = blockIdx.x;
    const int h = blockIdx.y, H = a.H, t = threadIdx.x;
    if (*a.status || c >= a.cu_chunks[a.n_seqs]) return;
    const ChunkPos p = chunk_pos<C>(a.cu_seqlens, a.cu_chunks, a.n_seqs, c);
    load_tile<DK, TK, C>(Kt, static_cast<const T*>(a.k), p.t0, p.len, H, h);
    load_tile<DK, TK, C>(Qt, static_cast<const T*>(a.q), p.t0, p.len, H, h);
    load_tile<DV, TV, C>(Ot, static_cast<const T*>(a.d_out), p.t0, p.len, H, h);
    if (t < C) {
        g_in[t] = t < p.len ? a.g[(p.t0 + t) * H + h] : 0.0f;
        v.beta[t] = t < p.len ? a.beta[(p.t0 + t) * H + h] : 0.0f;
    }
    __syncthreads();
    chunk_common<DK, C, TK, NN>(Kt, Qt, g_in, v, nnL, nnP, nnT, W);  // W's region is free until W

    using MK = NDMap<C, DK>;
    {  // W = T diag(beta gam) K
        float w[MK::TM][MK::TN];
        zero(w);
        mm<MK::TM, MK::TN, C>(w, [&](int i, int k) { return nnT[MK::row(t, i) * NN + k]; },
                              [&](int k, int j) { return __fmul_rn(__fmul_rn(v.beta[k], v.gam[k]),
                                                                   ld_f32(Kt + k * TK + MK::col(t, j))); });
#pragma unroll
        for (int i = 0; i < MK::TM; ++i)
#pragma unroll
            for (int j = 0; j < MK::TN; ++j) W[MK::row(t, i) * ND + MK::col(t, j)] = w[i][j];
    }
    __syncthreads();
    {  // Qt = diag(gam) Q - Pm W
        float w[MK::TM][MK::TN];
        zero(w);
        mm<MK::TM, MK::TN, C>(w, [&](int i, int k) { return nnP[MK::row(t, i) * NN + k]; },
                              [&](int k, int j) { return W[k * ND + MK::col(t, j)]; });
#pragma unroll
        for (int i = 0; i < MK::TM; ++i) {
            const int r = MK::row(t, i);
#pragma unroll
            for (int j = 0; j < MK::TN; ++j) {
                const int cc = MK::col(t, j);
                Qw[r * ND + cc] = __fsub_rn(__fmul_rn(v.gam[r], ld_f32(Qt + r * TK + cc)), w[i][j]);
            }
        }
    }
    __syncthreads();
    const size_t ch = (size_t)c * H + h;
    {  // M[c][c'] = gam_last [c' == c] - sum_r d_r K[r][c'] W[r][c]
        constexpr int TM = DK / 16, TN = DK / 16;
        constexpr uint32_t SPLIT = DK * DK * 2;
        float m[TM][TN];
        zero(m);
        const int r0 = (t >> 4) * TM, cg = t & 15;  // rows c' = r0 + i, columns c = 16 j + cg
        mm<TM, TN, C>(m, [&](int i, int k) { return __fmul_rn(v.dd[k], ld_f32(Kt + k * TK + r0 + i)); },
                      [&](int k, int j) { return W[k * ND + 16 * j + cg]; });
        unsigned char* img = a.mt + ch * 2 * SPLIT;
        const float gl = v.gam[C - 1];
        // the thread's TM values of column c are TM consecutive K elements of one core-matrix
        // row (TM divides 8): stored as 32-bit words of bf16 pairs
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int cc = 16 * j + cg;
            uint32_t hw[TM / 2], lw[TM / 2];
#pragma unroll
            for (int i = 0; i < TM; i += 2) {
                float h0, l0, h1, l1;
                tc::split_f32((r0 + i == cc) ? __fsub_rn(gl, m[i][j]) : -m[i][j], h0, l0);
                tc::split_f32((r0 + i + 1 == cc) ? __fsub_rn(gl, m[i + 1][j]) : -m[i + 1][j], h1, l1);
                hw[i / 2] = tc::pack_upper(h0, h1);
                lw[i / 2] = tc::pack_upper(l0, l1);
            }
            const uint32_t off = tc::tile_off<2>(cc, r0, DK);
            uint32_t* hd = reinterpret_cast<uint32_t*>(img + off);
            uint32_t* ld = reinterpret_cast<uint32_t*>(img + SPLIT + off);
            if constexpr (TM == 8) {
                *reinterpret_cast<uint4*>(hd) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(ld) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            } else {
#pragma unroll
                for (int e = 0; e < TM / 2; ++e) {
                    hd[e] = hw[e];
                    ld[e] = lw[e];
                }
            }
        }
    }
    {  // C_b stored [c][i] = sum_t Qt[t][c] dO[t][i]
        constexpr int TM = DK / 16, TN = DV / 16;
        float m[TM][TN];
        zero(m);
        const int r0 = (t >> 4) * TM, cg = t & 15;  // rows r0 + i, columns 16 j + cg
        mm<TM, TN, C>(m, [&](int i, int k) { return Qw[k * ND + r0 + i]; },
                      [&](int k, int j) { return ld_f32(Ot + k * TV + 16 * j + cg); });
        float* dst = a.cb + ch * DK * DV;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) dst[(size_t)(r0 + i) * DV + 16 * j + cg] = m[i][j];
    }
}

// ------------------------------------------------------------------------------------
// kb2: the reverse chains, one CTA per (sequence, head) (reverse_chain.cuh).
// ------------------------------------------------------------------------------------
template <int DK, int DV>
__global__ void __launch_bounds__(kBwdThreads, 1) kb2_reverse_chain(BackwardArgs a)
{
    extern __shared__ __align__(1024) unsigned char smc[];
    __shared__ uint32_t tslot;
    constexpr uint32_t COLS = RevChainCfg<DK, DV>::TMEM_COLS;
    if (*a.status || (int)blockIdx.x >= a.n_seqs * a.H) return;
    if ((threadIdx.x >> 5) == 0) tc::tmem_alloc(&tslot, COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tslot;
    reverse_chain<DK, DV>(a, blockIdx.x, smc, tmem, nullptr);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if ((threadIdx.x >> 5) == 0) tc::tmem_dealloc(tmem, COLS);
}

// ------------------------------------------------------------------------------------
// kb3: one chunk's adjoint in the WY form, given S_b (boundary state) and dS_end (the
// chain's).  Order of work (shared-memory regions in brackets):
//   a. tiles K, Q, V, dO; G, gam, d; L [nL], Pm [nP], T [nT]
//   b. S_b by halves of its key rows [BIG]: KS = K S_b^T (registers), Y = dO S_b:
//      dq += diag(gam) Y, dgam += rowsum(Y o Q);  then R = V - diag(gam) KS [ND1]
//   c. U = T diag(beta) R [ND2];  dgam_last = <dS_end, S_b>
//   d. dPm = (dO U^T) o lower [BIG];  ED += dPm o Pm (row and column sums);
//      dU = Pm^T dO (registers);  dQK = dPm o E:  dq += dQK K, dk += dQK^T Q
//   e. dS_end by halves [BIG]: dU += diag(d) K dS_end^T;  UdS = U dS_end:
//      dk += diag(d) UdS, dd = rowsum(UdS o K);  dU -> [ND2]
//   f. dT = dU (diag(beta) R)^T [nP];  TdU = T^T dU: dv = diag(beta) TdU,
//      dbeta = rowsum(TdU o R);  TdU -> [ND1]
//   g. S_b by halves [BIG]: Z = TdU S_b:  dk -= diag(beta gam) Z,
//      dgam -= beta rowsum(K o Z)
//   h. X = T^T dT [BIG];  dA = -(X T^T) o strict lower:  dbeta += rowsum(dA o L),
//      dL = diag(beta) dA, ED += dL o L, dKK = dL o E [nP];  dk += (dKK + dKK^T) K
//   i. dG = gam dgam - d dd + rowsum(ED) - colsum(ED), the last token adding
//      gam_last dgam_last + sum_r d_r dd_r;  dg = reverse cumulative sum of dG
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
struct Kb3Cfg {
    using Geo = BwdGeo<DK, DV, C, T>;
    static constexpr size_t K_OFF = 0, Q_OFF = Geo::TILE_K, V_OFF = 2 * Geo::TILE_K,
                            O_OFF = 2 * Geo::TILE_K + Geo::TILE_V;
    static constexpr size_t L_OFF = 2 * Geo::TILE_K + 2 * Geo::TILE_V, P_OFF = L_OFF + Geo::NNB,
                            T_OFF = P_OFF + Geo::NNB;
    static constexpr size_t BIG_OFF = T_OFF + Geo::NNB, N1_OFF = BIG_OFF + Geo::BIGB, N2_OFF = N1_OFF + Geo::NDB;
    static constexpr size_t VEC_OFF = N2_OFF + Geo::NDB;
    static constexpr size_t bytes = VEC_OFF + Geo::VEC + 64;
};

template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1) kb3_chunk_grads(BackwardArgs a)
{
    using Geo = BwdGeo<DK, DV, C, T>;
    using F = Kb3Cfg<DK, DV, C, T>;
    constexpr int TK = Geo::TK, TV = Geo::TV, NN = Geo::NN, NV = Geo::NDV;
    extern __shared__ __align__(16) unsigned char smd[];
    T* Kt = reinterpret_cast<T*>(smd + F::K_OFF);
    T* Qt = reinterpret_cast<T*>(smd + F::Q_OFF);
    T* Vt = reinterpret_cast<T*>(smd + F::V_OFF);
    T* Ot = reinterpret_cast<T*>(smd + F::O_OFF);
    float* nL = reinterpret_cast<float*>(smd + F::L_OFF);
    float* nP = reinterpret_cast<float*>(smd + F::P_OFF);
    float* nT = reinterpret_cast<float*>(smd + F::T_OFF);
    float* big = reinterpret_cast<float*>(smd + F::BIG_OFF);
    float* n1 = reinterpret_cast<float*>(smd + F::N1_OFF);
    float* n2 = reinterpret_cast<float*>(smd + F::N2_OFF);
    Vecs v(reinterpret_cast<float*>(smd + F::VEC_OFF), C);
    float* red = reinterpret_cast<float*>(smd + F::VEC_OFF + Geo::VEC);  // block-reduction scratch [8]
    float* g_in = v.dG;

    const int64_t c = blockIdx.x;
    const int h = blockIdx.y, H = a.H, t = threadIdx.x;
    if (*a.status || c >= a.cu_chunks[a.n_seqs]) return;
    const ChunkPos p = chunk_pos<C>(a.cu_seqlens, a.cu_chunks, a.n_seqs, c);
    const size_t ch = (size_t)c * H + h, SSZ = (size_t)DK * DV;
    const float* Sb = a.boundary + ch * SSZ;  // [c][i] = S_b[i][c]
    const float* dSe = a.d_end + ch * SSZ;

    // ---- a
    load_tile<DK, TK, C>(Kt, static_cast<const T*>(a.k), p.t0, p.len, H, h);
    load_tile<DK, TK, C>(Qt, static_cast<const T*>(a.q), p.t0, p.len, H, h);
    load_tile<DV, TV, C>(Vt, static_cast<const T*>(a.v), p.t0, p.len, H, h);
    load_tile<DV, TV, C>(Ot, static_cast<const T*>(a.d_out), p.t0, p.len, H, h);
    if (t < C) {
        g_in[t] = t < p.len ? a.g[(p.t0 + t) * H + h] : 0.0f;
        v.beta[t] = t < p.len ? a.beta[(p.t0 + t) * H + h] : 0.0f;
        v.edrow[t] = 0.0f;
    }
    __syncthreads();
    chunk_common<DK, C, TK, NN>(Kt, Qt, g_in, v, nL, nP, nT, big);  // big is free until step b

    using MK = NDMap<C, DK>;  // n x dk tiles (dq, dk)
    using MV = NDMap<C, DV>;  // n x dv tiles (R, U, dU, TdU)
    using MN = NNMap<C>;
    constexpr int TM = MK::TM;
    static_assert(MK::TM == MV::TM, "one row mapping");
    float dq[TM][MK::TN], dk[TM][MK::TN];
    zero(dq);
    zero(dk);
    float dgam[TM], ddr[TM], dbeta[TM];
#pragma unroll
    for (int i = 0; i < TM; ++i) dgam[i] = ddr[i] = dbeta[i] = 0.0f;

    // loads rows [h * DK/2, (h+1) * DK/2) of a stored state into big[cc][i]
    auto load_half = [&](const float* src, int hh) {
        __syncthreads();
        for (int idx = t; idx < (DK / 2) * DV; idx += kBwdThreads) {
            const int cc = idx / DV, i = idx % DV;
            big[cc * NV + i] = __ldg(src + (size_t)(hh * (DK / 2) + cc) * DV + i);
        }
        __syncthreads();
    };

    // ---- b
    float ks[TM][MV::TN];
    zero(ks);
    for (int hh = 0; hh < 2; ++hh) {
        load_half(Sb, hh);
        mm<TM, MV::TN, DK / 2>(ks, [&](int i, int k) { return ld_f32(Kt + MV::row(t, i) * TK + hh * (DK / 2) + k); },
                               [&](int k, int j) { return big[k * NV + MV::col(t, j)]; });
        float y[TM][MK::HN];
        zero(y);
        mm<TM, MK::HN, DV>(y, [&](int i, int k) { return ld_f32(Ot + MK::row(t, i) * TV + k); },
                           [&](int k, int j) { return big[MK::hlocal(t, j) * NV + k]; });
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = MK::row(t, i);
#pragma unroll
            for (int j = 0; j < MK::HN; ++j) {
                const int cc = MK::hcol(t, hh, j);
                dq[i][hh * MK::HN + j] = __fmul_rn(v.gam[r], y[i][j]);
                dgam[i] = __fmaf_rn(y[i][j], ld_f32(Qt + r * TK + cc), dgam[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {  // R = V - diag(gam) KS
        const int r = MV::row(t, i);
#pragma unroll
        for (int j = 0; j < MV::TN; ++j) {
            const int cc = MV::col(t, j);
            n1[r * NV + cc] = __fsub_rn(ld_f32(Vt + r * TV + cc), __fmul_rn(v.gam[r], ks[i][j]));
        }
    }
    __syncthreads();
    // ---- c: U = T diag(beta) R
    {
        float u[TM][MV::TN];
        zero(u);
        mm<TM, MV::TN, C>(u, [&](int i, int k) { return __fmul_rn(nT[MV::row(t, i) * NN + k], v.beta[k]); },
                          [&](int k, int j) { return n1[k * NV + MV::col(t, j)]; });
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < MV::TN; ++j) n2[MV::row(t, i) * NV + MV::col(t, j)] = u[i][j];
    }
    // dgam_last = <dS_end, S_b>: fixed per-thread order, then a fixed tree over the CTA
    {
        float sacc = 0.0f;
        for (size_t idx = t; idx < SSZ; idx += kBwdThreads) sacc = __fmaf_rn(__ldg(dSe + idx), __ldg(Sb + idx), sacc);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sacc = __fadd_rn(sacc, __shfl_xor_sync(0xffffffffu, sacc, o));
        if ((t & 31) == 0) red[t >> 5] = sacc;
    }
    __syncthreads();
    // ---- d: dPm = (dO U^T) o lower, into big (stride NN), column partials after it
    float* dpm = big;
    float* colp = big + C * NN;  // [16][C]
    {
        float m[MN::TM][MN::TM];
        zero(m);
        mm<MN::TM, MN::TM, DV>(m, [&](int i, int k) { return ld_f32(Ot + MN::row(t, i) * TV + k); },
                               [&](int k, int j) { return n2[MN::col(t, j) * NV + k]; });
        float rowp[MN::TM], colq[MN::TM];
#pragma unroll
        for (int j = 0; j < MN::TM; ++j) colq[j] = 0.0f;
#pragma unroll
        for (int i = 0; i < MN::TM; ++i) {
            const int r = MN::row(t, i);
            rowp[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < MN::TM; ++j) {
                const int cc = MN::col(t, j);
                const float x = cc <= r ? m[i][j] : 0.0f;
                const float ed = __fmul_rn(x, nP[r * NN + cc]);
                rowp[i] = __fadd_rn(rowp[i], ed);
                colq[j] = __fadd_rn(colq[j], ed);
                // dQK = dPm o E
                dpm[r * NN + cc] = cc <= r ? __fmul_rn(x, decay_exp(__fsub_rn(v.G[r], v.G[cc]))) : 0.0f;
            }
        }
#pragma unroll
        for (int i = 0; i < MN::TM; ++i) {
            const float s = rowgroup_sum(rowp[i]);
            if ((t & 15) == 0) v.edrow[MN::row(t, i)] = s;
        }
#pragma unroll
        for (int j = 0; j < MN::TM; ++j) colp[(t >> 4) * C + MN::col(t, j)] = colq[j];
    }
    float du[TM][MV::TN];  // dU = Pm^T dO (+ diag(d) K dS_end^T below)
    zero(du);
    mm<TM, MV::TN, C>(du, [&](int i, int k) { return nP[k * NN + MV::row(t, i)]; },
                      [&](int k, int j) { return ld_f32(Ot + k * TV + MV::col(t, j)); });
    __syncthreads();
    if (t < C) {  // column sums of dPm o Pm in a fixed order
        float s = 0.0f;
        for (int q = 0; q < 16; ++q) s = __fadd_rn(s, colp[q * C + t]);
        v.edcol[t] = s;
    }
    mm<TM, MK::TN, C>(dq, [&](int i, int k) { return dpm[MK::row(t, i) * NN + k]; },
                      [&](int k, int j) { return ld_f32(Kt + k * TK + MK::col(t, j)); });
    mm<TM, MK::TN, C>(dk, [&](int i, int k) { return dpm[k * NN + MK::row(t, i)]; },
                      [&](int k, int j) { return ld_f32(Qt + k * TK + MK::col(t, j)); });
    // ---- e: dS_end by halves
    for (int hh = 0; hh < 2; ++hh) {
        load_half(dSe, hh);
        mm<TM, MV::TN, DK / 2>(du, [&](int i, int k) {
            const int r = MV::row(t, i);
            return __fmul_rn(v.dd[r], ld_f32(Kt + r * TK + hh * (DK / 2) + k)); },
                               [&](int k, int j) { return big[k * NV + MV::col(t, j)]; });
        float y[TM][MK::HN];
        zero(y);
        mm<TM, MK::HN, DV>(y, [&](int i, int k) { return n2[MK::row(t, i) * NV + k]; },
                           [&](int k, int j) { return big[MK::hlocal(t, j) * NV + k]; });
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = MK::row(t, i);
#pragma unroll
            for (int j = 0; j < MK::HN; ++j) {
                const int cc = MK::hcol(t, hh, j);
                dk[i][hh * MK::HN + j] = __fmaf_rn(v.dd[r], y[i][j], dk[i][hh * MK::HN + j]);
                ddr[i] = __fmaf_rn(y[i][j], ld_f32(Kt + r * TK + cc), ddr[i]);
            }
        }
    }
    __syncthreads();  // U is dead: dU takes its place
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < MV::TN; ++j) n2[MV::row(t, i) * NV + MV::col(t, j)] = du[i][j];
    __syncthreads();
    // ---- f: dT = dU (diag(beta) R)^T into nP (Pm is dead);  TdU = T^T dU
    {
        float m[MN::TM][MN::TM];
        zero(m);
        mm<MN::TM, MN::TM, DV>(m, [&](int i, int k) { return n2[MN::row(t, i) * NV + k]; },
                               [&](int k, int j) { return n1[MN::col(t, j) * NV + k]; });
#pragma unroll
        for (int i = 0; i < MN::TM; ++i)
#pragma unroll
            for (int j = 0; j < MN::TM; ++j) nP[MN::row(t, i) * NN + MN::col(t, j)] = __fmul_rn(m[i][j], v.beta[MN::col(t, j)]);
    }
    float tdu[TM][MV::TN];
    zero(tdu);
    mm<TM, MV::TN, C>(tdu, [&](int i, int k) { return nT[k * NN + MV::row(t, i)]; },
                      [&](int k, int j) { return n2[k * NV + MV::col(t, j)]; });
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int r = MV::row(t, i);
        const bool live = r < p.len;
        float* dvrow = a.dv + ((p.t0 + r) * H + h) * DV;
#pragma unroll
        for (int j = 0; j < MV::TN; ++j) {
            const int cc = MV::col(t, j);
            dbeta[i] = __fmaf_rn(tdu[i][j], n1[r * NV + cc], dbeta[i]);
            if (live) dvrow[cc] = __fmul_rn(v.beta[r], tdu[i][j]);
        }
    }
    __syncthreads();  // R and dU readers are done
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < MV::TN; ++j) n1[MV::row(t, i) * NV + MV::col(t, j)] = tdu[i][j];
    // ---- g: S_b by halves again: Z = TdU S_b
    for (int hh = 0; hh < 2; ++hh) {
        load_half(Sb, hh);
        float y[TM][MK::HN];
        zero(y);
        mm<TM, MK::HN, DV>(y, [&](int i, int k) { return n1[MK::row(t, i) * NV + k]; },
                           [&](int k, int j) { return big[MK::hlocal(t, j) * NV + k]; });
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = MK::row(t, i);
            const float bg = __fmul_rn(v.beta[r], v.gam[r]);
            float kz = 0.0f;
#pragma unroll
            for (int j = 0; j < MK::HN; ++j) {
                const int cc = MK::hcol(t, hh, j);
                dk[i][hh * MK::HN + j] = __fmaf_rn(-bg, y[i][j], dk[i][hh * MK::HN + j]);
                kz = __fmaf_rn(y[i][j], ld_f32(Kt + r * TK + cc), kz);
            }
            dgam[i] = __fmaf_rn(-v.beta[r], kz, dgam[i]);
        }
    }
    __syncthreads();
    // ---- h: X = T^T dT into big;  dA = -(X T^T) o strict lower
    {
        float m[MN::TM][MN::TM];
        zero(m);
        mm<MN::TM, MN::TM, C>(m, [&](int i, int k) { return nT[k * NN + MN::row(t, i)]; },
                              [&](int k, int j) { return nP[k * NN + MN::col(t, j)]; });
#pragma unroll
        for (int i = 0; i < MN::TM; ++i)
#pragma unroll
            for (int j = 0; j < MN::TM; ++j) big[MN::row(t, i) * NN + MN::col(t, j)] = m[i][j];
    }
    __syncthreads();
    {
        float m[MN::TM][MN::TM];
        zero(m);
        mm<MN::TM, MN::TM, C>(m, [&](int i, int k) { return big[MN::row(t, i) * NN + k]; },
                              [&](int k, int j) { return nT[MN::col(t, j) * NN + k]; });
        float rowp[MN::TM], rowb[MN::TM], colq[MN::TM];
#pragma unroll
        for (int j = 0; j < MN::TM; ++j) colq[j] = 0.0f;
        __syncthreads();  // every reader of dT (nP) and X (big) is done
#pragma unroll
        for (int i = 0; i < MN::TM; ++i) {
            const int r = MN::row(t, i);
            rowp[i] = rowb[i] = 0.0f;
#pragma unroll
            for (int j = 0; j < MN::TM; ++j) {
                const int cc = MN::col(t, j);
                const float da = cc < r ? -m[i][j] : 0.0f;
                const float l = nL[r * NN + cc];
                rowb[i] = __fmaf_rn(da, l, rowb[i]);
                const float dl = __fmul_rn(v.beta[r], da);
                const float ed = __fmul_rn(dl, l);
                rowp[i] = __fadd_rn(rowp[i], ed);
                colq[j] = __fadd_rn(colq[j], ed);
                nP[r * NN + cc] = cc < r ? __fmul_rn(dl, decay_exp(__fsub_rn(v.G[r], v.G[cc]))) : 0.0f;  // dKK
            }
        }
#pragma unroll
        for (int i = 0; i < MN::TM; ++i) {
            const float s = rowgroup_sum(rowp[i]);
            const float sb = rowgroup_sum(rowb[i]);
            if ((t & 15) == 0) {
                v.edrow[MN::row(t, i)] = __fadd_rn(v.edrow[MN::row(t, i)], s);
                v.dbeta[MN::row(t, i)] = sb;
            }
        }
#pragma unroll
        for (int j = 0; j < MN::TM; ++j) colp[(t >> 4) * C + MN::col(t, j)] = colq[j];
    }
    __syncthreads();
    if (t < C) {
        float s = 0.0f;
        for (int q = 0; q < 16; ++q) s = __fadd_rn(s, colp[q * C + t]);
        v.edcol[t] = __fadd_rn(v.edcol[t], s);
    }
    mm<TM, MK::TN, C>(dk, [&](int i, int k) {
        const int r = MK::row(t, i);
        return __fadd_rn(nP[r * NN + k], nP[k * NN + r]); },
                      [&](int k, int j) { return ld_f32(Kt + k * TK + MK::col(t, j)); });
    // ---- i: per-token sums, then the gates
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const float sg = rowgroup_sum(dgam[i]);
        const float sd = rowgroup_sum(ddr[i]);
        const float sb = rowgroup_sum(dbeta[i]);
        if ((t & 15) == 0) {
            const int r = MK::row(t, i);
            v.dgam[r] = sg;
            v.ddv[r] = sd;
            v.dbeta[r] = __fadd_rn(v.dbeta[r], sb);
        }
    }
    __syncthreads();
    if (t == 0) {
        float dlast = 0.0f;
        for (int w = 0; w < kBwdThreads / 32; ++w) dlast = __fadd_rn(dlast, red[w]);
        float sdd = 0.0f;
        for (int r = 0; r < C; ++r) sdd = __fmaf_rn(v.dd[r], v.ddv[r], sdd);
        float acc = 0.0f;  // reverse cumulative sum of dG
        for (int r = C - 1; r >= 0; --r) {
            float dG = __fmul_rn(v.gam[r], r == C - 1 ? __fadd_rn(v.dgam[r], dlast) : v.dgam[r]);
            dG = __fsub_rn(dG, __fmul_rn(v.dd[r], v.ddv[r]));
            dG = __fadd_rn(dG, __fsub_rn(v.edrow[r], v.edcol[r]));
            if (r == C - 1) dG = __fadd_rn(dG, sdd);
            acc = __fadd_rn(acc, dG);
            v.dG[r] = acc;
        }
    }
    __syncthreads();
    if (t < p.len) {
        a.dg[(p.t0 + t) * H + h] = v.dG[t];
        a.dbeta[(p.t0 + t) * H + h] = v.dbeta[t];
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int r = MK::row(t, i);
        if (r >= p.len) continue;
        float* qrow = a.dq + ((p.t0 + r) * H + h) * DK;
        float* krow = a.dk + ((p.t0 + r) * H + h) * DK;
#pragma unroll
        for (int j = 0; j < MK::TN; ++j) {
            qrow[MK::col(t, j)] = dq[i][j];
            krow[MK::col(t, j)] = dk[i][j];
        }
    }
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

template <int DK, int DV, int C, typename T>
bool backward_fits()
{
    return Kb3Cfg<DK, DV, C, T>::bytes <= 232448 && Kb1Cfg<DK, DV, C, T>::bytes <= 232448;
}

template <int DK, int DV, int C, typename T>
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s)
{
    if constexpr (Kb3Cfg<DK, DV, C, T>::bytes > 232448 || Kb1Cfg<DK, DV, C, T>::bytes > 232448) {
        return cudaErrorInvalidConfiguration;
    } else {
        PrefillArgs pa{};
        pa.cu_seqlens = a.cu_seqlens;
        pa.n_seqs = a.n_seqs;
        pa.total_tokens = a.total_tokens;
        pa.boundary_capacity = a.boundary_capacity;
        pa.cu_chunks = a.cu_chunks;
        pa.status = a.status;
        pa.ready = a.ready;  // (k0 zeroes the hand-off counters)
        pa.max_chunks = a.max_chunks;
        pa.H = a.H;
        profile_mark(0, s);
        cudaError_t e = launch_chunk_index(pa, C, nullptr, nullptr, nullptr, s);
        if (e != cudaSuccess) return e;
        profile_mark(1, s);
        constexpr bool kTc = DK == 128 && DV == 128 && C == 64 && std::is_same<T, __nv_bfloat16>::value;
        const dim3 grid((unsigned)a.max_chunks, (unsigned)a.H);
        if constexpr (kTc) {
            e = launch_chunk_maps_tc(a, s);  // the tensor-core form of kb1 for this shape
        } else {
            auto k1 = kb1_chunk_maps<DK, DV, C, T>;
            if ((e = set_smem(k1, Kb1Cfg<DK, DV, C, T>::bytes)) != cudaSuccess) return e;
            k1<<<grid, kBwdThreads, Kb1Cfg<DK, DV, C, T>::bytes, s>>>(a);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
        profile_mark(2, s);
        if constexpr (kTc) {
            // the chain and the tensor-core form of kb3 in one launch (the chain's and the
            // gradients' times are not separable: both events mark its end)
            profile_mark(3, s);
            e = launch_chain_and_grads_tc(a, s);
        } else {
            auto k2 = kb2_reverse_chain<DK, DV>;
            // (the dynamic shared memory also caps the CTAs per SM so their TMEM columns fit)
            const size_t sm2 = std::max<size_t>(RevChainCfg<DK, DV>::bytes, tmem_cap_smem(RevChainCfg<DK, DV>::TMEM_COLS));
            if ((e = set_smem(k2, sm2)) != cudaSuccess) return e;
            k2<<<(unsigned)((int64_t)a.n_seqs * a.H), kBwdThreads, sm2, s>>>(a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            profile_mark(3, s);
            auto k3 = kb3_chunk_grads<DK, DV, C, T>;
            if ((e = set_smem(k3, Kb3Cfg<DK, DV, C, T>::bytes)) != cudaSuccess) return e;
            k3<<<grid, kBwdThreads, Kb3Cfg<DK, DV, C, T>::bytes, s>>>(a);
            e = cudaGetLastError();
        }
        profile_mark(4, s);
        return e;
    }
}

#define CPR_INST_BACKWARD(DK, DV, C)                                                                 \
    template cudaError_t launch_backward<DK, DV, C, float>(const BackwardArgs&, cudaStream_t);      \
    template cudaError_t launch_backward<DK, DV, C, __nv_bfloat16>(const BackwardArgs&, cudaStream_t); \
    template bool backward_fits<DK, DV, C, float>();                                                 \
    template bool backward_fits<DK, DV, C, __nv_bfloat16>();
CPR_FOR_EACH_SHAPE(CPR_INST_BACKWARD)

}  // namespace cpr
