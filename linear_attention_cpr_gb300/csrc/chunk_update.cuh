// chunk_update.cuh — the state-independent half of the chunk update U, as CTA-wide
// device routines called both by prefill's chunk-prep kernel and by decode's resync
// kernel.  Element sequences are those of numerics.cuh.
#pragma once

#include <type_traits>

#include "numerics.cuh"
#include "tc.cuh"

namespace cpr {

// Shared-memory scratch of one chunk's prep: keys (fp32, row stride DK + 4), A, and the
// per-token vectors.  `g_in` holds the chunk's g on entry and G on exit.
template <int DK, int C>
struct PrepSmem {
    static constexpr int KS = DK + 4;
    static constexpr size_t floats = (size_t)C * KS + (size_t)C * C + 4 * (size_t)C;
    float* kf;   // [C][KS]
    float* A;    // [C][C], transposed: A[i * C + r] = A_ri
    float* G;    // [C]  g on entry, G (sequential cumulative sum) after chunk_decays_and_A
    float* be;   // [C]  beta_r * e_r
    float* bs;   // [C]  beta_r
    float* dvs;  // [C]  d_r
    __device__ explicit PrepSmem(float* base)
        : kf(base), A(base + C * KS), G(A + C * C), be(G + C), bs(be + C), dvs(bs + C) {}
    // keys and A at `base`, the four per-token vectors at `vec`
    __device__ PrepSmem(float* base, float* vec)
        : kf(base), A(base + C * KS), G(vec), be(vec + C), bs(vec + 2 * C), dvs(vec + 3 * C) {}
};

// The key Gram matrix kk = K K^T of one chunk on the tensor cores: one M = 64, N = C,
// K = DK tcgen05 product (rows r, columns i) of the keys' bf16 splits.  bf16 keys are
// their own hi split (lo = 0), so one product is the whole sum; fp32 keys, and keys
// normalised in the kernel, take three (hi*hi + hi*lo + lo*hi).  The tile holds C rows per split; rows C..63 of the M = 64
// A operand read whatever follows (their accumulator rows are never used), so the
// region must span SPAN bytes.
template <int DK, int C, typename T>
struct KKCfg {
    static constexpr int NSPLIT = std::is_same<T, __nv_bfloat16>::value ? 1 : 2;
    static constexpr uint32_t SPLIT = C * DK * 2;
    static constexpr uint32_t SPAN = SPLIT + 64 * DK * 2;  // fp32 keys, the larger case
    static constexpr uint32_t idesc = tc::idesc_bf16(64, C);
};

// G, e, d, beta*e and the strictly lower-triangular A (stored transposed: At[i][r] =
// A_ri) from kf, g (in G) and beta (in bs); ktile: scratch of KKCfg::SPAN bytes for the
// key tile; TMEM columns [tmem, tmem + C) hold kk; the product's completion arrives on
// mbar with the given parity.  KEYS_AS_GIVEN: kf holds the keys exactly as stored (not
// normalised in the kernel).  All DK + DV threads; contains __syncthreads.  Returns
// false (uniformly) when the product's wait timed out; A is then undefined.
template <int DK, int DV, int C, typename T, bool KEYS_AS_GIVEN>
__device__ __forceinline__ bool chunk_decays_and_A(const PrepSmem<DK, C>& s, unsigned char* ktile, uint32_t tmem,
                                                   uint64_t* mbar, uint32_t parity)
{
    using KC = KKCfg<DK, C, T>;
    constexpr bool three = KC::NSPLIT == 2 || !KEYS_AS_GIVEN;
    constexpr int KS = PrepSmem<DK, C>::KS;
    constexpr int NWARP = (DK + DV) / 32;
    static_assert(NWARP >= 4 || C <= 16 * NWARP, "every TMEM lane quadrant holding kk rows needs a warp");
    const int tid = threadIdx.x;
    __syncthreads();
    for (int idx = tid; idx < C * (DK / 8); idx += DK + DV) {
        const int r = idx % C, c0 = (idx / C) * 8;
        float xs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = s.kf[r * KS + c0 + e];
        const uint32_t off = tc::tile_off<2>(r, c0, DK);
        tc::split8_store(xs, ktile + off, three ? ktile + KC::SPLIT + off : nullptr);
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t SBO = (DK / 8) * 128;
        const uint32_t ko = tc::smem_u32(ktile);
        const uint32_t ha[3] = {0u, 0u, 1u}, hb[3] = {0u, 1u, 0u};
#pragma unroll
        for (int p = 0; p < (three ? 3 : 1); ++p)
#pragma unroll
            for (int k = 0; k < DK / 16; ++k)
                tc::mma_bf16(tmem, tc::sdesc(ko + ha[p] * KC::SPLIT + k * 256, 128, SBO),
                             tc::sdesc(ko + hb[p] * KC::SPLIT + k * 256, 128, SBO), KC::idesc, (p | k) ? 1u : 0u);
        tc::commit(mbar);
        // sequential cumulative sum, in registers, while the product runs
        float gr[C];
#pragma unroll
        for (int r = 0; r < C; r += 4) {
            const float4 g4 = *reinterpret_cast<const float4*>(s.G + r);
            gr[r] = g4.x;
            gr[r + 1] = g4.y;
            gr[r + 2] = g4.z;
            gr[r + 3] = g4.w;
        }
#pragma unroll
        for (int r = 1; r < C; ++r) gr[r] = __fadd_rn(gr[r - 1], gr[r]);
#pragma unroll
        for (int r = 0; r < C; r += 4) *reinterpret_cast<float4*>(s.G + r) = make_float4(gr[r], gr[r + 1], gr[r + 2], gr[r + 3]);
    }
    __syncthreads();
    if (tid < C) {
        s.be[tid] = __fmul_rn(s.bs[tid], decay_exp(s.G[tid]));
        s.dvs[tid] = decay_exp(__fsub_rn(s.G[C - 1], s.G[tid]));
    }
    const bool ok = __syncthreads_and(tc::mbar_wait(mbar, parity));
    if (ok) {
        tc::fence_after_sync();
        constexpr int WPQ = NWARP >= 8 ? 2 : 1;  // warps per TMEM lane quadrant
        constexpr int CPW = C / WPQ, CPT = CPW / 2;
        const int warp = tid >> 5, q = warp & 3, hh = warp >> 2;
        if (warp < 4 * WPQ && 16 * q < C) {  // warp-uniform
            float kk[CPT];
            tc::tmem_ld_16x2<CPT>(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(hh * CPW), kk);
            const int r = 16 * q + (tid & 15), i0 = hh * CPW + ((tid >> 4) & 1) * CPT;
            const float br = s.bs[r], Gr = s.G[r];
#pragma unroll
            for (int e = 0; e < CPT; ++e)
                if (i0 + e < r) s.A[(i0 + e) * C + r] = a_entry(br, Gr, s.G[i0 + e], kk[e]);
        }
        tc::fence_before_sync();
    }
    __syncthreads();
    return ok;
}

// Column `col` of the right-hand sides [W0 | U0] (col < DK: W0_r[col] = (beta_r e_r)
// k_r[col], else U0_r[n] = beta_r v_r[n] with n = col - DK).  V element (r, n) of the
// chunk is vbase[r * vstride + n].
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
}

// ======================================================================================
// Tensor-core half of the chunk update.  With W = T W0 and U~ = T U0 (the WY relations
// above; T = (I + A)^-1, W0_r = (beta_r e_r) k_r, U0_r = beta_r v_r), U is applied in the
// matrix form
//     S_new = S_b M + B,   M = gamma I - W^T (D K),   B = U~^T (D K),   D = diag(d_r),
// with W^T (D K) = W0^T Z and U~^T (D K) = U0^T Z, Z = T^T (D K):
//   prep (state independent), tcgen05 products with K = C:
//        Z^T = (D K)^T T   (M = 128 rows c, N = C)
//        X = Z^T W0        (M = 128 rows c, N = DK)   ->  Mt = gamma I - X   (Mt[c][c'] = M[c'][c])
//        B = U0^T Z        (M = 128 rows i, N = DK)
//        bf16 hi/lo splits of every operand (tc::split_f32), three products
//        hi*hi + hi*lo + lo*hi accumulated in fp32 in TMEM; Mt is split the same way
//        (the chain's B operand image), B kept fp32, stored [DK][DV] like a state.
//   chain step: D = S_b M as one tcgen05 product per (sequence, head) (M = 128 value
//        rows, N = DK, K = DK), the state tile holding S_b's bf16 splits, three products
//        as above; then S_new[i][c] = D[i][c] + B[i][c] (one add).
// Both products have a fixed instruction sequence, so prefill's kernels and decode's
// resync produce the same bits.  Rows beyond DK (or DV) of the M = 128 products are zero.
// ======================================================================================
template <int DK, int DV, int C>
struct UCfg {
    static constexpr int MPAD = 128;
    static constexpr int NB = DK + DV;
    static constexpr uint32_t AOP_SPLIT = MPAD * C * 2;  // bf16 (D K)^T tile, one split
    static constexpr uint32_t BOP_SPLIT = NB * C * 2;    // bf16 [W | U~]^T tile, one split
    static constexpr uint32_t MT_SPLIT = DK * DK * 2;    // bf16 Mt tile [DK][DK], one split
    static constexpr uint32_t MT_BYTES = 2 * MT_SPLIT;
    static constexpr uint32_t BT_BYTES = DK * DV * 4;    // fp32 B, stored [DK][DV] like a state
    // prep shared memory: R1 = keys + A (FP32 phase), later the [W | U~] operand
    static constexpr uint32_t R1A = (uint32_t)(sizeof(float) * ((size_t)C * PrepSmem<DK, C>::KS + (size_t)C * C));
    static constexpr uint32_t mx(uint32_t x, uint32_t y) { return x > y ? x : y; }
    // R1 also stages the prep outputs (M^T image, then B) before their bulk stores
    static constexpr uint32_t R1 = mx(mx(R1A, 2 * BOP_SPLIT), mx(2 * DK * DK * 2, DK * DV * 4));
    static constexpr uint32_t AOP_OFF = (R1 + 1023) / 1024 * 1024;
    // the (D K)^T operand region first holds the key tile of the kk product
    static constexpr uint32_t AOP_REGION = mx(2 * AOP_SPLIT, KKCfg<DK, C, float>::SPAN);
    static constexpr uint32_t VEC_OFF = AOP_OFF + AOP_REGION;
    // the (D K)^T region also holds T (fp32, row stride C + 1) and the blocked inversion's
    // scratch while T is computed
    static_assert((uint32_t)(4 * (((C * (C + 1) + 3) / 4) * 4 + 256 * (C / 16 - 1))) <= AOP_REGION,
                  "T and its scratch fit the operand region");
    static constexpr uint32_t PREP_BYTES = VEC_OFF + 4 * C * 4;
    static constexpr uint32_t TMEM_COLS = mx(2 * DK, C) <= 32 ? 32 : mx(2 * DK, C) <= 64 ? 64 : mx(2 * DK, C) <= 128 ? 128 : 256;
    // decode resync (prep and one chain step in one CTA): [R1 | Mt] [Aop | Bt] [vectors] [values]
    static constexpr uint32_t up1k(uint32_t x) { return (x + 1023) / 1024 * 1024; }
    static constexpr uint32_t RS_BT_OFF = up1k(R1 > MT_BYTES ? R1 : MT_BYTES);
    static constexpr uint32_t RS_VEC_OFF = up1k(RS_BT_OFF + mx(AOP_REGION, BT_BYTES));
    static constexpr uint32_t RS_BAR_OFF = up1k(RS_VEC_OFF + 4 * C * 4);
    static constexpr uint32_t RS_V_OFF = RS_BAR_OFF + 64;  // the chunk's values, as stored
    static constexpr uint32_t rs_bytes(uint32_t value_bytes) { return RS_V_OFF + C * DV * value_bytes; }
    static constexpr uint32_t PREP_BAR_OFF = (PREP_BYTES + 15) / 16 * 16;
    static constexpr uint32_t PREP_SMEM = PREP_BAR_OFF + 64;
    static constexpr uint32_t prep_idesc = tc::idesc_bf16(MPAD, DK);
};

// Build both prep operands in shared memory from the chunk's keys (s.kf, fp32), g (s.G)
// and beta (s.bs); V element (r, n) at vbase[r * vstride + n]; KEYS_AS_GIVEN as for
// chunk_decays_and_A.  All DK + DV threads;
// contains __syncthreads.  Three phases of mbar (the key Gram product, the Z product),
// counted by `phase`; TMEM columns [tmem, tmem + C) are scratch.  On a true return aop
// holds Z^T = (D K)^T T and bop the right-hand sides [W0 | U0]^T, both as bf16 splits
// visible to the tensor cores; false (uniform) means a product timed out.
template <int DK, int DV, int C, typename T, bool KEYS_AS_GIVEN>
__device__ __forceinline__ bool prep_operands(const PrepSmem<DK, C>& s, unsigned char* aop, unsigned char* bop,
                                              const T* vbase, size_t vstride, uint32_t tmem, uint64_t* mbar,
                                              uint32_t& phase)
{
    using U = UCfg<DK, DV, C>;
    constexpr int KS = PrepSmem<DK, C>::KS;
    constexpr uint32_t TT_SPLIT = C * C * 2;  // one bf16 split of the T^T tile
    const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
    if (!chunk_decays_and_A<DK, DV, C, T, KEYS_AS_GIVEN>(s, aop, tmem, mbar, phase & 1)) return false;
    ++phase;
    // T = (I + A)^-1 by blocks with every thread (numerics.cuh), into the (D K)^T operand's
    // region, which the key Gram product no longer needs
    constexpr int TS = C + 1;
    float* tfull = reinterpret_cast<float*>(aop);
    invert_unit_lower<C, TS>(s.A, tfull, tfull + ((C * TS + 3) / 4) * 4, tid, nt);
    // A is dead: its space holds T^T (rows j, K = r), bf16 splits
    unsigned char* tt = reinterpret_cast<unsigned char*>(s.A);
    float x[C];
    if (tid < C) {
#pragma unroll
        for (int r = 0; r < C; ++r) x[r] = tfull[r * TS + tid];
#pragma unroll
        for (int r0 = 0; r0 < C; r0 += 8) {
            const uint32_t off = tc::tile_off<2>(tid, r0, C);
            tc::split8_store(*reinterpret_cast<const float(*)[8]>(x + r0), tt + off, tt + TT_SPLIT + off);
        }
    }
    __syncthreads();  // T is read: its region takes the (D K)^T operand
    // (D K)^T rows c: d_r * k_r[c] (zero rows beyond DK)
    for (int row = tid; row < U::MPAD; row += nt) {
#pragma unroll
        for (int r0 = 0; r0 < C; r0 += 8) {
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = row < DK ? __fmul_rn(s.dvs[r0 + e], s.kf[(r0 + e) * KS + row]) : 0.0f;
            const uint32_t off = tc::tile_off<2>(row, r0, C);
            tc::split8_store(xs, aop + off, aop + U::AOP_SPLIT + off);
        }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {  // Z^T = (D K)^T T into TMEM columns [0, C): M = 128 rows c, N = C, K = C
        tc::fence_after_sync();
        constexpr uint32_t SBO = (C / 8) * 128;
        constexpr uint32_t idesc = tc::idesc_bf16(U::MPAD, C);
        const uint32_t ao = tc::smem_u32(aop), to = tc::smem_u32(tt);
        const uint32_t ha[3] = {0u, 0u, 1u}, hb[3] = {0u, 1u, 0u};
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
            for (int k = 0; k < C / 16; ++k)
                tc::mma_bf16(tmem, tc::sdesc(ao + ha[p] * U::AOP_SPLIT + k * 256, 128, SBO),
                             tc::sdesc(to + hb[p] * TT_SPLIT + k * 256, 128, SBO), idesc, (p | k) ? 1u : 0u);
        tc::commit(mbar);
    }
    chunk_column<DK, DV, C, T>(s, tid, vbase, vstride, x);  // this thread's row of [W0 | U0]^T, while Z runs
    bool ok = __syncthreads_and(tc::mbar_wait(mbar, phase & 1));
    ++phase;
    if (!ok) return false;
    // Z^T (fp32 in TMEM, row c = lane) -> bf16 splits over the (D K)^T operand
    tc::fence_after_sync();
    {
        const int q = warp & 3, row = q * 32 + lane;
        for (int g = warp >> 2; g * 32 < C; g += (nt / 32 + 3) / 4) {  // warp-uniform
            float v[32];
            tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(g * 32), v);
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {
                if (g * 32 + e8 < C) {
                    const uint32_t off = tc::tile_off<2>(row, g * 32 + e8, C);
                    tc::split8_store(*reinterpret_cast<const float(*)[8]>(v + e8), aop + off, aop + U::AOP_SPLIT + off);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();  // keys and T^T are dead: their space becomes the [W0 | U0]^T operand
#pragma unroll
    for (int r0 = 0; r0 < C; r0 += 8) {
        const uint32_t off = tc::tile_off<2>(tid, r0, C);
        tc::split8_store(*reinterpret_cast<const float(*)[8]>(x + r0), bop + off, bop + U::BOP_SPLIT + off);
    }
    tc::fence_proxy_async();
    __syncthreads();
    return true;
}

// One thread: both prep products (X into TMEM columns [0, DK), B into [DK, 2 DK)), then
// commit to mbar.  aop = Z^T tile (128 rows c, K = C); bop = [W0 | U0]^T tile (rows
// 0..DK-1 = W0^T, rows DK.. = U0^T).
template <int DK, int DV, int C>
__device__ __forceinline__ void prep_mma(uint32_t tmem, const unsigned char* aop, const unsigned char* bop,
                                         uint64_t* mbar)
{
    using U = UCfg<DK, DV, C>;
    constexpr uint32_t SBO = (C / 8) * 128;
    const uint32_t ao = tc::smem_u32(aop), bo = tc::smem_u32(bop);
    const uint32_t uo = bo + (DK / 8) * SBO;  // U~^T rows start after the DK rows of W^T
    const uint32_t ha[3] = {0u, 0u, 1u}, hb[3] = {0u, 1u, 0u};  // hi*hi, hi*lo, lo*hi
    tc::fence_after_sync();
#pragma unroll
    for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
            tc::mma_bf16(tmem, tc::sdesc(ao + ha[p] * U::AOP_SPLIT + k * 256, 128, SBO),
                         tc::sdesc(bo + hb[p] * U::BOP_SPLIT + k * 256, 128, SBO), U::prep_idesc, (p | k) ? 1u : 0u);
#pragma unroll
    for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int k = 0; k < C / 16; ++k)
            tc::mma_bf16(tmem + DK, tc::sdesc(uo + ha[p] * U::BOP_SPLIT + k * 256, 128, SBO),
                         tc::sdesc(ao + hb[p] * U::AOP_SPLIT + k * 256, 128, SBO), U::prep_idesc, (p | k) ? 1u : 0u);
    tc::commit(mbar);
}

// All threads, after the prep products completed: the Mt image (bf16 splits; rows c,
// K = c') and B (fp32, element (i, c) at c * DV + i, the layout of a state).  With a
// shared-memory staging area of at least Mt's bytes (its previous contents dead), Mt is
// assembled there and written to the global destination with bulk copies; without one
// (staging NULL) it is written directly.  B is written directly (consecutive lanes hold
// consecutive rows i, so each warp store is 128 contiguous bytes).  Contains
// __syncthreads.
template <int DK, int DV, int C>
__device__ __forceinline__ void prep_epilogue(uint32_t tmem, float gamma, unsigned char* mt_out, float* b_out,
                                              unsigned char* staging)
{
    using U = UCfg<DK, DV, C>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    tc::fence_after_sync();
    constexpr int NG = 2 * DK / 32;  // 32-column groups: X then B
    const int q = warp & 3;
    const int row = q * 32 + lane;  // this thread's TMEM lane
    for (int part = 0; part < 2; ++part) {  // 0: Mt, 1: B
        unsigned char* mt_dst = staging ? staging : mt_out;
        float* b_dst = b_out;
        if (q * 32 < (part == 0 ? DK : DV)) {
            for (int g = warp >> 2; g < NG; g += (nw + 3) / 4) {
                if ((g < DK / 32) != (part == 0)) continue;
                float v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(g * 32), v);
                if (part == 0) {  // Mt[c][c'] = gamma [c == c'] - X[c][c'], row c = this lane
                    if (row >= DK) continue;
                    const int col0 = g * 32;
#pragma unroll
                    for (int e8 = 0; e8 < 32; e8 += 8) {
                        float xs[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int cc = col0 + e8 + e;
                            xs[e] = (cc == row) ? __fsub_rn(gamma, v[e8 + e]) : -v[e8 + e];
                        }
                        const uint32_t off = tc::tile_off<2>(row, col0 + e8, DK);
                        tc::split8_store(xs, mt_dst + off, mt_dst + U::MT_SPLIT + off);
                    }
                } else {  // B[i][c] at c * DV + i, row i = this lane (a warp writes 128 contiguous bytes)
                    if (row >= DV) continue;
                    float* dst = b_dst + (size_t)(g * 32 - DK) * DV + row;
#pragma unroll
                    for (int e = 0; e < 32; ++e) dst[(size_t)e * DV] = v[e];
                }
            }
        }
        if (staging && part == 0) {  // bulk stores of the assembled Mt, in flight while B is stored
            tc::fence_proxy_async();
            __syncthreads();
            if (tid == 0) {
                for (uint32_t off = 0; off < U::MT_BYTES; off += 16384)
                    tc::bulk_s2g(mt_out + off, staging + off, min(16384u, U::MT_BYTES - off));
                tc::bulk_commit();
            }
        }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
}

// The chain product: one M = 128 product per (sequence, head), value row i in TMEM lane i
// (rows beyond DV read a zero state tile and are never stored), the same instruction
// shape in prefill's chain CTAs and in decode's resync.
constexpr int kChainRows = 128;

// One thread: the chain product D = S M into TMEM columns [tmem_d, tmem_d + DK), with S as
// the A operand in TMEM (bf16 hi in columns [tmem_a, tmem_a + DK/2), lo in
// [tmem_a + DK/2, tmem_a + DK), row i in lane i, written by chain_put_a) and the M^T
// image mt (bf16 hi / lo [DK][DK], K-major) as B; three products hi*hi + hi*lo + lo*hi;
// commit to mbar.
template <int DK>
__device__ __forceinline__ void chain_mma(uint32_t tmem_d, uint32_t tmem_a, const unsigned char* mt, uint64_t* mbar)
{
    constexpr uint32_t SBO = (DK / 8) * 128, MT_SPLIT = DK * DK * 2;
    constexpr uint32_t idesc = tc::idesc_bf16(kChainRows, DK);
    const uint32_t mo = tc::smem_u32(mt);
    const uint32_t ha[3] = {0u, 0u, DK / 2}, hm[3] = {0u, 1u, 0u};
    tc::fence_after_sync();
#pragma unroll
    for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int k = 0; k < DK / 16; ++k)
            tc::mma_bf16_ta(tmem_d, tmem_a + ha[p] + k * 8, tc::sdesc(mo + hm[p] * MT_SPLIT + k * 256, 128, SBO), idesc,
                            (p | k) ? 1u : 0u);
    tc::commit(mbar);
}

// Epilogue of the chain product across NW warps: warp w reads TMEM lane quadrant w % 4
// (rows 32 (w % 4) .. +31, one per lane) and column part w / QW of CP parts; thread t takes
// row 32 ((t / 32) % 4) + t % 32 and the CPT consecutive columns from (t / 32 / QW) CPT.
// With fewer than four warps only the first NW quadrants (rows < 32 NW) are covered.
template <int DK, int NW>
struct ChainMap {
    static constexpr int QW = NW < 4 ? NW : 4;
    static constexpr int CP = NW / QW;
    static constexpr int CPT = DK / CP;                    // values per thread
    static constexpr int BLK = CPT < 32 ? CPT : 32;        // columns per tcgen05.ld 32x32b
    static constexpr int ROWS = 32 * QW;                   // rows covered
    static_assert(CPT % 16 == 0 && CPT % BLK == 0, "whole 32x32b blocks of paired columns");
    static __device__ __forceinline__ int row(int t) { return 32 * ((t >> 5) & 3) + (t & 31); }
    static __device__ __forceinline__ int col0(int t) { return ((t >> 5) / QW) * CPT; }
    static __device__ __forceinline__ uint32_t lanes(int t) { return (uint32_t)(((t >> 5) & 3) * 32) << 16; }
};

// This thread's accumulator values from TMEM columns at tmem_col.
template <int DK, int NW>
__device__ __forceinline__ void chain_acc(uint32_t tmem_col, int t, float (&v)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
#pragma unroll
    for (int b = 0; b < Mp::CPT / Mp::BLK; ++b) {
        float x[Mp::BLK];
        tc::tmem_ld_32x32b<Mp::BLK>(tmem_col + Mp::lanes(t) + (uint32_t)(Mp::col0(t) + b * Mp::BLK), x);
#pragma unroll
        for (int e = 0; e < Mp::BLK; ++e) v[b * Mp::BLK + e] = x[e];
    }
}

// This thread's B values read from global memory: bt is a chunk's B (element (i, c) at
// c * DV + i); rows beyond DV get zeros (never stored).
template <int DK, int DV, int NW>
__device__ __forceinline__ void chain_load_b(const float* __restrict__ bt, int t, float (&b)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
    const int i = Mp::row(t), c0 = Mp::col0(t);
#pragma unroll
    for (int e = 0; e < Mp::CPT; ++e) b[e] = i < DV ? __ldg(bt + (size_t)(c0 + e) * DV + i) : 0.0f;
}

// S_new = D + B for this thread's values, B already in registers (as chain_values).
template <int DK, int NW>
__device__ __forceinline__ void chain_values_reg(uint32_t tmem_col, int t, const float (&b)[ChainMap<DK, NW>::CPT],
                                                 float (&v)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
    chain_acc<DK, NW>(tmem_col, t, v);
#pragma unroll
    for (int e = 0; e < Mp::CPT; ++e) v[e] = __fadd_rn(v[e], b[e]);
}

// S_new = D + B for this thread's values, B read from a [DK][DV] fp32 image in shared
// memory (element (c, i) of B at c * DV + i; rows beyond DV add zero and are never stored).
template <int DK, int DV, int NW>
__device__ __forceinline__ void chain_values_smem(uint32_t tmem_col, int t, const float* sb,
                                                  float (&v)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
    chain_acc<DK, NW>(tmem_col, t, v);
    const int i = Mp::row(t), c0 = Mp::col0(t);
#pragma unroll
    for (int e = 0; e < Mp::CPT; ++e) v[e] = __fadd_rn(v[e], i < DV ? sb[(c0 + e) * DV + i] : 0.0f);
}

// This thread's values of a stored [DK][DV] fp32 state; zeros beyond DV or for a NULL
// source.
template <int DK, int DV, int NW>
__device__ __forceinline__ void chain_load_state(const float* src, int t, float (&v)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
    const int i = Mp::row(t), c0 = Mp::col0(t);
#pragma unroll
    for (int e = 0; e < Mp::CPT; ++e) v[e] = (src && i < DV) ? src[(size_t)(c0 + e) * DV + i] : 0.0f;
}

// Write this thread's values as its row of the A operand in TMEM: bf16 hi / lo splits
// (tc::split_f32, lo truncated to its upper 16 bits), two values per 32-bit column (the
// value of column c in TMEM column c / 2, even c in the low half), hi in
// [tmem_a, tmem_a + DK/2), lo in [tmem_a + DK/2, tmem_a + DK); then wait for the stores.
template <int DK, int NW>
__device__ __forceinline__ void chain_put_a(uint32_t tmem_a, int t, const float (&v)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
    constexpr int W = Mp::BLK / 2;
#pragma unroll
    for (int b = 0; b < Mp::CPT / Mp::BLK; ++b) {
        uint32_t hi[W], lo[W];
#pragma unroll
        for (int e = 0; e < W; ++e) {
            float h0, l0, h1, l1;
            tc::split_f32(v[b * Mp::BLK + 2 * e], h0, l0);
            tc::split_f32(v[b * Mp::BLK + 2 * e + 1], h1, l1);
            hi[e] = tc::pack_upper(h0, h1);
            lo[e] = tc::pack_upper(l0, l1);
        }
        const uint32_t base = tmem_a + Mp::lanes(t) + (uint32_t)((Mp::col0(t) + b * Mp::BLK) / 2);
        tc::tmem_st_32x32b<W>(base, hi);
        tc::tmem_st_32x32b<W>(base + DK / 2, lo);
    }
    tc::tmem_wait_st();
}

// Block b of this thread's values (columns col0 + b BLK .. + BLK) of a stored [DK][DV]
// state written as its part of the A operand: the blockwise form of chain_load_state and
// chain_put_a (fewer live registers; the same values and TMEM contents).
template <int DK, int DV, int NW>
__device__ __forceinline__ void chain_put_state_block(const float* src, uint32_t tmem_a, int t, int b)
{
    using Mp = ChainMap<DK, NW>;
    constexpr int W = Mp::BLK / 2;
    const int i = Mp::row(t), c0 = Mp::col0(t) + b * Mp::BLK;
    float v[Mp::BLK];
#pragma unroll
    for (int e = 0; e < Mp::BLK; ++e) v[e] = (src && i < DV) ? src[(size_t)(c0 + e) * DV + i] : 0.0f;
    uint32_t hi[W], lo[W];
#pragma unroll
    for (int e = 0; e < W; ++e) {
        float h0, l0, h1, l1;
        tc::split_f32(v[2 * e], h0, l0);
        tc::split_f32(v[2 * e + 1], h1, l1);
        hi[e] = tc::pack_upper(h0, h1);
        lo[e] = tc::pack_upper(l0, l1);
    }
    const uint32_t base = tmem_a + Mp::lanes(t) + (uint32_t)(c0 / 2);
    tc::tmem_st_32x32b<W>(base, hi);
    tc::tmem_st_32x32b<W>(base + DK / 2, lo);
}

// Block b of this thread's values of S_new = D + B (B element (i, c) at c * DV + i),
// stored into two [DK][DV] states: the blockwise form of chain_values and chain_store.
template <int DK, int DV, int NW>
__device__ __forceinline__ void chain_store_block(uint32_t tmem_col, const float* bsrc, float* dst0, float* dst1, int t,
                                                  int b)
{
    using Mp = ChainMap<DK, NW>;
    const int i = Mp::row(t), c0 = Mp::col0(t) + b * Mp::BLK;
    float v[Mp::BLK];
    tc::tmem_ld_32x32b<Mp::BLK>(tmem_col + Mp::lanes(t) + (uint32_t)c0, v);
    if (i >= DV) return;
#pragma unroll
    for (int e = 0; e < Mp::BLK; ++e) {
        const float x = __fadd_rn(v[e], bsrc[(size_t)(c0 + e) * DV + i]);
        dst0[(size_t)(c0 + e) * DV + i] = x;
        dst1[(size_t)(c0 + e) * DV + i] = x;
    }
}

// Store this thread's values into a [DK][DV] state (element (c, row)).
template <int DK, int DV, int NW>
__device__ __forceinline__ void chain_store(float* dst, int t, const float (&v)[ChainMap<DK, NW>::CPT])
{
    using Mp = ChainMap<DK, NW>;
    const int i = Mp::row(t), c0 = Mp::col0(t);
    if (i >= DV) return;
#pragma unroll
    for (int e = 0; e < Mp::CPT; ++e) dst[(size_t)(c0 + e) * DV + i] = v[e];
}

}  // namespace cpr
