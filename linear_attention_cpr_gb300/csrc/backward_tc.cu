// backward_tc.cu — the CPR backward's per-chunk gradients on the 5th-generation tensor
// cores, for bf16 inputs with dk = dv = 128 and C = 64 (the trainer's and the rollouts'
// shape).  It computes what kb3_chunk_grads (backward.cu) computes, in the same WY form
// and order of steps (see that file's header for the algebra), with every product a
// tcgen05 MMA instead of FP32 FMAs.
//
// "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section "Chunkwise-Parallel
// Recurrent (CPR) Gated DeltaNet", per-layer table, row "Trainer Fwd+Bwd": the pages time a
// CPR backward; this is the chunk-local part of its adjoint.
//
// One CTA of 8 warps per (chunk, head).  Every product is D[128 x 64] (+)= A[128 x K] *
// B[64 x K]^T with K = 128 or 64: the 128-row side is a key or value index (products of
// n x n results use 64 rows of A and zero rows after them), the 64-column side a token.
// Operands are written by the threads into shared memory as bf16 tiles in the tensor
// cores' K-major core-matrix layout: bf16 inputs exactly (one split), everything derived in
// fp32 as Dekker hi/lo splits (tc::split_f32), and each product is the sum of the split
// products hi*hi (+ hi*lo) (+ lo*hi), accumulated in fp32 in TMEM (about 2^-16 relative per
// term).  A tile can also be read MN-major (the descriptor's transpose bit), so the chunk's
// keys, its dO and each state are written once and serve as a matrix and its transpose:
// the products that read S_b both ways (and dS_end both ways) share one run.  Results
// come back with tcgen05.ld, one accumulator row (TMEM lane) and 32
// columns per thread; dq^T and dk^T accumulate in registers across products.  Sums over
// the 128 rows (a key or value index) of a result use a fixed butterfly over the warp's
// lanes and a fixed sum over the four lane quadrants, so the gradients are reproducible
// and independent of packing, as for the FP32 kernels.  All waits are bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "handoff.cuh"
#include "numerics.cuh"
#include "reverse_chain.cuh"
#include "tc.cuh"

namespace cpr {

namespace {

constexpr int kD = 128;   // dk = dv
constexpr int kN = 64;    // C, the tokens of a chunk
constexpr int kT = 256;   // threads
constexpr int kNN = kN + 1;

// Shared memory (bytes).
constexpr uint32_t KP_OFF = 0;                  // bf16 K [64][128] as stored (zero rows past the chunk)
constexpr uint32_t OP_OFF = KP_OFF + 16384;     // bf16 dO [64][128]
constexpr uint32_t TA_OFF = OP_OFF + 16384;     // A operand tiles (64 KB)
constexpr uint32_t TB_OFF = TA_OFF + 65536;     // B operand tiles (32 KB)
constexpr uint32_t TU_OFF = TB_OFF + 32768;     // U tile, later dT^T (32 KB)
constexpr uint32_t PM_OFF = TU_OFF + 32768;     // fp32 Pm [64][65], later dKK
constexpr uint32_t TM_OFF = PM_OFF + 16640;     // fp32 T [64][65] (first A^T [64][64])
constexpr uint32_t LM_OFF = TM_OFF + 16640;     // fp32 L [64][65]
constexpr uint32_t VEC_OFF = LM_OFF + 16640;    // 16 per-token vectors of 64 floats
constexpr uint32_t RED_OFF = VEC_OFF + 4096;    // reduction partials [8][64]
constexpr uint32_t BAR_OFF = RED_OFF + 2048;
constexpr uint32_t kSmem = BAR_OFF + 64;
static_assert(kSmem <= 232448, "one CTA's shared memory");

// TMEM accumulators (columns)
constexpr uint32_t P0 = 0, P1 = 64, P2 = 128, P3 = 192;
constexpr uint32_t kTmemCols = 256;

template <int K>
__device__ __forceinline__ uint32_t toff(int row, int k)
{
    return tc::tile_off<2>(row, k, K);
}

// D (TMEM) (+)= A (128 x K tile at a) * B (64 x K tile at b)^T; NA, NB: splits present in
// each tile (1: hi only, exact bf16; 2: hi and lo).  Products hi*hi, then hi*lo (NB = 2),
// then lo*hi (NA = 2), K ascending in each; the first instruction overwrites D unless
// `accumulate`.
template <int K, int NA, int NB>
__device__ __forceinline__ void mma_ab(uint32_t d, uint32_t a, uint32_t b, bool accumulate)
{
    constexpr uint32_t SBO = (K / 8) * 128, ASPL = 128 * K * 2, BSPL = 64 * K * 2;
    constexpr uint32_t idesc = tc::idesc_bf16(128, 64);
    const uint32_t pa[3] = {0u, 0u, 1u}, pb[3] = {0u, 1u, 0u};
#pragma unroll
    for (int p = 0; p < 3; ++p) {
        if ((p == 1 && NB != 2) || (p == 2 && NA != 2)) continue;
#pragma unroll
        for (int k = 0; k < K / 16; ++k)
            tc::mma_bf16(d, tc::sdesc(a + pa[p] * ASPL + k * 256, 128, SBO),
                         tc::sdesc(b + pb[p] * BSPL + k * 256, 128, SBO), idesc,
                         (accumulate || p != 0 || k != 0) ? 1u : 0u);
    }
}

// One operand of a product in shared memory: its hi split at `base` (lo at base + split),
// the descriptor's LBO and SBO, the byte step per 16 K elements, and whether the tensor
// cores read it MN-major (the instruction descriptor's transpose bit for A or B).
struct Opnd {
    uint32_t base, split, lbo, sbo, kstep;
    bool mn;
};
// A K-major tile of `rows` rows x K elements (toff<K>(row, k)): rows are the operand's M or N.
__device__ __forceinline__ Opnd kmaj(const unsigned char* p, int rows, int K)
{
    return Opnd{tc::smem_u32(p), (uint32_t)(rows * K * 2), 128u, (uint32_t)(K / 8 * 128), 256u, false};
}
// The same kind of tile, X[a][b] at toff<W>(a, b) with `rows` rows a, read MN-major: the
// operand's M or N index is b and its K index a (LBO steps 8 rows a, SBO 8 columns b), so
// one image serves a matrix and its transpose.
__device__ __forceinline__ Opnd mnview(const unsigned char* p, int rows, int W)
{
    return Opnd{tc::smem_u32(p), (uint32_t)(rows * W * 2), (uint32_t)(W / 8 * 128), 128u, (uint32_t)(W * 32), true};
}

// D (TMEM, 128 x 64) (+)= A * B^T over K elements, the split products as in mma_ab.
template <int K, int NA, int NB>
__device__ __forceinline__ void mma2(uint32_t d, const Opnd& A, const Opnd& B, bool accumulate)
{
    const uint32_t idesc = tc::idesc_bf16(128, 64) | (A.mn ? 1u << 15 : 0u) | (B.mn ? 1u << 16 : 0u);
    const uint32_t pa[3] = {0u, 0u, 1u}, pb[3] = {0u, 1u, 0u};
#pragma unroll
    for (int p = 0; p < 3; ++p) {
        if ((p == 1 && NB != 2) || (p == 2 && NA != 2)) continue;
#pragma unroll
        for (int k = 0; k < K / 16; ++k)
            tc::mma_bf16(d, tc::sdesc(A.base + pa[p] * A.split + k * A.kstep, A.lbo, A.sbo),
                         tc::sdesc(B.base + pb[p] * B.split + k * B.kstep, B.lbo, B.sbo), idesc,
                         (accumulate || p != 0 || k != 0) ? 1u : 0u);
    }
}

// The 16-byte group idx of a 64-row K-major tile with kD elements per row: its row and first
// column, chosen so that toff<kD>(row, col) = 16 idx (consecutive threads touch consecutive
// shared-memory bytes: no bank conflicts).
__device__ __forceinline__ int img_row(int idx) { return (idx & 7) | ((idx >> 7) << 3); }
__device__ __forceinline__ int img_col(int idx) { return ((idx >> 3) & 15) * 8; }

// Lane l of the warp gets the sum over the warp's 32 lanes of v[l] (a fixed butterfly:
// each round keeps one half of the remaining columns and adds the partner's copy).
__device__ __forceinline__ float colsum32(float (&v)[32])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool upper = (lane & k) != 0;
#pragma unroll
        for (int j = 0; j < k; ++j) {
            const float send = upper ? v[j] : v[j + k];
            const float recv = __shfl_xor_sync(0xffffffffu, send, k);
            v[j] = __fadd_rn(upper ? v[j + k] : v[j], recv);
        }
    }
    return v[0];
}

struct V16 {
    float *G, *gam, *dd, *beta, *dgam1, *dgam2, *ddv, *dbeta1, *dbeta2, *edr1, *edr2, *edc1, *edc2, *dG, *gin, *misc;
    __device__ explicit V16(float* p)
        : G(p), gam(p + 64), dd(p + 128), beta(p + 192), dgam1(p + 256), dgam2(p + 320), ddv(p + 384),
          dbeta1(p + 448), dbeta2(p + 512), edr1(p + 576), edr2(p + 640), edc1(p + 704), edc2(p + 768),
          dG(p + 832), gin(p + 896), misc(p + 960) {}
};

// The chunk gradients of one (chunk, head) item by the CTA's 8 warps.  TMEM columns
// [tmem, tmem + 256) and the mbarrier at BAR_OFF (initialised; its next phase `phase`)
// belong to the caller.  Starts and ends with every thread at a barrier; returns false
// (uniformly) after a product did not complete in time, with the status word set.
__device__ __forceinline__ bool chunk_grads_item(const BackwardArgs& a, int64_t c, int h, unsigned char* sm,
                                                 uint32_t tmem, uint32_t& phase)
{
    // the chunk's K and dO as K-major images (rows r, K = c: toff<kD>(r, c)), read in both
    // orientations by the products
    unsigned char* KI = sm + KP_OFF;
    unsigned char* OI = sm + OP_OFF;
    unsigned char* TA = sm + TA_OFF;
    unsigned char* TB = sm + TB_OFF;
    unsigned char* TU = sm + TU_OFF;
    float* Pm = reinterpret_cast<float*>(sm + PM_OFF);
    float* Tm = reinterpret_cast<float*>(sm + TM_OFF);
    float* Lm = reinterpret_cast<float*>(sm + LM_OFF);
    V16 v(reinterpret_cast<float*>(sm + VEC_OFF));
    float* red = reinterpret_cast<float*>(sm + RED_OFF);  // [8][64]
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
    volatile int* okf = reinterpret_cast<volatile int*>(sm + BAR_OFF + 12);

    const int H = a.H, t = threadIdx.x;
    const int n = find_seq(a.cu_chunks, a.n_seqs, c);
    const int64_t j = c - a.cu_chunks[n];
    const int64_t t0 = (int64_t)a.cu_seqlens[n] + j * kN;
    const int len = (int)min((int64_t)kN, (int64_t)a.cu_seqlens[n + 1] - t0);
    const size_t ch = (size_t)c * H + h, SSZ = (size_t)kD * kD;
    const float* Sb = a.boundary + ch * SSZ;  // [c][i] = S_b[i][c]
    const float* dSe = a.d_end + ch * SSZ;
    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(a.v);
    const __nv_bfloat16* go = static_cast<const __nv_bfloat16*>(a.d_out);

    // epilogue mapping: accumulator row m (TMEM lane), columns [32 hc, 32 hc + 32)
    const int w = t >> 5, lane = t & 31, q = w & 3, hc = w >> 2, m = 32 * q + lane;

    // ---- a: the chunk's K and dO as stored (zero rows past its tokens), g, beta
    for (int idx = t; idx < kN * 16; idx += kT) {
        const int r = img_row(idx), cv = img_col(idx);
        uint4 wk = make_uint4(0u, 0u, 0u, 0u), wo = wk;
        if (r < len) {
            wk = __ldg(reinterpret_cast<const uint4*>(gk + ((t0 + r) * H + h) * kD + cv));
            wo = __ldg(reinterpret_cast<const uint4*>(go + ((t0 + r) * H + h) * kD + cv));
        }
        *reinterpret_cast<uint4*>(KI + toff<kD>(r, cv)) = wk;
        *reinterpret_cast<uint4*>(OI + toff<kD>(r, cv)) = wo;
    }
    if (t < kN) {
        v.gin[t] = t < len ? a.g[(t0 + t) * H + h] : 0.0f;
        v.beta[t] = t < len ? a.beta[(t0 + t) * H + h] : 0.0f;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    auto kp = [&](int r, int c) { return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(KI + toff<kD>(r, c))); };
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    if (t == 0) {
        float G = 0.0f;
        for (int r = 0; r < kN; ++r) {
            G = r == 0 ? v.gin[0] : __fadd_rn(G, v.gin[r]);
            v.G[r] = G;
        }
    }
    __syncthreads();
    if (t < kN) {
        v.gam[t] = decay_exp(v.G[t]);
        v.dd[t] = decay_exp(__fsub_rn(v.G[kN - 1], v.G[t]));
    }

    bool alive = true;
    // Every writer has stored its tiles: make them visible to the tensor cores, let thread 0
    // issue the products and wait for them, then every thread may read the accumulators.
    auto run_begin = [&](auto issue) {
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (t == 0) {
            tc::fence_after_sync();
            issue();
            tc::commit(mbar);
        }
    };
    auto run_end = [&]() {
        if (t == 0) *okf = tc::mbar_wait(mbar, phase) ? 1 : 0;
        phase ^= 1u;
        __syncthreads();
        tc::fence_after_sync();
        alive = alive && *okf != 0;
    };
    // the products of one step: issued by thread 0 once every thread's tiles are written,
    // and done for every thread on return
    auto run = [&](auto issue) {
        run_begin(issue);
        run_end();
    };
    auto acc = [&](uint32_t col, float (&x)[32]) { tc::tmem_ld32(tmem + lanes + col + 32 * hc, x); };
    auto e_of = [&](int r, int i) { return decay_exp(__fsub_rn(v.G[r], v.G[i])); };
    // zero rows [64, 128) of a tile of K elements per row (hi and, if lo_too, lo)
    auto zero_upper = [&](unsigned char* base, int K, bool lo_too) {
        const uint32_t half = 64u * K * 2;  // rows 64.. start half-way into each split
        const int nv = (int)(half / 16);
        for (int idx = t; idx < nv * (lo_too ? 2 : 1); idx += kT) {
            const int s = idx / nv, o = idx % nv;
            *reinterpret_cast<uint4*>(base + s * (2 * half) + half + o * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    // A tile (128 rows x K = 128, hi/lo) from a stored state src[c][i] (128 x 128 fp32):
    // transposed (rows i, K = c) or as stored (rows c, K = i).  Consecutive threads take
    // consecutive rows of one 8-element K group, so each warp's 16-byte stores fill whole
    // 128-byte core-matrix rows (no bank conflicts); all eight loads of a thread are issued
    // before its splits are stored.
    auto state_tile = [&](const float* src, bool transposed) {
        float xs[8][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = t + u * kT, row = idx % kD, k8 = (idx / kD) * 8;
            if (transposed) {
#pragma unroll
                for (int e = 0; e < 8; ++e) xs[u][e] = __ldg(src + (size_t)(k8 + e) * kD + row);
            } else {
                const float4 p0 = __ldg(reinterpret_cast<const float4*>(src + (size_t)row * kD + k8));
                const float4 p1 = __ldg(reinterpret_cast<const float4*>(src + (size_t)row * kD + k8 + 4));
                xs[u][0] = p0.x, xs[u][1] = p0.y, xs[u][2] = p0.z, xs[u][3] = p0.w;
                xs[u][4] = p1.x, xs[u][5] = p1.y, xs[u][6] = p1.z, xs[u][7] = p1.w;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = t + u * kT, row = idx % kD, k8 = (idx / kD) * 8;
            tc::split8_store(xs[u], TA + toff<kD>(row, k8), TA + 32768 + toff<kD>(row, k8));
        }
    };
    if (t == 0) {  // both states are read several times: into L2 now
        tc::prefetch_l2(Sb, (uint32_t)(SSZ * 4));
        tc::prefetch_l2(dSe, (uint32_t)(SSZ * 4));
    }
    if (t < 2 * kN && (t & 63) < len) {  // the chunk's query and value rows (read column-wise later)
        const __nv_bfloat16* row = (t < kN ? gq : gv) + ((t0 + (t & 63)) * H + h) * kD;
        tc::prefetch_l2(row, kD * 2);
    }

    // ---- F1, F2: K K^T and Q K^T (n x n)
    {
        for (int idx = t; idx < kN * 16; idx += kT) {  // A: K and Q, rows t < 64 (zero rows after)
            const int r = img_row(idx), cv = img_col(idx);
            const uint4 kw = *reinterpret_cast<const uint4*>(KI + toff<kD>(r, cv));
            uint4 qw = make_uint4(0u, 0u, 0u, 0u);
            if (r < len) qw = __ldg(reinterpret_cast<const uint4*>(gq + ((t0 + r) * H + h) * kD + cv));
            *reinterpret_cast<uint4*>(TA + toff<kD>(r, cv)) = kw;
            *reinterpret_cast<uint4*>(TA + 32768 + toff<kD>(r, cv)) = qw;
        }
        zero_upper(TA, kD, false);
        zero_upper(TA + 32768, kD, false);
        run([&] {
            mma2<kD, 1, 1>(tmem + P0, kmaj(TA, 128, kD), kmaj(KI, kN, kD), false);
            mma2<kD, 1, 1>(tmem + P1, kmaj(TA + 32768, 128, kD), kmaj(KI, kN, kD), false);
        });
        if (q < 2) {  // rows t < 64
            float kk[32], qk[32];
            acc(P0, kk);
            acc(P1, qk);
            const float br = v.beta[m];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int r = 32 * hc + jj;
                const float e = r <= m ? e_of(m, r) : 0.0f;
                const float l = r < m ? __fmul_rn(kk[jj], e) : 0.0f;
                Lm[m * kNN + r] = l;
                Tm[r * kN + m] = __fmul_rn(br, l);  // A transposed for the substitution
                Pm[m * kNN + r] = __fmul_rn(qk[jj], e);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        // T = (I + A)^-1 by blocks, with every thread, into TU (free until F4's epilogue)
        invert_unit_lower<kN, kNN>(Tm, reinterpret_cast<float*>(TU), reinterpret_cast<float*>(TU + 16896), t, kT);
        {
            const float* X = reinterpret_cast<const float*>(TU);
            for (int idx = t; idx < kN * kN; idx += kT) Tm[(idx >> 6) * kNN + (idx & 63)] = X[(idx >> 6) * kNN + (idx & 63)];
        }
        __syncthreads();
    }
    float dqT[32], dkT[32], RT[32];  // row m (key index for dq/dk, value index for R), columns 32 hc + jj

    // ---- F3 and B1 in one run, both from one image of S_b as stored (rows c, K = i), F3
    //      reading it MN-major:
    //      F3: KS^T = S_b K^T;  R^T = V^T - KS^T diag(gam)
    //      B1: Y^T = S_b^T dO^T:  dq^T = Y^T diag(gam);  dgam = colsum(Y^T o Q^T)
    if (alive) {
        float vv[32];  // issued first: their latency overlaps the gather of S_b
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            vv[jj] = r < len ? __bfloat162float(gv[((t0 + r) * H + h) * kD + m]) : 0.0f;
        }
        state_tile(Sb, false);
        run_begin([&] {
            mma2<kD, 2, 1>(tmem + P0, mnview(TA, kD, kD), kmaj(KI, kN, kD), false);
            mma2<kD, 2, 1>(tmem + P1, kmaj(TA, kD, kD), kmaj(OI, kN, kD), false);
        });
        {  // dgam_last = <dS_end, S_b> while the products run: a fixed order per thread (four
           // component sums over its float4s, eight of each state's loads in flight), then
           // fixed trees
            float4 a4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float4 xd[8], xs[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i4 = t + (8 * b + u) * kT;
                    xd[u] = __ldg(reinterpret_cast<const float4*>(dSe) + i4);
                    xs[u] = __ldg(reinterpret_cast<const float4*>(Sb) + i4);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    a4.x = __fmaf_rn(xd[u].x, xs[u].x, a4.x);
                    a4.y = __fmaf_rn(xd[u].y, xs[u].y, a4.y);
                    a4.z = __fmaf_rn(xd[u].z, xs[u].z, a4.z);
                    a4.w = __fmaf_rn(xd[u].w, xs[u].w, a4.w);
                }
            }
            float sd = __fadd_rn(__fadd_rn(a4.x, a4.y), __fadd_rn(a4.z, a4.w));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) sd = __fadd_rn(sd, __shfl_xor_sync(0xffffffffu, sd, o));
            if (lane == 0) red[256 + w] = sd;
        }
        float qv[32];  // (their latency overlaps the products' end)
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            qv[jj] = r < len ? __bfloat162float(gq[((t0 + r) * H + h) * kD + m]) : 0.0f;
        }
        run_end();
        if (t == 0) {
            float d = 0.0f;
            for (int i = 0; i < 8; ++i) d = __fadd_rn(d, red[256 + i]);
            v.misc[0] = d;
        }
        {
            float ks[32];
            acc(P0, ks);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) RT[jj] = __fsub_rn(vv[jj], __fmul_rn(v.gam[32 * hc + jj], ks[jj]));
        }
        float y[32];
        acc(P1, y);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            dqT[jj] = __fmul_rn(v.gam[32 * hc + jj], y[jj]);
            qv[jj] = __fmul_rn(y[jj], qv[jj]);
            dkT[jj] = 0.0f;
        }
        red[q * 64 + 32 * hc + lane] = colsum32(qv);
        __syncthreads();
        if (t < kN) v.dgam1[t] = __fadd_rn(__fadd_rn(red[t], red[64 + t]), __fadd_rn(red[128 + t], red[192 + t]));
    }
    // ---- F4: U^T = (R^T diag(beta)) T^T  -> the U^T image (rows i, 64 columns t), B of B2
    //      and B4 read MN-major
    if (alive) {
#pragma unroll
        for (int e8 = 0; e8 < 32; e8 += 8) {  // A: rows i, K = r (this thread's row)
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = __fmul_rn(RT[e8 + e], v.beta[32 * hc + e8 + e]);
            tc::split8_store(xs, TA + toff<kN>(m, 32 * hc + e8), TA + 16384 + toff<kN>(m, 32 * hc + e8));
        }
        for (int idx = t; idx < kN * 8; idx += kT) {  // B: T, rows t, K = r
            const int r = idx >> 3, k8 = (idx & 7) * 8;
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = Tm[r * kNN + k8 + e];
            tc::split8_store(xs, TB + toff<kN>(r, k8), TB + 8192 + toff<kN>(r, k8));
        }
        run([&] { mma_ab<kN, 2, 2>(tmem + P0, tc::smem_u32(TA), tc::smem_u32(TB), false); });
        float u[32];
        acc(P0, u);
#pragma unroll
        for (int e8 = 0; e8 < 32; e8 += 8) {
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = u[e8 + e];
            tc::split8_store(xs, TU + toff<kN>(m, 32 * hc + e8), TU + 16384 + toff<kN>(m, 32 * hc + e8));
        }
    }
    // ---- B2: dPm = (dO U^T) o lower;  ED += dPm o Pm;  dQK = dPm o E  (tiles for B5, B6)
    if (alive) {
        for (int idx = t; idx < kN * 16; idx += kT)  // A: dO, rows t < 64 (its image), zero rows after
            reinterpret_cast<uint4*>(TA)[idx] = reinterpret_cast<const uint4*>(OI)[idx];
        zero_upper(TA, kD, false);
        run([&] { mma2<kD, 1, 2>(tmem + P0, kmaj(TA, 128, kD), mnview(TU, kD, kN), false); });
        if (q < 2) {
            float dp[32], col[32], rowp = 0.0f;
            acc(P0, dp);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int r = 32 * hc + jj;
                const float x = r <= m ? dp[jj] : 0.0f;
                const float ed = __fmul_rn(x, Pm[m * kNN + r]);
                rowp = __fadd_rn(rowp, ed);
                col[jj] = ed;
                dp[jj] = r <= m ? __fmul_rn(x, e_of(m, r)) : 0.0f;  // dQK
            }
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {  // the dQK image: rows t, K = r (B6 reads it MN-major)
                float xs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) xs[e] = dp[e8 + e];
                tc::split8_store(xs, TB + toff<kN>(m, 32 * hc + e8), TB + 8192 + toff<kN>(m, 32 * hc + e8));
            }
            red[q * 64 + 32 * hc + lane] = colsum32(col);
            red[256 + hc * 64 + m] = rowp;
        }
        __syncthreads();
        if (t < kN) {
            v.edc1[t] = __fadd_rn(red[t], red[64 + t]);
            v.edr1[t] = __fadd_rn(red[256 + t], red[320 + t]);
        }
    }
    // ---- B5, B6: dq += dQK K and dk += dQK^T Q, as dq^T = K^T dQK^T-side and dk^T = Q^T
    //      dQK-side: K^T and Q^T are the K image and a Q image (rows t, K = c), and dQK^T the
    //      dQK image, each read MN-major
    if (alive) {
        for (int idx = t; idx < kN * 16; idx += kT) {
            const int r = img_row(idx), cv = img_col(idx);
            uint4 qw = make_uint4(0u, 0u, 0u, 0u);
            if (r < len) qw = __ldg(reinterpret_cast<const uint4*>(gq + ((t0 + r) * H + h) * kD + cv));
            *reinterpret_cast<uint4*>(TA + toff<kD>(r, cv)) = qw;
        }
        run([&] {
            mma2<kN, 1, 2>(tmem + P0, mnview(KI, kN, kD), kmaj(TB, kN, kN), false);
            mma2<kN, 1, 2>(tmem + P1, mnview(TA, kN, kD), mnview(TB, kN, kN), false);
        });
        float x[32];
        acc(P0, x);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) dqT[jj] = __fadd_rn(dqT[jj], x[jj]);
        acc(P1, x);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) dkT[jj] = __fadd_rn(dkT[jj], x[jj]);
    }
    // ---- B3a and B4 in one run, both from one image of dS_end as stored (rows c, K = i),
    //      B3a reading it MN-major:
    //      B3a: dU^T = dS_end (diag(d) K)^T  (B3b adds dO^T Pm below)
    //      B4:  UdS^T = dS_end^T U-side:  dk^T += UdS^T diag(d);  dd = colsum(UdS^T o K^T)
    float DUT[32];
    if (alive) {
        state_tile(dSe, false);
        for (int idx = t; idx < kN * 16; idx += kT) {  // B of B3a: diag(d) K, rows r, K = c
            const int r = img_row(idx), c8 = img_col(idx);
            const uint4 kw = *reinterpret_cast<const uint4*>(KI + toff<kD>(r, c8));
            const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kw);
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = __fmul_rn(v.dd[r], __bfloat162float(kb[e]));
            tc::split8_store(xs, TB + toff<kD>(r, c8), TB + 16384 + toff<kD>(r, c8));
        }
        run([&] {
            mma2<kD, 2, 2>(tmem + P2, mnview(TA, kD, kD), kmaj(TB, kN, kD), false);
            mma2<kD, 2, 2>(tmem + P0, kmaj(TA, kD, kD), mnview(TU, kD, kN), false);
        });
        float x[32];
        acc(P0, x);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            dkT[jj] = __fmaf_rn(v.dd[r], x[jj], dkT[jj]);
            x[jj] = __fmul_rn(x[jj], kp(r, m));
        }
        red[q * 64 + 32 * hc + lane] = colsum32(x);
        __syncthreads();
        if (t < kN) v.ddv[t] = __fadd_rn(__fadd_rn(red[t], red[64 + t]), __fadd_rn(red[128 + t], red[192 + t]));
    }
    // ---- B3b: dU^T += dO^T Pm (dO^T: the dO image read MN-major)
    if (alive) {
        for (int idx = t; idx < kN * 8; idx += kT) {  // B: Pm^T rows r, K = t
            const int r = idx % kN, k8 = (idx / kN) * 8;
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = Pm[(k8 + e) * kNN + r];
            tc::split8_store(xs, TB + toff<kN>(r, k8), TB + 8192 + toff<kN>(r, k8));
        }
        run([&] { mma2<kN, 1, 2>(tmem + P2, mnview(OI, kN, kD), kmaj(TB, kN, kN), true); });
        acc(P2, DUT);
    }
    // ---- B7: dT = dU (diag(beta) R)^T (n x n): A = dU from the dU^T image (rows i, 128
    //      columns t, zero past 64) and B = beta R from the (beta R)^T image (rows i, 64
    //      columns r), both read MN-major; dT -> the dT image (rows t, K = t') for B10
    if (alive) {
        __syncthreads();  // every reader of the last reductions' partials and of TA is done
        {
            float br[8];
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {
#pragma unroll
                for (int e = 0; e < 8; ++e) br[e] = DUT[e8 + e];
                tc::split8_store(br, TA + toff<kD>(m, 32 * hc + e8), TA + 32768 + toff<kD>(m, 32 * hc + e8));
                *reinterpret_cast<uint4*>(TA + toff<kD>(m, 64 + 32 * hc + e8)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(TA + 32768 + toff<kD>(m, 64 + 32 * hc + e8)) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int e = 0; e < 8; ++e) br[e] = __fmul_rn(v.beta[32 * hc + e8 + e], RT[e8 + e]);
                tc::split8_store(br, TB + toff<kN>(m, 32 * hc + e8), TB + 16384 + toff<kN>(m, 32 * hc + e8));
            }
        }
        run([&] { mma2<kD, 2, 2>(tmem + P0, mnview(TA, kD, kD), mnview(TB, kD, kN), false); });
        if (q < 2) {
            float x[32];
            acc(P0, x);
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {
                float xs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) xs[e] = x[e8 + e];
                tc::split8_store(xs, TU + toff<kN>(m, 32 * hc + e8), TU + 8192 + toff<kN>(m, 32 * hc + e8));
            }
        }
    }
    // ---- B8: TdU^T = dU^T T:  dv = diag(beta) TdU;  dbeta = colsum(TdU^T o R^T)  (A: the dU^T
    //      image, K-major; TdU^T -> its image, rows i, 64 columns r, for B9)
    if (alive) {
        for (int idx = t; idx < kN * 8; idx += kT) {  // B: T^T rows r, K = t
            const int r = idx % kN, k8 = (idx / kN) * 8;
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = Tm[(k8 + e) * kNN + r];
            tc::split8_store(xs, TB + toff<kN>(r, k8), TB + 8192 + toff<kN>(r, k8));
        }
        run([&] { mma2<kN, 2, 2>(tmem + P1, kmaj(TA, kD, kD), kmaj(TB, kN, kN), false); });
        float x[32];
        acc(P1, x);
#pragma unroll
        for (int e8 = 0; e8 < 32; e8 += 8) {
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = x[e8 + e];
            tc::split8_store(xs, TB + toff<kN>(m, 32 * hc + e8), TB + 16384 + toff<kN>(m, 32 * hc + e8));
        }
        float* dvb = a.dv + ((size_t)t0 * H + h) * kD + m;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            if (r < len) dvb[(size_t)r * H * kD] = __fmul_rn(v.beta[r], x[jj]);
            x[jj] = __fmul_rn(x[jj], RT[jj]);
        }
        red[q * 64 + 32 * hc + lane] = colsum32(x);
        __syncthreads();
        if (t < kN) v.dbeta1[t] = __fadd_rn(__fadd_rn(red[t], red[64 + t]), __fadd_rn(red[128 + t], red[192 + t]));
    }
    // ---- B9: Z^T = S_b^T TdU^T:  dk^T -= Z^T diag(beta gam);  dgam -= beta colsum(Z^T o K^T)
    if (alive) {
        state_tile(Sb, false);  // A: S_b^T rows c, K = i (as stored)
        run([&] { mma2<kD, 2, 2>(tmem + P0, kmaj(TA, kD, kD), mnview(TB, kD, kN), false); });
        float x[32];
        acc(P0, x);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            dkT[jj] = __fmaf_rn(-__fmul_rn(v.beta[r], v.gam[r]), x[jj], dkT[jj]);
            x[jj] = __fmul_rn(x[jj], kp(r, m));
        }
        red[q * 64 + 32 * hc + lane] = colsum32(x);
        __syncthreads();
        if (t < kN)
            v.dgam2[t] = __fmul_rn(-v.beta[t], __fadd_rn(__fadd_rn(red[t], red[64 + t]),
                                                         __fadd_rn(red[128 + t], red[192 + t])));
    }
    // ---- B10: X = T^T dT (n x n; dT from its image read MN-major) -> the X tile (rows r,
    //      K = t) for B11
    if (alive) {
        __syncthreads();
        for (int idx = t; idx < kN * 8; idx += kT) {  // A: T^T rows r, K = t
            const int r = idx % kN, k8 = (idx / kN) * 8;
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = Tm[(k8 + e) * kNN + r];
            tc::split8_store(xs, TA + toff<kN>(r, k8), TA + 16384 + toff<kN>(r, k8));
        }
        zero_upper(TA, kN, true);
        run([&] { mma2<kN, 2, 2>(tmem + P1, kmaj(TA, 128, kN), mnview(TU, kN, kN), false); });
        if (q < 2) {
            float x[32];
            acc(P1, x);
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {
                float xs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) xs[e] = x[e8 + e];
                tc::split8_store(xs, TA + toff<kN>(m, 32 * hc + e8), TA + 16384 + toff<kN>(m, 32 * hc + e8));
            }
        }
    }
    // ---- B11: dA = -(X T^T) o strictly lower:  dbeta += rowsum(dA o L);  dL = beta dA;
    //      ED += dL o L;  dKK = dL o E  -> Ssym = dKK + dKK^T tile for B12
    if (alive) {
        for (int idx = t; idx < kN * 8; idx += kT) {  // B: T rows i, K = t
            const int r = idx >> 3, k8 = (idx & 7) * 8;
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = Tm[r * kNN + k8 + e];
            tc::split8_store(xs, TB + toff<kN>(r, k8), TB + 8192 + toff<kN>(r, k8));
        }
        run([&] { mma_ab<kN, 2, 2>(tmem + P0, tc::smem_u32(TA), tc::smem_u32(TB), false); });
        if (q < 2) {
            float x[32], col[32], rowb = 0.0f, rowe = 0.0f;
            acc(P0, x);
            const float br = v.beta[m];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int i = 32 * hc + jj;
                const float da = i < m ? -x[jj] : 0.0f;
                const float l = Lm[m * kNN + i];
                rowb = __fmaf_rn(da, l, rowb);
                const float dl = __fmul_rn(br, da);
                const float ed = __fmul_rn(dl, l);
                rowe = __fadd_rn(rowe, ed);
                col[jj] = ed;
                Pm[m * kNN + i] = i < m ? __fmul_rn(dl, e_of(m, i)) : 0.0f;  // dKK (Pm is dead)
            }
            red[q * 64 + 32 * hc + lane] = colsum32(col);
            red[256 + hc * 64 + m] = rowe;
            red[384 + hc * 64 + m] = rowb;
        }
        __syncthreads();
        if (t < kN) {
            v.edc2[t] = __fadd_rn(red[t], red[64 + t]);
            v.edr2[t] = __fadd_rn(red[256 + t], red[320 + t]);
            v.dbeta2[t] = __fadd_rn(red[384 + t], red[448 + t]);
        }
        for (int idx = t; idx < kN * 8; idx += kT) {  // B: Ssym rows r, K = i
            const int r = idx >> 3, k8 = (idx & 7) * 8;
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = __fadd_rn(Pm[r * kNN + k8 + e], Pm[(k8 + e) * kNN + r]);
            tc::split8_store(xs, TB + toff<kN>(r, k8), TB + 8192 + toff<kN>(r, k8));
        }
    }
    // ---- B12: dk^T += K^T Ssym^T-side (dk += (dKK + dKK^T) K; K^T: the K image read MN-major)
    if (alive) {
        run([&] { mma2<kN, 1, 2>(tmem + P1, mnview(KI, kN, kD), kmaj(TB, kN, kN), false); });
        float x[32];
        acc(P1, x);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) dkT[jj] = __fadd_rn(dkT[jj], x[jj]);
    }
    // ---- the gates and the stores
    if (alive) {
        __syncthreads();
        if (t == 0) {
            const float dlast = v.misc[0];
            float sdd = 0.0f;
            for (int r = 0; r < kN; ++r) sdd = __fmaf_rn(v.dd[r], v.ddv[r], sdd);
            float accg = 0.0f;
            for (int r = kN - 1; r >= 0; --r) {
                float dgam = __fadd_rn(v.dgam1[r], v.dgam2[r]);
                if (r == kN - 1) dgam = __fadd_rn(dgam, dlast);
                float dG = __fmul_rn(v.gam[r], dgam);
                dG = __fsub_rn(dG, __fmul_rn(v.dd[r], v.ddv[r]));
                dG = __fadd_rn(dG, __fsub_rn(__fadd_rn(v.edr1[r], v.edr2[r]), __fadd_rn(v.edc1[r], v.edc2[r])));
                if (r == kN - 1) dG = __fadd_rn(dG, sdd);
                accg = __fadd_rn(accg, dG);
                v.dG[r] = accg;
            }
        }
        __syncthreads();
        if (t < len) {
            a.dg[(t0 + t) * H + h] = v.dG[t];
            a.dbeta[(t0 + t) * H + h] = __fadd_rn(v.dbeta1[t], v.dbeta2[t]);
        }
        float* dqb = a.dq + ((size_t)t0 * H + h) * kD + m;
        float* dkb = a.dk + ((size_t)t0 * H + h) * kD + m;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            if (r < len) {
                dqb[(size_t)r * H * kD] = dqT[jj];
                dkb[(size_t)r * H * kD] = dkT[jj];
            }
        }
    } else if (t == 0) {
        atomicOr(a.status, CPR_DEV_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    return alive;
}

// ------------------------------------------------------------------------------------
// The reverse chain and the chunk gradients in one cooperative launch of one CTA per SM:
// CTAs [0, n_chain) run the reverse chains (reverse_chain.cuh), one (sequence, head) at a
// time, publishing each chunk's state adjoint d_end as soon as it is stored; then every
// CTA takes (chunk, head) items of the chunk gradients in reverse chunk order from a
// counter, each starting once its chunk's d_end is published.  The gradients of late
// chunks thus run while the chain is still stepping back through the early ones.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kT, 1) kb23_chain_and_grads_tc(BackwardArgs a, int n_chain)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ uint32_t tslot_s, claimed_s;
    __shared__ int wait_ok_s;
    static_assert(RevChainCfg<kD, kD>::bytes <= BAR_OFF, "the chain's shared memory stays clear of the items' mbarrier");
    const int t = threadIdx.x, w = t >> 5;
    if (*a.status) return;
    if (w == 0) tc::tmem_alloc(&tslot_s, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tslot_s;
    bool ok = true;
    if ((int)blockIdx.x < n_chain)
        for (int ci = blockIdx.x; ci < a.n_seqs * a.H && ok; ci += n_chain)
            ok = reverse_chain<kD, kD>(a, ci, sm, tmem, a.ready);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
    if (t == 0) {
        tc::mbar_init(mbar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    const uint32_t nchunks = (uint32_t)a.cu_chunks[a.n_seqs], items = nchunks * (uint32_t)a.H;
    uint32_t* next_item = a.ready + (size_t)a.max_chunks * a.H;
    uint32_t phase = 0;
    while (ok) {
        if (t == 0) claimed_s = atomicAdd(next_item, 1u);
        __syncthreads();
        const uint32_t u = claimed_s;
        if (u >= items) break;
        const int64_t c = (int64_t)(nchunks - 1 - u / (uint32_t)a.H);
        const int h = (int)(u % (uint32_t)a.H);
        if (t == 0)
            wait_ok_s = wait_published(a.ready + (size_t)c * a.H + h, 1u + a.wait_extra, a.status, a.wait_limit_ns);
        __syncthreads();
        if (!wait_ok_s) {
            if (t == 0) atomicOr(a.status, CPR_DEV_TIMEOUT);
            break;
        }
        ok = chunk_grads_item(a, c, h, sm, tmem, phase);  // (ends at a barrier)
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (t == 0) tc::mbar_inval(mbar);
    if (w == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------
// kb1 on the tensor cores: one chunk's coefficients of the reverse chain (what
// kb1_chunk_maps computes, backward.cu), one CTA of 8 warps per (chunk, head), with the
// products as tcgen05 MMAs of bf16 splits (the conventions above); accumulator rows are
// key indices c, columns tokens r or key/value indices:
//   F1, F2   K K^T and Q K^T -> Pm and A^T in shared memory; T = (I + A)^-1 by blocks
//   W        W^T = (diag(beta gam) K)^T T^T
//   Qt, M    (Pm W)^T = W^T Pm^T, then Qt^T = Q^T diag(gam) - (Pm W)^T;
//            M = gam_last I - W^T diag(d) K (two 64-column halves)
//   C_b      C_b = Qt^T dO, stored [c][i] like a state (two 64-column halves)
// M goes out as the reverse chain's B operand image (bf16 hi / lo, row c, K index c').
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kT, 1) kb1_chunk_maps_tc(BackwardArgs a)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    __nv_bfloat16* Kp = reinterpret_cast<__nv_bfloat16*>(sm + KP_OFF);
    __nv_bfloat16* Op = reinterpret_cast<__nv_bfloat16*>(sm + OP_OFF);
    unsigned char* TA = sm + TA_OFF;
    unsigned char* TB = sm + TB_OFF;
    unsigned char* TU = sm + TU_OFF;
    float* Pm = reinterpret_cast<float*>(sm + PM_OFF);
    float* Tm = reinterpret_cast<float*>(sm + TM_OFF);
    V16 v(reinterpret_cast<float*>(sm + VEC_OFF));
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 1);
    volatile int* okf = reinterpret_cast<volatile int*>(tslot + 1);

    const int64_t c = blockIdx.x;
    const int h = blockIdx.y, H = a.H, t = threadIdx.x;
    if (*a.status || c >= a.cu_chunks[a.n_seqs]) return;
    const int n = find_seq(a.cu_chunks, a.n_seqs, c);
    const int64_t j = c - a.cu_chunks[n];
    const int64_t t0 = (int64_t)a.cu_seqlens[n] + j * kN;
    const int len = (int)min((int64_t)kN, (int64_t)a.cu_seqlens[n + 1] - t0);
    const size_t ch = (size_t)c * H + h;
    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* go = static_cast<const __nv_bfloat16*>(a.d_out);
    const int w = t >> 5, lane = t & 31, q = w & 3, hc = w >> 2, m = 32 * q + lane;

    if (w == 0) tc::tmem_alloc(tslot, kTmemCols);
    if (t == 0) {
        tc::mbar_init(mbar, 1);
        tc::fence_mbar_init();
    }
    // the chunk's K and dO as stored (zero rows past its tokens), g, beta
    for (int idx = t; idx < kN * 16; idx += kT) {
        const int r = idx >> 4, cv = (idx & 15) * 8;
        uint4 wk = make_uint4(0u, 0u, 0u, 0u), wo = wk;
        if (r < len) {
            wk = __ldg(reinterpret_cast<const uint4*>(gk + ((t0 + r) * H + h) * kD + cv));
            wo = __ldg(reinterpret_cast<const uint4*>(go + ((t0 + r) * H + h) * kD + cv));
        }
        *reinterpret_cast<uint4*>(Kp + r * kD + cv) = wk;
        *reinterpret_cast<uint4*>(Op + r * kD + cv) = wo;
    }
    if (t < kN) {
        v.gin[t] = t < len ? a.g[(t0 + t) * H + h] : 0.0f;
        v.beta[t] = t < len ? a.beta[(t0 + t) * H + h] : 0.0f;
    }
    if (t < kN && t < len) tc::prefetch_l2(gq + ((t0 + t) * H + h) * kD, kD * 2);  // read column-wise later
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t lanes = (uint32_t)(32 * q) << 16;
    if (t == 0) {
        float G = 0.0f;
        for (int r = 0; r < kN; ++r) {
            G = r == 0 ? v.gin[0] : __fadd_rn(G, v.gin[r]);
            v.G[r] = G;
        }
    }
    __syncthreads();
    if (t < kN) {
        v.gam[t] = decay_exp(v.G[t]);
        v.dd[t] = decay_exp(__fsub_rn(v.G[kN - 1], v.G[t]));
        v.misc[t] = __fmul_rn(v.beta[t], v.gam[t]);  // the key scale of W (after gam is written)
    }

    uint32_t phase = 0;
    bool alive = true;
    auto run = [&](auto issue) {
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (t == 0) {
            tc::fence_after_sync();
            issue();
            tc::commit(mbar);
            *okf = tc::mbar_wait(mbar, phase) ? 1 : 0;
        }
        phase ^= 1u;
        __syncthreads();
        tc::fence_after_sync();
        alive = alive && *okf != 0;
    };
    auto acc = [&](uint32_t col, float (&x)[32]) { tc::tmem_ld32(tmem + lanes + col + 32 * hc, x); };
    // A tile of `rows` rows (c, K = the 64 tokens r, K-major) with element s_r X[r][c0 + c],
    // X a [64][128] bf16 tile in shared memory: hi / lo splits (lo at dst + lo_off), or
    // for s == NULL the exact bf16 values, hi only
    auto tokens_tile = [&](const __nv_bfloat16* X, int c0, int rows, const float* s, unsigned char* dst,
                           uint32_t lo_off) {
        for (int idx = t; idx < rows * 8; idx += kT) {
            const int cc = idx % rows, k8 = (idx / rows) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xv = __bfloat162float(X[(k8 + e) * kD + c0 + cc]);
                x[e] = s ? __fmul_rn(s[k8 + e], xv) : xv;
            }
            const uint32_t off = toff<kN>(cc, k8);
            tc::split8_store(x, dst + off, s ? dst + lo_off + off : nullptr);
        }
    };
    // a 64 x 64 fp32 tile X (row stride kNN) as a B operand (rows r, K = k; hi / lo)
    auto nn_tile = [&](const float* X, unsigned char* dst) {
        for (int idx = t; idx < kN * 8; idx += kT) {
            const int r = idx >> 3, k8 = (idx & 7) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = X[r * kNN + k8 + e];
            tc::split8_store(x, dst + toff<kN>(r, k8), dst + 8192 + toff<kN>(r, k8));
        }
    };

    // ---- F1, F2: K K^T and Q K^T (n x n) -> Pm, A^T
    {
        for (int idx = t; idx < kN * 16; idx += kT) {
            const int r = idx >> 4, cv = (idx & 15) * 8;
            const uint4 kw = *reinterpret_cast<const uint4*>(Kp + r * kD + cv);
            uint4 qw = make_uint4(0u, 0u, 0u, 0u);
            if (r < len) qw = __ldg(reinterpret_cast<const uint4*>(gq + ((t0 + r) * H + h) * kD + cv));
            *reinterpret_cast<uint4*>(TA + toff<kD>(r, cv)) = kw;
            *reinterpret_cast<uint4*>(TA + 32768 + toff<kD>(r, cv)) = qw;
            *reinterpret_cast<uint4*>(TB + toff<kD>(r, cv)) = kw;
        }
        for (int idx = t; idx < 2 * 1024; idx += kT) {  // rows [64, 128) of both A tiles: zero
            const int s = idx >> 10, o = idx & 1023;
            *reinterpret_cast<uint4*>(TA + s * 32768 + 16384 + o * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        run([&] {
            mma_ab<kD, 1, 1>(tmem + P0, tc::smem_u32(TA), tc::smem_u32(TB), false);
            mma_ab<kD, 1, 1>(tmem + P1, tc::smem_u32(TA + 32768), tc::smem_u32(TB), false);
        });
        if (alive && q < 2) {  // rows t < 64
            float kk[32], qk[32];
            acc(P0, kk);
            acc(P1, qk);
            const float br = v.beta[m];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int r = 32 * hc + jj;
                const float e = r <= m ? decay_exp(__fsub_rn(v.G[m], v.G[r])) : 0.0f;
                const float l = r < m ? __fmul_rn(kk[jj], e) : 0.0f;
                Tm[r * kN + m] = __fmul_rn(br, l);  // A transposed for the inversion
                Pm[m * kNN + r] = __fmul_rn(qk[jj], e);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        // T = (I + A)^-1 by blocks, with every thread (scratch in TU)
        invert_unit_lower<kN, kNN>(Tm, reinterpret_cast<float*>(TU), reinterpret_cast<float*>(TU + 16896), t, kT);
        {
            const float* X = reinterpret_cast<const float*>(TU);
            for (int idx = t; idx < kN * kN; idx += kT) Tm[(idx >> 6) * kNN + (idx & 63)] = X[(idx >> 6) * kNN + (idx & 63)];
        }
    }
    // ---- W^T = (diag(beta gam) K)^T T^T: A rows c, K = r;  B = T, rows r', K = r
    if (alive) {
        tokens_tile(Kp, 0, kD, v.misc, TA, 16384);
        __syncthreads();  // (Tm complete)
        nn_tile(Tm, TB);
        run([&] { mma_ab<kN, 2, 2>(tmem + P2, tc::smem_u32(TA), tc::smem_u32(TB), false); });
    }
    // ---- Qt and M: A = W^T (rows c, K = r); B = Pm (rows r', K = r) and diag(d) K halves
    if (alive) {
        float wt[32];
        acc(P2, wt);
#pragma unroll
        for (int e8 = 0; e8 < 32; e8 += 8) {
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = wt[e8 + e];
            tc::split8_store(xs, TA + toff<kN>(m, 32 * hc + e8), TA + 16384 + toff<kN>(m, 32 * hc + e8));
        }
        nn_tile(Pm, TB);
        for (int idx = t; idx < 2 * 64 * 8; idx += kT) {  // B: d_r K[r][c'] (rows c' of each half, K = r)
            const int half = idx >> 9, cc = idx & 63, k8 = ((idx >> 6) & 7) * 8;
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                x[e] = __fmul_rn(v.dd[k8 + e], __bfloat162float(Kp[(k8 + e) * kD + 64 * half + cc]));
            unsigned char* dst = TU + half * 16384;
            tc::split8_store(x, dst + toff<kN>(cc, k8), dst + 8192 + toff<kN>(cc, k8));
        }
        run([&] {
            mma_ab<kN, 2, 2>(tmem + P0, tc::smem_u32(TA), tc::smem_u32(TB), false);
            mma_ab<kN, 2, 2>(tmem + P1, tc::smem_u32(TA), tc::smem_u32(TU), false);
            mma_ab<kN, 2, 2>(tmem + P3, tc::smem_u32(TA), tc::smem_u32(TU + 16384), false);
        });
    }
    // ---- Qt^T = Q^T diag(gam) - (Pm W)^T -> A tile (rows c, K = r);  M -> its image;
    //      C_b = Qt^T dO in two halves (B = dO^T, rows i, K = r, exact bf16)
    if (alive) {
        float pw[32];
        acc(P0, pw);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int r = 32 * hc + jj;
            const float qv = r < len ? __bfloat162float(gq[((t0 + r) * H + h) * kD + m]) : 0.0f;
            pw[jj] = __fsub_rn(__fmul_rn(v.gam[r], qv), pw[jj]);
        }
#pragma unroll
        for (int e8 = 0; e8 < 32; e8 += 8) {
            float xs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[e] = pw[e8 + e];
            tc::split8_store(xs, TA + 32768 + toff<kN>(m, 32 * hc + e8), TA + 49152 + toff<kN>(m, 32 * hc + e8));
        }
        tokens_tile(Op, 0, kN, nullptr, TB, 0);
        tokens_tile(Op, 64, kN, nullptr, TB + 16384, 0);
        // M[c][c'] = gam_last [c == c'] - (W^T diag(d) K)[c][c'] into the image (row c, K = c')
        unsigned char* img = a.mt + ch * (size_t)(4 * kD * kD);
        const float gl = v.gam[kN - 1];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float mv[32];
            acc(half ? P3 : P1, mv);
#pragma unroll
            for (int e8 = 0; e8 < 32; e8 += 8) {
                float xs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int cp = 64 * half + 32 * hc + e8 + e;
                    xs[e] = cp == m ? __fsub_rn(gl, mv[e8 + e]) : -mv[e8 + e];
                }
                const uint32_t off = tc::tile_off<2>(m, 64 * half + 32 * hc + e8, kD);
                tc::split8_store(xs, img + off, img + 2 * kD * kD + off);
            }
        }
        run([&] {
            mma_ab<kN, 2, 1>(tmem + P0, tc::smem_u32(TA + 32768), tc::smem_u32(TB), false);
            mma_ab<kN, 2, 1>(tmem + P2, tc::smem_u32(TA + 32768), tc::smem_u32(TB + 16384), false);
        });
    }
    // ---- C_b stored [c][i]
    if (alive) {
        float* dst = a.cb + ch * (size_t)(kD * kD) + (size_t)m * kD;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float cv[32];
            acc(half ? P2 : P0, cv);
#pragma unroll
            for (int e4 = 0; e4 < 32; e4 += 4)
                *reinterpret_cast<float4*>(dst + 64 * half + 32 * hc + e4) =
                    make_float4(cv[e4], cv[e4 + 1], cv[e4 + 2], cv[e4 + 3]);
        }
    } else if (t == 0) {
        atomicOr(a.status, CPR_DEV_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (w == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// The reverse chain and the tensor-core chunk gradients (bf16, dk = dv = 128, C = 64) in
// one cooperative launch, in place of kb2 and kb3.
cudaError_t launch_chain_and_grads_tc(const BackwardArgs& a, cudaStream_t s)
{
    auto kern = kb23_chain_and_grads_tc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kT, kSmem)) != cudaSuccess) return e;
    if (per_sm < 1 || a.num_sms < 2) return cudaErrorInvalidConfiguration;
    const int grid = per_sm * a.num_sms;
    const int n_chain = std::max(1, std::min(a.n_seqs * a.H, grid / 2));
    BackwardArgs args = a;
    int nc = n_chain;
    void* params[] = {&args, &nc};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kT), params, kSmem, s);
}

// The tensor-core chunk coefficients (bf16, dk = dv = 128, C = 64) in place of kb1.
cudaError_t launch_chunk_maps_tc(const BackwardArgs& a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(kb1_chunk_maps_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    kb1_chunk_maps_tc<<<dim3((unsigned)a.max_chunks, (unsigned)a.H), kT, kSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace cpr
