// decode.cu — CPR decode: one token per sequence, with a resync every C tokens.
//
// "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section
// "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": decode runs the recurrent form
// and resynchronises the hidden state every C tokens, which keeps its rounding rhythm
// the same as prefill's.  Kernels, on the caller's stream:
//   k4_decode_step   the token step of every (sequence, head) whose token does not
//                    complete a chunk, on the state in HBM (the same per-element
//                    operations as prefill's intra-chunk kernel): the output, the new
//                    state and the token's slot in the ring
//   k5_resync        on a second stream, for sequences whose token completes a chunk:
//                    the token's output by the same operations, then U(ring S_b, ring
//                    chunk) by the same routines as prefill's chunk prep and chain; the
//                    result replaces both the state and ring S_b
//   k6_ring_fill     builds a ring from a prefill's results
//   k8_chunk_fill    (continuation) steps the tokens that fill each sequence's current
//                    chunk, several per sequence, on the state held in registers
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "chunk_update.cuh"
#include "common.cuh"
#include "numerics.cuh"

namespace cpr {

template <int VPT>
struct VecF;
template <>
struct VecF<1> {
    static __device__ __forceinline__ void load(const float* p, float* d) { d[0] = *p; }
    static __device__ __forceinline__ void store(float* p, const float* d) { *p = d[0]; }
};
template <>
struct VecF<2> {
    static __device__ __forceinline__ void load(const float* p, float* d)
    {
        const float2 x = *reinterpret_cast<const float2*>(p);
        d[0] = x.x;
        d[1] = x.y;
    }
    static __device__ __forceinline__ void store(float* p, const float* d)
    {
        *reinterpret_cast<float2*>(p) = make_float2(d[0], d[1]);
    }
};
template <>
struct VecF<4> {
    static __device__ __forceinline__ void load(const float* p, float* d)
    {
        const float4 x = *reinterpret_cast<const float4*>(p);
        d[0] = x.x;
        d[1] = x.y;
        d[2] = x.z;
        d[3] = x.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* d)
    {
        *reinterpret_cast<float4*>(p) = make_float4(d[0], d[1], d[2], d[3]);
    }
};

// ------------------------------------------------------------------------------------
// The token step of k4 (the same operations in the same order) as a routine, for the
// chunk fill, on a state held in registers by 8 warps: warp m owns key rows
// [m*DK/8, (m+1)*DK/8) (chain m of the canonical dot), lane l value columns
// [l*DV/32, (l+1)*DV/32); s[t][e] = S[m DK/8 + t][l DV/32 + e].  kf, qf: the token's key
// and query (fp32, shared); part, part2: [8][DV] shared scratch; v: the token's values;
// st: NULL, or where the stepped state goes (row stride DV, this thread's first element).
// Partial chains meet in shared memory and every value column's dot is finished by the
// canonical tree; warp 0 writes o.  Contains two __syncthreads (the callers' shared inputs
// must be written before the call).
// ------------------------------------------------------------------------------------
template <int DK, int DV, typename T>
__device__ __forceinline__ void token_step(float (&s)[DK / 8][DV / 32], const float* __restrict__ kf,
                                           const float* __restrict__ qf, float (*__restrict__ part)[DV],
                                           float (*__restrict__ part2)[DV], float alpha, float beta,
                                           const T* __restrict__ v, T* __restrict__ out, float* __restrict__ st)
{
    constexpr int L = DK / 8, VPT = DV / 32;
    const int m = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int e = 0; e < VPT; ++e) {
        float c = __fmul_rn(s[0][e], kf[m * L]);
#pragma unroll
        for (int t = 1; t < L; ++t) c = __fmaf_rn(s[t][e], kf[m * L + t], c);
        part[m][lane * VPT + e] = c;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < VPT; ++e) {
        const int i = lane * VPT + e;
        const float x = tree8(part[0][i], part[1][i], part[2][i], part[3][i], part[4][i], part[5][i], part[6][i],
                              part[7][i]);
        const float u = step_u(alpha, beta, to_f32<T>(v[i]), x);
#pragma unroll
        for (int t = 0; t < L; ++t) s[t][e] = step_s(s[t][e], alpha, u, kf[m * L + t]);
        float c = __fmul_rn(s[0][e], qf[m * L]);
#pragma unroll
        for (int t = 1; t < L; ++t) c = __fmaf_rn(s[t][e], qf[m * L + t], c);
        part2[m][i] = c;
    }
    if (st) {
#pragma unroll
        for (int t = 0; t < L; ++t) VecF<VPT>::store(st + (size_t)t * DV, s[t]);
    }
    __syncthreads();
    if (m == 0) {
#pragma unroll
        for (int e = 0; e < VPT; ++e) {
            const int i = lane * VPT + e;
            const float o = tree8(part2[0][i], part2[1][i], part2[2][i], part2[3][i], part2[4][i], part2[5][i],
                                  part2[6][i], part2[7][i]);
            out[i] = from_f32<T>(o);
        }
    }
}

// The token's key and query (shared, fp32) L2-normalised in place by the whole CTA: the
// two inverse norms by two threads of different warps (into scratch[0..1]), then one
// product per entry (two for the query) -- the arithmetic of l2_normalise_row.  Contains
// two __syncthreads.
template <int DK>
__device__ __forceinline__ void l2_normalise_qk(float* kf, float* qf, float* scratch)
{
    const int tid = threadIdx.x;
    if (tid == 0) scratch[0] = l2_inv<DK>([&](int c) { return kf[c]; });
    if (tid == 32) scratch[1] = l2_inv<DK>([&](int c) { return qf[c]; });
    __syncthreads();
    for (int c = tid; c < DK; c += blockDim.x) {
        kf[c] = __fmul_rn(kf[c], scratch[0]);
        qf[c] = __fmul_rn(__fmul_rn(qf[c], scratch[1]), query_scale<DK>());
    }
    __syncthreads();
}

// ------------------------------------------------------------------------------------
// k4: decode step.  NS CTAs per (sequence, head) (below), 8 warps each: warp m owns key
// rows [m*DK/8, (m+1)*DK/8) of the stored state (chain m of the canonical dot) and lane l
// owns value columns [l*DVS/32, (l+1)*DVS/32) of the CTA's DVS = DV/NS columns.  Partial
// chains meet in shared memory and every value column's dot is finished by the canonical
// tree.  Sequences whose token completes a chunk are left to k5 (their stepped state is
// replaced by the resync).
// ------------------------------------------------------------------------------------
// k4 runs NS CTAs per (sequence, head), split by value columns: CTA `cp` covers columns
// [cp DV/NS, (cp + 1) DV/NS) of every key row.  Each column's dots still take all DK keys
// in the eight canonical chains, so the values do not depend on NS; smaller CTAs (58
// registers a thread at DV = 128) keep four per SM resident, and more state loads in
// flight (the step is bound by moving the state through HBM).
template <int DV>
__host__ __device__ constexpr int k4_splits() { return DV >= 64 ? 2 : 1; }

template <int DK, int DV, int C, typename T, bool QK_NORM>
__global__ void __launch_bounds__(256) k4_decode_step(DecodeArgs a)
{
    constexpr int NS = k4_splits<DV>(), DVS = DV / NS;
    constexpr int L = DK / 8, VPT = DVS / 32;
    __shared__ __align__(16) float kf[DK];
    __shared__ __align__(16) float qf[DK];
    __shared__ __align__(16) float part[8][DVS];
    __shared__ __align__(16) float part2[8][DVS];
    __shared__ float sc[4];

    // grid (sequence x column part, query/key head, value head within its group)
    const int b = blockIdx.x / NS, cp = blockIdx.x % NS, h = blockIdx.y * gridDim.z + blockIdx.z;
    const int tid = threadIdx.x, H = a.H, i0 = cp * DVS;
    const int m = tid >> 5, lane = tid & 31;
    const int p = a.pos[b];
    if (p < 0) {
        if (tid == 0 && h == 0 && cp == 0) atomicOr(a.status, CPR_DEV_BAD_POS);
        return;
    }
    const int r = p % C;
    if (r == C - 1) return;  // k5 steps this token and resynchronises the state
    const size_t bh = (size_t)b * H + h;
    const size_t bhk = (size_t)b * a.Hk + blockIdx.y;
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* rk = static_cast<T*>(a.ring.k);
    T* rv = static_cast<T*>(a.ring.v);

    // the state's loads first: their latency overlaps the token's loads below (the ring's
    // stores there could otherwise keep them from being issued early)
    float s[L][VPT];
    float* st = a.state + bh * DK * DV + (size_t)(m * L) * DV + i0 + lane * VPT;
#pragma unroll
    for (int t = 0; t < L; ++t) VecF<VPT>::load(st + (size_t)t * DV, s[t]);
    for (int idx = tid; idx < DK; idx += 256) {
        const T kk = k[bhk * DK + idx];
        kf[idx] = to_f32<T>(kk);
        qf[idx] = to_f32<T>(q[bhk * DK + idx]);
        if (cp == 0) rk[(bh * C + r) * DK + idx] = kk;
    }
    for (int idx = tid; idx < DVS; idx += 256) rv[(bh * C + r) * DV + i0 + idx] = v[bh * DV + i0 + idx];
    if (tid == 0) {
        const float gg = a.g[bh], bb = a.beta[bh];
        sc[0] = decay_exp(gg);
        sc[1] = bb;
        if (cp == 0) {
            a.ring.g[bh * C + r] = gg;
            a.ring.beta[bh * C + r] = bb;
        }
    }
    __syncthreads();
    if (QK_NORM) l2_normalise_qk<DK>(kf, qf, sc + 2);  // (a separate build: the usual one is untouched)

    const float alpha = sc[0], beta = sc[1];
#pragma unroll
    for (int e = 0; e < VPT; ++e) {
        float c = __fmul_rn(s[0][e], kf[m * L]);
#pragma unroll
        for (int t = 1; t < L; ++t) c = __fmaf_rn(s[t][e], kf[m * L + t], c);
        part[m][lane * VPT + e] = c;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < VPT; ++e) {
        const int i = lane * VPT + e;
        const float x = tree8(part[0][i], part[1][i], part[2][i], part[3][i], part[4][i], part[5][i], part[6][i],
                              part[7][i]);
        const float u = step_u(alpha, beta, to_f32<T>(v[bh * DV + i0 + i]), x);
#pragma unroll
        for (int t = 0; t < L; ++t) s[t][e] = step_s(s[t][e], alpha, u, kf[m * L + t]);
        float c = __fmul_rn(s[0][e], qf[m * L]);
#pragma unroll
        for (int t = 1; t < L; ++t) c = __fmaf_rn(s[t][e], qf[m * L + t], c);
        part2[m][i] = c;
    }
#pragma unroll
    for (int t = 0; t < L; ++t) VecF<VPT>::store(st + (size_t)t * DV, s[t]);
    __syncthreads();
    if (m == 0) {
        T* out = static_cast<T*>(a.out);
#pragma unroll
        for (int e = 0; e < VPT; ++e) {
            const int i = lane * VPT + e;
            const float o = tree8(part2[0][i], part2[1][i], part2[2][i], part2[3][i], part2[4][i], part2[5][i],
                                  part2[6][i], part2[7][i]);
            out[bh * DV + i0 + i] = from_f32<T>(o);
        }
    }
}

// ------------------------------------------------------------------------------------
// k8: chunk fill for a continuation.  One CTA per (sequence, head), k4's mapping: the
// sequence's first skip[n] tokens (those that fill the chunk it is in, from position
// pos0[n]) are stepped one after another by k4's token step on the state held in
// registers; each token goes to its ring slot and its output to `out`.  The stepped state
// is written back; when the chunk completes, the resync (k5) then replaces it.  2-byte
// inputs arrive up front as one tensor-map box each for the keys, queries and values of
// the sequence's first C tokens (with g and beta by plain loads), so the steps read only
// shared memory; 4-byte inputs are loaded token by token.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(256) k8_chunk_fill(DecodeArgs a, const int32_t* __restrict__ cu_seqlens,
                                                     const int32_t* __restrict__ pos0,
                                                     const int32_t* __restrict__ skip,
                                                     const __grid_constant__ ChunkMaps maps)
{
    constexpr int L = DK / 8, VPT = DV / 32;
    constexpr bool kBoxes = sizeof(T) == 2;
    // token t uses buffer t & 1 of the key, query, scalars and partial sums, so the next
    // token's staging may start while warp 0 still finishes this token's output
    __shared__ __align__(16) float kf2[2][DK];
    __shared__ __align__(16) float qf2[2][DK];
    __shared__ __align__(16) float pa2[2][8][DV];
    __shared__ __align__(16) float pb2[2][8][DV];
    __shared__ float sc2[2][4];
    __shared__ float sg[C], sbeta[C];
    __shared__ uint64_t tile_bar;
    extern __shared__ __align__(128) unsigned char sm8[];  // (2-byte inputs) keys, queries, values [C][d]

    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, H = a.H;
    const int m = tid >> 5, lane = tid & 31;
    const int f = skip[n];
    if (*a.status || f <= 0) return;
    const int r0 = pos0[n] % C;
    const size_t nh = (size_t)n * H + h;
    const int hk = qk_head(h, H, a.Hk);
    const int64_t t0 = cu_seqlens[n];
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* out = static_cast<T*>(a.out);
    T* rk = static_cast<T*>(a.ring.k);
    T* rv = static_cast<T*>(a.ring.v);
    T* sk = reinterpret_cast<T*>(sm8);
    T* sq = sk + C * DK;
    T* sv = sq + C * DK;

    if constexpr (kBoxes) {
        if (tid == 0) {
            tc::mbar_init(&tile_bar, 1);
            tc::fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            tc::mbar_arrive_expect_tx(&tile_bar, (uint32_t)(2 * DK + DV) * C * 2);
            tc::tma_load_3d(sk, &maps.k, 0, hk, (int32_t)t0, &tile_bar);
            tc::tma_load_3d(sq, &maps.q, 0, hk, (int32_t)t0, &tile_bar);
            tc::tma_load_3d(sv, &maps.v, 0, h, (int32_t)t0, &tile_bar);
        }
        if (tid < f) {
            sg[tid] = a.g[(t0 + tid) * H + h];
            sbeta[tid] = a.beta[(t0 + tid) * H + h];
        }
    }
    float s[L][VPT];
    float* st = a.state + nh * DK * DV + (size_t)(m * L) * DV + lane * VPT;
#pragma unroll
    for (int t = 0; t < L; ++t) VecF<VPT>::load(st + (size_t)t * DV, s[t]);
    if constexpr (kBoxes) {
        const bool landed = tc::mbar_wait(&tile_bar, 0);
        if (!__syncthreads_and(landed)) {  // (the boxes land, bounded, before the CTA leaves)
            if (tid == 0) {
                atomicOr(a.status, CPR_DEV_TIMEOUT);
                if (!landed) tc::mbar_wait(&tile_bar, 0, 1u << 16);
            }
            return;
        }
    }
    for (int t = 0; t < f; ++t) {
        const size_t tok = ((size_t)t0 + t) * H + h;  // packed token index x H + h
        const int r = r0 + t;                          // its ring slot
        float* kf = kf2[t & 1];
        float* qf = qf2[t & 1];
        float* sc = sc2[t & 1];
        if constexpr (kBoxes) {
            for (int idx = tid; idx < DK; idx += 256) {
                const T kk = sk[t * DK + idx];
                kf[idx] = to_f32<T>(kk);
                qf[idx] = to_f32<T>(sq[t * DK + idx]);
                rk[(nh * C + r) * DK + idx] = kk;
            }
            for (int idx = tid; idx < DV; idx += 256) rv[(nh * C + r) * DV + idx] = sv[t * DV + idx];
            if (tid == 0) {
                const float gg = sg[t], bb = sbeta[t];
                sc[0] = decay_exp(gg);
                sc[1] = bb;
                a.ring.g[nh * C + r] = gg;
                a.ring.beta[nh * C + r] = bb;
            }
        } else {
            const size_t tokk = ((size_t)t0 + t) * a.Hk + hk;
            for (int idx = tid; idx < DK; idx += 256) {
                const T kk = k[tokk * DK + idx];
                kf[idx] = to_f32<T>(kk);
                qf[idx] = to_f32<T>(q[tokk * DK + idx]);
                rk[(nh * C + r) * DK + idx] = kk;
            }
            for (int idx = tid; idx < DV; idx += 256) rv[(nh * C + r) * DV + idx] = v[tok * DV + idx];
            if (tid == 0) {
                const float gg = a.g[tok], bb = a.beta[tok];
                sc[0] = decay_exp(gg);
                sc[1] = bb;
                a.ring.g[nh * C + r] = gg;
                a.ring.beta[nh * C + r] = bb;
            }
        }
        __syncthreads();
        if (a.qk_norm) l2_normalise_qk<DK>(kf, qf, sc + 2);
        token_step<DK, DV, T>(s, kf, qf, pa2[t & 1], pb2[t & 1], sc[0], sc[1], kBoxes ? sv + t * DV : v + tok * DV,
                              out + tok * DV, t + 1 == f ? st : nullptr);
        // (no barrier: the next token writes the other buffers; this token's were last read
        // before a barrier the next token's threads pass, or by warp 0 before it reaches the
        // next token's first barrier)
    }
}

// ------------------------------------------------------------------------------------
// k5: resync, on a second stream while k4 steps every sequence.  A grid of at most one
// wave walks the (sequence, head) pairs of the sequences whose token completes a chunk
// (found from pos), DK + DV threads per CTA.  Each pair runs the same routines as prefill:
// the key Gram product, the FP32 phase and the prep products of k1_chunk_prep
// (prep_operands, prep_mma, prep_epilogue, here into shared memory), then the chain
// product and epilogue of the chain role (chain_mma, chain_values) on the ring's S_b.
// The result replaces ring S_b and the state.  The chunk's last token (this step's) is
// read from the step's inputs; k4 leaves these sequences alone.
// ------------------------------------------------------------------------------------

// The output of this step's token for (b, h), from the state before the step, by the
// element sequence of k4 (per value column i: the eight chains of S k as fmul then fma
// over their DK/8 rows, the canonical tree, u, then the chains of S' q over the stepped
// rows).  Threads i < DV take column i; the stepped state itself is not kept.  The state
// is read from a shared-memory copy (Ssm, laid out as stored) whose bulk copy completes on
// mbar's phase `phase` (the step kernel keeps HBM busy meanwhile, so one copy in flight
// beats a round trip per chain).  kf, qf: DK floats of shared scratch each, part: 8 DV
// (the key normalisation's scratch, then the chains of each value column).  Returns false
// (uniformly) if the copy did not land in time.
// Ends with a barrier.
template <int DK, int DV, int C, typename T, bool QK_NORM>
__device__ __forceinline__ bool completing_token_output(const DecodeArgs& a, size_t bh, const float* Ssm, float* kf,
                                                        float* qf, float* part, uint64_t* mbar, uint32_t& phase)
{
    constexpr int L = DK / 8;
    const int tid = threadIdx.x;
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const size_t bhk = a.Hk == a.H ? bh : (bh / a.H) * a.Hk + qk_head((int)(bh % a.H), a.H, a.Hk);
    for (int idx = tid; idx < DK; idx += blockDim.x) {
        kf[idx] = to_f32<T>(k[bhk * DK + idx]);
        qf[idx] = to_f32<T>(q[bhk * DK + idx]);
    }
    float g = 0.0f, beta = 0.0f, vi = 0.0f;
    if (tid < DV) {
        g = a.g[bh];
        beta = a.beta[bh];
        vi = to_f32<T>(static_cast<const T*>(a.v)[bh * DV + tid]);
    }
    const bool ok = __syncthreads_and(tc::mbar_wait(mbar, phase & 1));
    if (!ok) {  // the copy still lands (bounded) before the CTA gives up its shared memory
        if (threadIdx.x == 0) tc::mbar_wait(mbar, phase & 1, 1u << 16);
        ++phase;
        return false;
    }
    ++phase;
    if (QK_NORM) l2_normalise_qk<DK>(kf, qf, part);
    if (tid < DV) {
        const int i = tid;
        const float* S = Ssm + i;  // S[c][i] at c * DV
        const float alpha = decay_exp(g);
        float* c = part + i;  // chain m at c[m * DV]
#pragma unroll 1
        for (int m = 0; m < 8; ++m) {
            float acc = __fmul_rn(S[(m * L) * DV], kf[m * L]);
#pragma unroll
            for (int t = 1; t < L; ++t) acc = __fmaf_rn(S[(m * L + t) * DV], kf[m * L + t], acc);
            c[m * DV] = acc;
        }
        const float x = tree8(c[0], c[DV], c[2 * DV], c[3 * DV], c[4 * DV], c[5 * DV], c[6 * DV], c[7 * DV]);
        const float u = step_u(alpha, beta, vi, x);
#pragma unroll 1
        for (int m = 0; m < 8; ++m) {
            float acc = __fmul_rn(step_s(S[(m * L) * DV], alpha, u, kf[m * L]), qf[m * L]);
#pragma unroll
            for (int t = 1; t < L; ++t) acc = __fmaf_rn(step_s(S[(m * L + t) * DV], alpha, u, kf[m * L + t]), qf[m * L + t], acc);
            c[m * DV] = acc;
        }
        const float o = tree8(c[0], c[DV], c[2 * DV], c[3 * DV], c[4 * DV], c[5 * DV], c[6 * DV], c[7 * DV]);
        static_cast<T*>(a.out)[bh * DV + i] = from_f32<T>(o);
    }
    __syncthreads();  // every read of the copy is done before its space is reused
    return true;
}
template <int DK, int DV, int C, typename T, bool QK_NORM>
__device__ __forceinline__ bool resync_one(const DecodeArgs& a, int b, int h, unsigned char* sm5, uint32_t tmem,
                                           uint64_t* mbar, uint32_t& phase)
{
    using U = UCfg<DK, DV, C>;
    const PrepSmem<DK, C> s(reinterpret_cast<float*>(sm5), reinterpret_cast<float*>(sm5 + U::RS_VEC_OFF));
    constexpr int KS = PrepSmem<DK, C>::KS;
    unsigned char* bop = sm5;                    // then the M^T image
    unsigned char* aop = sm5 + U::RS_BT_OFF;     // then B^T
    unsigned char* mt = sm5;
    float* bt = reinterpret_cast<float*>(sm5 + U::RS_BT_OFF);
    T* vsm = reinterpret_cast<T*>(sm5 + U::RS_V_OFF);

    const int tid = threadIdx.x, H = a.H;
    const size_t bh = (size_t)b * H + h;
    const size_t SS = (size_t)DK * DV;
    const T* rk = static_cast<const T*>(a.ring.k) + bh * C * DK;
    const T* rv = static_cast<const T*>(a.ring.v) + bh * C * DV;
    // tokens 0..C-2 of the chunk come from the ring, token C-1 (this step's) from the inputs:
    // the step kernel writes its ring slot concurrently (a continuation's fill has written
    // every slot, and has produced the token's output)
    const size_t bhk = (size_t)b * a.Hk + qk_head(h, H, a.Hk);
    const T* tk = a.resync_only ? rk + (size_t)(C - 1) * DK : static_cast<const T*>(a.k) + bhk * DK;
    const T* tv = a.resync_only ? rv + (size_t)(C - 1) * DV : static_cast<const T*>(a.v) + bh * DV;
    float* Ssm = reinterpret_cast<float*>(sm5 + U::RS_BT_OFF);  // the state's copy (the prep's later regions)
    if (tid == 0) {
        tc::prefetch_l2(a.ring.S_b + bh * SS, (uint32_t)(SS * sizeof(float)));  // read by the chain step
        if (!a.resync_only) {
            constexpr uint32_t BYTES = (uint32_t)(DK * DV * sizeof(float)), PIECE = 16384;
            tc::fence_proxy_async();  // (the previous pair's generic accesses to the region)
            tc::mbar_arrive_expect_tx(mbar, BYTES);
            for (uint32_t off = 0; off < BYTES; off += PIECE)
                tc::bulk_g2s(reinterpret_cast<unsigned char*>(Ssm) + off,
                             reinterpret_cast<const unsigned char*>(a.state + bh * SS) + off, min(PIECE, BYTES - off),
                             mbar);
        }
    }
    // the chunk's keys and values, 16 bytes a load, every load of a thread in flight at once
    // (issued before the token's output, stored after it)
    constexpr int VE = 16 / (int)sizeof(T), KV = DK / VE, VV = DV / VE;
    constexpr int NKV = C * KV, NVEC = NKV + C * VV, PT = (NVEC + DK + DV - 1) / (DK + DV);
    uint4 w[PT];
#pragma unroll
    for (int e = 0; e < PT; ++e) {
        const int idx = tid + e * (DK + DV);
        if (idx < NKV) {
            const int r = idx / KV, j = (idx % KV) * VE;
            w[e] = __ldg(reinterpret_cast<const uint4*>((r < C - 1 ? rk + (size_t)r * DK : tk) + j));
        } else if (idx < NVEC) {
            const int r = (idx - NKV) / VV, n = ((idx - NKV) % VV) * VE;
            w[e] = __ldg(reinterpret_cast<const uint4*>((r < C - 1 ? rv + (size_t)r * DV : tv) + n));
        }
    }
    if (!a.resync_only &&
        !completing_token_output<DK, DV, C, T, QK_NORM>(a, bh, Ssm, reinterpret_cast<float*>(sm5),
                                                        reinterpret_cast<float*>(sm5) + DK,
                                                        reinterpret_cast<float*>(sm5) + 2 * DK, mbar, phase))
        return false;
#pragma unroll
    for (int e = 0; e < PT; ++e) {
        const int idx = tid + e * (DK + DV);
        if (idx < NKV) {
            const int r = idx / KV, j = (idx % KV) * VE;
            const T* x = reinterpret_cast<const T*>(&w[e]);
#pragma unroll
            for (int q = 0; q < VE; ++q) s.kf[r * KS + j + q] = to_f32<T>(x[q]);
        } else if (idx < NVEC) {
            const int r = (idx - NKV) / VV, n = ((idx - NKV) % VV) * VE;
            *reinterpret_cast<uint4*>(vsm + (size_t)r * DV + n) = w[e];
        }
    }
    if (tid < C) {
        const bool ring_slot = tid < C - 1 || a.resync_only;
        s.G[tid] = ring_slot ? a.ring.g[bh * C + tid] : a.g[bh];
        s.bs[tid] = ring_slot ? a.ring.beta[bh * C + tid] : a.beta[bh];
    }
    if (QK_NORM) {  // the chunk's keys L2-normalised in place, one row per thread
        __syncthreads();
        if (tid < C) l2_normalise_row<DK>(s.kf + tid * KS, [](int cc) { return cc; }, false);
    }
    tc::fence_before_sync();
    bool ok = prep_operands<DK, DV, C, T, !QK_NORM>(s, aop, bop, vsm, (size_t)DV, tmem, mbar, phase);
    if (!ok) return false;
    tc::fence_after_sync();
    if (tid == 0) prep_mma<DK, DV, C>(tmem, aop, bop, mbar);
    ok = __syncthreads_and(tc::mbar_wait(mbar, phase & 1));
    ++phase;
    if (ok) prep_epilogue<DK, DV, C>(tmem, decay_exp(s.G[C - 1]), mt, bt, nullptr);
    __syncthreads();
    if (!ok) return false;
    // the chain product of prefill's chain CTAs: ring S_b as the A operand in TMEM columns
    // [DK, 2 DK), the product into [0, DK) (the prep products' columns are free again)
    constexpr int NW = (DK + DV) / 32;
    static_assert(ChainMap<DK, NW>::ROWS >= DV, "the warps cover every value row");
    constexpr int NB = ChainMap<DK, NW>::CPT / ChainMap<DK, NW>::BLK;  // column blocks per thread
    tc::fence_after_sync();
#pragma unroll 1
    for (int b = 0; b < NB; ++b) chain_put_state_block<DK, DV, NW>(a.ring.S_b + bh * SS, tmem + DK, tid, b);
    tc::tmem_wait_st();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) chain_mma<DK>(tmem, tmem + DK, mt, mbar);
    ok = __syncthreads_and(tc::mbar_wait(mbar, phase & 1));
    ++phase;
    if (!ok) return false;
    tc::fence_after_sync();
#pragma unroll 1
    for (int b = 0; b < NB; ++b)
        chain_store_block<DK, DV, NW>(tmem, bt, a.ring.S_b + bh * SS, a.state + bh * SS, tid, b);
    tc::fence_before_sync();
    __syncthreads();  // TMEM and shared memory are free for the next pair
    tc::fence_after_sync();
    return true;
}

// At most 192 registers a thread (none spilled): with 256 threads that leaves room on the
// SM for one CTA of the step kernel, which runs beside the resync.
template <int DK, int DV, int C, typename T, bool QK_NORM>
__global__ void __maxnreg__(192) k5_resync(DecodeArgs a)
{
    using U = UCfg<DK, DV, C>;
    extern __shared__ __align__(1024) unsigned char sm5[];
    __shared__ int warp_cnt[(DK + DV) / 32];
    __shared__ int found;
    // the sequences whose token completes a chunk, in ascending order: rank n <-> the n-th b
    // with pos[b] % C == C - 1 (pos >= 0); every CTA counts them from pos
    if (a.resync_only && *a.status) return;  // a continuation whose index step failed
    auto completes = [&](int b) { const int p = a.pos[b]; return p >= 0 && p % C == C - 1; };
    int total = 0;
    for (int b0 = 0; b0 < a.B; b0 += blockDim.x)
        total += __syncthreads_count((int)threadIdx.x + b0 < a.B && completes((int)threadIdx.x + b0));
    const uint32_t items = (uint32_t)total * (uint32_t)a.H;
    if (blockIdx.x >= items) return;
    // b of rank n: a block-wide scan over pos (all threads)
    auto seq_of_rank = [&](int n) -> int {
        const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
        int before = 0;
        for (int b0 = 0; b0 < a.B; b0 += blockDim.x) {
            const bool q = tid + b0 < a.B && completes(tid + b0);
            const unsigned m = __ballot_sync(0xffffffffu, q);
            if (lane == 0) warp_cnt[wid] = __popc(m);
            if (tid == 0) found = -1;
            __syncthreads();
            int rank = before + __popc(m & ((1u << lane) - 1u));
            for (int w = 0; w < wid; ++w) rank += warp_cnt[w];
            if (q && rank == n) found = tid + b0;
            int chunk_total = 0;
            for (int w = 0; w < nw; ++w) chunk_total += warp_cnt[w];
            __syncthreads();
            const int f = found;
            __syncthreads();
            if (f >= 0) return f;
            before += chunk_total;
        }
        return 0;  // not reached: n < total
    };
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm5 + U::RS_BAR_OFF);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 1);
    const int tid = threadIdx.x;
    if (tid < 32) tc::tmem_alloc(tslot, U::TMEM_COLS);
    if (tid == 0) {
        tc::mbar_init(mbar, 1);  // phases per pair: kk, Z, prep, chain
        tc::fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    uint32_t phase = 0;
    for (uint32_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int b = seq_of_rank((int)(it / a.H));
        if (!resync_one<DK, DV, C, T, QK_NORM>(a, b, (int)(it % a.H), sm5, tmem, mbar, phase)) {
            if (tid == 0) atomicOr(a.status, CPR_DEV_TIMEOUT);
            break;  // uniform: the barrier's phase is unknown after a timeout
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid < 32) tc::tmem_dealloc(tmem, U::TMEM_COLS);
}

// ------------------------------------------------------------------------------------
// k6: ring fill from a prefill.  One CTA per (sequence, head).
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(256) k6_ring_fill(RingArgs a)
{
    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, H = a.H;
    __shared__ long long cbase;
    __shared__ int valid;
    if (a.status && *a.status) return;
    if (tid == 0) {
        long long acc = 0;
        int ok = a.cu_seqlens[0] == 0;
        for (int m = 0; m < n; ++m) {
            const int64_t Lm = a.cu_seqlens[m + 1] - seq_begin(a.cu_seqlens, a.skip, m);
            ok &= (Lm >= 0);
            acc += (Lm > 0) ? (Lm + C - 1) / C : 0;
        }
        cbase = acc;
        valid = ok && a.cu_seqlens[n + 1] >= seq_begin(a.cu_seqlens, a.skip, n) &&
                (int64_t)a.cu_seqlens[n + 1] <= a.total_tokens;
    }
    __syncthreads();
    if (!valid) return;
    const int64_t t0 = seq_begin(a.cu_seqlens, a.skip, n);
    const int64_t L = a.cu_seqlens[n + 1] - t0;
    if (a.skip && L == 0) return;  // a continuation that stayed in its chunk: the fill kept the ring
    const int rem = (int)(L % C);
    const size_t nh = (size_t)n * H + h;
    const size_t SS = (size_t)DK * DV;
    const float* src = (rem != 0) ? a.boundary + ((size_t)(cbase + (L + C - 1) / C - 1) * H + h) * SS
                                   : a.state_out + nh * SS;
    float* dst = a.ring.S_b + nh * SS;
    for (size_t idx = tid; idx < SS / 4; idx += blockDim.x)
        reinterpret_cast<float4*>(dst)[idx] = reinterpret_cast<const float4*>(src)[idx];
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* rk = static_cast<T*>(a.ring.k);
    T* rv = static_cast<T*>(a.ring.v);
    const int64_t tf = t0 + L - rem;  // first token of the final partial chunk
    for (int idx = tid; idx < rem * DK; idx += blockDim.x) {
        const int r = idx / DK, jj = idx % DK;
        rk[(nh * C + r) * DK + jj] = k[((size_t)(tf + r) * a.Hk + qk_head(h, H, a.Hk)) * DK + jj];
    }
    for (int idx = tid; idx < rem * DV; idx += blockDim.x) {
        const int r = idx / DV, jj = idx % DV;
        rv[(nh * C + r) * DV + jj] = v[((size_t)(tf + r) * H + h) * DV + jj];
    }
    if (tid < rem) {
        a.ring.g[nh * C + tid] = a.g[(size_t)(tf + tid) * H + h];
        a.ring.beta[nh * C + tid] = a.beta[(size_t)(tf + tid) * H + h];
    }
}

namespace {
// Per-device side stream and fork/join events of the decode launch (created on first use).
// The side stream has the device's greatest priority: its few resync CTAs are placed as
// soon as an SM has room, ahead of the step kernel's waiting CTAs, so they run beside the
// step instead of after it.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex use;  // held by one call from its fork to its join
};
cudaError_t side_stream(SideStream*& out)
{
    static SideStream per_device[64];
    static std::mutex create;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    SideStream& ss = per_device[dev];
    std::lock_guard<std::mutex> lock(create);
    if (!ss.join) {
        int least = 0, greatest = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
        if (!ss.stream && (e = cudaStreamCreateWithPriority(&ss.stream, cudaStreamNonBlocking, greatest)) != cudaSuccess)
            return e;
        if (!ss.fork && (e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    out = &ss;
    return cudaSuccess;
}
}  // namespace

template <int DK, int DV, int C, typename T>
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    SideStream* ss = nullptr;
    if ((e = side_stream(ss)) != cudaSuccess) return e;
    // calls from several host threads take turns on the shared side stream and its events
    std::lock_guard<std::mutex> turn(ss->use);
    profile_mark(0, s);
    // fork: the resync runs on the side stream while the step kernel runs on s
    if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->stream, ss->fork, 0)) != cudaSuccess) return e;
    // dynamic shared memory also caps the CTAs per SM so their TMEM columns fit in 512
    const size_t sm5 = std::max<size_t>(UCfg<DK, DV, C>::rs_bytes(sizeof(T)), tmem_cap_smem(UCfg<DK, DV, C>::TMEM_COLS));
    auto k5 = a.qk_norm ? k5_resync<DK, DV, C, T, true> : k5_resync<DK, DV, C, T, false>;
    e = cudaFuncSetAttribute(k5, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm5);
    if (e != cudaSuccess) return e;
    // at most half the SMs, so the step kernel keeps the rest while the resync runs
    const int grid = std::max(1, std::min(a.B * a.H, std::max(1, a.num_sms / 2) * (int)(232448 / sm5)));
    k5<<<grid, DK + DV, sm5, ss->stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (a.qk_norm)
        k4_decode_step<DK, DV, C, T, true><<<dim3(a.B * k4_splits<DV>(), a.Hk, a.H / a.Hk), 256, 0, s>>>(a);
    else
        k4_decode_step<DK, DV, C, T, false><<<dim3(a.B * k4_splits<DV>(), a.Hk, a.H / a.Hk), 256, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_mark(1, s);
    // join: work issued on s after this call sees the resync's results
    if ((e = cudaEventRecord(ss->join, ss->stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, ss->join, 0)) != cudaSuccess) return e;
    profile_mark(2, s);
    return cudaSuccess;
}

template <int DK, int DV, int C, typename T>
cudaError_t launch_ring_from_prefill(const RingArgs& a, cudaStream_t s)
{
    k6_ring_fill<DK, DV, C, T><<<dim3(a.n_seqs, a.H), 256, 0, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// Continuation prefill: the chunk index (which also takes each sequence's fill tokens);
// then, on the library's side stream, the fill (k8) and the resync of the chunks it
// completes (k5, resync only, after k8), while the remainder's chunk prep (k1) runs on the
// caller's stream; once both are done, k23 runs the remaining tokens from the resulting
// states in place, and k6 fills the ring for the final partial chunks.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
cudaError_t launch_prefill_continue(const PrefillArgs& a, const int32_t* pos0, float* state,
                                    const cpr_gdn_ring& ring, cudaStream_t s)
{
    int32_t* skip = const_cast<int32_t*>(a.skip);
    int32_t* pos_last = reinterpret_cast<int32_t*>(a.ws + PrefillLayout(a.total_tokens, a.n_seqs, a.H, DK, DV, C).pos_last);
    cudaError_t e = launch_chunk_index(a, C, pos0, skip, pos_last, s);
    if (e != cudaSuccess) return e;
    DecodeArgs d{};
    d.q = a.q;
    d.k = a.k;
    d.v = a.v;
    d.g = a.g;
    d.beta = a.beta;
    d.state = state;
    d.ring = ring;
    d.pos = pos_last;
    d.B = a.n_seqs;
    d.H = a.H;
    d.Hk = a.Hk;
    d.qk_norm = a.qk_norm;
    d.out = a.out;
    d.status = a.status;
    d.num_sms = a.num_sms;
    d.resync_only = 1;
    // the fill and its resync (which update the states) run on the side stream while the
    // remainder's chunk prep (which reads only the inputs) runs on s; k23 waits for both
    SideStream* ss = nullptr;
    if ((e = side_stream(ss)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> turn(ss->use);
    if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->stream, ss->fork, 0)) != cudaSuccess) return e;
    ChunkMaps maps{};
    size_t sm8 = 0;
    if (sizeof(T) == 2 && a.total_tokens > 0) {
        if (!chunk_maps(&maps, a.q, a.k, a.v, a.total_tokens, a.H, a.Hk, DK, DV, C)) return cudaErrorInvalidValue;
        sm8 = (size_t)(2 * DK + DV) * C * sizeof(T);
        e = cudaFuncSetAttribute(k8_chunk_fill<DK, DV, C, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm8);
        if (e != cudaSuccess) return e;
    }
    k8_chunk_fill<DK, DV, C, T>
        <<<dim3((unsigned)a.n_seqs, a.H), 256, sm8, ss->stream>>>(d, a.cu_seqlens, pos0, skip, maps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t sm5 = std::max<size_t>(UCfg<DK, DV, C>::rs_bytes(sizeof(T)), tmem_cap_smem(UCfg<DK, DV, C>::TMEM_COLS));
    auto k5 = d.qk_norm ? k5_resync<DK, DV, C, T, true> : k5_resync<DK, DV, C, T, false>;
    e = cudaFuncSetAttribute(k5, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm5);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(a.n_seqs * a.H, a.num_sms * (int)(232448 / sm5)));
    k5<<<grid, DK + DV, sm5, ss->stream>>>(d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    PrefillArgs p = a;
    p.state_in = state;
    p.state_out = state;
    if ((e = launch_chunk_prep<DK, DV, C, T>(p, s)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ss->join, ss->stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, ss->join, 0)) != cudaSuccess) return e;
    if ((e = launch_chain_and_intra<DK, DV, C, T>(p, s)) != cudaSuccess) return e;
    RingArgs ra;
    ra.k = a.k;
    ra.v = a.v;
    ra.g = a.g;
    ra.beta = a.beta;
    ra.cu_seqlens = a.cu_seqlens;
    ra.skip = a.skip;
    ra.n_seqs = a.n_seqs;
    ra.total_tokens = a.total_tokens;
    ra.H = a.H;
    ra.Hk = a.Hk;
    ra.boundary = a.boundary;
    ra.state_out = state;
    ra.ring = ring;
    ra.status = a.status;
    return launch_ring_from_prefill<DK, DV, C, T>(ra, s);
}

#define CPR_INST_DECODE(DK, DV, C)                                                                         \
    template cudaError_t launch_decode<DK, DV, C, float>(const DecodeArgs&, cudaStream_t);                \
    template cudaError_t launch_decode<DK, DV, C, __nv_bfloat16>(const DecodeArgs&, cudaStream_t);        \
    template cudaError_t launch_ring_from_prefill<DK, DV, C, float>(const RingArgs&, cudaStream_t);       \
    template cudaError_t launch_ring_from_prefill<DK, DV, C, __nv_bfloat16>(const RingArgs&, cudaStream_t); \
    template cudaError_t launch_prefill_continue<DK, DV, C, float>(const PrefillArgs&, const int32_t*, float*, \
                                                                   const cpr_gdn_ring&, cudaStream_t);      \
    template cudaError_t launch_prefill_continue<DK, DV, C, __nv_bfloat16>(const PrefillArgs&, const int32_t*, \
                                                                           float*, const cpr_gdn_ring&, cudaStream_t);
CPR_FOR_EACH_SHAPE(CPR_INST_DECODE)

}  // namespace cpr
