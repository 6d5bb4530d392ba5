// prefill.cu — CPR prefill / training forward over a packed batch.
//
// "SkyRL IsoExec: vLLM 与 Megatron 的 logprob 差 ...", section "Gated DeltaNet 的第三条路：
// chunkwise-parallel recurrent": training and prefill first compute the recurrent
// state at each chunk boundary, then a parallel recurrent scan produces the outputs
// inside each chunk.  Four kernels, all on the caller's stream:
//   k0_chunk_index   cu_chunks[n] = sum_{m<n} ceil(L_m / C), with device-side checks
//   k1_chunk_prep    the state-independent half of U for every full chunk (parallel):
//                    G, decays, A, and W, U~ by forward substitution
//   k2_chain         the state-dependent half of U, sequential over each sequence's
//                    chunks, one CTA per (sequence, head, slice of value rows): writes
//                    every boundary state (and state_out when L is a multiple of C)
//   k3_intra_chunk   the token recurrence inside every chunk from its boundary state,
//                    one CTA per (chunk, head), one thread per value row holding that
//                    row of the state in registers; writes o (and state_out for a
//                    final partial chunk)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "chunk_update.cuh"
#include "numerics.cuh"

namespace cpr {

// ------------------------------------------------------------------------------------
// k0: chunk index.  One CTA of 1024 threads; each thread owns a contiguous range of
// sequences.  On invalid cu_seqlens (or too many chunks) every cu_chunks entry is 0,
// so the later kernels find no chunk, and the status word records why.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k0_chunk_index(const int32_t* __restrict__ cu, int32_t n_seqs,
                                                      int64_t total_tokens, int32_t C, int64_t capacity,
                                                      int32_t* __restrict__ cu_chunks,
                                                      uint32_t* __restrict__ status)
{
    __shared__ long long part[1024];
    __shared__ unsigned bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = (cu[0] != 0 || (int64_t)cu[n_seqs] != total_tokens) ? CPR_DEV_BAD_CU_SEQLENS : 0u;
    __syncthreads();
    const int per = (n_seqs + 1023) / 1024;
    const int n0 = min(n_seqs, tid * per), n1 = min(n_seqs, n0 + per);
    long long s = 0;
    for (int n = n0; n < n1; ++n) {
        const int L = cu[n + 1] - cu[n];
        if (L < 0) atomicOr(&bad, CPR_DEV_BAD_CU_SEQLENS);
        s += (L > 0) ? (L + C - 1) / C : 0;
    }
    part[tid] = s;
    __syncthreads();
    if (tid == 0) {
        long long run = 0;
        for (int t = 0; t < 1024; ++t) {
            const long long x = part[t];
            part[t] = run;
            run += x;
        }
        if (!bad && run > capacity) bad = CPR_DEV_BOUNDARY_CAPACITY;
        if (!bad && run > 0x7fffffffLL) bad = CPR_DEV_BOUNDARY_CAPACITY;
    }
    __syncthreads();
    const bool ok = (bad == 0);
    long long run = part[tid];
    for (int n = n0; n < n1; ++n) {
        cu_chunks[n] = ok ? (int32_t)run : 0;
        const int L = cu[n + 1] - cu[n];
        run += (L > 0) ? (L + C - 1) / C : 0;
    }
    if (tid == 1023) cu_chunks[n_seqs] = ok ? (int32_t)run : 0;  // part[1023] + its own range = total
    if (tid == 0) *status = bad;
}

// ------------------------------------------------------------------------------------
// k1: chunk prep.  One CTA per (chunk, head), DK + DV threads (one per column of
// [W | U~]).  Exits for partial chunks.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(DK + DV) k1_chunk_prep(PrefillArgs a)
{
    extern __shared__ __align__(16) float sm1[];
    const PrepSmem<DK, C> s(sm1);
    constexpr int KS = PrepSmem<DK, C>::KS;

    const int64_t c = blockIdx.x;
    const int h = blockIdx.y, tid = threadIdx.x, H = a.H;
    if (c >= a.cu_chunks[a.n_seqs]) return;
    const int n = find_seq(a.cu_chunks, a.n_seqs, c);
    const int64_t j = c - a.cu_chunks[n];
    const int64_t L = a.cu_seqlens[n + 1] - a.cu_seqlens[n];
    if ((j + 1) * C > L) return;  // partial chunk: no update
    const int64_t t0 = a.cu_seqlens[n] + j * C;
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);

    for (int idx = tid; idx < C * DK; idx += blockDim.x) {
        const int r = idx / DK, jj = idx % DK;
        s.kf[r * KS + jj] = to_f32<T>(k[((t0 + r) * H + h) * DK + jj]);
    }
    if (tid < C) {
        s.G[tid] = a.g[(t0 + tid) * H + h];
        s.bs[tid] = a.beta[(t0 + tid) * H + h];
    }
    chunk_decays_and_A<DK, C>(s);
    float x[C];
    const int col = tid;
    chunk_column<DK, DV, C, T>(s, col, v + ((size_t)t0 * H + h) * DV, (size_t)H * DV, x);
    const size_t ch = (size_t)c * H + h;
    if (col < DK) {
        float4* dst = reinterpret_cast<float4*>(a.wt + (ch * DK + col) * C);
#pragma unroll
        for (int r = 0; r < C; r += 4) dst[r / 4] = make_float4(x[r], x[r + 1], x[r + 2], x[r + 3]);
    } else {
        float* dst = a.ut + ch * C * DV + (col - DK);
#pragma unroll
        for (int r = 0; r < C; ++r) dst[(size_t)r * DV] = x[r];
    }
    if (tid < C) a.dvec[ch * (C + 4) + tid] = s.dvs[tid];
    if (tid == 0) a.dvec[ch * (C + 4) + C] = decay_exp(s.G[C - 1]);
}

// ------------------------------------------------------------------------------------
// k2: boundary chain.  One CTA per (sequence, head, slice of NS value rows).  The
// slice of the state lives in shared memory (storage order [DK][NS]); the next
// chunk's W^T, U~ slice, decays and keys are prefetched with cp.async while the
// current chunk is applied.  Slicing the value rows changes no bit: each state row
// evolves on its own.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int DK, int DV, int C, typename T>
struct K2Cfg {
    static constexpr int NS = 16;
    static constexpr int DT = (C / 4) * (NS / 4);   // delta tiles
    static constexpr int ST = (NS / 4) * (DK / 4);  // S_new tiles
    static constexpr int THREADS = ((DT > ST ? DT : ST) + 31) / 32 * 32;
    // one prefetch buffer: Wt [DK][C], Us [C][NS], dv [C + 4], kraw [C][DK] (T)
    static constexpr size_t BUF_FLOATS = (size_t)DK * C + (size_t)C * NS + (C + 4);
    static constexpr size_t KRAW_BYTES = (size_t)C * DK * sizeof(T);
    static constexpr size_t BUF_BYTES = BUF_FLOATS * sizeof(float) + KRAW_BYTES;
    static constexpr size_t bytes = 2 * BUF_BYTES + sizeof(float) * ((size_t)C * DK + (size_t)DK * NS + (size_t)C * NS);
};

template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(K2Cfg<DK, DV, C, T>::THREADS) k2_chain(PrefillArgs a)
{
    using Cf = K2Cfg<DK, DV, C, T>;
    constexpr int NS = Cf::NS;
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char* bufp[2] = {smraw, smraw + Cf::BUF_BYTES};
    float* kf = reinterpret_cast<float*>(smraw + 2 * Cf::BUF_BYTES);  // [C][DK]
    float* St = kf + C * DK;                                           // [DK][NS]
    float* dd = St + DK * NS;                                          // [C][NS]

    const int H = a.H, tid = threadIdx.x;
    const int n = blockIdx.x / H, h = blockIdx.x % H, n0 = blockIdx.y * NS;
    if (*a.status) return;
    const int64_t t0 = a.cu_seqlens[n];
    const int64_t L = a.cu_seqlens[n + 1] - t0;
    const int64_t nfull = L / C, nch = a.cu_chunks[n + 1] - a.cu_chunks[n], cbase = a.cu_chunks[n];
    const T* k = static_cast<const T*>(a.k);
    const size_t SS = (size_t)DK * DV;

    for (int idx = tid; idx < DK * NS; idx += blockDim.x) {
        const int jj = idx / NS, nn = idx % NS;
        St[idx] = a.state_in ? a.state_in[((size_t)n * H + h) * SS + (size_t)jj * DV + n0 + nn] : 0.0f;
    }
    __syncthreads();
    auto store_state = [&](float* dst) {  // dst: a [DK][DV] state; write our slice
        for (int idx = tid; idx < DK * NS / 4; idx += blockDim.x) {
            const int jj = idx / (NS / 4), q4 = idx % (NS / 4);
            *reinterpret_cast<float4*>(dst + (size_t)jj * DV + n0 + 4 * q4) =
                *reinterpret_cast<const float4*>(St + jj * NS + 4 * q4);
        }
    };
    if (L == 0) {
        store_state(a.state_out + ((size_t)n * H + h) * SS);
        return;
    }
    store_state(a.boundary + ((size_t)cbase * H + h) * SS);
    if (nfull == 0) return;

    auto issue = [&](int64_t jc, unsigned char* buf) {
        const size_t ch = (size_t)(cbase + jc) * H + h;
        float* Wt = reinterpret_cast<float*>(buf);
        float* Us = Wt + DK * C;
        float* dv = Us + C * NS;
        unsigned char* kraw = buf + Cf::BUF_FLOATS * sizeof(float);
        const float* gW = a.wt + ch * DK * C;
        for (int idx = tid; idx < DK * C / 4; idx += blockDim.x) cp_async16(Wt + 4 * idx, gW + 4 * idx);
        for (int idx = tid; idx < C * NS / 4; idx += blockDim.x) {
            const int r = idx / (NS / 4), q4 = idx % (NS / 4);
            cp_async16(Us + r * NS + 4 * q4, a.ut + (ch * C + r) * DV + n0 + 4 * q4);
        }
        for (int idx = tid; idx < (C + 4) / 4; idx += blockDim.x) cp_async16(dv + 4 * idx, a.dvec + ch * (C + 4) + 4 * idx);
        constexpr int ROW16 = DK * (int)sizeof(T) / 16;
        const int64_t tk = t0 + jc * C;
        for (int idx = tid; idx < C * ROW16; idx += blockDim.x) {
            const int r = idx / ROW16, q16 = idx % ROW16;
            cp_async16(kraw + ((size_t)r * DK * sizeof(T)) + 16 * q16,
                       reinterpret_cast<const unsigned char*>(k + ((tk + r) * H + h) * DK) + 16 * q16);
        }
    };

    issue(0, bufp[0]);
    cp_async_commit();
    for (int64_t jc = 0; jc < nfull; ++jc) {
        if (jc + 1 < nfull) issue(jc + 1, bufp[(jc + 1) & 1]);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        unsigned char* buf = bufp[jc & 1];
        const float* Wt = reinterpret_cast<const float*>(buf);
        const float* Us = Wt + DK * C;
        const float* dv = Us + C * NS;
        const T* kraw = reinterpret_cast<const T*>(buf + Cf::BUF_FLOATS * sizeof(float));
        for (int idx = tid; idx < C * DK; idx += blockDim.x) kf[idx] = to_f32<T>(kraw[idx]);
        const float gamma = dv[C];
        for (int t = tid; t < Cf::DT; t += blockDim.x) {
            const int r0 = (t / (NS / 4)) * 4, m0 = (t % (NS / 4)) * 4;
            float o[4][4];
            delta_tile<DK>(Wt, C, St, NS, Us, NS, dv, r0, m0, o);
#pragma unroll
            for (int aa = 0; aa < 4; ++aa)
                *reinterpret_cast<float4*>(dd + (r0 + aa) * NS + m0) = make_float4(o[aa][0], o[aa][1], o[aa][2], o[aa][3]);
        }
        __syncthreads();
        for (int t = tid; t < Cf::ST; t += blockDim.x) {
            const int c0 = (t % (DK / 4)) * 4, m0 = (t / (DK / 4)) * 4;
            float o[4][4];
            snew_tile<C>(St, NS, dd, NS, kf, DK, gamma, m0, c0, o);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<float4*>(St + (c0 + cc) * NS + m0) = make_float4(o[cc][0], o[cc][1], o[cc][2], o[cc][3]);
        }
        __syncthreads();
        if (jc + 1 < nch)
            store_state(a.boundary + ((size_t)(cbase + jc + 1) * H + h) * SS);
        else
            store_state(a.state_out + ((size_t)n * H + h) * SS);
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------
// k3: intra-chunk token recurrence.  One CTA per (chunk, head), DV threads; thread i
// holds row i of the state as DK/2 pairs (S[p], S[p + DK/2]) so that the two halves of
// the canonical dot's chains (chain m and chain m+4) advance in one paired FMA.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C>
struct K3Smem {
    static constexpr size_t bytes = sizeof(float) * ((size_t)2 * C * DK + (size_t)C * DV + 2 * C);
};

template <int DK, bool NEXT>
__device__ __forceinline__ void k3_token(float2 (&Sp)[DK / 2], const float2* __restrict__ kr,
                                         const float2* __restrict__ qr, const float2* __restrict__ kn,
                                         float alpha, float u, float& o, float& xn)
{
    constexpr int L = DK / 8;
    const float2 a2 = make_float2(alpha, alpha), u2 = make_float2(u, u);
    float2 co[4], cx[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int t = 0; t < L; t += 2) {
            const int p = m * L + t;
            const float4 k4 = *reinterpret_cast<const float4*>(kr + p);
            const float4 q4 = *reinterpret_cast<const float4*>(qr + p);
            const float2 k0 = make_float2(k4.x, k4.y), k1 = make_float2(k4.z, k4.w);
            const float2 q0 = make_float2(q4.x, q4.y), q1 = make_float2(q4.z, q4.w);
            const float2 s0 = __ffma2_rn(u2, k0, __fmul2_rn(a2, Sp[p]));
            const float2 s1 = __ffma2_rn(u2, k1, __fmul2_rn(a2, Sp[p + 1]));
            Sp[p] = s0;
            Sp[p + 1] = s1;
            co[m] = (t == 0) ? __fmul2_rn(s0, q0) : __ffma2_rn(s0, q0, co[m]);
            co[m] = __ffma2_rn(s1, q1, co[m]);
            if (NEXT) {
                const float4 n4 = *reinterpret_cast<const float4*>(kn + p);
                const float2 n0 = make_float2(n4.x, n4.y), n1 = make_float2(n4.z, n4.w);
                cx[m] = (t == 0) ? __fmul2_rn(s0, n0) : __ffma2_rn(s0, n0, cx[m]);
                cx[m] = __ffma2_rn(s1, n1, cx[m]);
            }
        }
    }
    o = tree8_pairs(co[0], co[1], co[2], co[3]);
    if (NEXT) xn = tree8_pairs(cx[0], cx[1], cx[2], cx[3]);
}

template <int DK>
__device__ __forceinline__ float k3_dot(const float2 (&Sp)[DK / 2], const float2* __restrict__ w)
{
    constexpr int L = DK / 8;
    float2 c[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int t = 0; t < L; t += 2) {
            const int p = m * L + t;
            const float4 w4 = *reinterpret_cast<const float4*>(w + p);
            const float2 w0 = make_float2(w4.x, w4.y), w1 = make_float2(w4.z, w4.w);
            c[m] = (t == 0) ? __fmul2_rn(Sp[p], w0) : __ffma2_rn(Sp[p], w0, c[m]);
            c[m] = __ffma2_rn(Sp[p + 1], w1, c[m]);
        }
    }
    return tree8_pairs(c[0], c[1], c[2], c[3]);
}

template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(DV, 2) k3_intra_chunk(PrefillArgs a)
{
    static_assert(DK % 16 == 0, "DK must be a multiple of 16");
    extern __shared__ __align__(16) float sm3[];
    float2* kp = reinterpret_cast<float2*>(sm3);   // [C][DK/2] pairs (k[p], k[p + DK/2])
    float2* qp = kp + C * (DK / 2);                 // [C][DK/2]
    float* vs = reinterpret_cast<float*>(qp + C * (DK / 2));  // [C][DV]
    float* al = vs + C * DV;                        // [C]
    float* bt = al + C;                             // [C]

    const int64_t c = blockIdx.x;
    const int h = blockIdx.y, i = threadIdx.x, H = a.H;
    if (c >= a.cu_chunks[a.n_seqs]) return;
    const int n = find_seq(a.cu_chunks, a.n_seqs, c);
    const int64_t j = c - a.cu_chunks[n];
    const int64_t L = a.cu_seqlens[n + 1] - a.cu_seqlens[n];
    const int64_t t0 = a.cu_seqlens[n] + j * C;
    const int len = (int)min((int64_t)C, L - j * C);
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    T* out = static_cast<T*>(a.out);

    // stage the chunk's keys, queries (as pairs) and values in shared memory
    for (int idx = i; idx < len * DK; idx += DV) {
        const int r = idx / DK, jj = idx % DK;
        const size_t g = ((size_t)(t0 + r) * H + h) * DK + jj;
        float* kd = reinterpret_cast<float*>(kp + r * (DK / 2) + (jj % (DK / 2))) + (jj / (DK / 2));
        float* qd = reinterpret_cast<float*>(qp + r * (DK / 2) + (jj % (DK / 2))) + (jj / (DK / 2));
        *kd = to_f32<T>(k[g]);
        *qd = to_f32<T>(q[g]);
    }
    for (int r = 0; r < len; ++r) vs[r * DV + i] = to_f32<T>(v[((size_t)(t0 + r) * H + h) * DV + i]);
    if (i < len) {
        al[i] = decay_exp(a.g[(t0 + i) * H + h]);
        bt[i] = a.beta[(t0 + i) * H + h];
    }
    // the chunk's boundary state, row i
    float2 Sp[DK / 2];
    const float* bsrc = a.boundary + ((size_t)c * H + h) * DK * DV + i;
#pragma unroll
    for (int p = 0; p < DK / 2; ++p) Sp[p] = make_float2(bsrc[(size_t)p * DV], bsrc[(size_t)(p + DK / 2) * DV]);
    __syncthreads();

    float x = k3_dot<DK>(Sp, kp);
    T* orow = out + ((size_t)t0 * H + h) * DV + i;
    for (int r = 0; r < len; ++r) {
        const float alpha = al[r];
        const float u = step_u(alpha, bt[r], vs[r * DV + i], x);
        float o, xn = 0.0f;
        if (r + 1 < len)
            k3_token<DK, true>(Sp, kp + r * (DK / 2), qp + r * (DK / 2), kp + (r + 1) * (DK / 2), alpha, u, o, xn);
        else
            k3_token<DK, false>(Sp, kp + r * (DK / 2), qp + r * (DK / 2), kp, alpha, u, o, xn);
        orow[(size_t)r * H * DV] = from_f32<T>(o);
        x = xn;
    }
    if (j * C + len == L && len < C) {  // final partial chunk: the stepped state is state_out
        float* dst = a.state_out + ((size_t)n * H + h) * DK * DV + i;
#pragma unroll
        for (int p = 0; p < DK / 2; ++p) {
            dst[(size_t)p * DV] = Sp[p].x;
            dst[(size_t)(p + DK / 2) * DV] = Sp[p].y;
        }
    }
}

// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T>
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s)
{
    profile_mark(0, s);
    k0_chunk_index<<<1, 1024, 0, s>>>(a.cu_seqlens, a.n_seqs, a.total_tokens, C, a.boundary_capacity,
                                      a.cu_chunks, a.status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    profile_mark(1, s);

    const size_t sm1 = sizeof(float) * PrepSmem<DK, C>::floats;
    e = cudaFuncSetAttribute(k1_chunk_prep<DK, DV, C, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    if (e != cudaSuccess) return e;
    k1_chunk_prep<DK, DV, C, T><<<dim3((unsigned)a.max_chunks, a.H), DK + DV, sm1, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    profile_mark(2, s);

    using Cf = K2Cfg<DK, DV, C, T>;
    e = cudaFuncSetAttribute(k2_chain<DK, DV, C, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::bytes);
    if (e != cudaSuccess) return e;
    k2_chain<DK, DV, C, T><<<dim3((unsigned)(a.n_seqs * a.H), DV / Cf::NS), Cf::THREADS, Cf::bytes, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    profile_mark(3, s);

    const size_t sm3 = K3Smem<DK, DV, C>::bytes;
    e = cudaFuncSetAttribute(k3_intra_chunk<DK, DV, C, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3);
    if (e != cudaSuccess) return e;
    k3_intra_chunk<DK, DV, C, T><<<dim3((unsigned)a.max_chunks, a.H), DV, sm3, s>>>(a);
    e = cudaGetLastError();
    profile_mark(4, s);
    return e;
}

#define CPR_INST_PREFILL(DK, DV, C)                                                                     \
    template cudaError_t launch_prefill<DK, DV, C, float>(const PrefillArgs&, cudaStream_t);           \
    template cudaError_t launch_prefill<DK, DV, C, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);
CPR_FOR_EACH_SHAPE(CPR_INST_PREFILL)

}  // namespace cpr
