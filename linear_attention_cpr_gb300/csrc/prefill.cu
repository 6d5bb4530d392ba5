// prefill.cu — CPR prefill / training forward over a packed batch.
//
// "SkyRL IsoExec: vLLM 与 Megatron 的 logprob 差 ...", section "Gated DeltaNet 的第三条路：
// chunkwise-parallel recurrent": training and prefill first compute the recurrent
// state at each chunk boundary, then a parallel recurrent scan produces the outputs
// inside each chunk.  Three kernels, all on the caller's stream:
//   k0_chunk_index   cu_chunks[n] = sum_{m<n} ceil(L_m / C), with device-side checks
//   k1_chunk_prep    the state-independent half of U for every full chunk (parallel):
//                    G, decays, A, and W, U~ by forward substitution
//   k23_chain_and_intra  one cooperative launch with two roles:
//                    chain CTAs: the state-dependent half of U, sequential over each
//                    sequence's chunks, one CTA per (sequence, head) at a time: every
//                    boundary state (and state_out when L is a multiple
//                    of C), each published as soon as it is stored;
//                    item groups: the token recurrence inside every chunk from its
//                    boundary state, one group of DV threads per (chunk, head), one thread
//                    per two value rows holding them in registers; writes o (and
//                    state_out for a final partial chunk)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "chunk_update.cuh"
#include "handoff.cuh"
#include "numerics.cuh"

namespace cpr {

// ------------------------------------------------------------------------------------
// k0: chunk index.  One CTA of 1024 threads; each thread owns a contiguous range of
// sequences (a shuffle scan gives each range's first chunk).  It also zeroes k23's
// publication counters.  On invalid cu_seqlens (or too many chunks) every cu_chunks entry is 0,
// so the later kernels find no chunk, and the status word records why.  For a continuation
// (pos0 non-NULL) it first takes from each sequence the tokens that fill its current chunk
// (skip[n] of them; pos_last[n] = the position of the last, or -1) and indexes the chunks of
// the rest.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k0_chunk_index(const int32_t* __restrict__ cu, int32_t n_seqs,
                                                      int64_t total_tokens, int32_t C, int64_t capacity,
                                                      int32_t* __restrict__ cu_chunks,
                                                      uint32_t* __restrict__ status, uint32_t* __restrict__ ready,
                                                      int64_t n_ready, const int32_t* __restrict__ pos0,
                                                      int32_t* __restrict__ skip, int32_t* __restrict__ pos_last)
{
    __shared__ long long warp_sum[32];
    __shared__ unsigned bad;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int64_t i = tid; i < n_ready; i += 1024) ready[i] = 0u;  // the chain/item counters of k23
    if (tid == 0) bad = (cu[0] != 0 || (int64_t)cu[n_seqs] != total_tokens) ? CPR_DEV_BAD_CU_SEQLENS : 0u;
    __syncthreads();
    const int per = (n_seqs + 1023) / 1024;
    const int n0 = min(n_seqs, tid * per), n1 = min(n_seqs, n0 + per);
    long long s = 0;
    for (int n = n0; n < n1; ++n) {
        int L = cu[n + 1] - cu[n];
        if (L < 0) atomicOr(&bad, CPR_DEV_BAD_CU_SEQLENS);
        if (pos0) {
            const int p = pos0[n];
            int f = 0;
            if (p < 0)
                atomicOr(&bad, CPR_DEV_BAD_POS);
            else if (p % C != 0)
                f = min(C - p % C, max(L, 0));
            skip[n] = f;
            pos_last[n] = f > 0 ? p + f - 1 : -1;
            L -= f;
        }
        s += (L > 0) ? (L + C - 1) / C : 0;
    }
    // exclusive prefix sum of s over the 1024 threads: warp scans, then a scan of the warp sums
    long long incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        long long w = warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const long long total = warp_sum[31];
    if (tid == 0) {
        if (!bad && total > capacity) bad = CPR_DEV_BOUNDARY_CAPACITY;
        if (!bad && total > 0x7fffffffLL) bad = CPR_DEV_BOUNDARY_CAPACITY;
    }
    __syncthreads();
    const bool ok = (bad == 0);
    long long run = incl - s + (wid > 0 ? warp_sum[wid - 1] : 0);
    for (int n = n0; n < n1; ++n) {
        cu_chunks[n] = ok ? (int32_t)run : 0;
        const int L = cu[n + 1] - cu[n] - (pos0 ? skip[n] : 0);
        run += (L > 0) ? (L + C - 1) / C : 0;
    }
    if (tid == 1023) cu_chunks[n_seqs] = ok ? (int32_t)total : 0;
    if (tid == 0) *status = bad;
}

// ------------------------------------------------------------------------------------
// k1: chunk prep.  One CTA per (chunk, head), DK + DV threads.  The key Gram product on
// the tensor cores, the FP32 phase (decays, A, T = (I + A)^-1 by forward substitution)
// and the Z product are followed by one tcgen05 product giving
// M^T and B^T of the chunk (chunk_update.cuh), written to the workspace: M^T as the
// shared-memory image the chain kernel copies in one piece, B^T as fp32 rows.
// Exits for partial chunks.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C, typename T, bool GROUPED, bool QK_NORM>
__global__ void __launch_bounds__(DK + DV) k1_chunk_prep(PrefillArgs a)
{
    using U = UCfg<DK, DV, C>;
    static_assert(U::R1 >= U::MT_BYTES, "R1 stages the M^T image");
    extern __shared__ __align__(1024) unsigned char sm1[];
    const PrepSmem<DK, C> s(reinterpret_cast<float*>(sm1), reinterpret_cast<float*>(sm1 + U::VEC_OFF));
    constexpr int KS = PrepSmem<DK, C>::KS;
    unsigned char* aop = sm1 + U::AOP_OFF;
    unsigned char* bop = sm1;  // reuses the key / A space once the FP32 phase is done
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm1 + U::PREP_BAR_OFF);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 1);

    const int64_t c = blockIdx.x;
    // grid (chunk, query/key head, value head within its group) when grouped, else
    // (chunk, head): no division for the head either way
    const int h = GROUPED ? blockIdx.y * gridDim.z + blockIdx.z : blockIdx.y, tid = threadIdx.x, H = a.H;
    if (c >= a.cu_chunks[a.n_seqs]) return;
    const int n = find_seq(a.cu_chunks, a.n_seqs, c);
    const int64_t j = c - a.cu_chunks[n];
    const int64_t tb = seq_begin(a.cu_seqlens, a.skip, n);
    const int64_t L = a.cu_seqlens[n + 1] - tb;
    if ((j + 1) * C > L) return;  // partial chunk: no update
    const int64_t t0 = tb + j * C;
    const T* k = static_cast<const T*>(a.k);
    const int kH = GROUPED ? a.Hk : H, kh = GROUPED ? (int)blockIdx.y : h;  // query/key heads, this one
    const T* v = static_cast<const T*>(a.v);

    if (tid < 32) tc::tmem_alloc(tslot, U::TMEM_COLS);
    if (tid == 0) {
        tc::mbar_init(mbar, 1);
        tc::fence_mbar_init();
    }
    {
        constexpr int VE = 16 / (int)sizeof(T), KV = DK / VE, NK = (C * KV + DK + DV - 1) / (DK + DV);
        uint4 kr[NK];
#pragma unroll
        for (int q4 = 0; q4 < NK; ++q4) {
            const int idx = tid + q4 * (DK + DV);
            if (idx < C * KV)
                kr[q4] = __ldg(reinterpret_cast<const uint4*>(k + ((t0 + idx / KV) * kH + kh) * DK + (idx % KV) * VE));
        }
#pragma unroll
        for (int q4 = 0; q4 < NK; ++q4) {
            const int idx = tid + q4 * (DK + DV);
            if (idx < C * KV) {
                const T* ke = reinterpret_cast<const T*>(&kr[q4]);
#pragma unroll
                for (int e = 0; e < VE; ++e) s.kf[(idx / KV) * KS + (idx % KV) * VE + e] = to_f32<T>(ke[e]);
            }
        }
    }
    if (tid < C) {
        s.G[tid] = a.g[(t0 + tid) * H + h];
        s.bs[tid] = a.beta[(t0 + tid) * H + h];
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (QK_NORM) {  // the keys L2-normalised in place, one row per thread
        if (tid < C) l2_normalise_row<DK>(s.kf + tid * KS, [](int cc) { return cc; }, false);
        __syncthreads();
    }
    const uint32_t tmem = *tslot;
    uint32_t phase = 0;
    bool ok = prep_operands<DK, DV, C, T, !QK_NORM>(s, aop, bop, v + ((size_t)t0 * H + h) * DV, (size_t)H * DV, tmem,
                                                   mbar, phase);
    tc::fence_after_sync();
    if (ok && tid == 0) prep_mma<DK, DV, C>(tmem, aop, bop, mbar);
    ok = __syncthreads_and(ok && tc::mbar_wait(mbar, phase & 1));  // uniform: the epilogue's TMEM loads are warp-wide
    if (ok) {
        const size_t ch = (size_t)c * H + h;
        // the operand space (R1) is dead once the products completed: it stages the outputs
        prep_epilogue<DK, DV, C>(tmem, decay_exp(s.G[C - 1]), a.mt + ch * U::MT_BYTES, a.bt + ch * DK * DV, sm1);
    } else if (tid == 0) {
        atomicOr(a.status, CPR_DEV_TIMEOUT);
    }
    __syncthreads();
    if (tid == 0) tc::bulk_wait_all();
    tc::fence_after_sync();
    if (tid < 32) tc::tmem_dealloc(tmem, U::TMEM_COLS);
}

// ------------------------------------------------------------------------------------
// Boundary chain of one (sequence, head), by a CTA of 8 warps.  Each step, the epilogue
// warps read the accumulator (value row i in TMEM lane i), add B (from shared memory),
// write the bf16-split state tile back into TMEM and arrive on an mbarrier; lane 0 of
// warp 7 is also the producer: it bulk-copies each chunk's M^T image into one of two
// shared-memory stages one chunk ahead, issues the tcgen05 chain product (M = 128) once
// every epilogue thread has arrived; as soon as every thread has read a chunk's B (an
// mbarrier of its own, before the tile is written), it bulk-copies the next chunk's B
// into the B buffer, ahead of the next M^T copy; both images are prefetched into L2 a few
// chunks ahead of their copies.  The boundary
// state is stored while the next product runs and published for the intra-chunk items one
// step later by a thread that neither polls nor produces.  All waits are bounded; a
// timeout is reported in the status word.  A chain CTA runs its chains one after another;
// its mbarrier phases continue across them.
// ------------------------------------------------------------------------------------
template <int DK, int DV>
struct K2Cfg {
    static_assert(DV <= kChainRows, "one chain product covers every value row");
    static constexpr int NSLICE = 1;  // publications per boundary state
    static constexpr uint32_t MT_BYTES = 2 * DK * DK * 2;
    static constexpr int NSTAGE = 2;  // M^T images in flight: the one in use and one ahead
    static constexpr uint32_t STAGE = MT_BYTES;
    static constexpr uint32_t BT_BYTES = DK * DV * 4;  // one chunk's B (fp32, laid out like a state)
    static constexpr uint32_t B_OFF = NSTAGE * STAGE;
    static constexpr uint32_t BAR_OFF = B_OFF + BT_BYTES;
    static constexpr uint32_t bytes = BAR_OFF + 128;
    // TMEM: the accumulator in columns [0, DK), the state tile (A operand) in [DK, 2 DK)
    static constexpr uint32_t TMEM_COLS = 2 * DK <= 64 ? 64 : 2 * DK <= 128 ? 128 : 256;
    static constexpr uint32_t PIECE = 16384;
    static constexpr int THREADS = 256;
    static constexpr int NW = THREADS / 32;  // epilogue warps (all)
};

// How many chain steps ahead the producer prefetches a chunk's M^T and B images into L2
// (k1 wrote them long before, so they come from HBM; the shared-memory copies one step
// ahead then hit in L2).
constexpr int kPrefetchAhead = 3;

template <int DK, int DV, int C, typename T>
__device__ __forceinline__ void chain_role(const PrefillArgs& a, unsigned char* sm2, int cta, int ncta)
{
    using Cf = K2Cfg<DK, DV>;
    using Mp = ChainMap<DK, Cf::NW>;
    uint64_t* mbar_ld = reinterpret_cast<uint64_t*>(sm2 + Cf::BAR_OFF);  // [NSTAGE] stage landed
    uint64_t* mbar_mma = mbar_ld + Cf::NSTAGE;                           // product done
    uint64_t* mbar_tile = mbar_mma + 1;                                  // state tile ready (all threads)
    uint64_t* mbar_b = mbar_tile + 1;                                    // the chunk's B landed
    uint64_t* mbar_bread = mbar_b + 1;                                   // every thread read the chunk's B
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar_bread + 1);
    const float* sb = reinterpret_cast<const float*>(sm2 + Cf::B_OFF);  // [DK][DV]
    volatile int* mma_ok = reinterpret_cast<volatile int*>(tslot + 1);  // [2] thread 0's wait results, by step parity

    const int H = a.H, tid = threadIdx.x, warp = tid >> 5;
    const bool producer = (tid == Cf::THREADS - 32);
    const bool publisher = (tid == 32);  // neither the poller (thread 0) nor in the producer's warp
    const size_t SS = (size_t)DK * DV;
    if (warp == 0) tc::tmem_alloc(tslot, Cf::TMEM_COLS);
    if (tid == 0) {
        for (int b = 0; b < Cf::NSTAGE; ++b) tc::mbar_init(&mbar_ld[b], 1);
        tc::mbar_init(mbar_mma, 1);
        tc::mbar_init(mbar_tile, Cf::THREADS);
        tc::mbar_init(mbar_b, 1);
        tc::mbar_init(mbar_bread, Cf::THREADS);
        tc::fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    int64_t G = 0;   // chain steps this CTA has run: the phase count of its mbarriers
    int64_t RB = 0;  // completed phases of mbar_bread (one per step that has a successor)
    bool failed = false;
    const int nchains = a.n_seqs * H;
    for (int ci = cta; ci < nchains && !failed; ci += ncta) {
        const int n = ci / H, h = ci % H;
        const int64_t t0 = seq_begin(a.cu_seqlens, a.skip, n);
        const int64_t L = a.cu_seqlens[n + 1] - t0;
        const int64_t nfull = L / C, nch = a.cu_chunks[n + 1] - a.cu_chunks[n], cbase = a.cu_chunks[n];
        const size_t nh = (size_t)n * H + h;
        const float* s_in = a.state_in ? a.state_in + nh * SS : nullptr;
        uint32_t* ready = a.ready + (size_t)cbase * H + h;  // + jc * H for chunk cbase + jc

        auto copy_state = [&](float* dst) {
            for (size_t idx = tid; idx < SS; idx += Cf::THREADS) dst[idx] = s_in ? s_in[idx] : 0.0f;
        };
        if (L == 0) {  // empty sequence: state_out = state_in
            copy_state(a.state_out + nh * SS);
            continue;
        }
        copy_state(a.boundary + ((size_t)cbase * H + h) * SS);
        __syncthreads();
        if (publisher) publish(ready);
        if (nfull == 0) continue;

        // producer (one thread): M^T stage loads and the chain products
        int64_t issued = 0;
        auto issue_load = [&](int64_t jc) {
            const size_t ch = (size_t)(cbase + jc) * H + h;
            const unsigned char* src = a.mt + ch * Cf::MT_BYTES;
            const int b = (int)((G + jc) % Cf::NSTAGE);
            unsigned char* dst = sm2 + b * Cf::STAGE;
            tc::mbar_arrive_expect_tx(&mbar_ld[b], Cf::STAGE);
            for (uint32_t off = 0; off < Cf::MT_BYTES; off += Cf::PIECE)
                tc::bulk_g2s(dst + off, src + off, min(Cf::PIECE, Cf::MT_BYTES - off), &mbar_ld[b]);
        };
        auto ld_parity = [&](int64_t jc) { return (uint32_t)(((G + jc) / Cf::NSTAGE) & 1); };
        int64_t b_issued = 0;
        auto issue_b = [&](int64_t jc) {  // chunk jc's B into the B buffer (every thread read the last one)
            const unsigned char* src = reinterpret_cast<const unsigned char*>(a.bt + ((size_t)(cbase + jc) * H + h) * SS);
            unsigned char* dst = sm2 + Cf::B_OFF;
            tc::mbar_arrive_expect_tx(mbar_b, Cf::BT_BYTES);
            for (uint32_t off = 0; off < Cf::BT_BYTES; off += Cf::PIECE)
                tc::bulk_g2s(dst + off, src + off, min(Cf::PIECE, Cf::BT_BYTES - off), mbar_b);
            ++b_issued;
        };
        // both images of chunk jc into L2 a few steps before their shared-memory copies
        auto prefetch = [&](int64_t jc) {
            if (jc >= nfull) return;
            const size_t ch = (size_t)(cbase + jc) * H + h;
            tc::prefetch_l2(a.mt + ch * Cf::MT_BYTES, Cf::MT_BYTES);
            tc::prefetch_l2(a.bt + ch * SS, Cf::BT_BYTES);
        };
        auto produce = [&](int64_t jc) -> bool {  // step jc's product, once its state tile is written
            if (!tc::mbar_wait(mbar_tile, (uint32_t)((G + jc) & 1))) return false;
            if (!tc::mbar_wait(&mbar_ld[(G + jc) % Cf::NSTAGE], ld_parity(jc))) return false;
            chain_mma<DK>(tmem, tmem + DK, sm2 + ((G + jc) % Cf::NSTAGE) * Cf::STAGE, mbar_mma);
            if (issued < nfull) issue_load(issued++);  // product jc-1 is done: its stage is free
            prefetch(jc + kPrefetchAhead);
            return true;
        };

        bool pfail = false;
        {
            float v0[Mp::CPT];
            chain_load_state<DK, DV, Cf::NW>(s_in, tid, v0);
            tc::fence_after_sync();  // the previous chain's products are done (behind a barrier)
            chain_put_a<DK, Cf::NW>(tmem + DK, tid, v0);
            tc::fence_before_sync();
            tc::mbar_arrive(mbar_tile);
        }
        if (producer) {
            for (int64_t jc = 1; jc < kPrefetchAhead; ++jc) prefetch(jc);
            for (; issued < Cf::NSTAGE - 1 && issued < nfull; ++issued) issue_load(issued);
            issue_b(0);
            pfail = !produce(0);
        }
        __syncwarp();
        // A wait that times out ends the chain for every thread: the producer then issues no
        // product, so thread 0's wait for it times out too and every thread reads the same
        // result after the barrier.
        bool ok = true;
        for (int64_t jc = 0; jc < nfull; ++jc) {
            // one thread polls the product's mbarrier, the others meet it at a hardware
            // barrier (polling by every warp would compete with the product for shared memory)
            if (tid == 0)
                mma_ok[jc & 1] = (tc::mbar_wait(mbar_mma, (uint32_t)((G + jc) & 1)) &&
                                  tc::mbar_wait(mbar_b, (uint32_t)((G + jc) & 1))) ? 1 : 0;
            __syncthreads();
            ok = mma_ok[jc & 1] != 0;
            if (!ok) break;
            tc::fence_after_sync();
            float v[Mp::CPT];
            chain_values_smem<DK, DV, Cf::NW>(tmem, tid, sb, v);
            if (jc + 1 < nfull) {
                tc::mbar_arrive(mbar_bread);
                if (warp == Cf::NW - 1) {  // the producer's warp stays converged around its wait
                    __syncwarp();
                    // chunk jc+1's B into the buffer as soon as every thread has read chunk jc's
                    if (producer && !pfail) {
                        pfail = !tc::mbar_wait(mbar_bread, (uint32_t)(RB & 1));
                        if (!pfail) issue_b(jc + 1);
                    }
                    __syncwarp();
                }
                ++RB;
                chain_put_a<DK, Cf::NW>(tmem + DK, tid, v);
            }
            tc::fence_before_sync();
            if (jc + 1 < nfull) tc::mbar_arrive(mbar_tile);
            // the boundary state completed one step ago: every store to it was issued before
            // the barrier above
            if (publisher && jc >= 1) publish(ready + (size_t)jc * H);
            if (jc + 1 < nfull) {
                // the producer issues the next product before its own loads and stores
                if (producer) pfail = !produce(jc + 1);
                __syncwarp();
            }
            float* dst = (jc + 1 < nch) ? a.boundary + ((size_t)(cbase + jc + 1) * H + h) * SS
                                        : a.state_out + nh * SS;
            chain_store<DK, DV, Cf::NW>(dst, tid, v);
        }
        // the last step's stores are issued; every thread holds the same ok
        failed = __syncthreads_or(!ok || pfail) != 0;
        if (!failed && publisher && nfull < nch) publish(ready + (size_t)nfull * H);
        if (failed && producer) {  // let copies still in flight land before the CTA exits
            for (int64_t jc = 0; jc < issued; ++jc)
                tc::mbar_wait(&mbar_ld[(G + jc) % Cf::NSTAGE], ld_parity(jc), 1u << 16);
            if (b_issued > 0) tc::mbar_wait(mbar_b, (uint32_t)((G + b_issued - 1) & 1), 1u << 16);
        }
        G += nfull;
    }
    __syncthreads();
    if (failed && tid == 0) atomicOr(a.status, CPR_DEV_TIMEOUT);
    if (tid == 0) {  // the shared memory is reused by the items
        for (int b = 0; b < Cf::NSTAGE; ++b) tc::mbar_inval(&mbar_ld[b]);
        tc::mbar_inval(mbar_mma);
        tc::mbar_inval(mbar_tile);
        tc::mbar_inval(mbar_b);
        tc::mbar_inval(mbar_bread);
    }
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, Cf::TMEM_COLS);
    __syncthreads();
}

// ------------------------------------------------------------------------------------
// Intra-chunk token recurrence of one (chunk, head) item, by a group of DV threads.
// Thread (warp w, lane l) owns two value rows, i0 = 16w + (l & 15) and i1 = i0 + DV/2,
// over one half of the key columns, h = l >> 4 (columns [h*DK/2, (h+1)*DK/2)).  It keeps
// them as pairs (S[i][c], S[i][c + DK/4]) so that chains m and m+2 of its half advance in
// one paired FMA; each key/query value loaded from shared memory serves both rows (two
// distinct addresses per warp-wide load, one per half).  The half-warps hold the two
// halves of the canonical tree, ((c0+c1)+(c2+c3)) and ((c4+c5)+(c6+c7)), and add them
// after one shuffle.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C>
struct K3Smem {
    // key/query rows: half 0's DK/4 pairs, 4 floats of padding, half 1's pairs, 4 floats
    // (the padding puts the two half-warps' broadcast loads in different banks)
    static constexpr int ROW = DK + 8;
    static constexpr int NT = DV;  // threads of a group
    // keys and queries (fp32 pairs), values as stored (at most fp32), alpha and beta
    static constexpr size_t bytes = sizeof(float) * ((size_t)2 * C * ROW + (size_t)C * DV + 2 * C);
    // 2-byte inputs arrive as tensor-map boxes: the key and query tiles as stored ([C][DK])
    // land in the tails of the key and query regions, and are converted from there
    static constexpr uint32_t REGION = 4u * C * ROW;  // bytes of the key (or the query) region
    static constexpr uint32_t RAW = 2u * C * DK;      // bytes of a 2-byte tile
    static constexpr uint32_t RAW_OFF = REGION - RAW;
    // the fp32 rows of the first C/2 keys end before the tile begins, so those rows convert
    // in place in any order; the other rows go through registers
    static_assert(4u * (C / 2) * ROW <= RAW_OFF, "first half of the rows clear of the tile");
    static_assert(RAW_OFF % 128 == 0 && REGION % 128 == 0, "tensor-map destinations 128-byte aligned");
    static constexpr int UNITS = C * DK / 16;  // conversion units of a tile: 8 pairs each
};

// One conversion unit: pairs [8m, 8m + 8) of half hh of tile row r, i.e. 8 columns from
// hh*DK/2 + 8m (the pairs' first members) and 8 from hh*DK/2 + DK/4 + 8m (their second).
template <int DK, typename T>
__device__ __forceinline__ void unit_read(const T* raw, int u, uint4& x, uint4& y)
{
    constexpr int UPR = DK / 16, MH = DK / 32;  // units per row, per half
    const int r = u / UPR, hh = (u % UPR) / MH, m = u % MH;
    const T* src = raw + r * DK + hh * (DK / 2) + 8 * m;
    x = *reinterpret_cast<const uint4*>(src);
    y = *reinterpret_cast<const uint4*>(src + DK / 4);
}

template <int DK, int ROW, typename T>
__device__ __forceinline__ void unit_write(float* region, int u, const uint4& x, const uint4& y)
{
    constexpr int UPR = DK / 16, MH = DK / 32;
    const int r = u / UPR, hh = (u % UPR) / MH, m = u % MH;
    float4* d = reinterpret_cast<float4*>(region + r * ROW + hh * (DK / 2 + 4) + 16 * m);
    const T* xe = reinterpret_cast<const T*>(&x);
    const T* ye = reinterpret_cast<const T*>(&y);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = make_float4(to_f32<T>(xe[2 * i]), to_f32<T>(ye[2 * i]), to_f32<T>(xe[2 * i + 1]),
                           to_f32<T>(ye[2 * i + 1]));
}

// bar.sync of a named barrier that also returns whether p held in every participating thread.
__device__ __forceinline__ bool named_bar_all(int id, int nthreads, bool p)
{
    uint32_t r;
    asm volatile(
        "{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\nbarrier.cta.red.and.pred po, %2, %3, pi;\n"
        "selp.u32 %0, 1, 0, po;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int DK>
struct K3Row {
    static constexpr int NP = DK / 4;  // pairs per row per thread (half of DK columns)
};

// Partial (this half) of the canonical dot of both rows with w (pairs of this half).
template <int DK>
__device__ __forceinline__ void k3_half_dot(const float2 (&S0)[DK / 4], const float2 (&S1)[DK / 4],
                                            const float2* __restrict__ w, float& d0, float& d1)
{
    constexpr int L = DK / 8;  // pair p is chain p/L (x) and p/L + 2 (y)
    float2 a0[2], a1[2];
#pragma unroll
    for (int t = 0; t < L; t += 2) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int p = m * L + t;
            const float4 w4 = *reinterpret_cast<const float4*>(w + p);
            const float2 w0 = make_float2(w4.x, w4.y), w1 = make_float2(w4.z, w4.w);
            const bool first = (t == 0);
            a0[m] = first ? __fmul2_rn(S0[p], w0) : __ffma2_rn(S0[p], w0, a0[m]);
            a1[m] = first ? __fmul2_rn(S1[p], w0) : __ffma2_rn(S1[p], w0, a1[m]);
            a0[m] = __ffma2_rn(S0[p + 1], w1, a0[m]);
            a1[m] = __ffma2_rn(S1[p + 1], w1, a1[m]);
        }
    }
    // chains (c0, c2) in a[0] and (c1, c3) in a[1]: (c0 + c1) + (c2 + c3)
    const float2 s0 = __fadd2_rn(a0[0], a0[1]), s1 = __fadd2_rn(a1[0], a1[1]);
    d0 = __fadd_rn(s0.x, s0.y);
    d1 = __fadd_rn(s1.x, s1.y);
}

template <int DK, bool NEXT>
__device__ __forceinline__ void k3_token(float2 (&S0)[DK / 4], float2 (&S1)[DK / 4], const float2* __restrict__ kr,
                                         const float2* __restrict__ qr, const float2* __restrict__ kn, float alpha,
                                         float u0, float u1, float& o0, float& o1, float& x0, float& x1)
{
    constexpr int L = DK / 8;  // pairs [0, L) carry chains (0, 2); pairs [L, 2L) chains (1, 3)
    const float2 a2 = make_float2(alpha, alpha), u02 = make_float2(u0, u0), u12 = make_float2(u1, u1);
    float2 co0[2], co1[2], cx0[2], cx1[2];
#pragma unroll
    for (int t = 0; t < L; t += 2) {
        const bool first = (t == 0);
#pragma unroll
        for (int m = 0; m < 2; ++m) {  // both chain blocks in one pass: 8 independent chains in flight
            const int p = m * L + t;
            const float4 k4 = *reinterpret_cast<const float4*>(kr + p);
            const float4 q4 = *reinterpret_cast<const float4*>(qr + p);
            const float2 k0 = make_float2(k4.x, k4.y), k1 = make_float2(k4.z, k4.w);
            const float2 q0 = make_float2(q4.x, q4.y), q1 = make_float2(q4.z, q4.w);
            const float2 s00 = __ffma2_rn(u02, k0, __fmul2_rn(a2, S0[p]));
            const float2 s10 = __ffma2_rn(u12, k0, __fmul2_rn(a2, S1[p]));
            const float2 s01 = __ffma2_rn(u02, k1, __fmul2_rn(a2, S0[p + 1]));
            const float2 s11 = __ffma2_rn(u12, k1, __fmul2_rn(a2, S1[p + 1]));
            S0[p] = s00;
            S1[p] = s10;
            S0[p + 1] = s01;
            S1[p + 1] = s11;
            co0[m] = first ? __fmul2_rn(s00, q0) : __ffma2_rn(s00, q0, co0[m]);
            co1[m] = first ? __fmul2_rn(s10, q0) : __ffma2_rn(s10, q0, co1[m]);
            if (NEXT) {
                const float4 n4 = *reinterpret_cast<const float4*>(kn + p);
                const float2 n0 = make_float2(n4.x, n4.y), n1 = make_float2(n4.z, n4.w);
                cx0[m] = first ? __fmul2_rn(s00, n0) : __ffma2_rn(s00, n0, cx0[m]);
                cx1[m] = first ? __fmul2_rn(s10, n0) : __ffma2_rn(s10, n0, cx1[m]);
                cx0[m] = __ffma2_rn(s01, n1, cx0[m]);
                cx1[m] = __ffma2_rn(s11, n1, cx1[m]);
            }
            co0[m] = __ffma2_rn(s01, q1, co0[m]);
            co1[m] = __ffma2_rn(s11, q1, co1[m]);
        }
    }
    {
        const float2 t0 = __fadd2_rn(co0[0], co0[1]), t1 = __fadd2_rn(co1[0], co1[1]);
        o0 = __fadd_rn(t0.x, t0.y);
        o1 = __fadd_rn(t1.x, t1.y);
    }
    if (NEXT) {
        const float2 t0 = __fadd2_rn(cx0[0], cx0[1]), t1 = __fadd2_rn(cx1[0], cx1[1]);
        x0 = __fadd_rn(t0.x, t0.y);
        x1 = __fadd_rn(t1.x, t1.y);
    }
}

// Both halves end with the same value: left half + right half (the canonical tree's root).
__device__ __forceinline__ float k3_join(float mine, int half)
{
    const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
    return half == 0 ? __fadd_rn(mine, other) : __fadd_rn(other, mine);
}

// Returns false when the item's boxes did not land in time (the group then stops).
template <int DK, int DV, int C, typename T>
__device__ __forceinline__ bool intra_item(const PrefillArgs& a, const ChunkMaps& maps, int64_t c, int hd, int tid,
                                           float* sm3, int bar, uint64_t* tbar, uint32_t& tphase)
{
    static_assert(DK % 32 == 0 && DV % 32 == 0, "DK and DV must be multiples of 32");
    using S3 = K3Smem<DK, DV, C>;
    constexpr int NT = S3::NT, NP = DK / 4, ROW = S3::ROW;
    // keys and queries: row r, half h, pair p at float offset r*ROW + h*(DK/2 + 4) + 2p,
    // holding (x[h*DK/2 + p], x[h*DK/2 + p + DK/4])
    float* kp = sm3;                                      // [C][ROW]
    float* qp = kp + C * ROW;                             // [C][ROW]
    T* vs = reinterpret_cast<T*>(qp + C * ROW);           // [C][DV], as stored
    float* al = reinterpret_cast<float*>(vs + C * DV);    // [C]
    float* bt = al + C;                                   // [C]

    const int H = a.H;
    const int n = find_seq(a.cu_chunks, a.n_seqs, c);
    const int64_t j = c - a.cu_chunks[n];
    const int64_t tb = seq_begin(a.cu_seqlens, a.skip, n);
    const int64_t Ls = a.cu_seqlens[n + 1] - tb;
    const int64_t t0 = tb + j * C;
    const int len = (int)min((int64_t)C, Ls - j * C);
    const int hk = qk_head(hd, H, a.Hk);
    T* out = static_cast<T*>(a.out);

    if constexpr (sizeof(T) == 2) {
        // stage the chunk: one tensor-map box each for its keys, queries and values (the
        // values stay as stored and are converted when used); keys and queries are then
        // converted into fp32 pairs
        unsigned char* base = reinterpret_cast<unsigned char*>(sm3);
        const T* rk = reinterpret_cast<const T*>(base + S3::RAW_OFF);
        const T* rq = reinterpret_cast<const T*>(base + S3::REGION + S3::RAW_OFF);
        if (tid == 0) {
            tc::mbar_arrive_expect_tx(tbar, 2 * S3::RAW + 2u * C * DV);
            tc::tma_load_3d(base + S3::RAW_OFF, &maps.k, 0, hk, (int32_t)t0, tbar);
            tc::tma_load_3d(base + S3::REGION + S3::RAW_OFF, &maps.q, 0, hk, (int32_t)t0, tbar);
            tc::tma_load_3d(vs, &maps.v, 0, hd, (int32_t)t0, tbar);
        }
        if (tid < len) {
            al[tid] = decay_exp(a.g[(t0 + tid) * H + hd]);
            bt[tid] = a.beta[(t0 + tid) * H + hd];
        }
        const bool landed = tc::mbar_wait(tbar, tphase);
        tphase ^= 1u;
        constexpr int HALF = S3::UNITS / 2;  // units of rows [0, C/2)
        constexpr int NB = (HALF + NT - 1) / NT;
        if (landed) {  // rows [0, C/2): straight into their fp32 rows, clear of both tiles
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                const int u = tid + i * NT;
                if (u < HALF) {
                    uint4 x, y;
                    unit_read<DK, T>(rk, u, x, y);
                    unit_write<DK, ROW, T>(kp, u, x, y);
                    unit_read<DK, T>(rq, u, x, y);
                    unit_write<DK, ROW, T>(qp, u, x, y);
                }
            }
        }
        // rows [C/2, C): read every unit before any thread writes over the tiles
        uint4 kx[NB], ky[NB], qx[NB], qy[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int u = HALF + tid + i * NT;
            if (landed && u < S3::UNITS) {
                unit_read<DK, T>(rk, u, kx[i], ky[i]);
                unit_read<DK, T>(rq, u, qx[i], qy[i]);
            }
        }
        if (!named_bar_all(bar, NT, landed)) {
            // a box still in flight lands (bounded wait) before the group stops
            if (tid == 0) {
                atomicOr(a.status, CPR_DEV_TIMEOUT);
                if (!landed) tc::mbar_wait(tbar, tphase ^ 1u, 1u << 16);
            }
            named_bar(bar, NT);
            return false;
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int u = HALF + tid + i * NT;
            if (u < S3::UNITS) {
                unit_write<DK, ROW, T>(kp, u, kx[i], ky[i]);
                unit_write<DK, ROW, T>(qp, u, qx[i], qy[i]);
            }
        }
    } else {
        // 4-byte inputs: values by 16-byte asynchronous copies, keys and queries by loads
        // issued a few at a time, then placed as fp32 pairs
        const T* q = static_cast<const T*>(a.q);
        const T* k = static_cast<const T*>(a.k);
        const T* v = static_cast<const T*>(a.v);
        constexpr int VE = 16 / (int)sizeof(T);
        constexpr int KV = DK / VE, VV = DV / VE;
        constexpr int NK = (C * KV + NT - 1) / NT, NV = (C * VV + NT - 1) / NT;
#pragma unroll
        for (int s = 0; s < NV; ++s) {
            const int idx = tid + s * NT, r = idx / VV, cc = idx % VV;
            if (r < len) tc::cp_async16(vs + r * DV + cc * VE, v + ((size_t)(t0 + r) * H + hd) * DV + cc * VE);
        }
        constexpr int P = NK < 2 ? NK : 2;  // loads in flight per pass
#pragma unroll
        for (int s0 = 0; s0 < NK; s0 += P) {
            uint4 kr[P], qr[P];
#pragma unroll
            for (int s = 0; s < P; ++s) {
                const int idx = tid + (s0 + s) * NT, r = idx / KV, cc = idx % KV;
                if (s0 + s < NK && r < len) {
                    const size_t g = ((size_t)(t0 + r) * a.Hk + hk) * DK + cc * VE;
                    kr[s] = __ldg(reinterpret_cast<const uint4*>(k + g));
                    qr[s] = __ldg(reinterpret_cast<const uint4*>(q + g));
                }
            }
#pragma unroll
            for (int s = 0; s < P; ++s) {
                const int idx = tid + (s0 + s) * NT, r = idx / KV, cc = idx % KV;
                if (s0 + s < NK && r < len) {
                    const T* ke = reinterpret_cast<const T*>(&kr[s]);
                    const T* qe = reinterpret_cast<const T*>(&qr[s]);
#pragma unroll
                    for (int e = 0; e < VE; ++e) {
                        const int jj = cc * VE + e, hh = jj / (DK / 2), jl = jj % (DK / 2);
                        const int pidx = r * ROW + hh * (DK / 2 + 4) + 2 * (jl % NP) + jl / NP;
                        kp[pidx] = to_f32<T>(ke[e]);
                        qp[pidx] = to_f32<T>(qe[e]);
                    }
                }
            }
        }
        tc::cp_async_wait_all();
        if (tid < len) {
            al[tid] = decay_exp(a.g[(t0 + tid) * H + hd]);
            bt[tid] = a.beta[(t0 + tid) * H + hd];
        }
    }
    if (a.qk_norm) {  // keys and queries L2-normalised in place, one row per thread
        named_bar(bar, NT);
        if (tid < 2 * len) {
            const bool query = tid >= len;
            float* row = query ? qp + (tid - len) * ROW : kp + tid * ROW;
            l2_normalise_row<DK>(row, [](int cc) {
                const int hh = cc / (DK / 2), jl = cc % (DK / 2);
                return hh * (DK / 2 + 4) + 2 * (jl % (DK / 4)) + jl / (DK / 4);
            }, query);
        }
    }
    // the chunk's boundary state comes from the chain CTAs of this launch: wait until it is
    // published (bounded)
    __shared__ int wait_ok[8];
    const int gi = bar - 1;
    if (tid == 0)
        wait_ok[gi] = wait_published(a.ready + (size_t)c * H + hd, (uint32_t)K2Cfg<DK, DV>::NSLICE + a.wait_extra,
                                     a.status, a.wait_limit_ns);
    named_bar(bar, NT);
    if (!wait_ok[gi]) {
        if (tid == 0) atomicOr(a.status, CPR_DEV_TIMEOUT);
        named_bar(bar, NT);
        return true;
    }
    const int w = tid >> 5, lane = tid & 31, half = lane >> 4;
    const int i0 = w * 16 + (lane & 15), i1 = i0 + DV / 2;
    // the chunk's boundary state: rows i0, i1 over this half's columns
    float2 S0[NP], S1[NP];
    {
        const float* bsrc = a.boundary + ((size_t)c * H + hd) * DK * DV + (size_t)(half * (DK / 2)) * DV;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            S0[p] = make_float2(bsrc[(size_t)p * DV + i0], bsrc[(size_t)(p + NP) * DV + i0]);
            S1[p] = make_float2(bsrc[(size_t)p * DV + i1], bsrc[(size_t)(p + NP) * DV + i1]);
        }
    }

    const float2* kph = reinterpret_cast<const float2*>(kp + half * (DK / 2 + 4));
    const float2* qph = reinterpret_cast<const float2*>(qp + half * (DK / 2 + 4));
    constexpr int RP = ROW / 2;  // row stride in pairs
    float x0, x1;
    k3_half_dot<DK>(S0, S1, kph, x0, x1);
    x0 = k3_join(x0, half);
    x1 = k3_join(x1, half);
    T* orow = out + ((size_t)t0 * H + hd) * DV;
    for (int r = 0; r < len; ++r) {
        const float alpha = al[r], beta = bt[r];
        const float u0 = step_u(alpha, beta, to_f32<T>(vs[r * DV + i0]), x0);
        const float u1 = step_u(alpha, beta, to_f32<T>(vs[r * DV + i1]), x1);
        float o0, o1;
        if (r + 1 < len)
            k3_token<DK, true>(S0, S1, kph + r * RP, qph + r * RP, kph + (r + 1) * RP, alpha, u0, u1, o0, o1, x0, x1);
        else
            k3_token<DK, false>(S0, S1, kph + r * RP, qph + r * RP, kph, alpha, u0, u1, o0, o1, x0, x1);
        o0 = k3_join(o0, half);
        o1 = k3_join(o1, half);
        if (r + 1 < len) {
            x0 = k3_join(x0, half);
            x1 = k3_join(x1, half);
        }
        // both halves hold both outputs: half 0 stores row i0, half 1 row i1 (no branch)
        orow[(size_t)r * H * DV + (half ? i1 : i0)] = from_f32<T>(half ? o1 : o0);
    }
    if (j * C + len == Ls && len < C) {  // final partial chunk: the stepped state is state_out
        float* dst = a.state_out + ((size_t)n * H + hd) * DK * DV + (size_t)(half * (DK / 2)) * DV;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            dst[(size_t)p * DV + i0] = S0[p].x;
            dst[(size_t)(p + NP) * DV + i0] = S0[p].y;
            dst[(size_t)p * DV + i1] = S1[p].x;
            dst[(size_t)(p + NP) * DV + i1] = S1[p].y;
        }
    }
    named_bar(bar, NT);  // the group's shared memory is reused by its next item
    return true;
}

// ------------------------------------------------------------------------------------
// k23: boundary chain and intra-chunk recurrence in one cooperative launch of one CTA per
// SM slot, 8 warps each.  CTAs [0, n_chain) run the chains (chain_role) and then join the
// others on the (chunk, head) items of the intra-chunk recurrence: 256 / DV groups of DV
// threads per CTA claim items in chunk order from a counter, each item starting as soon
// as its boundary state is published.  The chain's latency-bound steps thus overlap the FP32-bound items.
// ------------------------------------------------------------------------------------
template <int DK, int DV, int C>
struct K23Cfg {
    static constexpr int GROUPS = K2Cfg<DK, DV>::THREADS / K3Smem<DK, DV, C>::NT;
    static constexpr size_t GROUP_BYTES = (K3Smem<DK, DV, C>::bytes + 1023) / 1024 * 1024;
    static constexpr size_t bytes = K2Cfg<DK, DV>::bytes > GROUPS * GROUP_BYTES ? K2Cfg<DK, DV>::bytes : GROUPS * GROUP_BYTES;
    static_assert(GROUPS >= 1 && GROUPS <= 8, "item groups use named barriers 1..8");
};

template <int DK, int DV, int C, typename T>
__global__ void __launch_bounds__(K2Cfg<DK, DV>::THREADS, 1)
    k23_chain_and_intra(PrefillArgs a, int n_chain, const __grid_constant__ ChunkMaps maps)
{
    using F = K23Cfg<DK, DV, C>;
    constexpr int NT = K3Smem<DK, DV, C>::NT;
    extern __shared__ __align__(1024) unsigned char sm23[];
    __shared__ uint64_t tile_bar[F::GROUPS];  // each group's boxes landed
    __shared__ uint32_t claimed[F::GROUPS];
    if (*a.status) return;
    if (threadIdx.x < F::GROUPS) tc::mbar_init(&tile_bar[threadIdx.x], 1);
    tc::fence_mbar_init();
    __syncthreads();
    // chain CTAs join the items once their chains are done
    if ((int)blockIdx.x < n_chain) chain_role<DK, DV, C, T>(a, sm23, blockIdx.x, n_chain);
    const int g = threadIdx.x / NT, gtid = (int)threadIdx.x % NT;
    const uint32_t items = (uint32_t)a.cu_chunks[a.n_seqs] * (uint32_t)a.H;
    uint32_t* next_item = a.ready + (size_t)a.max_chunks * a.H;
    float* smg = reinterpret_cast<float*>(sm23 + g * F::GROUP_BYTES);
    uint32_t tphase = 0;
    for (;;) {  // items are claimed in chunk order, one group at a time
        // this thread's shared-memory accesses (the last item's, or the chain's) come before
        // the boxes the next item's copies write
        tc::fence_proxy_async();
        if (gtid == 0) claimed[g] = atomicAdd(next_item, 1u);
        named_bar(1 + g, NT);
        const uint32_t t = claimed[g];
        if (t >= items) break;
        // (ends with a group barrier)
        if (!intra_item<DK, DV, C, T>(a, maps, t / a.H, (int)(t % a.H), gtid, smg, 1 + g, &tile_bar[g], tphase))
            break;
    }
}

// ------------------------------------------------------------------------------------
cudaError_t launch_chunk_index(const PrefillArgs& a, int32_t C, const int32_t* pos0, int32_t* skip,
                               int32_t* pos_last, cudaStream_t s)
{
    k0_chunk_index<<<1, 1024, 0, s>>>(a.cu_seqlens, a.n_seqs, a.total_tokens, C, a.boundary_capacity, a.cu_chunks,
                                      a.status, a.ready, (int64_t)a.max_chunks * a.H + 1, pos0, skip, pos_last);
    return cudaGetLastError();
}

template <int DK, int DV, int C, typename T>
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s)
{
    profile_mark(0, s);
    if (!a.skip)  // (a continuation has run the chunk index itself)
        k0_chunk_index<<<1, 1024, 0, s>>>(a.cu_seqlens, a.n_seqs, a.total_tokens, C, a.boundary_capacity,
                                          a.cu_chunks, a.status, a.ready, (int64_t)a.max_chunks * a.H + 1, nullptr,
                                          nullptr, nullptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    profile_mark(1, s);
    if ((e = launch_chunk_prep<DK, DV, C, T>(a, s)) != cudaSuccess) return e;
    profile_mark(2, s);
    e = launch_chain_and_intra<DK, DV, C, T>(a, s);
    profile_mark(3, s);
    return e;
}

template <int DK, int DV, int C, typename T>
cudaError_t launch_chunk_prep(const PrefillArgs& a, cudaStream_t s)
{
    cudaError_t e;
    // dynamic shared memory also caps the CTAs per SM so their TMEM columns fit in 512
    const size_t sm1 = std::max<size_t>(UCfg<DK, DV, C>::PREP_SMEM, tmem_cap_smem(UCfg<DK, DV, C>::TMEM_COLS));
    // separate builds for grouped heads and for normalised keys: the usual one is untouched
    auto k1 = (a.Hk == a.H) ? (a.qk_norm ? k1_chunk_prep<DK, DV, C, T, false, true> : k1_chunk_prep<DK, DV, C, T, false, false>)
                            : (a.qk_norm ? k1_chunk_prep<DK, DV, C, T, true, true> : k1_chunk_prep<DK, DV, C, T, true, false>);
    e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    if (e != cudaSuccess) return e;
    k1<<<dim3((unsigned)a.max_chunks, a.Hk, a.H / a.Hk), DK + DV, sm1, s>>>(a);
    return cudaGetLastError();
}

bool chunk_maps(ChunkMaps* m, const void* q, const void* k, const void* v, int64_t total_tokens, int32_t H,
                int32_t Hk, int32_t dk, int32_t dv, int32_t C)
{
    const EncodeTiledFn f = tensor_map_encoder();
    if (!f || total_tokens < 1 || total_tokens > 0x7fffffff || C < 1 || C > 256) return false;
    auto enc = [&](CUtensorMap* map, const void* base, int d, int heads) {
        if (d < 8 || d > 256 || d % 8 != 0 || ((uintptr_t)base & 15u)) return false;
        const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)total_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
        const cuuint32_t box[3] = {(cuuint32_t)d, 1, (cuuint32_t)C}, estr[3] = {1, 1, 1};
        return f(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    return enc(&m->k, k, dk, Hk) && enc(&m->q, q, dk, Hk) && enc(&m->v, v, dv, H);
}

template <int DK, int DV, int C, typename T>
cudaError_t launch_chain_and_intra(const PrefillArgs& a, cudaStream_t s)
{
    cudaError_t e;
    using Cf = K2Cfg<DK, DV>;
    auto kern = k23_chain_and_intra<DK, DV, C, T>;
    const size_t sm23 = std::max<size_t>(K23Cfg<DK, DV, C>::bytes, tmem_cap_smem(Cf::TMEM_COLS));
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm23);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cf::THREADS, sm23);
    if (e != cudaSuccess) return e;
    if (per_sm < 1 || a.num_sms < 2) return cudaErrorInvalidConfiguration;
    const int grid = per_sm * a.num_sms;
    const int chains = a.n_seqs * a.H;
    const int n_chain = std::max(1, std::min(chains, grid / 2));
    PrefillArgs args = a;
    int nc = n_chain;
    ChunkMaps maps{};
    // (no tokens: no items, and the maps stay unused)
    if (sizeof(T) == 2 && a.total_tokens > 0 &&
        !chunk_maps(&maps, a.q, a.k, a.v, a.total_tokens, a.H, a.Hk, DK, DV, C))
        return cudaErrorInvalidValue;
    void* params[] = {&args, &nc, &maps};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(Cf::THREADS), params, sm23,
                                       s);
}

#define CPR_INST_PREFILL(DK, DV, C)                                                                     \
    template cudaError_t launch_prefill<DK, DV, C, float>(const PrefillArgs&, cudaStream_t);           \
    template cudaError_t launch_prefill<DK, DV, C, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);   \
    template cudaError_t launch_chunk_prep<DK, DV, C, float>(const PrefillArgs&, cudaStream_t);        \
    template cudaError_t launch_chunk_prep<DK, DV, C, __nv_bfloat16>(const PrefillArgs&, cudaStream_t); \
    template cudaError_t launch_chain_and_intra<DK, DV, C, float>(const PrefillArgs&, cudaStream_t);   \
    template cudaError_t launch_chain_and_intra<DK, DV, C, __nv_bfloat16>(const PrefillArgs&, cudaStream_t);
CPR_FOR_EACH_SHAPE(CPR_INST_PREFILL)

}  // namespace cpr
