// reverse_chain.cuh — the CPR backward's reverse chain of one (sequence, head).
//
// With S_end = S_b M + B per chunk (backward.cu's header), the adjoint of a chunk's start
// is dS_b = dS_end M^T + C_b.  For j = last .. 0 the chain stores dS (the adjoint at chunk
// j's end) into d_end[j], then steps it to chunk j's start by the forward chain's routines
// (chunk_update.cuh): dS as the A operand in TMEM (bf16 hi / lo, value row i in lane i),
// chunk j's M image (written by kb1) as B, three tcgen05 products hi*hi + hi*lo + lo*hi
// accumulated in fp32, C_j added in the epilogue.  The images come by bulk copies two
// chunks deep; each chunk's C_j loads and d_end stores run while its product does.  The
// start value is d_state_out (zero if absent); the end value is d_state_in.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "chunk_update.cuh"
#include "common.cuh"
#include "handoff.cuh"
#include "tc.cuh"

namespace cpr {

template <int DK, int DV>
struct RevChainCfg {
    static constexpr int THREADS = 256;
    static constexpr int NW = THREADS / 32;
    static constexpr uint32_t IMG = 2u * DK * DK * 2;  // one chunk's M image (bf16 hi, lo)
    static constexpr uint32_t PIECE = 16384;
    static constexpr uint32_t BAR_OFF = 2 * IMG;       // two stages
    static constexpr size_t bytes = BAR_OFF + 64;
    // TMEM: the accumulator in columns [0, DK), the A operand in [DK, 2 DK)
    static constexpr uint32_t TMEM_COLS = 2 * DK <= 64 ? 64 : 2 * DK <= 128 ? 128 : 256;
};

// The chain of (sequence, head) nh = n H + h by all 256 threads of the CTA.  sm: at least
// RevChainCfg::bytes of shared memory (its mbarriers, at BAR_OFF, are initialised here and
// invalidated before the return); tmem: 2 DK allocated columns.  When ready is non-NULL,
// chunk j's d_end is published at ready[j H + h] (handoff.cuh) once every thread has
// stored it.  Every wait is bounded: returns false (uniformly) after a timeout, with the
// status word set and no copy or product still in flight.  Starts and ends at a barrier.
template <int DK, int DV>
__device__ __forceinline__ bool reverse_chain(const BackwardArgs& a, int nh, unsigned char* sm, uint32_t tmem,
                                              uint32_t* ready)
{
    using F = RevChainCfg<DK, DV>;
    using Mp = ChainMap<DK, F::NW>;
    uint64_t* mbar_ld = reinterpret_cast<uint64_t*>(sm + F::BAR_OFF);  // [2] stage landed
    uint64_t* mbar_mma = mbar_ld + 2;                                  // product done
    volatile int* ok_s = reinterpret_cast<volatile int*>(mbar_mma + 1);  // thread 0's wait result

    const int n = nh / a.H, h = nh % a.H, t = threadIdx.x;
    const int64_t cb = a.cu_chunks[n], nch = (int64_t)a.cu_chunks[n + 1] - cb;
    const size_t SSZ = (size_t)DK * DV;
    const float* ds_out = a.d_state_out ? a.d_state_out + (size_t)nh * SSZ : nullptr;
    float v[Mp::CPT];
    chain_load_state<DK, DV, F::NW>(ds_out, t, v);
    if (nch == 0) {  // no chunk: d_state_in = d_state_out
        if (a.d_state_in) chain_store<DK, DV, F::NW>(a.d_state_in + (size_t)nh * SSZ, t, v);
        __syncthreads();
        return true;
    }
    if (t == 0) {
        tc::mbar_init(&mbar_ld[0], 1);
        tc::mbar_init(&mbar_ld[1], 1);
        tc::mbar_init(mbar_mma, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();

    int64_t issued = 0;    // (thread 0) image copies issued, step jj into stage jj & 1
    int64_t products = 0;  // (thread 0) products issued
    auto issue = [&]() {
        const int64_t jj = issued++, j = nch - 1 - jj;
        const unsigned char* src = a.mt + ((size_t)(cb + j) * a.H + h) * F::IMG;
        unsigned char* dst = sm + (jj & 1) * F::IMG;
        tc::mbar_arrive_expect_tx(&mbar_ld[jj & 1], F::IMG);
        for (uint32_t off = 0; off < F::IMG; off += F::PIECE)
            tc::bulk_g2s(dst + off, src + off, min(F::PIECE, F::IMG - off), &mbar_ld[jj & 1]);
    };
    if (t == 0) {
        tc::fence_proxy_async();  // (the CTA's earlier shared-memory accesses, before the copies)
        issue();
        if (nch > 1) issue();
    }
    tc::fence_after_sync();  // (an earlier user of the TMEM columns is done: behind a barrier)
    chain_put_a<DK, F::NW>(tmem + DK, t, v);
    tc::fence_before_sync();
    __syncthreads();
    bool ok = true;
    for (int64_t jj = 0; jj < nch; ++jj) {
        const int64_t j = nch - 1 - jj;
        const size_t ch = (size_t)(cb + j) * a.H + h;
        bool landed = true;
        if (t == 0) {
            landed = tc::mbar_wait(&mbar_ld[jj & 1], (uint32_t)((jj >> 1) & 1));
            if (landed) {
                chain_mma<DK>(tmem, tmem + DK, sm + (jj & 1) * F::IMG, mbar_mma);
                ++products;
            }
        }
        chain_store<DK, DV, F::NW>(a.d_end + ch * SSZ, t, v);  // dS at the chunk's end
        float b[Mp::CPT];
        chain_load_b<DK, DV, F::NW>(a.cb + ch * SSZ, t, b);
        if (t == 0) ok_s[0] = (landed && tc::mbar_wait(mbar_mma, (uint32_t)(jj & 1))) ? 1 : 0;
        __syncthreads();  // (every thread's d_end stores for chunk j are issued)
        ok = ok_s[0] != 0;
        if (!ok) break;
        if (ready && t == 32) publish(ready + (size_t)(cb + j) * a.H + h);
        tc::fence_after_sync();
        if (t == 0 && issued < nch) issue();  // the product is done: its stage is free
        chain_values_reg<DK, F::NW>(tmem, t, b, v);
        if (jj + 1 < nch) chain_put_a<DK, F::NW>(tmem + DK, t, v);
        tc::fence_before_sync();
        __syncthreads();  // (every thread has read ok_s)
    }
    if (ok) {
        if (a.d_state_in) chain_store<DK, DV, F::NW>(a.d_state_in + (size_t)nh * SSZ, t, v);
    } else if (t == 0) {  // copies and a product still in flight end before the return
        atomicOr(a.status, CPR_DEV_TIMEOUT);
        for (int64_t jj = 0; jj < issued; ++jj) tc::mbar_wait(&mbar_ld[jj & 1], (uint32_t)((jj >> 1) & 1), 1u << 16);
        if (products > 0) tc::mbar_wait(mbar_mma, (uint32_t)((products - 1) & 1), 1u << 16);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (t == 0) {  // the shared memory is reused by the caller
        tc::mbar_inval(&mbar_ld[0]);
        tc::mbar_inval(&mbar_ld[1]);
        tc::mbar_inval(mbar_mma);
    }
    __syncthreads();
    return ok;
}

}  // namespace cpr
