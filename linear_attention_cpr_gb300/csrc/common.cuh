// common.cuh — launch arguments, workspace layout and chunk bookkeeping shared by the
// CPR Gated DeltaNet kernels and the C-ABI host code.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/cpr_gdn.h"

namespace cpr {

// Shapes built into the library: X(DK, DV, C).
#define CPR_FOR_EACH_SHAPE(X) \
    X(32, 32, 16)             \
    X(64, 64, 32)             \
    X(128, 128, 16)           \
    X(128, 128, 32)           \
    X(128, 128, 64)

constexpr size_t kAlign = 256;
__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Upper bound on the chunks of a batch of n_seqs sequences with total_tokens tokens.
__host__ __device__ inline int64_t max_chunks_bound(int64_t total_tokens, int32_t n_seqs, int32_t C)
{
    return total_tokens / C + n_seqs;
}

// Prefill workspace:
//   [0, 256)       status word (uint32) and padding
//   cu_chunks      int32 [n_seqs + 1]
//   Wt             fp32 [max_chunks, H, DK, C]   (W of every full chunk, transposed)
//   Ut             fp32 [max_chunks, H, C, DV]   (U~ of every full chunk)
//   dvec           fp32 [max_chunks, H, C + 4]   (d_r for r < C, gamma at index C)
struct PrefillLayout {
    size_t cu_chunks, wt, ut, dvec, total;
    __host__ __device__ PrefillLayout(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk, int32_t dv,
                                      int32_t C)
    {
        const int64_t mc = max_chunks_bound(total_tokens, n_seqs, C);
        cu_chunks = kAlign;
        wt = align_up(cu_chunks + sizeof(int32_t) * (size_t)(n_seqs + 1), kAlign);
        ut = align_up(wt + sizeof(float) * (size_t)mc * H * dk * C, kAlign);
        dvec = align_up(ut + sizeof(float) * (size_t)mc * H * C * dv, kAlign);
        total = align_up(dvec + sizeof(float) * (size_t)mc * H * (C + 4), kAlign);
    }
};

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu_seqlens;
    int32_t n_seqs;
    int64_t total_tokens;
    int32_t H;
    const float* state_in;
    void* out;
    float* state_out;
    float* boundary;
    int64_t boundary_capacity;
    unsigned char* ws;
    uint32_t* status;
    int32_t* cu_chunks;
    float* wt;
    float* ut;
    float* dvec;
    int64_t max_chunks;
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    float* state;
    cpr_gdn_ring ring;
    const int32_t* pos;
    int32_t B;
    int32_t H;
    void* out;
    uint32_t* status;
};

struct RingArgs {
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu_seqlens;
    int32_t n_seqs;
    int64_t total_tokens;
    int32_t H;
    const float* boundary;
    const float* state_out;
    cpr_gdn_ring ring;
};

// Index of the sequence owning global chunk c: the n with cu_chunks[n] <= c < cu_chunks[n+1].
__device__ __forceinline__ int find_seq(const int32_t* cu_chunks, int n_seqs, int64_t c)
{
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)cu_chunks[mid] <= c)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Event recorded after the i-th kernel of a call when the profiling hook is on (else null).
cudaEvent_t profile_event(int i);
inline void profile_mark(int i, cudaStream_t s)
{
    if (cudaEvent_t e = profile_event(i)) cudaEventRecord(e, s);
}

template <int DK, int DV, int C, typename T> cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
template <int DK, int DV, int C, typename T> cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
template <int DK, int DV, int C, typename T> cudaError_t launch_ring_from_prefill(const RingArgs& a, cudaStream_t s);

}  // namespace cpr
