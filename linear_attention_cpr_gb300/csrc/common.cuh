// common.cuh — launch arguments, workspace layout and chunk bookkeeping shared by the
// CPR Gated DeltaNet kernels and the C-ABI host code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/cpr_gdn.h"

namespace cpr {

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime (the library does
// not link libcuda); NULL when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Tensor maps of a call's 2-byte (bf16) inputs for chunk boxes: keys and queries as
// [T][Hk][dk], values as [T][H][dv]; one box is C consecutive tokens of one head (rows past
// the last token read zeros).  False if the encoder is missing or refuses the layout.
struct ChunkMaps {
    CUtensorMap k, q, v;
};
bool chunk_maps(ChunkMaps* m, const void* q, const void* k, const void* v, int64_t total_tokens, int32_t H,
                int32_t Hk, int32_t dk, int32_t dv, int32_t C);

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
//   mt             [max_chunks, H] tiles of 2 * dk * dk bf16: the chunk's M^T, bf16 hi/lo
//                  splits, in the tensor cores' shared-memory image
//   bt             fp32 [max_chunks, H, dk, dv]: the chunk's B (laid out like a state)
//   ready          uint32 [max_chunks, H]: publications of each boundary state, then
//                  one uint32: the next intra-chunk item to claim
//   skip, pos_last int32 [n_seqs] each (continuation only): tokens that fill each
//                  sequence's current chunk, and the position of the last of them (-1: none)
struct PrefillLayout {
    size_t cu_chunks, mt, bt, ready, skip, pos_last, total, mt_bytes, bt_bytes;
    __host__ __device__ PrefillLayout(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk, int32_t dv,
                                      int32_t C)
    {
        const int64_t mc = max_chunks_bound(total_tokens, n_seqs, C);
        mt_bytes = (size_t)2 * dk * dk * 2;
        bt_bytes = (size_t)dk * dv * 4;
        cu_chunks = kAlign;
        mt = align_up(cu_chunks + sizeof(int32_t) * (size_t)(n_seqs + 1), kAlign);
        bt = align_up(mt + mt_bytes * (size_t)mc * H, kAlign);
        ready = align_up(bt + bt_bytes * (size_t)mc * H, kAlign);
        skip = align_up(ready + sizeof(uint32_t) * ((size_t)mc * H + 1), kAlign);
        pos_last = align_up(skip + sizeof(int32_t) * (size_t)n_seqs, kAlign);
        total = align_up(pos_last + sizeof(int32_t) * (size_t)n_seqs, kAlign);
    }
};

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu_seqlens;
    const int32_t* skip;  // NULL, or tokens of each sequence already consumed (continuation)
    int32_t n_seqs;
    int64_t total_tokens;
    int32_t H;   // value heads (states, v, g, beta, o)
    int32_t Hk;  // query/key heads: value head h reads q/k head h / (H / Hk)
    int32_t qk_norm;  // queries and keys L2-normalised in the kernels (CPR_QK_L2NORM)
    const float* state_in;
    void* out;
    float* state_out;
    float* boundary;
    int64_t boundary_capacity;
    unsigned char* ws;
    uint32_t* status;
    int32_t* cu_chunks;
    unsigned char* mt;
    float* bt;
    uint32_t* ready;
    int64_t max_chunks;
    int num_sms;
    // the items' wait for a published boundary state: the count it waits for is
    // NSLICE + wait_extra (0 except in the timeout test, where nothing reaches it), and it
    // gives up after wait_limit_ns (0: the default of about 4 s)
    uint32_t wait_extra;
    uint64_t wait_limit_ns;
};

// Backward workspace:
//   [0, 256)       status word (uint32) and padding
//   cu_chunks      int32 [n_seqs + 1]
//   mt             [max_chunks, H] x 4 dk^2 bytes: each chunk's M as the B operand of the
//                  reverse chain's product (bf16 hi, then lo, [dk][dk] K-major core matrices)
//   cb             fp32 [max_chunks, H, dk, dv]: each chunk's C_b = dO^T Qt, laid out like a state
//   d_end          fp32 [max_chunks, H, dk, dv]: the adjoint of the state at each chunk's end
//   ready          uint32 [max_chunks, H] + 1: publication counters of d_end and the item
//                  counter (the fused chain-and-gradients launch), zeroed by k0
struct BackwardLayout {
    size_t cu_chunks, mt, cb, d_end, ready, total;
    __host__ __device__ BackwardLayout(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk, int32_t dv,
                                       int32_t C)
    {
        const int64_t mc = max_chunks_bound(total_tokens, n_seqs, C);
        cu_chunks = kAlign;
        mt = align_up(cu_chunks + sizeof(int32_t) * (size_t)(n_seqs + 1), kAlign);
        cb = align_up(mt + (size_t)dk * dk * 4 * (size_t)mc * H, kAlign);
        d_end = align_up(cb + (size_t)dk * dv * 4 * (size_t)mc * H, kAlign);
        ready = align_up(d_end + (size_t)dk * dv * 4 * (size_t)mc * H, kAlign);
        total = align_up(ready + 4 * ((size_t)mc * H + 1), kAlign);
    }
};

struct BackwardArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu_seqlens;
    int32_t n_seqs;
    int64_t total_tokens;
    int32_t H;
    const float* boundary;     // the forward's boundary states [n_chunks, H, dk, dv]
    int64_t boundary_capacity;
    const void* d_out;         // [T, H, dv], the element type of q, k, v
    const float* d_state_out;  // [N, H, dk, dv] or NULL (zero)
    float* dq;
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* d_state_in;         // [N, H, dk, dv] or NULL (not wanted)
    uint32_t* status;
    uint32_t* ready;           // the hand-off counters (layout `ready`)
    int32_t* cu_chunks;
    unsigned char* mt;  // each chunk's M image for the reverse chain's products
    float* cb;
    float* d_end;
    int64_t max_chunks;
    int num_sms;
    // the chunk gradients' wait for a published d_end (fused launch): the count it waits
    // for is 1 + wait_extra (0 except in the timeout test), limit as PrefillArgs
    uint32_t wait_extra;
    uint64_t wait_limit_ns;
};

// Decode workspace: [0, 256) status word.
inline size_t decode_workspace_bytes(int32_t) { return kAlign; }

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
    int32_t Hk;       // as PrefillArgs::Hk
    int32_t qk_norm;  // as PrefillArgs::qk_norm
    void* out;
    uint32_t* status;
    int num_sms;
    int resync_only;  // continuation: every token of a completed chunk is in the ring, no output
};

struct RingArgs {
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu_seqlens;
    const int32_t* skip;      // as PrefillArgs::skip
    const uint32_t* status;   // NULL, or a status word: nonzero means do nothing
    int32_t n_seqs;
    int64_t total_tokens;
    int32_t H;
    int32_t Hk;               // as PrefillArgs::Hk
    const float* boundary;
    const float* state_out;
    cpr_gdn_ring ring;
};

// The query/key head that value head h reads (H value heads over Hk query/key heads).  The
// division sits in a separate call so that the usual case, Hk = H, runs none of it.
static __device__ __noinline__ int qk_head_grouped(int h, int H, int Hk) { return h / (H / Hk); }
__device__ __forceinline__ int qk_head(int h, int H, int Hk) { return Hk == H ? h : qk_head_grouped(h, H, Hk); }

// First token of sequence n's part of a batch: cu_seqlens[n], plus skip[n] when a
// continuation has already consumed that many of its tokens.
__device__ __forceinline__ int64_t seq_begin(const int32_t* cu, const int32_t* skip, int n)
{
    return (int64_t)cu[n] + (skip ? skip[n] : 0);
}

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

// Dynamic shared memory that keeps at most 512 / tmem_cols CTAs on one SM (233,472 bytes
// of shared memory per SM, 1 KB reserved per CTA), so the TMEM columns they allocate fit.
constexpr size_t tmem_cap_smem(uint32_t tmem_cols)
{
    return 233472 / (512 / tmem_cols + 1) - 1024 + 16;
}

// k0 alone: the chunk index (and, for a continuation, each sequence's fill tokens).
cudaError_t launch_chunk_index(const PrefillArgs& a, int32_t C, const int32_t* pos0, int32_t* skip,
                               int32_t* pos_last, cudaStream_t s);
template <int DK, int DV, int C, typename T> cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
// The two halves of a prefill after its chunk index: k1 (state independent) and k23.
template <int DK, int DV, int C, typename T> cudaError_t launch_chunk_prep(const PrefillArgs& a, cudaStream_t s);
template <int DK, int DV, int C, typename T> cudaError_t launch_chain_and_intra(const PrefillArgs& a, cudaStream_t s);
// Continuation (pos0: absolute position of each sequence's first token): the chunk index
// with the fill lengths, the fill of each sequence's current chunk and its resync, then
// the prefill of the rest and the ring.
template <int DK, int DV, int C, typename T>
cudaError_t launch_prefill_continue(const PrefillArgs& a, const int32_t* pos0, float* state, const cpr_gdn_ring& ring,
                                    cudaStream_t s);
template <int DK, int DV, int C, typename T> cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
template <int DK, int DV, int C, typename T> cudaError_t launch_ring_from_prefill(const RingArgs& a, cudaStream_t s);
// The CPR backward (k0, then the chunk maps, the reverse chain and the chunk gradients).
template <int DK, int DV, int C, typename T> cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s);
// The chunk gradients of the backward on the tensor cores (bf16, dk = dv = 128, C = 64).
cudaError_t launch_chain_and_grads_tc(const BackwardArgs& a, cudaStream_t s);
cudaError_t launch_chunk_maps_tc(const BackwardArgs& a, cudaStream_t s);
// Whether the backward's chunk kernels fit one CTA's shared memory for this shape and type.
template <int DK, int DV, int C, typename T> bool backward_fits();

}  // namespace cpr
