/*
 * cpr_gdn.h — C ABI of the Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet layer
 * for one GB300 GPU (sm_103a).
 *
 * The method: "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section
 * "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet", and "SkyRL IsoExec: vLLM 与
 * Megatron 的 logprob 差 ...", section "Gated DeltaNet 的第三条路：chunkwise-parallel
 * recurrent".  CPR keeps the token recurrence of Gated DeltaNet
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t,
 *     alpha_t = exp(g_t)
 * (S is dv x dk, fp32) as the function that produces every output, and evaluates it
 * in three steps:
 *   1. the state at every chunk boundary (every C tokens from each sequence's start)
 *      is produced by one fixed-order fp32 chunk-update function U(S_b, chunk);
 *   2. the outputs inside each chunk are produced by the token recurrence starting
 *      from the chunk's boundary state, all chunks in parallel;
 *   3. decode runs the same token recurrence one token at a time and, when a token
 *      completes a chunk, replaces its state by U(S_b, chunk) — the same U.
 * Consequently prefill, training-forward and decode give bit-identical outputs and
 * states, and no result depends on batch composition, packing or batch position.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers (unless the name ends in _host), on the
 *     current CUDA device, row-major and contiguous.  The caller owns every buffer;
 *     the library allocates no memory and reads no host memory during a call, and all
 *     work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - dtype selects the element type of q, k, v, out and the ring's k, v:
 *     CPR_DTYPE_BF16 (2 bytes) or CPR_DTYPE_F32 (4 bytes).  g, beta and every state
 *     are fp32.
 *   - A state is stored per (sequence, head) as [dk, dv]: element (j, i) holds S[i][j]
 *     (row i of S is the value index).
 *   - Supported shapes: dk == dv in {32, 64, 128}; C in {16, 32, 64} (not every pair
 *     is built: cpr_gdn_supported() answers).  Other shapes return
 *     CPR_ERR_UNSUPPORTED_SHAPE.
 *   - Alignment: q, k, v, out, states, boundary states, ring buffers and the
 *     workspace must be 16-byte aligned (CPR_ERR_MISALIGNED otherwise); g, beta,
 *     cu_seqlens and pos 4-byte aligned.
 *   - Errors: a negative return value means nothing was enqueued (argument checks)
 *     or a launch failed (CPR_ERR_CUDA).  Checks that need device data (cu_seqlens,
 *     pos) run on the device: they skip the offending work and record a bit in the
 *     workspace status word, read with cpr_gdn_device_status().  Asynchronous CUDA
 *     errors surface at the caller's next synchronisation.
 */
#ifndef CPR_GDN_H
#define CPR_GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define CPR_OK 0
#define CPR_ERR_INVALID_ARG (-1)       /* null pointer, negative size, bad dtype, ... */
#define CPR_ERR_UNSUPPORTED_SHAPE (-2) /* (dk, dv, C) not built into this library */
#define CPR_ERR_MISALIGNED (-3)        /* a pointer breaks the alignment rule above */
#define CPR_ERR_WORKSPACE (-4)         /* workspace missing or smaller than required */
#define CPR_ERR_CUDA (-5)              /* a kernel launch or CUDA runtime call failed */

/* Bits of the device status word (cpr_gdn_device_status). */
#define CPR_DEV_BAD_CU_SEQLENS 1u /* cu_seqlens[0] != 0, decreasing, or last != total_tokens */
#define CPR_DEV_BOUNDARY_CAPACITY 2u /* more chunks than boundary_capacity */
#define CPR_DEV_BAD_POS 4u        /* a decode position is negative */
#define CPR_DEV_TIMEOUT 8u        /* a bounded device wait gave up (the work behind it skipped) */

/* Element types of q, k, v, out and the ring's k, v. */
#define CPR_DTYPE_BF16 0
#define CPR_DTYPE_F32 1

/*
 * Decode ring: what decode keeps per (sequence, head) between calls so that it can
 * resynchronise at the end of the current chunk.  All device pointers, caller-owned:
 *   S_b   fp32  [B, H, dk, dv]  state at the start of the sequence's current chunk
 *   k     dtype [B, H, C, dk]   keys of the current chunk so far (slot = position % C)
 *   v     dtype [B, H, C, dv]   values of the current chunk so far
 *   g     fp32  [B, H, C]       log-decays of the current chunk so far
 *   beta  fp32  [B, H, C]       write strengths of the current chunk so far
 * Decode reads and writes it in place; cpr_gdn_ring_from_prefill() fills it.
 */
typedef struct cpr_gdn_ring {
    float* S_b;
    void* k;
    void* v;
    float* g;
    float* beta;
} cpr_gdn_ring;

/* 1 if (dk, dv, C, dtype) is built into this library, else 0. */
int cpr_gdn_supported(int32_t dk, int32_t dv, int32_t C, int32_t dtype);

/* Library ABI version (incremented on any change of these declarations). */
int32_t cpr_gdn_version(void);

/* Human-readable text of a return code. Never NULL; the string is static. */
const char* cpr_gdn_strerror(int32_t code);

/*
 * Number of chunks of a packed batch: sum over sequences of ceil(L_n / C), where
 * L_n = cu_seqlens_host[n+1] - cu_seqlens_host[n].  HOST pointer.  This is the row
 * count of boundary_states.  Returns a negative code on invalid input.
 */
int64_t cpr_gdn_num_chunks(const int32_t* cu_seqlens_host, int32_t n_seqs, int32_t C);

/*
 * Bytes of device workspace cpr_gdn_prefill needs for a batch of n_seqs sequences
 * holding total_tokens tokens (an upper bound: it does not depend on how the tokens
 * are split between sequences).  0 on invalid arguments.
 */
size_t cpr_gdn_prefill_workspace_size(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk,
                                      int32_t dv, int32_t C);

/* Bytes of device workspace cpr_gdn_decode needs (the status word). */
size_t cpr_gdn_decode_workspace_size(int32_t B, int32_t H, int32_t dk, int32_t dv, int32_t C);

/*
 * CPR prefill / training forward over a packed batch (CPR steps 1 and 2).
 *   q, k        dtype [total_tokens, H, dk]     (caller applies any q scaling / key norm)
 *   v           dtype [total_tokens, H, dv]
 *   g, beta     fp32  [total_tokens, H]          g = log(alpha) <= 0, beta in [0, 1]
 *   cu_seqlens  int32 [n_seqs + 1]  DEVICE; cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[n_seqs] = total_tokens.  Every sequence starts at its own
 *               position 0: the chunk grid is anchored there.
 *   state_in    fp32  [n_seqs, H, dk, dv] initial states, or NULL for zero states.
 * Outputs:
 *   out         dtype [total_tokens, H, dv]   o_t = S_t q_t (rounded to nearest even
 *               when dtype is bf16)
 *   state_out   fp32  [n_seqs, H, dk, dv]     state after each sequence's last token:
 *               U's result when L_n is a multiple of C, else the stepped state.
 *               (state_in when L_n = 0.)
 *   boundary_states fp32 [boundary_capacity, H, dk, dv]: row c holds the state at the
 *               start of chunk c (chunks numbered in packed order, sequence by sequence;
 *               row 0 of each sequence is its state_in).  Rows beyond the batch's chunk
 *               count are not written.  If the count exceeds boundary_capacity nothing
 *               is written and CPR_DEV_BOUNDARY_CAPACITY is recorded.
 *   workspace   >= cpr_gdn_prefill_workspace_size(...) bytes, 16-byte aligned; holds
 *               the status word of this call.  Calls sharing a workspace must not
 *               overlap on the device.
 * Buffers must not overlap each other, except that state_out may equal state_in.
 */
int32_t cpr_gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                        int32_t dk, int32_t dv, int32_t C, int32_t dtype, const float* state_in,
                        void* out, float* state_out, float* boundary_states, int64_t boundary_capacity,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * The CPR backward: gradients of a loss L with respect to the layer's inputs, given its
 * upstream gradients dL/do and dL/dS_T.  ("IsoExec: Eliminating Trainer-Inference
 * Mismatch in SkyRL", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet",
 * per-layer table, row "Trainer Fwd+Bwd": the pages time the trainer's backward but do
 * not describe it; this is the exact adjoint of the token recurrence above, run back
 * over the forward's chunk grid.)  Three steps on `stream`:
 *   1. per chunk, independent of the states: the chunk's linear map M (S_end = S_b M + B)
 *      and C_b = dO^T Qt, where row t of Qt is the chunk's query t carried back through
 *      the chunk's first t token transitions;
 *   2. per (sequence, head), from the last chunk to the first, the adjoint at every chunk
 *      boundary: dS_b = dS_end M^T + C_b (starting from d_state_out);
 *   3. per chunk, in parallel: the chunk's gradients from its boundary state (saved by the
 *      forward) and the adjoint at its end, through the WY form of the chunk.
 * All arithmetic is fp32 in a fixed order without atomics: results are reproducible and
 * independent of how sequences are packed or ordered in the batch.
 *   q, k, v, g, beta, cu_seqlens, n_seqs, total_tokens, H, dk, dv, C, dtype: as given to
 *               the forward (cpr_gdn_prefill) whose gradients are wanted
 *   boundary_states fp32 [boundary_capacity, H, dk, dv]: the forward's boundary states
 *               (the state at the start of every chunk, as cpr_gdn_prefill wrote them)
 *   d_out       dtype [total_tokens, H, dv]   dL/do
 *   d_state_out fp32 [n_seqs, H, dk, dv]      dL/d(state_out), or NULL for zero
 * Outputs (fp32, written, not accumulated):
 *   dq, dk_out  [total_tokens, H, dk];  dv_out [total_tokens, H, dv];
 *   dg, dbeta   [total_tokens, H]  (dg is dL/dg with g = log alpha)
 *   d_state_in  [n_seqs, H, dk, dv]  dL/d(state_in), or NULL if not wanted
 *   workspace   >= cpr_gdn_backward_workspace_size(...) bytes, 16-byte aligned; holds the
 *               status word (cpr_gdn_device_status)
 * Shapes: those cpr_gdn_backward_supported() accepts (every built (dk, dv, C) in bf16; fp32
 * where the chunk kernels fit one CTA's shared memory).  Returns CPR_OK or a negative
 * code as for cpr_gdn_prefill; device-side checks of cu_seqlens and boundary_capacity
 * record CPR_DEV_* bits and skip the work.
 */
size_t cpr_gdn_backward_workspace_size(int64_t total_tokens, int32_t n_seqs, int32_t H, int32_t dk, int32_t dv,
                                       int32_t C);
int cpr_gdn_backward_supported(int32_t dk, int32_t dv, int32_t C, int32_t dtype);
int32_t cpr_gdn_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                         int32_t dv, int32_t C, int32_t dtype, const float* boundary_states,
                         int64_t boundary_capacity, const void* d_out, const float* d_state_out, float* dq,
                         float* dk_out, float* dv_out, float* dg, float* dbeta, float* d_state_in, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Fill a decode ring from a prefill's results so that decode continues each sequence
 * at position L_n (CPR step 3 starts where prefill stopped).  Arguments as in
 * cpr_gdn_prefill; ring buffers are sized for B = n_seqs.  For each (n, h): ring S_b =
 * the boundary state of the sequence's last chunk if L_n % C != 0, else state_out
 * (state_in if L_n = 0); ring slots 0 .. (L_n % C) - 1 receive that chunk's tokens.
 * boundary_states and state_out are those the prefill wrote; cu_seqlens is DEVICE.
 * k, v, g, beta and boundary_states may be NULL when total_tokens is 0.  A sequence
 * whose cu_seqlens entries are decreasing or reach past total_tokens is skipped.
 */
int32_t cpr_gdn_ring_from_prefill(const void* k, const void* v, const float* g, const float* beta,
                                  const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                                  int32_t dv, int32_t C, int32_t dtype, const float* boundary_states,
                                  const float* state_out, const cpr_gdn_ring* ring, void* stream);

/*
 * One CPR decode step for B sequences (CPR step 3): every sequence b receives one
 * token at absolute position pos[b] (>= 0; the caller owns and advances pos).
 *   q, k   dtype [B, H, dk];  v dtype [B, H, dv];  g, beta fp32 [B, H]
 *   state  fp32 [B, H, dk, dv]  in/out: the sequence's recurrent state
 *   ring   in/out (see cpr_gdn_ring); the token goes to slot pos[b] % C
 *   pos    int32 [B] DEVICE
 *   out    dtype [B, H, dv]
 * The token is stepped by the same recurrence as prefill; when pos[b] % C == C - 1
 * the state (and ring S_b) become U(ring S_b, ring chunk).  A negative pos[b] skips
 * sequence b and records CPR_DEV_BAD_POS.  workspace >= cpr_gdn_decode_workspace_size.
 * The resync (and the step of those sequences' tokens) runs on a second stream owned by
 * the library (one per device, created on the first call) that forks from `stream` and
 * joins it again at the end of the call: work issued on `stream` after the call sees
 * every result.  Calls on one device share that stream; calls from several host threads
 * take turns on it (a lock held while each call enqueues its work).
 */
int32_t cpr_gdn_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       float* state, const cpr_gdn_ring* ring, const int32_t* pos, int32_t B, int32_t H,
                       int32_t dk, int32_t dv, int32_t C, int32_t dtype, void* out, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Continuation prefill (a rollout's chunked prefill): every sequence n continues from
 * absolute position pos0[n] with the state and ring that decode (or an earlier prefill
 * with cpr_gdn_ring_from_prefill) left, and receives the L_n = cu_seqlens[n + 1] -
 * cu_seqlens[n] tokens at positions pos0[n] .. pos0[n] + L_n - 1.  The results are those
 * of decode run token by token over the same tokens, bit for bit (and so those of one
 * prefill over each whole sequence):
 *   - the first tokens, up to the end of the chunk that pos0[n] lies in (none when pos0[n]
 *     is a multiple of C), are stepped from `state` by decode's token step and go to the
 *     ring; a chunk they complete is resynchronised as in decode;
 *   - the remaining tokens, which start at a chunk boundary, run as in cpr_gdn_prefill from
 *     the resulting state; boundary_states receives the start states of their chunks,
 *     indexed as cpr_gdn_prefill indexes chunks of those remainders (its capacity counts
 *     their chunks, cpr_gdn_num_chunks of the remaining lengths);
 *   - `state` and the ring end as decode leaves them at position pos0[n] + L_n.
 *   q, k, v, g, beta, cu_seqlens (DEVICE), out: as in cpr_gdn_prefill
 *   pos0   int32 [n_seqs] DEVICE, >= 0
 *   state  fp32 [n_seqs, H, dk, dv] in/out;  ring in/out (B = n_seqs)
 * workspace >= cpr_gdn_prefill_workspace_size(total_tokens, n_seqs, H, dk, dv, C).  A
 * negative pos0[n] records CPR_DEV_BAD_POS in the workspace's status word and the call
 * then leaves every output as it was.  The first tokens' steps and resync run on the
 * library's side stream (the one decode uses) while the remainder's chunk preparation
 * runs on `stream`; the call joins them again, so work issued on `stream` after it sees
 * every result.  Calls on one device take turns on that side stream.
 */
int32_t cpr_gdn_prefill_continue(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                 int32_t dk, int32_t dv, int32_t C, int32_t dtype, const int32_t* pos0, float* state,
                                 const cpr_gdn_ring* ring, void* out, float* boundary_states,
                                 int64_t boundary_capacity, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Grouped value heads and options: the four calls above with H value heads over Hk
 * query/key heads (Hk divides H; value head h reads query/key head h / (H / Hk)).  q and k
 * are then [.., Hk, dk]; v, g, beta, out, states and the ring keep H heads (the ring holds
 * each value head's copy of its keys, as given).  `flags` (prefill, decode, continuation):
 *   CPR_QK_L2NORM  the kernels L2-normalise every key and query row before use:
 *                  k / sqrt(sum k^2 + 1e-6) and q / sqrt(sum q^2 + 1e-6) * dk^-1/2, the sum
 *                  of squares in the canonical dot order, the square root and reciprocal
 *                  correctly rounded, so every path normalises to the same bits.  A decode
 *                  or continuation must use the flag its prefill used.
 * Every other argument, and the results per value head, are those of the call without the
 * suffix, which is the case Hk = H, flags = 0.
 */
#define CPR_QK_L2NORM 1u
int32_t cpr_gdn_prefill_grouped(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                int32_t Hk, uint32_t flags, int32_t dk, int32_t dv, int32_t C, int32_t dtype,
                                const float* state_in, void* out, float* state_out, float* boundary_states,
                                int64_t boundary_capacity, void* workspace, size_t workspace_bytes, void* stream);
int32_t cpr_gdn_ring_from_prefill_grouped(const void* k, const void* v, const float* g, const float* beta,
                                          const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                          int32_t Hk, int32_t dk, int32_t dv, int32_t C, int32_t dtype,
                                          const float* boundary_states, const float* state_out,
                                          const cpr_gdn_ring* ring, void* stream);
int32_t cpr_gdn_decode_grouped(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               float* state, const cpr_gdn_ring* ring, const int32_t* pos, int32_t B, int32_t H,
                               int32_t Hk, uint32_t flags, int32_t dk, int32_t dv, int32_t C, int32_t dtype,
                               void* out, void* workspace, size_t workspace_bytes, void* stream);
int32_t cpr_gdn_prefill_continue_grouped(const void* q, const void* k, const void* v, const float* g,
                                         const float* beta, const int32_t* cu_seqlens, int32_t n_seqs,
                                         int64_t total_tokens, int32_t H, int32_t Hk, uint32_t flags, int32_t dk,
                                         int32_t dv, int32_t C, int32_t dtype, const int32_t* pos0, float* state,
                                         const cpr_gdn_ring* ring, void* out, float* boundary_states,
                                         int64_t boundary_capacity, void* workspace, size_t workspace_bytes,
                                         void* stream);

/*
 * Prefill for callers that cannot allocate device memory.  (The pages have no
 * counterpart of this entry point; it belongs to this library's interface only.)
 *
 * Serving runtimes that reserve all device memory for their own pool, loops that must
 * not hit the device synchronisation an allocation can cause, and C hosts without a
 * device allocator cannot provide cpr_gdn_prefill's workspace.  This entry point takes
 * the same arguments minus the workspace and uses a scratch array of
 * CPR_GDN_NOALLOC_SCRATCH_BYTES owned by the library (a static device array: every GPU
 * that loads the library's device code holds it until the process exits).  It calls no
 * allocating routine.  The caller still provides every input and output buffer.
 *   - Problems whose cpr_gdn_prefill_workspace_size() exceeds
 *     CPR_GDN_NOALLOC_SCRATCH_BYTES are rejected with CPR_ERR_WORKSPACE before any work
 *     is enqueued (for dk = dv = 128, C = 64 that is about 120 chunk-heads, e.g. 16 heads
 *     x 7 chunks).
 *   - The first call on each device looks up the scratch's device address with that
 *     device current (this may load the library's device code): make it before any
 *     stream capture begins.  The address is remembered per device for the life of the
 *     process; cudaDeviceReset invalidates it, so do not call this entry point on a
 *     device after resetting it.
 *   - All calls share the scratch, which keeps the last call's contents (nothing in it
 *     needs to start at zero).  Calls that overlap on the GPU race on it: serialise them.
 *   - The device status word of the last call lives in that scratch; read it with
 *     cpr_gdn_prefill_noalloc_status.
 * Results are bit for bit those cpr_gdn_prefill returns for the same arguments.
 */
#define CPR_GDN_NOALLOC_SCRATCH_BYTES (16u << 20)
int32_t cpr_gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                const int32_t* cu_seqlens, int32_t n_seqs, int64_t total_tokens, int32_t H,
                                int32_t dk, int32_t dv, int32_t C, int32_t dtype, const float* state_in, void* out,
                                float* state_out, float* boundary_states, int64_t boundary_capacity, void* stream);

/*
 * Device status word of the last cpr_gdn_prefill_noalloc call on the current device (an
 * OR of CPR_DEV_* bits, 0 when every device-side check passed, e.g. CPR_DEV_TIMEOUT when
 * a bounded wait gave up and some outputs were not written).  Waits for `stream`, copies
 * the word from the library's scratch into *status_out and allocates nothing; the same
 * first-call and reset rules as cpr_gdn_prefill_noalloc apply.  Returns CPR_OK,
 * CPR_ERR_INVALID_ARG (status_out NULL) or CPR_ERR_CUDA.
 */
int32_t cpr_gdn_prefill_noalloc_status(uint32_t* status_out, void* stream);

/*
 * Profiling hook (used by the benchmark to time each kernel with CUDA events on the
 * stream it runs on).  events: n_events cudaEvent_t handles created by the caller, or
 * NULL to switch the hook off.  While it is on, every cpr_gdn_prefill records
 * events[0] before its first kernel and events[i] after its i-th kernel (i = 1..3:
 * chunk index, chunk prep, boundary chain with the intra-chunk recurrence; needs
 * n_events >= 4), every cpr_gdn_decode records events[0] before and events[1],
 * events[2] after its step and resync kernels, and every cpr_gdn_backward records
 * events[0] before its first kernel and events[1..4] after the chunk index, the chunk
 * maps, the reverse chain and the chunk gradients (needs n_events >= 5; where the last two
 * share one launch, events[3] is recorded before it).  Process-wide; not for concurrent
 * calls from several threads.
 */
int32_t cpr_gdn_set_profile_events(void* const* events, int32_t n_events);

/*
 * Test hook for the failure path of the device-side waits on other CTAs: the prefill's
 * (an intra-chunk item waiting for its boundary state to be published by the chain) and
 * the backward's where its chain and chunk gradients share one launch (dk = dv = 128,
 * C = 64, bf16: a chunk's gradients waiting for its state adjoint).  While
 * extra_publications > 0, every such item waits for that many publications more than the
 * chain ever makes, so each wait runs out after limit_ns nanoseconds (0: the default of
 * about 4 s), the item is skipped (its outputs are not written) and the call records
 * CPR_DEV_TIMEOUT in its status word; the context stays usable.
 * cpr_gdn_set_wait_test(0, 0) restores normal operation.  Process-wide, read when a
 * prefill or backward is enqueued; not for concurrent use with other calls.  Returns
 * CPR_OK.
 */
int32_t cpr_gdn_set_wait_test(uint32_t extra_publications, uint64_t limit_ns);

/*
 * Read the device status word of the last call that used `workspace` (waits for
 * `stream`).  *status_out receives an OR of CPR_DEV_* bits, 0 when all device-side
 * checks passed.  Returns CPR_OK or CPR_ERR_CUDA.
 */
int32_t cpr_gdn_device_status(const void* workspace, uint32_t* status_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CPR_GDN_H */
