/*
 * cpr_pik.h — C ABI of the deterministic K-split GEMM ("pik") for one GB300 GPU (sm_103a).
 *
 * The operation: "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section on
 * the fixed binary reduction tree (tensor parallelism, the pik implementation), and
 * "SkyRL IsoExec: vLLM 与 Megatron 的 logprob 差 ...", section on the unified model.  A
 * product Y = X W^T is reduced over K in a way that does not depend on how K is shared
 * among tensor-parallel ranks:
 *   - K is cut into n_leaves contiguous leaves of K / n_leaves elements (a fixed constant
 *     of the contract, a power of two up to 8);
 *   - each leaf's partial product is computed by tensor-core MMAs with fp32 accumulation
 *     in one fixed instruction order (K ascending, 16 elements per instruction, the
 *     first instruction of a leaf overwriting the accumulator);
 *   - the leaf partials are summed by one fixed binary tree: adjacent pairs first,
 *     ((P0 + P1) + (P2 + P3)) + ((P4 + P5) + (P6 + P7)), each addition an fp32 add
 *     rounded to nearest;
 *   - a rank owns a contiguous, aligned block of leaves (a complete subtree) and computes
 *     that subtree's root; cpr_pik_combine then finishes the same tree over the ranks'
 *     roots.  The result is therefore bit-identical for every rank count that divides
 *     n_leaves, including one rank computing everything in a single cpr_pik_gemm call.
 * Every call runs on one GPU, the current device, over that GPU's own memory.  The
 * library moves no partial sums between GPUs: a caller with several GPUs computes each
 * rank's subtree root on that rank's GPU, gathers the roots into one buffer with its own
 * transport, and then calls cpr_pik_combine there; on one GPU the roots are consecutive
 * buffers.
 *
 * Conventions (as in cpr_gdn.h): device pointers on the current device, row-major and
 * contiguous; the caller owns every buffer; all work is enqueued on `stream`; the
 * library allocates no memory.  A negative return value means nothing was enqueued
 * (argument checks) or a launch failed.  Error codes are those of cpr_gdn.h.
 */
#ifndef CPR_PIK_H
#define CPR_PIK_H

#include <stddef.h>
#include <stdint.h>

#include "cpr_gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of the device workspace of cpr_pik_gemm: one status word, read back with
 * cpr_gdn_device_status() (CPR_DEV_TIMEOUT if a tensor-core wait gave up; the tile of
 * that CTA is then not written). */
size_t cpr_pik_workspace_size(void);

/* Subtree root of leaves [leaf_lo, leaf_hi) of Y = X W^T.
 *   x          bf16 [M, K] (K contiguous), 16-byte aligned, device memory of the current device
 *   w          bf16 [N, K] (K contiguous: the layout of a linear layer's weight), 16-byte
 *              aligned, device memory of the current device (host, managed or another GPU's
 *              memory is rejected with CPR_ERR_INVALID_ARG: the operands are read through
 *              tensor maps that must describe this GPU's own buffers)
 *   y          fp32 [M, N], written (not accumulated); 4-byte aligned
 *   M, N       >= 1, any value (ragged tiles are masked)
 *   K          a multiple of 64 * n_leaves
 *   n_leaves   1, 2, 4 or 8: the contract's leaf count
 *   leaf_lo, leaf_hi   0 <= leaf_lo < leaf_hi <= n_leaves, leaf_hi - leaf_lo a power of two
 *              that divides leaf_lo (a complete subtree); (0, n_leaves) is the whole product
 *   workspace  cpr_pik_workspace_size() bytes, 16-byte aligned; its status word is reset
 * Host work per call: two TMA descriptors of x and w are encoded (the driver's tensor-map
 * encoder, found through the CUDA runtime; CPR_ERR_CUDA if it is unavailable).
 * Returns CPR_OK, CPR_ERR_INVALID_ARG, CPR_ERR_MISALIGNED, CPR_ERR_WORKSPACE or
 * CPR_ERR_CUDA.  Does not synchronise. */
int32_t cpr_pik_gemm(const void* x, const void* w, float* y, int32_t M, int32_t N, int32_t K, int32_t n_leaves,
                     int32_t leaf_lo, int32_t leaf_hi, void* workspace, void* stream);

/* The top of the tree over n_parts subtree roots: y[i] = tree over p of parts[p * count + i]
 * (pairs of adjacent parts first, fp32 adds rounded to nearest).
 *   parts      fp32 [n_parts, count], 16-byte aligned
 *   n_parts    1, 2, 4 or 8 (roots of equal, adjacent subtrees in leaf order)
 *   count      >= 0 elements per part (M * N)
 *   y          fp32 [count], 16-byte aligned; may equal parts (in place on the first part)
 * Returns CPR_OK, CPR_ERR_INVALID_ARG, CPR_ERR_MISALIGNED or CPR_ERR_CUDA. */
int32_t cpr_pik_combine(const float* parts, int32_t n_parts, int64_t count, float* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CPR_PIK_H */
