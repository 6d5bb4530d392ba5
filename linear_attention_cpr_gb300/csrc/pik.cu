// pik.cu — the deterministic K-split GEMM ("pik") on the 5th-generation tensor cores, and
// its C ABI (include/cpr_pik.h).
//
// "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section on the fixed binary
// reduction tree (tensor parallelism, the pik implementation): K is cut into contiguous
// leaves, each leaf is a tensor-core product with fp32 accumulation in a fixed order, and
// one binary tree over the leaves fixes how their partial sums meet, so the result does
// not depend on how the leaves are shared among ranks.
//
// k_pik_leaves: one CTA per 128 x 128 output tile.  A tile's operands are 128 rows of X
// and 128 rows of W per 64 K elements, each row 128 bytes in the tensor cores'
// 128-byte-swizzled K-major layout; each CTA loads its own X and W boxes (one TMA box of
// 128 rows each, into its own shared memory, completing on its own barrier).  Tiles are
// rastered in groups of kGroup tile rows, so the CTAs resident at one time share their
// operand rows in L2.  Warp 0 issues the loads into six stages, warp 1 issues the MMAs (4
// per stage, K = 16 each) and commits each stage to its stage-free barrier; warps 4-7
// merge partials and run the epilogue.  Up to four leaves: each leaf of the CTA's range
// accumulates in its own TMEM slot of 128 columns, the loop never waits for a reduction,
// and the epilogue sums the slots with the tree in registers.  Eight leaves: slot
// popcount(j) takes leaf j; when an odd leaf completes, warps 4-7 merge the finished pairs
// of the tree in TMEM (a binary counter: at most four live partials) before the next leaf
// starts, leaving the root in slot 0.  A leaf's instruction sequence, and so every bit of
// its partial, is the same whichever leaf range a call covers.
// k_pik_combine: the top of the same tree over the ranks' subtree roots (HBM-bound).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/cpr_pik.h"
#include "common.cuh"
#include "tc.cuh"

namespace cpr {
namespace {

constexpr int kBM = 128;       // tile rows (M of the MMA instruction; row i in TMEM lane i)
constexpr int kBN = 128;       // tile columns (N of the MMA instruction)
constexpr int kBK = 64;        // K elements per stage: one 128-byte swizzled row per operand row
constexpr int kStages = 6;     // shared-memory stages
constexpr int kThreads = 256;  // warp 0: loads, warp 1: MMAs, warps 4-7: merges and epilogue
constexpr int kGroup = 8;      // tile rows per raster group (concurrent tiles share operands in L2)
constexpr int kSlots = 512 / kBN;  // partial sums that fit in TMEM
constexpr uint32_t kOpBytes = 128 * 128;             // 128 rows of 128 bytes: one TMA box (16 KB)
constexpr uint32_t kStage = 2 * kOpBytes;            // X then W
constexpr size_t kBarOff = (size_t)kStages * kStage;
constexpr size_t kSmem = kBarOff + 256 + 1024;       // barriers, TMEM slot, alignment slack

struct PikArgs {
    float* y;
    int32_t M, N, K, n_leaves, leaf_lo, leaf_hi;
    int vec_store;  // y rows start 16-byte aligned: store 4 values at a time
    uint32_t* status;
};

// One 64-element x 128-row box of a [rows, K] bf16 tensor map at (k, row0), into this
// CTA's shared memory, completing its bytes on this CTA's mbar.
__device__ __forceinline__ void tma_box(void* dst, const CUtensorMap* map, int32_t k, int32_t row0, uint64_t* mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(k), "r"(row0), "r"(tc::smem_u32(mbar))
        : "memory");
}

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle: rows of 128 bytes,
// 8-row groups 1024 bytes apart (SBO), the tile 1024-byte aligned; the start address
// advances 32 bytes per 16 K elements inside the swizzled row.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;              // LBO: unused by a swizzled K-major operand
    d |= (uint64_t)(1024 >> 4) << 32;    // SBO
    d |= (uint64_t)1 << 46;              // descriptor version of the 5th-generation tensor cores
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// The fixed tree over n (a power of two) adjacent values: pairs of neighbours first.
template <int MAXL, int E>
__device__ __forceinline__ void leaf_tree(float (&v)[MAXL][E], int n)
{
#pragma unroll
    for (int wdt = 1; wdt < MAXL; wdt <<= 1)
#pragma unroll
        for (int l = 0; l + wdt < MAXL; l += 2 * wdt)
            if (wdt < n && l + wdt < n)
#pragma unroll
                for (int e = 0; e < E; ++e) v[l][e] = __fadd_rn(v[l][e], v[l + wdt][e]);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_pik_leaves(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw, const PikArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);  // [kStages] stage landed
    uint64_t* empty = full + kStages;                              // [kStages] stage read by the MMAs
    uint64_t* leaf_done = empty + kStages;                         // an odd leaf's products are done
    uint64_t* merged = leaf_done + 1;                              // its pairs are merged
    uint64_t* acc_done = merged + 1;                               // every product is done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_done + 1);
    const int tid = threadIdx.x, warp = tid >> 5;

    // grouped raster over tiles: kGroup tile rows walk the tile columns together
    const int tiles_m = (a.M + kBM - 1) / kBM, tiles_n = (a.N + kBN - 1) / kBN;
    const int c = blockIdx.x, per_group = kGroup * tiles_n;
    const int g0 = (c / per_group) * kGroup, gsz = min(kGroup, tiles_m - g0), r = c % per_group;
    const int mt = g0 + r % gsz, nt = r / gsz;
    const int32_t m0 = mt * kBM, n0 = nt * kBN;  // rows past M or N load zeros and are not stored

    const int nl = a.leaf_hi - a.leaf_lo;
    const bool merge = nl > kSlots;
    const int used = merge ? kSlots : nl;
    const uint32_t cols = used <= 1 ? 128u : used <= 2 ? 256u : 512u;
    if (warp == 0) tc::tmem_alloc(tslot, cols);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(leaf_done, 1);
        tc::mbar_init(merged, 128);
        tc::mbar_init(acc_done, 1);
        tc::fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    const int64_t KL = (int64_t)a.K / a.n_leaves;
    const int spl = (int)(KL / kBK), S = nl * spl;  // stages per leaf, in all
    const int32_t kbase = (int32_t)((int64_t)a.leaf_lo * KL);
    bool ok = true;

    if (tid == 0) {
        // producer: the tile's 128 X rows and 128 W rows of each 64-element K step
        for (int s = 0; s < S && ok; ++s) {
            const int b = s % kStages;
            if (s >= kStages) ok = tc::mbar_wait(&empty[b], (uint32_t)((s / kStages - 1) & 1));
            if (!ok) break;
            unsigned char* st = smem + (size_t)b * kStage;
            tc::mbar_arrive_expect_tx(&full[b], kStage);
            const int32_t k0 = kbase + s * kBK;
            tma_box(st, &tx, k0, m0, &full[b]);
            tma_box(st + kOpBytes, &tw, k0, n0, &full[b]);
        }
        // every arrival meant for this CTA's stage barriers has landed before it can exit
        for (int b = 0; b < kStages && b < S; ++b) {
            const int uses = (S - b + kStages - 1) / kStages;
            ok = tc::mbar_wait(&empty[b], (uint32_t)((uses - 1) & 1)) && ok;
        }
    } else if (tid == 32) {
        // MMA issuer
        constexpr uint32_t idesc = tc::idesc_bf16(kBM, kBN);
        int events = 0;
        for (int s = 0; s < S && ok; ++s) {
            const int b = s % kStages;
            ok = tc::mbar_wait(&full[b], (uint32_t)((s / kStages) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            const int j = s / spl;
            const uint32_t d = tmem + (uint32_t)((merge ? __popc(j) : j) * kBN);
            const uint32_t sx = tc::smem_u32(smem + (size_t)b * kStage), sw = sx + kOpBytes;
            const bool first = (s % spl) == 0;  // a leaf's first instruction overwrites its slot
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                tc::mma_bf16(d, sdesc_sw128(sx + k * 32), sdesc_sw128(sw + k * 32), idesc, (first && k == 0) ? 0u : 1u);
            tc::commit(&empty[b]);
            if (merge && s % spl == spl - 1 && (j & 1)) {
                tc::commit(leaf_done);
                ok = tc::mbar_wait(merged, (uint32_t)(events & 1));
                ++events;
                tc::fence_after_sync();
            }
        }
        tc::commit(acc_done);
    } else if (warp >= 4) {
        const int q = warp & 3;
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        if (merge) {
            for (int j = 1, e = 0; j < nl; j += 2, ++e) {
                ok = tc::mbar_wait(leaf_done, (uint32_t)(e & 1)) && ok;
                tc::fence_after_sync();
                for (int top = __popc(j), m = __ffs(j + 1) - 1; m > 0; --m, --top) {
#pragma unroll 1
                    for (int cb = 0; cb < kBN / 32; ++cb) {
                        float l[32], rr[32];
                        uint32_t o[32];
                        const uint32_t dst = tmem + lanes + (uint32_t)((top - 1) * kBN + cb * 32);
                        tc::tmem_ld_32x32b<32>(dst, l);
                        tc::tmem_ld_32x32b<32>(tmem + lanes + (uint32_t)(top * kBN + cb * 32), rr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__fadd_rn(l[i], rr[i]));
                        tc::tmem_st_32x32b<32>(dst, o);
                    }
                    tc::tmem_wait_st();
                }
                tc::fence_before_sync();
                tc::mbar_arrive(merged);
            }
        }
        ok = tc::mbar_wait(acc_done, 0u) && ok;
        tc::fence_after_sync();
    }
    const bool failed = __syncthreads_or(!ok) != 0;

    if (!failed && warp >= 4) {
        constexpr int E = 8;
        const int parts = merge ? 1 : nl;  // partials left in slots 0 .. parts-1
        const int row = (warp & 3) * 32 + (tid & 31);
        const int64_t gm = (int64_t)m0 + row;
        const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll 1
        for (int cb = 0; cb < kBN / E; ++cb) {
            float v[kSlots][E];
#pragma unroll
            for (int l = 0; l < kSlots; ++l)
                if (l < parts) tc::tmem_ld_32x32b<E>(tmem + lanes + (uint32_t)(l * kBN + cb * E), v[l]);
            leaf_tree<kSlots, E>(v, parts);
            const int64_t c0 = (int64_t)n0 + cb * E;
            if (gm < a.M) {
                float* dst = a.y + gm * a.N + c0;
                if (a.vec_store && c0 + E <= a.N) {
                    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
                    reinterpret_cast<float4*>(dst)[1] = make_float4(v[0][4], v[0][5], v[0][6], v[0][7]);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        if (c0 + e < a.N) dst[e] = v[0][e];
                }
            }
        }
    }
    if (failed && tid == 0) atomicOr(a.status, CPR_DEV_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, cols);
}

// y[i] = tree over the P parts (pairs of neighbours first).  vec: count % 4 == 0 and the
// buffers 16-byte aligned, four elements per thread and iteration.
template <int P>
__global__ void __launch_bounds__(256) k_pik_combine(const float* parts, int64_t count, float* y, int vec)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x, t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (vec) {
        const int64_t n4 = count / 4;
        for (int64_t i = t0; i < n4; i += stride) {
            float v[P][4];
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const float4 q = reinterpret_cast<const float4*>(parts + p * count)[i];
                v[p][0] = q.x, v[p][1] = q.y, v[p][2] = q.z, v[p][3] = q.w;
            }
            leaf_tree<P, 4>(v, P);
            reinterpret_cast<float4*>(y)[i] = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
        }
    } else {
        for (int64_t i = t0; i < count; i += stride) {
            float v[P][1];
#pragma unroll
            for (int p = 0; p < P; ++p) v[p][0] = parts[p * count + i];
            leaf_tree<P, 1>(v, P);
            y[i] = v[0][0];
        }
    }
}

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

// True when p is device memory of the current device (not host, managed or a peer GPU's
// memory): the tensor maps are only ever built over this GPU's own buffers.
bool on_this_device(const void* p)
{
    int dev = -1;
    cudaPointerAttributes at{};
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error an unknown pointer leaves
        return false;
    }
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}
bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Tensor map of a [rows, K] bf16 matrix whose box is 64 K elements x 128 rows, landing as
// 128 rows of 128 bytes in the 128-byte swizzle the MMA descriptors read.  Rows past the
// end read zeros.
bool box_map(CUtensorMap* m, const void* base, int32_t rows, int32_t K)
{
    const EncodeTiledFn f = tensor_map_encoder();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, 128}, es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace cpr

using namespace cpr;

extern "C" size_t cpr_pik_workspace_size(void) { return kAlign; }

extern "C" int32_t cpr_pik_gemm(const void* x, const void* w, float* y, int32_t M, int32_t N, int32_t K,
                                int32_t n_leaves, int32_t leaf_lo, int32_t leaf_hi, void* workspace, void* stream)
{
    if (!x || !w || !y || M < 1 || N < 1 || K < 1) return CPR_ERR_INVALID_ARG;
    if (!(n_leaves == 1 || n_leaves == 2 || n_leaves == 4 || n_leaves == 8)) return CPR_ERR_INVALID_ARG;
    if (K % (kBK * n_leaves) != 0) return CPR_ERR_INVALID_ARG;
    const int nl = leaf_hi - leaf_lo;
    if (leaf_lo < 0 || leaf_hi > n_leaves || !pow2(nl) || leaf_lo % nl != 0) return CPR_ERR_INVALID_ARG;
    if ((int64_t)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN) > 0x7fffffff / 2) return CPR_ERR_INVALID_ARG;
    if (!workspace) return CPR_ERR_WORKSPACE;
    if (!al16(x) || !al16(w) || !al16(workspace) || ((uintptr_t)y & 3u)) return CPR_ERR_MISALIGNED;
    if (!on_this_device(x) || !on_this_device(w)) return CPR_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PikArgs a{y, M, N, K, n_leaves, leaf_lo, leaf_hi, (al16(y) && N % 4 == 0) ? 1 : 0,
              static_cast<uint32_t*>(workspace)};
    CUtensorMap mx, mw;
    if (!box_map(&mx, x, M, K) || !box_map(&mw, w, N, K)) return CPR_ERR_CUDA;
    if (cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s) != cudaSuccess) return CPR_ERR_CUDA;
    if (cudaFuncSetAttribute(k_pik_leaves, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
        return CPR_ERR_CUDA;
    const int64_t tiles = (int64_t)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    k_pik_leaves<<<(unsigned)tiles, kThreads, kSmem, s>>>(mx, mw, a);
    return cudaGetLastError() == cudaSuccess ? CPR_OK : CPR_ERR_CUDA;
}

extern "C" int32_t cpr_pik_combine(const float* parts, int32_t n_parts, int64_t count, float* y, void* stream)
{
    if (!parts || !y || count < 0) return CPR_ERR_INVALID_ARG;
    if (!(n_parts == 1 || n_parts == 2 || n_parts == 4 || n_parts == 8)) return CPR_ERR_INVALID_ARG;
    if (!al16(parts) || !al16(y)) return CPR_ERR_MISALIGNED;
    if (count == 0) return CPR_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return CPR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int vec = count % 4 == 0;
    const int64_t work = vec ? count / 4 : count;
    const int64_t want = (work + 255) / 256;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 8));
    switch (n_parts) {
        case 1: k_pik_combine<1><<<grid, 256, 0, s>>>(parts, count, y, vec); break;
        case 2: k_pik_combine<2><<<grid, 256, 0, s>>>(parts, count, y, vec); break;
        case 4: k_pik_combine<4><<<grid, 256, 0, s>>>(parts, count, y, vec); break;
        default: k_pik_combine<8><<<grid, 256, 0, s>>>(parts, count, y, vec); break;
    }
    return cudaGetLastError() == cudaSuccess ? CPR_OK : CPR_ERR_CUDA;
}
