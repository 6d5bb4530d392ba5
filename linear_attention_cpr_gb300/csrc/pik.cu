// pik.cu — the deterministic K-split GEMM ("pik") on the 5th-generation tensor cores, and
// its C ABI (include/cpr_pik.h).
//
// "IsoExec: Eliminating Trainer-Inference Mismatch in SkyRL", section on the fixed binary
// reduction tree (tensor parallelism, the pik implementation): K is cut into contiguous
// leaves, each leaf is a tensor-core product with fp32 accumulation in a fixed order, and
// one binary tree over the leaves fixes how their partial sums meet, so the result does
// not depend on how the leaves are shared among ranks.
//
// k_pik_leaves: one CTA per 128 x 128 output tile.  Up to four leaves: each leaf of the
// CTA's range accumulates in its own TMEM slot of 128 columns, the main loop never waits
// for a reduction, and the epilogue sums the slots with the tree in registers.  Eight
// leaves: slot popcount(j) takes leaf j, and as each odd leaf completes the loop waits for
// its products and merges the finished pairs of the tree in TMEM (a binary counter: at
// most four live partials), leaving the root in slot 0.  Operands are staged by every thread
// with 16-byte cp.async into the no-swizzle K-major core-matrix layout (tc.cuh), six
// stages of 64 K elements, and one thread issues the MMAs (4 per stage, K = 16 each) and
// commits each stage to an mbarrier that frees it.  The leaf's instruction sequence, and
// so every bit of its partial, is the same whichever tile shape or leaf range a call uses.
// k_pik_combine: the top of the same tree over the ranks' subtree roots (HBM-bound).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/cpr_pik.h"
#include "common.cuh"
#include "tc.cuh"

namespace cpr {
namespace {

constexpr int kBM = 128;      // tile rows (M of the MMA instruction; row i in TMEM lane i)
constexpr int kBK = 64;       // K elements per stage
constexpr int kStages = 6;    // shared-memory stages
constexpr int kLag = 2;       // products kept queued before a stage is refilled
constexpr int kThreads = 128; // 4 warps: loads, epilogue (warp w reads lane quadrant w); thread 0 issues
constexpr int kGroupM = 8;    // m-tiles per raster group (the concurrently running tiles share operands in L2)

template <int BN>
struct PikCfg {
    static constexpr int SLOTS = 512 / BN;  // partial sums that fit in TMEM
    static constexpr uint32_t A_BYTES = kBM * kBK * 2, B_BYTES = BN * kBK * 2, STAGE = A_BYTES + B_BYTES;
    static constexpr uint32_t SBO = (kBK / 8) * 128;  // step between 8-row core groups
    static constexpr size_t BAR_OFF = (size_t)kStages * STAGE;
    static constexpr size_t SMEM = BAR_OFF + 128;
};

struct PikArgs {
    const __nv_bfloat16* x;
    const __nv_bfloat16* w;
    float* y;
    int32_t M, N, K, n_leaves, leaf_lo, leaf_hi;
    int vec_store;  // y rows start 16-byte aligned: store 4 values at a time
    uint32_t* status;
};

__device__ __forceinline__ void cp_async16_zfill(void* smem, const void* gmem, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(tc::smem_u32(smem)), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Rows [row0, row0 + ROWS) x K elements [k0, k0 + 64) of a [rows, K] bf16 matrix into a
// core-matrix tile: 16-byte piece c (8 K elements) is row 8 (c / 64) + c % 8, K piece
// (c / 8) % 8, and lands at byte 16 c of the tile.  Rows at or beyond `rows` read zeros.
template <int ROWS>
__device__ __forceinline__ void load_tile(unsigned char* dst, const __nv_bfloat16* src, int64_t row0, int rows,
                                          int64_t K, int64_t k0, int tid)
{
#pragma unroll
    for (int i = 0; i < ROWS * 8 / kThreads; ++i) {
        const int c = tid + i * kThreads;
        const int r = ((c >> 6) << 3) | (c & 7), kc = (c >> 3) & 7;
        const int64_t gr = row0 + r;
        const bool in = gr < rows;
        cp_async16_zfill(dst + c * 16, src + (in ? gr : 0) * K + k0 + kc * 8, in ? 16u : 0u);
    }
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

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) k_pik_leaves(const PikArgs a)
{
    using Cf = PikCfg<BN>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* mma_done = reinterpret_cast<uint64_t*>(smem + Cf::BAR_OFF);  // [kStages] stage read by its products
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_done + kStages);
    const int tid = threadIdx.x, warp = tid >> 5;

    // grouped raster: kGroupM m-tiles side by side walk the n-tiles together
    const int tiles_m = (a.M + kBM - 1) / kBM, tiles_n = (a.N + BN - 1) / BN;
    const int per_group = kGroupM * tiles_n, b = blockIdx.x;
    const int g0 = (b / per_group) * kGroupM, gsz = min(kGroupM, tiles_m - g0), r = b % per_group;
    const int64_t m0 = (int64_t)(g0 + r % gsz) * kBM, n0 = (int64_t)(r / gsz) * BN;

    const int nl = a.leaf_hi - a.leaf_lo;
    const bool merge = nl > Cf::SLOTS;  // more leaves than slots: merge pairs as they complete
    const int used = merge ? Cf::SLOTS : nl;
    const uint32_t cols = used * BN <= 32 ? 32u : used * BN <= 64 ? 64u : used * BN <= 128 ? 128u : used * BN <= 256 ? 256u : 512u;
    if (warp == 0) tc::tmem_alloc(tslot, cols);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) tc::mbar_init(&mma_done[s], 1);
        tc::fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    const int64_t K = a.K, KL = K / a.n_leaves, kbase = (int64_t)a.leaf_lo * KL;
    const int spl = (int)(KL / kBK), S = nl * spl;  // stages per leaf, in all
    auto load = [&](int s) {
        unsigned char* st = smem + (s % kStages) * Cf::STAGE;
        const int64_t k0 = kbase + (int64_t)s * kBK;
        load_tile<kBM>(st, a.x, m0, a.M, K, k0, tid);
        load_tile<BN>(st + Cf::A_BYTES, a.w, n0, a.N, K, k0, tid);
    };

    for (int s = 0; s < kStages - kLag; ++s) {  // one group per stage, empty past the end
        if (s < S) load(s);
        cp_async_commit();
    }
    bool ok = true;
    constexpr uint32_t idesc = tc::idesc_bf16(kBM, BN);
    for (int s = 0; s < S; ++s) {
        cp_async_wait_group<kStages - kLag - 1>();  // this thread's pieces of stage s have landed
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t sa = tc::smem_u32(smem + (s % kStages) * Cf::STAGE), sb = sa + Cf::A_BYTES;
            const int j = s / spl;  // leaf
            const uint32_t d = tmem + (uint32_t)((merge ? __popc(j) : j) * BN);
            const bool first = (s % spl) == 0;  // a leaf's first instruction overwrites its slot
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                tc::mma_bf16(d, tc::sdesc(sa + k * 256, 128, Cf::SBO), tc::sdesc(sb + k * 256, 128, Cf::SBO), idesc,
                             (first && k == 0) ? 0u : 1u);
            tc::commit(&mma_done[s % kStages]);
        }
        // refill the stage of step s - kLag (its products are done) with step s + kStages - kLag
        const int nxt = s + kStages - kLag;
        if (nxt < S) {
            if (s >= kLag) {
                const int p = s - kLag;
                ok = tc::mbar_wait(&mma_done[p % kStages], (uint32_t)((p / kStages) & 1)) && ok;
            }
            if (ok) load(nxt);
        }
        cp_async_commit();
        if (merge && s % spl == spl - 1 && ((s / spl) & 1)) {
            // leaf j (odd) is complete once its products are: merge the finished pairs, left
            // (earlier leaves) + right, ctz(j + 1) levels, into the lower slot
            const int j = s / spl;
            ok = tc::mbar_wait(&mma_done[s % kStages], (uint32_t)((s / kStages) & 1)) && ok;
            tc::fence_after_sync();
            const uint32_t lanes = (uint32_t)(warp * 32) << 16;
            for (int top = __popc(j), m = __ffs(j + 1) - 1; m > 0; --m, --top) {
#pragma unroll 1
                for (int cb = 0; cb < BN / 32; ++cb) {
                    float l[32], r[32];
                    uint32_t o[32];
                    const uint32_t dst = tmem + lanes + (uint32_t)((top - 1) * BN + cb * 32);
                    tc::tmem_ld_32x32b<32>(dst, l);
                    tc::tmem_ld_32x32b<32>(tmem + lanes + (uint32_t)(top * BN + cb * 32), r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__fadd_rn(l[e], r[e]));
                    tc::tmem_st_32x32b<32>(dst, o);
                }
                tc::tmem_wait_st();
            }
            tc::fence_before_sync();  // the next products are issued after the loop's barrier
        }
    }
    if (S > 0) ok = tc::mbar_wait(&mma_done[(S - 1) % kStages], (uint32_t)(((S - 1) / kStages) & 1)) && ok;
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    const bool failed = __syncthreads_or(!ok) != 0;
    tc::fence_after_sync();

    if (!failed) {
        constexpr int MAXL = Cf::SLOTS, E = 8;
        const int parts = merge ? 1 : nl;  // partials left in slots 0 .. parts-1
        const int row = warp * 32 + (tid & 31);
        const int64_t gm = m0 + row;
        const uint32_t lanes = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
        for (int cb = 0; cb < BN / E; ++cb) {
            float v[MAXL][E];
#pragma unroll
            for (int l = 0; l < MAXL; ++l)
                if (l < parts) tc::tmem_ld_32x32b<E>(tmem + lanes + (uint32_t)(l * BN + cb * E), v[l]);
            leaf_tree<MAXL, E>(v, parts);
            const int64_t c0 = n0 + cb * E;
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
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) tc::mbar_inval(&mma_done[s]);
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
bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

template <int BN>
cudaError_t launch_pik(const PikArgs& a, cudaStream_t s)
{
    using Cf = PikCfg<BN>;
    cudaError_t e = cudaFuncSetAttribute(k_pik_leaves<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)((a.M + kBM - 1) / kBM) * ((a.N + BN - 1) / BN);
    k_pik_leaves<BN><<<(unsigned)tiles, kThreads, Cf::SMEM, s>>>(a);
    return cudaGetLastError();
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
    if ((int64_t)((M + kBM - 1) / kBM) * ((N + 63) / 64) > 0x7fffffff) return CPR_ERR_INVALID_ARG;
    if (!workspace) return CPR_ERR_WORKSPACE;
    if (!al16(x) || !al16(w) || !al16(workspace) || ((uintptr_t)y & 3u)) return CPR_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    PikArgs a{static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), y, M, N, K, n_leaves,
              leaf_lo, leaf_hi, (al16(y) && N % 4 == 0) ? 1 : 0, static_cast<uint32_t*>(workspace)};
    if (cudaMemsetAsync(a.status, 0, sizeof(uint32_t), s) != cudaSuccess) return CPR_ERR_CUDA;
    const cudaError_t e = launch_pik<128>(a, s);
    return e == cudaSuccess ? CPR_OK : CPR_ERR_CUDA;
}

extern "C" int32_t cpr_pik_combine(const float* parts, int32_t n_parts, int64_t count, float* y, void* stream)
{
    if (!parts || !y || count < 0) return CPR_ERR_INVALID_ARG;
    if (!(n_parts == 1 || n_parts == 2 || n_parts == 4 || n_parts == 8)) return CPR_ERR_INVALID_ARG;
    if (!al16(parts) || !al16(y)) return CPR_ERR_MISALIGNED;
    if (count == 0) return CPR_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
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
