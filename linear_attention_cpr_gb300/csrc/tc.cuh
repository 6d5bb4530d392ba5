// tc.cuh — inline-PTX helpers for the 5th-generation tensor cores (tcgen05) of sm_103a:
// shared-memory matrix descriptors, instruction descriptors, TMEM allocation, MMA issue
// and commit, mbarriers with bounded waits, bulk global->shared copies, TMEM loads.
//
// Operand layout of the layer kernels (verified against a CPU reference on this GPU): no
// swizzle, K-major; a tile of R rows x K elements is made of "core matrices" of 8 rows x
// 16 bytes, core (i, kk) stored at byte (i * (K*esize/16) + kk) * 128, row r of a core at
// +16*r.  In the descriptor, LBO is the byte step between cores adjacent along K (128)
// and SBO the step between 8-row groups (K*esize/16 * 128).
// The same tile read MN-major (the instruction descriptor's transpose bit for A or B, bits
// 15 and 16): the operand's M or N index runs along the 16-byte rows, its K index across
// them; LBO is then the byte step between 8-element K groups and SBO the step between
// 8-element M or N groups (checked on this GPU against a CPU product).
// (pik.cu uses the 128-byte-swizzled K-major layout instead, with its own descriptor.)
// Accumulator layout: M = 128 -> row m in TMEM lane m; M = 64 -> rows 16q..16q+15 in
// lanes 32q..32q+15.  Column j of D is TMEM column (base + j).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace cpr {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of element (row, col) in a K-major core-matrix tile with K elements per row.
template <int ESIZE>
__host__ __device__ __forceinline__ uint32_t tile_off(int row, int col, int K)
{
    constexpr int EPC = 16 / ESIZE;  // elements per 16-byte core row
    return (uint32_t)(((row >> 3) * (K / EPC) + col / EPC) * 128 + (row & 7) * 16 + (col % EPC) * ESIZE);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version of the 5th-generation tensor cores
    return d;
}

// kind::f16 with bf16 A and B (both K-major), fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on mbar once every previously issued MMA of this thread has completed.
__device__ __forceinline__ void commit(uint64_t* mbar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     smem_u32(mbar))
                 : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(mbar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(mbar)), "r"(bytes)
                 : "memory");
}

// Wait for the phase with the given parity to complete; gives up after max_iters polls and
// returns false (the caller records a timeout and winds down).
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, uint32_t max_iters = 1u << 22)
{
    uint32_t done = 0;
    for (uint32_t it = 0; it < max_iters; ++it) {
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(mbar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// Invalidate an mbarrier whose shared memory is about to be reused for other data.
__device__ __forceinline__ void mbar_inval(uint64_t* mbar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_u32(mbar)) : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) global -> shared,
// completing as transaction bytes on mbar.
// 16-byte asynchronous copy global -> shared (both 16-byte aligned), and the wait for all
// of this thread's copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ void bulk_g2s(void* smem, const void* gmem, uint32_t bytes, uint64_t* mbar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(smem)),
        "l"(gmem), "r"(bytes), "r"(smem_u32(mbar))
        : "memory");
}

// One box of a 3-dimensional tensor map (a CUtensorMap in kernel-parameter, constant or
// global memory) at coordinates (x, y, z) into this CTA's shared memory (128-byte aligned),
// completing its bytes on mbar.  x times the element size must be a multiple of 16 bytes;
// elements outside the tensor land as zeros and still count towards the bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, int32_t x, int32_t y, int32_t z,
                                            uint64_t* mbar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(mbar))
        : "memory");
}

// Prefetch `bytes` (a multiple of 16, address 16-byte aligned) of global memory into L2
// (no completion to wait for: a hint that a later copy of the same bytes hits in L2).
__device__ __forceinline__ void prefetch_l2(const void* gmem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(gmem), "r"(bytes) : "memory");
}

// Bulk copy shared -> global (both 16-byte aligned, bytes a multiple of 16), tracked by
// this thread's bulk group: commit with bulk_commit, wait with bulk_wait_all.
__device__ __forceinline__ void bulk_s2g(void* gmem, const void* smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gmem), "r"(smem_u32(smem)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until every committed bulk store of this thread is complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// Allocation (one full warp).  The TMEM address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor cores.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32*(w%4) ..).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// tcgen05.ld 32x32b with N 32-bit columns: thread t of the warp reads TMEM lane
// (quadrant base + t), columns [taddr_col, taddr_col + N) (the layout of an M = 128
// accumulator, row = lane).
template <int N>
__device__ __forceinline__ void tmem_ld_32x32b(uint32_t taddr, float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_ld_32x32b<32>(uint32_t taddr, float (&v)[32])
{
    tmem_ld32(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld_32x32b<8>(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}
template <>
__device__ __forceinline__ void tmem_ld_32x32b<16>(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// tcgen05.st 32x32b with N 32-bit columns: thread t of the warp writes TMEM lane
// (quadrant base + t), columns [taddr_col, taddr_col + N).  The caller waits with
// tmem_wait_st() before the data is used.
template <int N>
__device__ __forceinline__ void tmem_st_32x32b(uint32_t taddr, const uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_st_32x32b<4>(uint32_t taddr, const uint32_t (&r)[4])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_32x32b<8>(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_32x32b<16>(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_32x32b<32>(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// tcgen05.mma kind::f16 with the A operand in TMEM (same lanes as the accumulator rows;
// each 32-bit column holds two consecutive K elements, the even one in the low half), B
// from a shared-memory descriptor.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// tcgen05.ld 16x32bx2 with N 32-bit columns per half: thread t of the warp reads TMEM
// lane (quadrant base + t % 16), columns [taddr_col + (t / 16) * N, + N) (verified on
// this GPU).  Used for M = 64 accumulators, whose rows occupy 16 lanes per quadrant.
template <int N>
__device__ __forceinline__ void tmem_ld_16x2(uint32_t taddr, float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_ld_16x2<4>(uint32_t taddr, float (&v)[4])
{
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x4.b32 {%0,%1,%2,%3}, [%4], 4;\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __uint_as_float(r[j]);
}

template <>
__device__ __forceinline__ void tmem_ld_16x2<8>(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], 8;\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}

template <>
__device__ __forceinline__ void tmem_ld_16x2<16>(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 16;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

template <>
__device__ __forceinline__ void tmem_ld_16x2<32>(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], 32;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* mbar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(mbar)) : "memory");
}

// Two-term bf16 split of an fp32 value, x = hi + lo + e.  hi is the head of Dekker's
// splitting (Veltkamp's method with the constant 2^16 + 1): a value with at most 8
// significant bits, so exactly a bf16, computed with three fp32 operations; lo = x - hi is
// exact in fp32 and is truncated to bf16 when packed (its upper 16 bits), so
// |e| < 2^-15 |x|.  Every step is an explicit round-to-nearest fp32 operation or a bit
// move, so all kernels produce the same splits.
__device__ __forceinline__ void split_f32(float x, float& hi, float& lo)
{
    const float t = __fmul_rn(x, 65537.0f);
    hi = __fsub_rn(t, __fsub_rn(t, x));
    lo = __fsub_rn(x, hi);
}

// bf16 pair (a in the low half, b in the high half) from the upper 16 bits of two fp32s.
__device__ __forceinline__ uint32_t pack_upper(float a, float b)
{
    return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
}

// Split 8 consecutive values into 16-byte hi and lo bf16 rows (lo_dst may be NULL).
__device__ __forceinline__ void split8_store(const float (&x)[8], unsigned char* hi_dst, unsigned char* lo_dst)
{
    float h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) split_f32(x[e], h[e], l[e]);
    *reinterpret_cast<uint4*>(hi_dst) =
        make_uint4(pack_upper(h[0], h[1]), pack_upper(h[2], h[3]), pack_upper(h[4], h[5]), pack_upper(h[6], h[7]));
    if (lo_dst)
        *reinterpret_cast<uint4*>(lo_dst) =
            make_uint4(pack_upper(l[0], l[1]), pack_upper(l[2], l[3]), pack_upper(l[4], l[5]), pack_upper(l[6], l[7]));
}

}  // namespace tc
}  // namespace cpr
