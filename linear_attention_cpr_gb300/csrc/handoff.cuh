// handoff.cuh — hand-off between the CTAs of one cooperative launch: a producer CTA
// publishes a finished piece of work through a counter in global memory, consumers wait
// for it (bounded).  Used by the forward's chain and items and by the backward's reverse
// chain and chunk gradients.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cpr_gdn.h"

namespace cpr {

// ------------------------------------------------------------------------------------
// ready[c * H + h] counts the publications of chunk c's result for head h (a boundary
// state, or the backward's state adjoint): the producing CTA's threads issue their stores,
// meet at a barrier, and one thread adds 1 with release semantics.  All CTAs of the launch
// are resident (cooperative launch) and producers wait on nothing but their own copies and
// products, so every wait below ends; it is still bounded (about 4 s) and reports a
// timeout instead of hanging.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void named_bar(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Wait until *flag >= target; gives up (returns 0) after limit_ns (0: about 4 s), or at
// once when another CTA of the launch has recorded a timeout in the status word.
__device__ __forceinline__ int wait_published(const uint32_t* flag, uint32_t target, const uint32_t* status,
                                              uint64_t limit_ns)
{
    if (ld_acquire(flag) >= target) return 1;
    const uint64_t limit = limit_ns ? limit_ns : 4000000000ull;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        __nanosleep(128);
        if (ld_acquire(flag) >= target) return 1;
        if ((ld_acquire(status) & CPR_DEV_TIMEOUT) || global_ns() - t0 > limit) break;
    }
    return 0;
}

// Publish a result: the CTA's stores to it were issued before a barrier this thread has
// passed; the release orders them before the count.
__device__ __forceinline__ void publish(uint32_t* flag)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(flag) : "memory");
}

}  // namespace cpr
