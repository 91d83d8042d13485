// fr_split_merge.cuh -- the bounded grid barrier of the decode attention
// kernels that merge their KV splits inside their own launch (fr_attn_sw.cu):
// every split's state must be stored before any CTA combines them.
#pragma once

#include <math.h>
#include <stdint.h>

#include "fr_sm100.cuh"

namespace fr {
namespace split_merge {

using namespace sm100;

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One thread per CTA, after the CTA's state is stored (and a CTA barrier):
// arrive with a release add (the state is visible before the count moves),
// then poll the count until every one of the n CTAs has arrived. Every CTA
// must be resident (cooperative launch). Returns false if the wait gave up
// after limit_ns. Each CTA calls grid_barrier_depart once it no longer needs
// the barrier (off the critical path, at its end): the last to depart returns
// both words to zero for the next call, whose CTAs arrive only after this grid
// is complete.
__device__ __forceinline__ bool grid_barrier(unsigned* barrier, unsigned n, uint64_t limit_ns) {
    unsigned* count = barrier;
    red_release_add_u32(count, 1u);
    const uint64_t t_start = global_ns();
    while (ld_acquire_u32(count) < n) {
        if (global_ns() - t_start > limit_ns) return false;
        __nanosleep(20);
    }
    return true;
}
__device__ __forceinline__ void grid_barrier_depart(unsigned* barrier, unsigned n) {
    unsigned* count = barrier;
    unsigned* departed = barrier + 1;
    if (atomicAdd(departed, 1u) == n - 1u) {
        *count = 0u;
        *departed = 0u;
    }
}

}  // namespace split_merge
}  // namespace fr
