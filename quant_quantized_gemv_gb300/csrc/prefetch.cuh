// prefetch.cuh -- a bulk L2 prefetch hint for the streaming GEMV kernels.
#pragma once

namespace mq {

// Hint: move [p, p + bytes) from HBM toward L2 (p 16-byte aligned, bytes a
// multiple of 16; one instruction per contiguous range, no completion to
// wait for).  A repacked tile-chunk is contiguous, so one call covers the
// chunk a warp will load next.
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

}  // namespace mq
