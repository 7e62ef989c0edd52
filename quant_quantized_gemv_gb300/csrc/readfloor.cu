// readfloor.cu -- a plain streaming read of n bytes in one launch: the floor
// against which a GEMV of the same bytes is judged.  A GEMV must at least
// read its weights once; this kernel does only that (16-byte non-coherent
// loads bypassing L1, two per lane in flight, one resident wave of 384-thread
// CTAs), so its time is what a single launch of that size costs on this GPU,
// launch ramp and tail included.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace mq {
namespace {

__device__ __forceinline__ uint4 ld_nc16(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(384, 1) read_floor_kernel(const uint4 *src, size_t n16,
                                                            unsigned *sink)
{
    const size_t nthr = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned acc = 0;
    for (; i + nthr < n16; i += 2 * nthr) {
        const uint4 a = ld_nc16(src + i), b = ld_nc16(src + i + nthr);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w;
    }
    if (i < n16) {
        const uint4 a = ld_nc16(src + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
    if (sink && acc == 0x9e3779b9u) *sink = acc;  // keeps the loads; practically never stores
}

}  // namespace

cudaError_t launch_read_floor(const void *src, size_t bytes, unsigned *sink, int sms, cudaStream_t st)
{
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, read_floor_kernel, 384, 0);
    if (e != cudaSuccess) return e;
    read_floor_kernel<<<sms * (per_sm > 0 ? per_sm : 1), 384, 0, st>>>(
        reinterpret_cast<const uint4 *>(src), bytes / 16, sink);
    return cudaGetLastError();
}

}  // namespace mq
