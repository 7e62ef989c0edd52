// copy.cu -- a copy between any two buffers the GPU can address (device
// memory, or pinned host memory mapped into the device's address space),
// done by a kernel rather than a copy engine.  In a decode step the input
// row comes from the host and the output goes back to it; as kernels these
// transfers sit in the same programmatic-dependent-launch chain as the
// producers and GEMVs instead of handing the stream to a copy engine and
// back (on GB300 the host's pinned memory is reached over NVLink-C2C).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace mq {
namespace {

// One 16-byte word per thread while the copy is small: a step's input or
// output is latency-bound, and a single round trip over the link is the
// floor (7B step with a 151 KB input: 15.1 us end to end, against 16.6 us
// with four words per thread).  Larger copies stride over at most 1216 CTAs
// (8 per SM).
constexpr int kCopyThreads = 128;
constexpr int kCopyMaxCtas = 1216;

// Wait for the preceding kernel (the source may be its output, or the
// destination its input), then move 16-byte words, grid-stride, 4 loads in
// flight per thread.
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4 *dst, const uint4 *src, size_t n16)
{
    griddep_launch_dependents();
    griddep_wait();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldcg(src + i), b = __ldcg(src + i + stride);
        const uint4 c = __ldcg(src + i + 2 * stride), d = __ldcg(src + i + 3 * stride);
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = __ldcg(src + i);
}

}  // namespace

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int pdl, cudaStream_t st)
{
    const size_t n16 = bytes / 16;
    size_t ctas = (n16 + kCopyThreads - 1) / kCopyThreads;
    if (ctas < 1) ctas = 1;
    if (ctas > kCopyMaxCtas) ctas = kCopyMaxCtas;
    return launch_maybe_pdl(copy_kernel, dim3((unsigned)ctas), dim3(kCopyThreads), 0, pdl, st,
                            (uint4 *)dst, (const uint4 *)src, n16);
}

}  // namespace mq
