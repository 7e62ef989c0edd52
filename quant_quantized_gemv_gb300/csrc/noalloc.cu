// noalloc.cu -- a q6_K decode GEMV entry point that needs no caller-provided
// workspace and allocates nothing.
//
// Who needs it: code that runs where it may not allocate device memory.
// Examples are a plugin or callback handed only input and output pointers
// by a host framework that owns every allocation, a real-time path that
// forbids allocation once it has started, and a caller inside a region
// where cudaMalloc is not allowed or would synchronize the device.  Such a
// caller cannot create the split-K workspace that mq_gemv_q6k_q8 expects.
//
// What it does: it runs the same GEMV kernel with the library's default
// plan.  When that plan splits tiles, the scratch (one arrival counter per
// 8-row tile, then 8 floats of partial sums per work item) lives in the
// file-scope device array below instead of a caller buffer.  Every GPU
// that loads the library keeps this array until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "kernels.h"
#include "layout.h"
#include "mq.h"

namespace {

using namespace mq;

// Largest scratch a call may use.  With one resident wave of at most 2432
// warps (152 SMs x 16 warps) a split plan needs at most 2432 x 32 B of
// partials plus 4 B per tile of counters, about 80 KB.
constexpr size_t kNoAllocScratchBytes = 128 * 1024;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDev];  // device address of the array, per device

// Look up (once per device, with that device current) the device address of
// the array.  In host code `g_noalloc_scratch` names a host-side stand-in,
// not device memory, so the kernel must be given this address instead.
int scratch_address(void **out)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDev) return MQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e2 = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e2 != cudaSuccess) return cuda_fail("cudaGetSymbolAddress(scratch)", e2);
        if (!p) return MQ_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MQ_OK;
}

// Zero the arrival counters at the head of the scratch.  A kernel rather
// than a memset so that a decode chain with programmatic dependent launch
// stays a chain: it waits for its predecessor (which may be the previous
// call still using the array) before it writes, and lets the GEMV behind it
// start streaming weights meanwhile.
__global__ void clear_counters_kernel(unsigned *cnt, int n)
{
    griddep_launch_dependents();
    griddep_wait();
    for (int i = threadIdx.x; i < n; i += blockDim.x) cnt[i] = 0u;
}

}  // namespace

extern "C" int mq_gemv_q6k_q8_noalloc(const void *Wp, const void *q8, float *y, int rows, int cols,
                                      void *stream)
{
    if (!Wp || !q8 || !y) return MQ_ERR_NULL;
    if (rows < 1 || cols < kQK || cols % kQK != 0 || (long long)rows * cols >= (1LL << 40))
        return MQ_ERR_SHAPE;
    if (((uintptr_t)Wp & 15u) || ((uintptr_t)q8 & 15u) || ((uintptr_t)y & 15u)) return MQ_ERR_ALIGN;
    int splits = 0, cps = 0, tpi = 0;
    const int pst = mq_gemv_plan(rows, cols, 6, &splits, &cps, &tpi);
    if (pst != MQ_OK) return pst;
    const size_t need = mq_gemv_workspace_bytes_for(rows, cols, splits, cps, tpi);
    if (need > kNoAllocScratchBytes) return MQ_ERR_WORKSPACE;  // plan too big for the array
    if (need == 0) return mq_gemv_q6k_q8_plan(Wp, q8, y, rows, cols, splits, cps, tpi, nullptr, 0,
                                              stream);
    void *ws = nullptr;
    const int st = scratch_address(&ws);
    if (st != MQ_OK) return st;
    // The counters must start at zero; a finished call leaves them at zero,
    // but clear them anyway so that an interrupted earlier call cannot leak.
    const int ncnt = ceil_div(rows, kTileRows);
    const cudaError_t e = launch_maybe_pdl(clear_counters_kernel, dim3(1), dim3(256), 0, pdl_setting(),
                                           (cudaStream_t)stream, (unsigned *)ws, ncnt);
    if (e != cudaSuccess) return cuda_fail("clearing the scratch counters", e);
    return mq_gemv_q6k_q8_plan(Wp, q8, y, rows, cols, splits, cps, tpi, ws, kNoAllocScratchBytes,
                               stream);
}
