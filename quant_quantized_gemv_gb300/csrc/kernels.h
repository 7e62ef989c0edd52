// kernels.h -- launch interface between the C ABI (api.cpp) and the CUDA
// kernels (gemv.cu, producers.cu).  Internal to the library.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mq {

// One GEMV launch.  The matrix is ntiles x nchunks chunk units (tile = 8
// rows, chunk = 4 super-blocks of those rows).  A work item (one warp)
// streams a contiguous range of them:
//   splits == 1: item i covers whole tiles [i*tpi, min((i+1)*tpi, ntiles));
//   splits > 1 (tall rows): item i is split s = i % splits of tile
//     t = i / splits and covers chunks [s*cps, min((s+1)*cps, nchunks)) of t.
//     Up to kMaxCtaSplits splits the splits of a tile are the warps of one
//     CTA and combine in shared memory; beyond that they combine through the
//     workspace, where the last one to finish adds the partials in ascending
//     split order.
struct GemvLaunch {
    const uint8_t *W;       // repacked weights (layout.h)
    const uint8_t *q8;      // q8 plane of cols values
    float *y;               // rows outputs
    int32_t *isums;         // sub-dot mode: rows * nb * {16 | 8} int32, else null
    unsigned *ws_cnt;       // arrival counters [ntiles] (splits > kMaxCtaSplits)
    float *ws_part;         // partials [n_items][8 rows] (splits > kMaxCtaSplits)
    int rows, nb, ntiles, nchunks;
    int splits, cps, tpi;   // the plan (see above)
    int n_items;
    size_t tile_bytes;
    unsigned q8_d_off, q8_sum_off;
    int pdl;                // launch with programmatic stream serialization
};

cudaError_t launch_gemv_q6k(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_gemv_q4k(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_subdots_q6k(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_subdots_q4k(const GemvLaunch &a, cudaStream_t st);

constexpr int kGemvWarpsPerBlock = 4;   // CTA of independent warps
constexpr int kMaxCtaSplits = 12;       // largest CTA whose warps are one tile's splits

// Warps per CTA for a plan with `splits` splits.
inline int gemv_cta_warps(int splits, bool subdots = false)
{
    return (!subdots && splits > 1 && splits <= kMaxCtaSplits) ? splits : kGemvWarpsPerBlock;
}

// Resident CTAs per SM of the GEMV kernel for format 6 (q6_K) or 4 (q4_K)
// with `warps_per_cta` warps, on the current device (0 on error).
int gemv_ctas_per_sm(int fmt, int warps_per_cta);

// Producers.  d_off / sum_off locate the q8 plane's fp16-scale and sum
// sections (layout.h q8_d_offset / q8_sum_offset).
cudaError_t launch_quantize_q8(const float *x, uint8_t *q8, int n, unsigned d_off,
                               unsigned sum_off, int pdl, cudaStream_t st);
cudaError_t launch_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y,
                                    uint8_t *q8, int n, unsigned d_off, unsigned sum_off, int pdl,
                                    cudaStream_t st);
cudaError_t launch_swiglu_quant_q8(const float *g, const float *u, float *y, uint8_t *q8, int n,
                                   unsigned d_off, unsigned sum_off, int pdl, cudaStream_t st);

// Launch `kernel` on `st`, with programmatic stream serialization when pdl
// is set (the kernel then may start before its predecessor in the stream
// finishes and must call griddep_wait() before touching dependent data).
template <class... KArgs, class... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, int pdl,
                             cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace mq

#ifdef __CUDACC__
// Programmatic dependent launch controls (no-ops without the attribute).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif
