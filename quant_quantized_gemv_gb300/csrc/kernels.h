// kernels.h -- launch interface between the C ABI (api.cpp) and the CUDA
// kernels (gemv.cu, producers.cu).  Internal to the library.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mq {

// One GEMV launch.  A work item is (tile t, split s): one warp streams chunks
// [s*cps, min((s+1)*cps, nchunks)) of the 8-row tile t.
struct GemvLaunch {
    const uint8_t *W;       // repacked weights (layout.h)
    const uint8_t *q8;      // q8 plane of cols values
    float *y;               // rows outputs
    int32_t *isums;         // sub-dot mode: rows * nb * {16 | 8} int32, else null
    unsigned *ws_cnt;       // split-K arrival counters [ntiles] (splits > 1)
    float *ws_part;         // split-K partials [splits][ntiles][8] (splits > 1)
    int rows, nb, ntiles, nchunks, splits, cps;
    long long n_items;      // ntiles * splits
    size_t tile_bytes;
    unsigned q8_d_off, q8_sum_off;
};

cudaError_t launch_gemv_q6k(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_gemv_q4k(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_subdots_q6k(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_subdots_q4k(const GemvLaunch &a, cudaStream_t st);

// Producers.  d_off / sum_off locate the q8 plane's fp16-scale and sum
// sections (layout.h q8_d_offset / q8_sum_offset).
cudaError_t launch_quantize_q8(const float *x, uint8_t *q8, int n, unsigned d_off,
                               unsigned sum_off, cudaStream_t st);
cudaError_t launch_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y,
                                    uint8_t *q8, int n, unsigned d_off, unsigned sum_off,
                                    cudaStream_t st);
cudaError_t launch_swiglu_quant_q8(const float *g, const float *u, float *y, uint8_t *q8, int n,
                                   unsigned d_off, unsigned sum_off, cudaStream_t st);

constexpr int kGemvWarpsPerBlock = 4;

}  // namespace mq
