// producers.cu -- the q8 activation producers for sm_103a: standalone
// quantize, rms_norm -> q8 and SwiGLU -> q8 (page "70 · D3-5 — fused-producer
// decode A-quantize", §2-§3).
//
// Quantization (§3.2 of that page, per 32-value block): am = max|v|,
// d = am / 127, di = d != 0 ? 1/d : 0, q = clamp(rint(v * di), -128, 127),
// fp16(d) stored, sum of q stored.  Built without fast-math, so the division,
// the reciprocal and the rounding are IEEE f32 exactly as the host computes
// them.  Here 8 consecutive lanes share a block (4 values each, one float4
// load): the max and the sum are taken with 3 xor-shuffles, which is exact for
// both (max is associative; integer addition too), so the bytes do not
// depend on the thread geometry.  Shuffles run on every lane unconditionally
// and only loads/stores are guarded (the page's §3.3 barrier pitfall).
//
// The fused producers quantize the f32 values they have just computed, in
// registers, so the q8 bytes are by construction the quantization of the f32
// output they write (the page's "constructive bitwise", §2.3).
//
// Inputs may be written by the preceding kernel, which under programmatic
// dependent launch is still running when these kernels start: every input
// is read after griddepcontrol.wait and with coherent loads (ld.global.cg),
// never the non-coherent path the compiler may hoist above the wait.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "kernels.h"

namespace mq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int q8_code(float v, float di)
{
    int q = __float2int_rn(v * di);  // round half to even, like rintf
    return max(-128, min(127, q));
}

// Quantize 4 values held by this lane; 8 lanes (aligned group) form a block.
// gid = global index of this lane's 4-value group (block = gid / 8).
__device__ __forceinline__ void quantize4(float4 v, bool valid, long long gid, uint8_t *q8,
                                          unsigned d_off, unsigned sum_off)
{
    float am = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    am = fmaxf(am, __shfl_xor_sync(kFull, am, 1));
    am = fmaxf(am, __shfl_xor_sync(kFull, am, 2));
    am = fmaxf(am, __shfl_xor_sync(kFull, am, 4));
    const float d = am / 127.0f;
    const float di = (d != 0.0f) ? 1.0f / d : 0.0f;
    const int q0 = q8_code(v.x, di), q1 = q8_code(v.y, di);
    const int q2 = q8_code(v.z, di), q3 = q8_code(v.w, di);
    int s = q0 + q1 + q2 + q3;
    s += __shfl_xor_sync(kFull, s, 1);
    s += __shfl_xor_sync(kFull, s, 2);
    s += __shfl_xor_sync(kFull, s, 4);
    if (!valid) return;
    const uint32_t packed = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8) |
                            ((uint32_t)(q2 & 0xff) << 16) | ((uint32_t)(q3 & 0xff) << 24);
    reinterpret_cast<uint32_t *>(q8)[gid] = packed;
    if ((gid & 7) == 0) {
        const long long b = gid >> 3;
        reinterpret_cast<__half *>(q8 + d_off)[b] = __float2half_rn(d);
        reinterpret_cast<int *>(q8 + sum_off)[b] = s;
    }
}

// Rows of n values (n4 = n / 4 lane groups each) are quantized into planes
// `stride` bytes apart: blockIdx.y is the row, blockIdx.x * blockDim.x +
// threadIdx.x the lane group within it.  n4 is a multiple of 8, so every
// 8-lane block lies in one row; lanes past the row's end only join the
// shuffles.
__global__ void __launch_bounds__(256) quantize_q8_kernel(const float *__restrict__ x,
                                                          uint8_t *__restrict__ q8, int n4,
                                                          unsigned stride, unsigned d_off,
                                                          unsigned sum_off)
{
    griddep_launch_dependents();
    griddep_wait();  // x may come from the preceding kernel
    const size_t row = blockIdx.y;
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = gid < n4;
    const float4 v = valid ? __ldcg(reinterpret_cast<const float4 *>(x) + row * n4 + gid)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    quantize4(v, valid, gid, q8 + row * stride, d_off, sum_off);
}

// y = (g / (1 + exp(-g))) * u, the swiglu body of the D3-5 page §3.2, over
// rows of n values; y may alias g or u (each lane reads its 4 values before
// writing them).
__global__ void __launch_bounds__(256) swiglu_quant_q8_kernel(const float *g, const float *u,
                                                              float *y, uint8_t *__restrict__ q8,
                                                              int n4, unsigned stride,
                                                              unsigned d_off, unsigned sum_off)
{
    griddep_launch_dependents();
    griddep_wait();  // g and u may come from the preceding kernels
    const size_t row = blockIdx.y;
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = gid < n4;
    const size_t at = row * n4 + gid;  // float4 index in the nt x n arrays
    float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
        const float4 gv = __ldcg(reinterpret_cast<const float4 *>(g) + at);
        const float4 uv = __ldcg(reinterpret_cast<const float4 *>(u) + at);
        out.x = (gv.x / (1.0f + expf(-gv.x))) * uv.x;
        out.y = (gv.y / (1.0f + expf(-gv.y))) * uv.y;
        out.z = (gv.z / (1.0f + expf(-gv.z))) * uv.z;
        out.w = (gv.w / (1.0f + expf(-gv.w))) * uv.w;
        reinterpret_cast<float4 *>(y)[at] = out;
    }
    quantize4(out, valid, gid, q8 + row * stride, d_off, sum_off);
}

// Each row (blockIdx.y) over a grid of CTAs with no inter-CTA communication: every CTA
// computes the whole sum of squares itself (the row is a few tens of KB and
// sits in L2, so the redundant reads cost less than a grid-wide exchange),
// in one fixed order -- per-thread serial, a fixed shuffle tree, then the
// per-warp partials added in warp order by every thread -- so all CTAs get
// the same bits.  scale = 1/sqrt(ss/n + eps) (IEEE sqrt and division), then
// each CTA writes y = (x * scale) * gain and its q8 blocks for its own slice.
// 512 threads (14B decode sweep 2.234 ms per step, against 2.298 ms with
// 256 threads and 2.227 ms with 1024, which is slower on the single-layer
// chains: rms -> gate||up -> down 28.85 against 28.58 us).  K: the float4
// groups per thread loaded before the sum chain starts (4 for rows up to
// 8192 values, else 8), so that a thread's loads are one round trip, not
// one per pair of groups.
constexpr int kRmsThreads = 512;
constexpr int kRmsMaxCtas = 64;

template <int K>
__global__ void __launch_bounds__(kRmsThreads) rmsnorm_quant_q8_kernel(
    const float *__restrict__ x, const float *__restrict__ gain, float eps, float *__restrict__ y,
    uint8_t *__restrict__ q8, int n, unsigned stride, unsigned d_off, unsigned sum_off)
{
    __shared__ float warp_ss[kRmsThreads / 32];
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n4 = n >> 2;
    const int first = blockIdx.x * kRmsThreads;  // this CTA's first float4
    const size_t row = blockIdx.y;
    const float4 *x4 = reinterpret_cast<const float4 *>(x + row * n);
    const float4 *g4 = reinterpret_cast<const float4 *>(gain);
    // the gain is a weight (never written by the preceding kernel): its first
    // slice is loaded before the wait, off the chain's critical path (14B
    // decode sweep 2.234 -> 2.214 ms per step)
    const float4 g_own = first + tid < n4 ? __ldg(g4 + first + tid) : make_float4(0.f, 0.f, 0.f, 0.f);
    griddep_wait();  // x may come from the preceding kernel
    y += row * n;
    q8 += row * stride;

    float ss = 0.0f;
    float4 own = make_float4(0.f, 0.f, 0.f, 0.f);  // x[first + tid], kept from the sum pass
    // The thread's first K groups are all requested before the first fmaf:
    // with the loop below alone (2-fold unrolled), the third group of a
    // 5120-value row waited for the first two's arithmetic, a second round
    // trip (14B decode sweep 2092.8 -> 2061.4 us per step, same bits).  A
    // group past the row adds fmaf(0, 0, ss) = ss, which leaves the bits
    // unchanged, so the per-lane order and result are the loop's.
    {
        float4 v[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int i = tid + k * kRmsThreads;
            v[k] = i < n4 ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (k * kRmsThreads == first) own = v[k];
            ss = fmaf(v[k].x, v[k].x, ss);
            ss = fmaf(v[k].y, v[k].y, ss);
            ss = fmaf(v[k].z, v[k].z, ss);
            ss = fmaf(v[k].w, v[k].w, ss);
        }
    }
#pragma unroll 2
    for (int i = tid + K * kRmsThreads; i < n4; i += kRmsThreads) {
        const float4 v = __ldcg(x4 + i);
        if (i == first + tid) own = v;
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
    if (lane == 0) warp_ss[wid] = ss;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kRmsThreads / 32; ++w) t += warp_ss[w];
    const float scale = 1.0f / sqrtf(t / (float)n + eps);

    // The slice loop's trip count is uniform across the CTA, so the
    // quantizer's shuffles always see full warps.
    // one slice per CTA up to 64 CTAs (256 K values): not unrolled
#pragma unroll 1
    for (int base = first; base < n4; base += gridDim.x * kRmsThreads) {
        const int i = base + tid;
        const bool valid = i < n4;
        float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) {
            const float4 v = base == first ? own : __ldcg(x4 + i);
            const float4 gv = base == first ? g_own : __ldg(g4 + i);
            out.x = (v.x * scale) * gv.x;
            out.y = (v.y * scale) * gv.y;
            out.z = (v.z * scale) * gv.z;
            out.w = (v.w * scale) * gv.w;
            reinterpret_cast<float4 *>(y)[i] = out;
        }
        quantize4(out, valid, i, q8, d_off, sum_off);
    }
}

inline unsigned blocks_for(long long threads, int per_block)
{
    return (unsigned)((threads + per_block - 1) / per_block);
}

}  // namespace

cudaError_t launch_quantize_q8(const float *x, uint8_t *q8, int n, int rows, unsigned stride,
                               unsigned d_off, unsigned sum_off, int pdl, cudaStream_t st)
{
    const int n4 = n / 4;
    return launch_maybe_pdl(quantize_q8_kernel, dim3(blocks_for(n4, 256), (unsigned)rows), dim3(256),
                            0, pdl, st, x, q8, n4, stride, d_off, sum_off);
}

cudaError_t launch_swiglu_quant_q8(const float *g, const float *u, float *y, uint8_t *q8, int n,
                                   int rows, unsigned stride, unsigned d_off, unsigned sum_off,
                                   int pdl, cudaStream_t st)
{
    const int n4 = n / 4;
    return launch_maybe_pdl(swiglu_quant_q8_kernel, dim3(blocks_for(n4, 256), (unsigned)rows),
                            dim3(256), 0, pdl, st, g, u, y, q8, n4, stride, d_off, sum_off);
}

cudaError_t launch_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y,
                                    uint8_t *q8, int n, int rows, unsigned stride, unsigned d_off,
                                    unsigned sum_off, int pdl, cudaStream_t st)
{
    const unsigned ctas = std::min(blocks_for(n / 4, kRmsThreads), (unsigned)kRmsMaxCtas);
    const auto kernel = n / 4 <= 4 * kRmsThreads ? rmsnorm_quant_q8_kernel<4> : rmsnorm_quant_q8_kernel<8>;
    return launch_maybe_pdl(kernel, dim3(ctas, (unsigned)rows), dim3(kRmsThreads), 0, pdl, st, x, gain,
                            eps, y, q8, n, stride, d_off, sum_off);
}

}  // namespace mq
