// gemv_gateup.cu -- the FFN's gate and up GEMVs with the SwiGLU -> q8
// producer fused into their epilogue: one launch reads the rms_norm'd
// hidden state's q8 plane, streams both weight matrices and writes
// act = silu(gate) * up (f32) together with act's q8 plane for ffn_down.
//
// The pages tried this fusion (page "76 · D4-4 — dpl dense split-plane q6_K
// decode MMVQ", §2 and §5: the concatenated gate||up launch with a SwiGLU
// epilogue) and closed it on GB10 because its grid ran 1.5 waves.  Here the
// grid is one resident wave by construction (below), and the per-row
// arithmetic is the single-token GEMV's whole-tile path, so act and its q8
// plane are bit for bit those of GEMV(gate), GEMV(up), then the SwiGLU
// producer (page "70 · D3-5 — fused-producer decode A-quantize", §3.2).
//
// Work: rows are cut into q8 blocks of 32 outputs = 4 tiles of gate and the
// same 4 tiles of up.  A CTA takes whole blocks (grid-stride); its W warps
// share a block's 8 tiles (warp w: tiles w, w + W, ...; even tiles are gate,
// odd are up), each streaming whole rows with two register buffers.  Row
// sums meet in shared memory; after one barrier a warp of the CTA forms act
// for the block's 32 rows (one per lane), writes it and quantizes it (max
// and sum by xor-shuffles: exact, so the bytes do not depend on the lane
// count).  The exchange buffer alternates with the block, so one barrier per
// block suffices.  The host picks W (1..8) so that the CTAs fit one wave.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "gemv_common.cuh"
#include "kernels.h"
#include "layout.h"

namespace mq {
namespace {

using namespace gemv_detail;

// Wait for the producer, stage the q8 plane in shared memory, meet at named
// barrier 1 (every warp calls this exactly once).
__device__ __forceinline__ void stage(const GemvLaunch &a, uint8_t *xs)
{
    griddep_wait();
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q8);
    uint4 *dst = reinterpret_cast<uint4 *>(xs);
    const int n16 = (int)(a.q8_bytes >> 4);
    // 2-fold: a 5120-value plane is ~3 copies per thread (unrolled 4-fold the
    // 14B decode sweep took 2120 against 2109 us per step, with the rms write
    // loop below not unrolled)
    for (int i = threadIdx.x; i < n16; i += blockDim.x) copy16_async(dst + i, src + i);
    copy_async_wait_all();
    asm volatile("bar.sync 1, %0;" ::"r"(blockDim.x) : "memory");
}

// act for 32 rows, one per lane, quantized as one q8 block ([D3-5] §3.2):
// am = max|v|, d = am / 127, di = d != 0 ? 1/d : 0, q = clamp(rint(v*di)).
__device__ __forceinline__ void quantize_block(float v, const GateUpLaunch &L, int blk, int lane)
{
    float am = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
    const float d = am / 127.0f;
    const float di = (d != 0.0f) ? 1.0f / d : 0.0f;
    const int q = max(-128, min(127, __float2int_rn(v * di)));
    int s = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    L.q8o[(size_t)blk * 32 + lane] = (uint8_t)(q & 0xff);
    if (lane == 0) {
        reinterpret_cast<__half *>(L.q8o + L.o_d_off)[blk] = __float2half_rn(d);
        reinterpret_cast<int *>(L.q8o + L.o_sum_off)[blk] = s;
    }
}

template <int FMT>
__device__ __forceinline__ void run_gateup(const GateUpLaunch &L, uint8_t *xs, int lane)
{
    __shared__ float sums[2][8][8];  // [block parity][tile of the block][row]
    using Regs = typename Fmt<FMT>::Regs;
    constexpr int kChunkBytes = Fmt<FMT>::kChunkBytes;
    const GemvLaunch &a = L.g;
    const int W = blockDim.x >> 5, w = threadIdx.x >> 5;
    const int nch = a.nchunks;
    const int tiles = (8 - w + W - 1) / W;  // this warp's tiles per block
    const int my_blocks = (L.nblk - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int n_units = my_blocks * tiles * nch;

    struct Cursor {
        int k, m, c;  // block iteration, this warp's tile index, chunk
    };
    auto unit_at = [&](const Cursor &q) {
        const int blk = (int)blockIdx.x + q.k * (int)gridDim.x;
        const int j = w + q.m * W;  // tile of the block: even gate, odd up
        return locate(a, a.part[j & 1], 4 * blk + (j >> 1), q.c, lane, kChunkBytes);
    };
    auto advance = [&](Cursor &q) {
        if (++q.c == nch) {
            q.c = 0;
            if (++q.m == tiles) { q.m = 0; ++q.k; }
        }
    };

    Regs A, B;
    Cursor next{0, 0, 0};
    Unit xa = unit_at(next), xb;
    load_w(xa, lane, A);  // weights do not depend on the preceding kernel
    stage(a, xs);         // the plane does
    load_x(a, xs, xa, lane, A);
    Cursor ca = next, cb;
    advance(next);

    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;

    // finish the unit at cursor q (tile end: park the row sums; block end:
    // meet the CTA and run the epilogue)
    auto finish = [&](const Cursor &q) {
        if (q.c != nch - 1) return;
        const float v = reduce8(acc, lane);
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
        const int j = w + q.m * W;
        if ((lane & 3) == 0) sums[q.k & 1][j][lane >> 2] = v;
        if (q.m != tiles - 1) return;
        asm volatile("bar.sync 2, %0;" ::"r"(blockDim.x) : "memory");
        if (w != q.k % W) return;
        const int blk = (int)blockIdx.x + q.k * (int)gridDim.x;
        const float g = sums[q.k & 1][2 * (lane >> 3)][lane & 7];
        const float u = sums[q.k & 1][2 * (lane >> 3) + 1][lane & 7];
        const float act = (g / (1.0f + expf(-g))) * u;
        L.act[(size_t)blk * 32 + lane] = act;
        quantize_block(act, L, blk, lane);
    };

    for (int u = 0; u < n_units; u += 2) {
        const bool has_b = u + 1 < n_units;
        if (has_b) {
            cb = next;
            xb = unit_at(next);
            load_w(xb, lane, B);
            load_x(a, xs, xb, lane, B);
            advance(next);
        }
        compute<false>(a, a.part[0], A, xa, lane, acc);
        finish(ca);
        if (!has_b) break;
        const bool has_a = u + 2 < n_units;
        if (has_a) {
            ca = next;
            xa = unit_at(next);
            load_w(xa, lane, A);
            load_x(a, xs, xa, lane, A);
            advance(next);
        }
        compute<false>(a, a.part[0], B, xb, lane, acc);
        finish(cb);
    }
}

// One kernel per format.  Unlike the single-token GEMV (gemv.cu), here the
// per-format kernels measured faster in a PDL decode chain (rms -> gate||up
// -> down: 30.5 us against 33.9 us with all three formats in one kernel).
template <int FMT>
__global__ void __launch_bounds__(32 * kMaxCtaSplits, 1)
    gateup_kernel(const __grid_constant__ GateUpLaunch L)
{
    extern __shared__ __align__(16) uint8_t xs[];  // the q8 plane
    griddep_launch_dependents();
    run_gateup<FMT>(L, xs, threadIdx.x & 31);
}

using KernelFn = void (*)(GateUpLaunch);

KernelFn gateup_kernel_for(int fmt)
{
    return fmt == 6 ? gateup_kernel<6> : fmt == 5 ? gateup_kernel<5> : gateup_kernel<4>;
}

}  // namespace

cudaError_t launch_gateup(const GateUpLaunch &L, int ctas, cudaStream_t st)
{
    return launch_maybe_pdl(gateup_kernel_for(L.g.part[0].fmt), dim3((unsigned)ctas),
                            dim3(32 * L.wpb), (size_t)L.g.q8_bytes, L.g.pdl, st, L);
}

int gateup_ctas_per_sm(int fmt, int warps_per_cta, size_t smem)
{
    int blocks = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &blocks, gateup_kernel_for(fmt), 32 * warps_per_cta, smem);
    if (e != cudaSuccess) cuda_fail("gate||up occupancy", e);
    return e == cudaSuccess ? blocks : 0;
}

bool gateup_opt_in(size_t max_plane)
{
    cudaError_t e = cudaSuccess;
    for (int fmt : {6, 4, 5})
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gateup_kernel_for(fmt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)max_plane);
    if (e != cudaSuccess) cuda_fail("gate||up shared-memory opt-in", e);
    return e == cudaSuccess;
}

}  // namespace mq
