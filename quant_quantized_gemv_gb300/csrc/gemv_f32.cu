// gemv_f32.cu -- batch-1 GEMV of repacked q6_K weights against an f32
// activation row: the dequantize-and-FMA family that the minfer pages keep
// beside the q8 MMVQ (page "67 · D3: 14B decode attribution + the D3b
// bitwise MMVQ triple", §2.3 and §3.3: the "padded f32" kernels, which won
// below od*id ~ 24M on GB10 because their reads were coalesced where the
// q8 kernel's unit loads were scattered).  No q8 producer runs before it.
//
// What is computed: y_r = sum_e w_{r,e} x_e with w = f16(d) * sc * (q - 32),
// in f32: per 16-weight sub-block two FMA chains over its even and odd
// weights, s = s_even + s_odd, then acc_r += (d * sc) * s.
//
// How (GB300 design).  The weights are the q8 path's repacked layout
// (layout.h), streamed the same way: tiles of 8 rows, chunks of 4
// super-blocks, lane i owns unit i (32 columns) of a chunk for all 8 rows,
// one register buffer at 128 registers so that 16 warps share an SM (two
// buffers at 168 registers and 12 warps measured slower: 149 against 125 us
// on the 152064 x 5120 head, 21.4 against 19.9 us on 3584 x 18944).
// What differs is the activation: 4 bytes per value instead of ~1.06, so
// every CTA stages the whole row in shared memory (up to 57856 values) and
// each activation value is read from there once per tile row.  The staged
// row is stored with the 16-byte slots of each unit XOR-swizzled by the
// unit index (slot j of unit U at U*8 + (j ^ (U & 7))): the 8 lanes of a
// shared-memory phase then hit 8 different slots, so the loads are free of
// bank conflicts although lanes read 128 bytes apart.  A code q in 0..63
// becomes the float q - 32 without a conversion instruction: the byte is
// placed in the low mantissa bits of 2^23 (0x4B0000qq = 2^23 + q, a byte
// permute) and 2^23 + 32 is subtracted, exactly.  The subtraction and the
// FMA run on pairs of values (Blackwell's f32x2 add and fma), each pair
// accumulating its own partial sum of the sub-block; the two are added
// before the scale is applied.  Measured against one value per instruction
// (two-buffer form): 149 against 167 us on the 152064 x 5120 head, 21.2
// against 23.6 us on 3584 x 18944.
//
// Plans are the single-token GEMV's (whole tiles per warp, or 2..12 splits
// of a tile as the warps of one CTA meeting in shared memory); there is no
// workspace mode.  Split sums are added in ascending split order.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemv_common.cuh"
#include "kernels.h"
#include "layout.h"
#include "prefetch.cuh"

namespace mq {
namespace {

using namespace gemv_detail;

// Stage x (cols floats, after the producer finished) with the swizzle
// above, then meet at named barrier 1 (every warp of the CTA calls this).
__device__ __forceinline__ void stage_x(const GemvLaunch &a, uint4 *xs)
{
    griddep_wait();
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q8);
    const int n16 = (int)(a.q8_bytes >> 4);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) {
        const int U = i >> 3;
        copy16_async(xs + ((i & ~7) | ((i ^ U) & 7)), src + i);
    }
    copy_async_wait_all();
    asm volatile("bar.sync 1, %0;" ::"r"(blockDim.x) : "memory");
}

// Packed f32 pairs (Blackwell f32x2 arithmetic): one instruction adds or
// multiplies-adds two lanes of values held in a 64-bit register pair.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    unsigned long long v;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(lo), "f"(hi));
    return v;
}
__device__ __forceinline__ float sum2(unsigned long long v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// 2^23 + code for bytes B and B + 1 of w, as a pair
template <int B>
__device__ __forceinline__ unsigned long long biased2(uint32_t w)
{
    return pack2(__int_as_float((int)__byte_perm(w, 0x4B000000u, 0x7540u | B)),
                 __int_as_float((int)__byte_perm(w, 0x4B000000u, 0x7540u | (B + 1))));
}

// Codes of row r, weights 16h + 4m .. 16h + 4m + 3 (one per byte).
template <int H>
__device__ __forceinline__ uint32_t codes_half(const Q6kW &R, int r, int m)
{
    const uint32_t hw = H == 0 ? ((r & 1) ? R.qh[r >> 1].z : R.qh[r >> 1].x)
                               : ((r & 1) ? R.qh[r >> 1].w : R.qh[r >> 1].y);
    const uint32_t w = H == 0 ? word(R.ql[r], m) : (word(R.ql[r], m) >> 4);
    return (w & kLo4) | (((hw >> (2 * m)) & 0x03030303u) << 4);
}

// One chunk of 8 rows against the lane's 32 activation values: sub-block
// half H (weights 16H .. 16H + 15 of the unit) for every row, in pairs.
template <int H>
__device__ __forceinline__ void compute_half(const Q6kW &R, const uint4 *xu, int sw, float (&acc)[8])
{
    const unsigned long long bias = pack2(-8388640.0f, -8388640.0f);  // -(2^23 + 32)
    unsigned long long s[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = 0ull;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint4 xv = xu[(4 * H + m) ^ sw];  // values 16H + 4m .. 16H + 4m + 3
        const unsigned long long x01 = pack2(__uint_as_float(xv.x), __uint_as_float(xv.y));
        const unsigned long long x23 = pack2(__uint_as_float(xv.z), __uint_as_float(xv.w));
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint32_t q = codes_half<H>(R, r, m);
            s[r] = fma2(add2(biased2<0>(q), bias), x01, s[r]);
            s[r] = fma2(add2(biased2<2>(q), bias), x23, s[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        int sc0, sc1;
        float d;
        q6k_scales(R, r, sc0, sc1, d);
        acc[r] = fmaf(d * (float)(H == 0 ? sc0 : sc1), sum2(s[r]), acc[r]);
    }
}

__device__ __forceinline__ void compute_f32(const Q6kW &R, const uint4 *xs, const Unit &x, int lane,
                                            float (&acc)[8])
{
    if (!x.active) return;  // zero weights and no activation: nothing to add
    const int U = 32 * x.c + lane;
    const uint4 *xu = xs + (size_t)U * 8;
    compute_half<0>(R, xu, U & 7, acc);
    compute_half<1>(R, xu, U & 7, acc);
}

// Tile t finished for this warp: write it (whole tile) or combine it with
// the tile's other splits (the warps of this CTA, ascending split order).
__device__ __forceinline__ void flush_f32(const GemvLaunch &a, const GemvPart &P, int t,
                                          float (&acc)[8], int lane)
{
    __shared__ float cta_part[kMaxCtaSplits][8];
    const float v = reduce8(acc, lane);
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    const int row0 = t * kTileRows;
    if (a.splits == 1) {
        if ((lane & 3) == 0 && row0 + (lane >> 2) < P.rows) P.y[row0 + (lane >> 2)] = v;
        return;
    }
    const int s = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float pk = __shfl_sync(kFull, v, 4 * k);
        if (lane == k) cta_part[s][k] = pk;
    }
    __syncthreads();
    if (s == 0 && lane < 8) {
        float sum = 0.0f;
        for (int j = 0; j < a.splits; ++j) sum += cta_part[j][lane];
        if (row0 + lane < P.rows) P.y[row0 + lane] = sum;
    }
}

__device__ __forceinline__ void run_f32(const GemvLaunch &a, const GemvPart &P, uint4 *xs, int u0,
                                        int u1, int lane)
{
    constexpr int kChunkBytes = kQ6kChunkPerBlock * kChunkBlocks;
    const int nch = a.nchunks;
    Q6kW A;
    int t = u0 / nch, c = u0 - t * nch;  // position of the next chunk to load
    Unit xa = locate(a, P, t, c, lane, kChunkBytes);
    load_w(xa, lane, A);  // weights do not depend on the preceding kernel
    stage_x(a, xs);       // the activation does
    if (++c == nch) { c = 0; ++t; }
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    for (int u = u0; u < u1; ++u) {
        const int tcur = xa.t;
        // Lane 0 asks L2 for chunk u + 1 (one bulk prefetch of its contiguous
        // bytes) before chunk u computes, so the register loads issued after
        // the compute find it there: 7B ffn_down 20.0 -> 18.5 us, 14B
        // ffn_down 32.4 -> 28.0 us, head 125.5 -> 122.5 us (shapes with one
        // chunk per warp issue none).
        if (lane == 0 && u + 1 < u1) {
            const Unit nx = locate(a, P, t, c, 0, kChunkBytes);
            prefetch_l2(nx.seg, (unsigned)(kChunkBytes / kChunkBlocks * nx.cb));
        }
        compute_f32(A, xs, xa, lane, acc);
        const bool more = u + 1 < u1;
        if (more) {  // the next chunk into the same registers
            xa = locate(a, P, t, c, lane, kChunkBytes);
            load_w(xa, lane, A);
            if (++c == nch) { c = 0; ++t; }
        }
        if (!more || xa.t != tcur) flush_f32(a, P, tcur, acc, lane);
    }
}

__global__ void __maxnreg__(kGemvMaxRegs)
    gemv_q6k_f32_kernel(const __grid_constant__ GemvLaunch a)
{
    extern __shared__ __align__(16) uint4 xs[];  // the activation row, swizzled
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    griddep_launch_dependents();
    if (item >= a.n_items) {  // only in the last CTA of a whole-tile grid
        stage_x(a, xs);
        return;
    }
    const GemvPart &P = a.part[0];
    const int nch = a.nchunks;
    int u0, u1;
    if (a.splits > 1) {
        const int tt = item / a.splits, s = item - tt * a.splits;
        u0 = tt * nch + s * a.cps;
        u1 = tt * nch + min(s * a.cps + a.cps, nch);
    } else {
        u0 = item * a.tpi * nch;
        u1 = min(u0 + a.tpi * nch, P.ntiles * nch);
    }
    run_f32(a, P, xs, u0, u1, lane);
}

}  // namespace

cudaError_t launch_gemv_f32(const GemvLaunch &a, cudaStream_t st)
{
    const int warps = gemv_cta_warps(a.splits);
    const long long blocks = (a.n_items + warps - 1) / warps;
    return launch_maybe_pdl(gemv_q6k_f32_kernel, dim3((unsigned)blocks), dim3(32 * warps),
                            (size_t)a.q8_bytes, a.pdl, st, a);
}

int gemv_f32_ctas_per_sm(int warps_per_cta, size_t smem)
{
    int blocks = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &blocks, gemv_q6k_f32_kernel, 32 * warps_per_cta, smem);
    if (e != cudaSuccess) cuda_fail("f32 GEMV occupancy", e);
    return e == cudaSuccess ? blocks : 0;
}

size_t gemv_f32_max_x_bytes()
{
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int limit = optin - 1024;  // room for the kernel's static shared memory
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_q6k_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (e != cudaSuccess) {
        cuda_fail("f32 GEMV shared-memory opt-in", e);
        return 0;
    }
    return (size_t)limit & ~(size_t)15;
}

}  // namespace mq
