// gemv.cu -- batch-1 decode GEMV of repacked q6_K / q4_K weights against a
// q8 activation plane (the "MMVQ" of the minfer pages), for sm_103a.
//
// What is computed (page "74 · D4-2 — B0 latent correctness fix", §3.2
// Excerpt C; page "67 · D3", §3.2): for every 16-weight (q6_K) or 32-weight
// (q4_K) sub-block an exact int32 dot product of the weight codes with the
// int8 activation codes (dp4a), then an f32 combine with the fp16 block
// scale(s), the int8/6-bit sub-block scale(s) and the fp16 activation scale.
//
// How (GB300 design; layout.h describes the byte order):
//   * The work is a pure HBM stream (page "67 · D3", §2.1: 93.4% of decode
//     kernel time is weight streaming), so there are no tensor cores and no
//     shared-memory staging: each lane issues 14 (q6_K) or 13 (q4_K)
//     independent 16-byte loads per chunk (224 B in flight per lane), every
//     warp-wide load instruction covers 512 contiguous bytes, and the weight
//     loads bypass L1 (ld.global.nc.L1::no_allocate) because each byte is used
//     once.
//   * A warp owns one work item: 8 rows (a tile) x a contiguous range of
//     4-super-block chunks.  Lane i owns unit i of every chunk for all 8 rows,
//     so its activation codes (32 B + fp16 scale) are loaded once per chunk
//     and reused 8 times from registers.
//   * Per row the lane accumulates in f32 over its chunks in ascending order;
//     the 8 row sums are then reduced across the warp with a fixed butterfly
//     (9 shuffles).  With S > 1 splits per tile the warp writes its 8
//     partials to a workspace and the split that arrives last (atomic ticket,
//     no waiting) adds the S partials in ascending split order: the result
//     does not depend on which split finishes first.  Page "74 · D4-2" (§2,
//     §6) is why the host proves, before launch, that the splits cover every
//     chunk exactly once.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "layout.h"

namespace mq {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kLo4 = 0x0f0f0f0fu;
constexpr uint32_t kOnes = 0x01010101u;

// 16-byte streaming load: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const uint8_t *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const uint8_t *p)
{
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int k)
{
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

__device__ __forceinline__ float half_lo(uint32_t w)
{
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t w)
{
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// Activation unit: the 32 int8 codes of q8 block U and its fp16 scale.
struct Act {
    uint4 xa, xb;  // codes 0..15, 16..31
    float d8;
};

__device__ __forceinline__ Act load_act(const GemvLaunch &a, int U)
{
    Act x;
    const uint4 *qs = reinterpret_cast<const uint4 *>(a.q8 + (size_t)U * 32);
    x.xa = __ldg(qs);
    x.xb = __ldg(qs + 1);
    const unsigned short dh =
        __ldg(reinterpret_cast<const unsigned short *>(a.q8 + a.q8_d_off) + U);
    x.d8 = __half2float(__ushort_as_half(dh));
    return x;
}

__device__ __forceinline__ int sum16(const uint4 &v)
{
    int s = __dp4a((int)v.x, (int)kOnes, 0);
    s = __dp4a((int)v.y, (int)kOnes, s);
    s = __dp4a((int)v.z, (int)kOnes, s);
    return __dp4a((int)v.w, (int)kOnes, s);
}

// ---- q6_K: one lane, one chunk, 8 rows --------------------------------------
// Unit codes for row r: QL word m holds the low 4 bits of weights 4m..4m+3
// (low nibbles) and 16+4m..16+4m+3 (high nibbles); QH word h byte k holds
// the 2-bit highs of weights 16h+4m+k at bits 2m.  q - 32 is never formed:
// isum = dot(q, x) - 32 * sum(x) is the same integer.
template <bool SUBDOTS>
__device__ __forceinline__ void q6k_chunk(const GemvLaunch &a, const uint8_t *seg, int cb,
                                          int lane, int c, int t, float (&acc)[8])
{
    const int nu = 8 * cb;
    const Act x = load_act(a, 32 * c + lane);
    const int xs0 = sum16(x.xa), xs1 = sum16(x.xb);

    uint4 ql[8], qh[4];
#pragma unroll
    for (int r = 0; r < 8; ++r) ql[r] = ld_stream16(seg + ((size_t)r * nu + lane) * 16);
#pragma unroll
    for (int p = 0; p < 4; ++p)
        qh[p] = ld_stream16(seg + (size_t)kQ6kQH * cb + ((size_t)p * nu + lane) * 16);
    const uint4 sc = ld_stream16(seg + (size_t)kQ6kSC * cb + (size_t)lane * 16);
    const uint4 dd = ld_stream16(seg + (size_t)kQ6kD * cb + (size_t)(lane >> 3) * 16);

#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const uint32_t h0 = (r & 1) ? qh[r >> 1].z : qh[r >> 1].x;
        const uint32_t h1 = (r & 1) ? qh[r >> 1].w : qh[r >> 1].y;
        int dot0 = 0, dot1 = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint32_t w = word(ql[r], m);
            const uint32_t q0 = (w & kLo4) | (((h0 >> (2 * m)) & 0x03030303u) << 4);
            const uint32_t q1 = ((w >> 4) & kLo4) | (((h1 >> (2 * m)) & 0x03030303u) << 4);
            dot0 = __dp4a((int)q0, (int)word(x.xa, m), dot0);
            dot1 = __dp4a((int)q1, (int)word(x.xb, m), dot1);
        }
        const int isum0 = dot0 - 32 * xs0;
        const int isum1 = dot1 - 32 * xs1;
        const uint32_t scw = word(sc, r >> 1) >> (16 * (r & 1));
        const int sc0 = (int)(int8_t)(scw & 0xffu);
        const int sc1 = (int)(int8_t)((scw >> 8) & 0xffu);
        if (SUBDOTS) {
            const int row = t * kTileRows + r;
            if (row < a.rows) {
                const int blk = kChunkBlocks * c + (lane >> 3), p = lane & 7;
                int32_t *o = a.isums + ((size_t)row * a.nb + blk) * 16 + 2 * p;
                o[0] = isum0;
                o[1] = isum1;
            }
        } else {
            const float d = (r & 1) ? half_hi(word(dd, r >> 1)) : half_lo(word(dd, r >> 1));
            acc[r] = fmaf(d * x.d8, (float)(sc0 * isum0 + sc1 * isum1), acc[r]);
        }
    }
}

// ---- q4_K: one lane, one chunk, 8 rows --------------------------------------
template <bool SUBDOTS>
__device__ __forceinline__ void q4k_chunk(const GemvLaunch &a, const uint8_t *seg, int cb,
                                          int lane, int c, int t, float (&acc)[8])
{
    const int nu = 8 * cb;
    const int U = 32 * c + lane;
    const Act x = load_act(a, U);
    const int qsum = __ldg(reinterpret_cast<const int *>(a.q8 + a.q8_sum_off) + U);

    uint4 qs[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) qs[r] = ld_stream16(seg + ((size_t)r * nu + lane) * 16);
    const uint8_t *smp = seg + (size_t)kQ4kSM * cb + (size_t)lane * 4;
    const uint32_t s0 = ld_stream4(smp);
    const uint32_t s1 = ld_stream4(smp + (size_t)nu * 4);
    const uint32_t s2 = ld_stream4(smp + (size_t)nu * 8);
    const uint8_t *dmp = seg + (size_t)kQ4kDM * cb + (size_t)(lane >> 3) * 32;
    const uint4 dm0 = ld_stream16(dmp);
    const uint4 dm1 = ld_stream16(dmp + 16);

#pragma unroll
    for (int r = 0; r < 8; ++r) {
        int dot = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint32_t w = word(qs[r], m);
            dot = __dp4a((int)(w & kLo4), (int)word(x.xa, m), dot);
            dot = __dp4a((int)((w >> 4) & kLo4), (int)word(x.xb, m), dot);
        }
        if (SUBDOTS) {
            const int row = t * kTileRows + r;
            if (row < a.rows) {
                const int blk = kChunkBlocks * c + (lane >> 3), k = lane & 7;
                a.isums[((size_t)row * a.nb + blk) * 8 + k] = dot;
            }
        } else {
            const int hi = (int)((s2 >> (4 * r)) & 15u);
            const int sc = (int)((s0 >> (4 * r)) & 15u) | ((hi & 3) << 4);
            const int mn = (int)((s1 >> (4 * r)) & 15u) | ((hi >> 2) << 4);
            const uint32_t dmw = word(r < 4 ? dm0 : dm1, r & 3);
            const float d = half_lo(dmw), dmin = half_hi(dmw);
            const float term = fmaf(d, (float)(sc * dot), -dmin * (float)(mn * qsum));
            acc[r] = fmaf(x.d8, term, acc[r]);
        }
    }
}

// Reduce acc[0..7] over the 32 lanes; returns the sum of row (lane >> 2) in
// every lane (the 4 lanes of a group hold the same value).
__device__ __forceinline__ float reduce8(const float (&acc)[8], int lane)
{
    float v4[4];
    const bool b4 = lane & 16;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = b4 ? acc[k] : acc[k + 4];
        const float keep = b4 ? acc[k + 4] : acc[k];
        v4[k] = keep + __shfl_xor_sync(kFull, send, 16);
    }
    float v2[2];
    const bool b3 = lane & 8;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = b3 ? v4[k] : v4[k + 2];
        const float keep = b3 ? v4[k + 2] : v4[k];
        v2[k] = keep + __shfl_xor_sync(kFull, send, 8);
    }
    const bool b2 = lane & 4;
    float v = (b2 ? v2[1] : v2[0]) + __shfl_xor_sync(kFull, b2 ? v2[0] : v2[1], 4);
    v += __shfl_xor_sync(kFull, v, 2);
    v += __shfl_xor_sync(kFull, v, 1);
    return v;
}

template <int FMT, bool SUBDOTS>  // FMT 6 = q6_K, 4 = q4_K
__global__ void __launch_bounds__(32 * kGemvWarpsPerBlock) gemv_kernel(const GemvLaunch a)
{
    const int lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * kGemvWarpsPerBlock + (threadIdx.x >> 5);
    if (item >= a.n_items) return;  // whole warp; the kernel has no block barrier
    const int t = (int)(item / a.splits);
    const int s = (int)(item - (long long)t * a.splits);
    const int c0 = s * a.cps;
    const int c1 = min(c0 + a.cps, a.nchunks);
    const uint8_t *tile = a.W + (size_t)t * a.tile_bytes;
    constexpr int kChunkBytes = (FMT == 6 ? kQ6kChunkPerBlock : kQ4kChunkPerBlock) * kChunkBlocks;

    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    for (int c = c0; c < c1; ++c) {
        const int cb = min(kChunkBlocks, a.nb - kChunkBlocks * c);
        if (lane < 8 * cb) {
            const uint8_t *seg = tile + (size_t)c * kChunkBytes;
            if (FMT == 6)
                q6k_chunk<SUBDOTS>(a, seg, cb, lane, c, t, acc);
            else
                q4k_chunk<SUBDOTS>(a, seg, cb, lane, c, t, acc);
        }
    }
    if (SUBDOTS) return;

    const float v = reduce8(acc, lane);
    const int row0 = t * kTileRows;
    if (a.splits == 1) {
        if ((lane & 3) == 0 && row0 + (lane >> 2) < a.rows) a.y[row0 + (lane >> 2)] = v;
        return;
    }
    // split-K: lane 0 publishes the 8 partials, then takes a ticket.
    float part[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) part[k] = __shfl_sync(kFull, v, 4 * k);
    int last = 0;
    if (lane == 0) {
        float4 *dst = reinterpret_cast<float4 *>(a.ws_part + ((size_t)s * a.ntiles + t) * 8);
        dst[0] = make_float4(part[0], part[1], part[2], part[3]);
        dst[1] = make_float4(part[4], part[5], part[6], part[7]);
        __threadfence();
        const unsigned prev = atomicAdd(a.ws_cnt + t, 1u);
        last = prev == (unsigned)(a.splits - 1);
    }
    last = __shfl_sync(kFull, last, 0);
    if (!last) return;
    __threadfence();
    if (lane < 8) {
        float sum = 0.0f;
        for (int k = 0; k < a.splits; ++k)
            sum += __ldcg(a.ws_part + ((size_t)k * a.ntiles + t) * 8 + lane);
        if (row0 + lane < a.rows) a.y[row0 + lane] = sum;
    }
    if (lane == 0) a.ws_cnt[t] = 0u;  // ready for the next call
}

template <int FMT, bool SUBDOTS>
cudaError_t launch(const GemvLaunch &a, cudaStream_t st)
{
    const long long blocks = (a.n_items + kGemvWarpsPerBlock - 1) / kGemvWarpsPerBlock;
    gemv_kernel<FMT, SUBDOTS><<<(unsigned)blocks, 32 * kGemvWarpsPerBlock, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_q6k(const GemvLaunch &a, cudaStream_t st) { return launch<6, false>(a, st); }
cudaError_t launch_gemv_q4k(const GemvLaunch &a, cudaStream_t st) { return launch<4, false>(a, st); }
cudaError_t launch_subdots_q6k(const GemvLaunch &a, cudaStream_t st) { return launch<6, true>(a, st); }
cudaError_t launch_subdots_q4k(const GemvLaunch &a, cudaStream_t st) { return launch<4, true>(a, st); }

}  // namespace mq
