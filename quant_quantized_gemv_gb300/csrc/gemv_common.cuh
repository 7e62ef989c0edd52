// gemv_common.cuh -- device pieces shared by the single-token GEMV (gemv.cu)
// and the small-batch GEMV (gemv_batch.cu): streaming loads, chunk location,
// the per-lane weight registers of one chunk and their decoding into dp4a
// operands, and the 8-row warp reduction.  Internal to the library.
//
// A lane owns one unit (32 weights of q6_K, 64 of q4_K; page "74 · D4-2 — B0
// latent correctness fix", §2) of the current chunk for the 8 rows of a
// tile; layout.h gives the byte order these loads and decoders follow.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.h"
#include "layout.h"

namespace mq {
namespace gemv_detail {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kLo4 = 0x0f0f0f0fu;
constexpr uint32_t kOnes = 0x01010101u;

// 16-byte streaming load: read-only path, no L1 allocation (each weight
// byte is used once).
__device__ __forceinline__ uint4 ld_stream16(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const uint8_t *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
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

// Sum of the 16 int8 codes in v.
__device__ __forceinline__ int sum16(const uint4 &v)
{
    int s = __dp4a((int)v.x, (int)kOnes, 0);
    s = __dp4a((int)v.y, (int)kOnes, s);
    s = __dp4a((int)v.z, (int)kOnes, s);
    return __dp4a((int)v.w, (int)kOnes, s);
}

struct Unit {
    const uint8_t *seg;  // chunk base
    int t, c, cb;        // tile, chunk within the tile, blocks in the chunk
    bool active;         // this lane owns a unit of the chunk
};

__device__ __forceinline__ Unit locate(const GemvLaunch &a, const GemvPart &P, int t, int c,
                                      int lane, int chunk_bytes)
{
    Unit x;
    x.t = t;
    x.c = c;
    x.cb = min(kChunkBlocks, a.nb - kChunkBlocks * c);
    x.seg = P.W + (size_t)t * P.tile_bytes_div16 * 16 + (size_t)c * chunk_bytes;
    x.active = lane < 8 * x.cb;
    return x;
}

// ---- q6_K ------------------------------------------------------------------
// Unit codes for row r: QL word m holds the low 4 bits of weights 4m..4m+3
// (low nibbles) and 16+4m..16+4m+3 (high nibbles); QH word h byte k holds
// the 2-bit highs of weights 16h+4m+k at bits 2m.  q - 32 is never formed:
// isum = dot(q, x) - 32 * sum(x) is the same integer.
struct Q6kW {
    uint4 ql[8], qh[4], sc, dd;  // weights of one chunk (8 rows)
};

__device__ __forceinline__ void load_w(const Unit &x, int lane, Q6kW &R)
{
    const int nu = 8 * x.cb, cb = x.cb;
    if (x.active) {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.ql[r] = ld_stream16(x.seg + ((size_t)r * nu + lane) * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p)
            R.qh[p] = ld_stream16(x.seg + (size_t)kQ6kQH * cb + ((size_t)p * nu + lane) * 16);
        R.sc = ld_stream16(x.seg + (size_t)kQ6kSC * cb + (size_t)lane * 16);
        R.dd = ld_stream16(x.seg + (size_t)kQ6kD * cb + (size_t)(lane >> 3) * 16);
    } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.ql[r] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int p = 0; p < 4; ++p) R.qh[p] = make_uint4(0, 0, 0, 0);
        R.sc = R.dd = make_uint4(0, 0, 0, 0);
    }
}

// The unsigned 6-bit codes of row r, weights 4m..4m+3 (q0, sub-block 0 of
// the unit) and 16+4m..16+4m+3 (q1, sub-block 1), one code per byte.
__device__ __forceinline__ void q6k_codes(const Q6kW &R, int r, int m, uint32_t &q0, uint32_t &q1)
{
    const uint32_t h0 = (r & 1) ? R.qh[r >> 1].z : R.qh[r >> 1].x;
    const uint32_t h1 = (r & 1) ? R.qh[r >> 1].w : R.qh[r >> 1].y;
    const uint32_t w = word(R.ql[r], m);
    q0 = (w & kLo4) | (((h0 >> (2 * m)) & 0x03030303u) << 4);
    q1 = ((w >> 4) & kLo4) | (((h1 >> (2 * m)) & 0x03030303u) << 4);
}

// Row r's two int8 sub-block scales and fp16 block scale d.
__device__ __forceinline__ void q6k_scales(const Q6kW &R, int r, int &sc0, int &sc1, float &d)
{
    const uint32_t scw = word(R.sc, r >> 1) >> (16 * (r & 1));
    sc0 = (int)(int8_t)(scw & 0xffu);
    sc1 = (int)(int8_t)((scw >> 8) & 0xffu);
    d = (r & 1) ? half_hi(word(R.dd, r >> 1)) : half_lo(word(R.dd, r >> 1));
}

// ---- q4_K ------------------------------------------------------------------
struct Q4kW {
    uint4 qs[8], dm0, dm1;       // nibbles of 8 rows; (d, dmin) of 8 rows
    uint32_t s0, s1, s2;         // 6-bit scales and mins of 8 rows, packed
};

// The QS, SM and DM planes (q4_K, and q5_K at other SM / DM offsets).
template <int SM, int DM>
__device__ __forceinline__ void load_w_q4like(const Unit &x, int lane, Q4kW &R)
{
    const int nu = 8 * x.cb, cb = x.cb;
    if (x.active) {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.qs[r] = ld_stream16(x.seg + ((size_t)r * nu + lane) * 16);
        const uint8_t *smp = x.seg + (size_t)SM * cb + (size_t)lane * 4;
        R.s0 = ld_stream4(smp);
        R.s1 = ld_stream4(smp + (size_t)nu * 4);
        R.s2 = ld_stream4(smp + (size_t)nu * 8);
        const uint8_t *dmp = x.seg + (size_t)DM * cb + (size_t)(lane >> 3) * 32;
        R.dm0 = ld_stream16(dmp);
        R.dm1 = ld_stream16(dmp + 16);
    } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.qs[r] = make_uint4(0, 0, 0, 0);
        R.s0 = R.s1 = R.s2 = 0;
        R.dm0 = R.dm1 = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void load_w(const Unit &x, int lane, Q4kW &R)
{
    load_w_q4like<kQ4kSM, kQ4kDM>(x, lane, R);
}

// Row r's codes for words m of the unit: weights 4m..4m+3 (lo, against the
// activation codes xa) and 16+4m..16+4m+3 (hi, against xb), one per byte.
__device__ __forceinline__ void codes(const Q4kW &R, int r, int m, uint32_t &lo, uint32_t &hi)
{
    const uint32_t w = word(R.qs[r], m);
    lo = w & kLo4;
    hi = (w >> 4) & kLo4;
}

// Row r's 6-bit scale and min and fp16 d, dmin.
__device__ __forceinline__ void q4k_scales(const Q4kW &R, int r, int &sc, int &mn, float &d,
                                           float &dmin)
{
    const int hi = (int)((R.s2 >> (4 * r)) & 15u);
    sc = (int)((R.s0 >> (4 * r)) & 15u) | ((hi & 3) << 4);
    mn = (int)((R.s1 >> (4 * r)) & 15u) | ((hi >> 2) << 4);
    const uint32_t dmw = word(r < 4 ? R.dm0 : R.dm1, r & 3);
    d = half_lo(dmw);
    dmin = half_hi(dmw);
}

// ---- q5_K: q4_K's fields plus each code's fifth bit -------------------------
struct Q5kW : Q4kW {
    uint4 qh[2];  // fifth-bit words H of rows 0..3 and 4..7
};

__device__ __forceinline__ void load_w(const Unit &x, int lane, Q5kW &R)
{
    load_w_q4like<kQ5kSM, kQ5kDM>(x, lane, R);
    if (x.active) {
        const uint8_t *hp = x.seg + (size_t)kQ5kQH * x.cb + (size_t)lane * 32;
        R.qh[0] = ld_stream16(hp);
        R.qh[1] = ld_stream16(hp + 16);
    } else {
        R.qh[0] = R.qh[1] = make_uint4(0, 0, 0, 0);
    }
}

// As for q4_K, with bit 4 of every byte taken from the fifth-bit word.
__device__ __forceinline__ void codes(const Q5kW &R, int r, int m, uint32_t &lo, uint32_t &hi)
{
    const uint32_t H = word(R.qh[r >> 2], r & 3);
    const uint32_t w = word(R.qs[r], m);
    lo = (w & kLo4) | (((H >> m) & 0x01010101u) << 4);
    hi = ((w >> 4) & kLo4) | (((H >> (m + 4)) & 0x01010101u) << 4);
}

// ---- single-token activation codes and chunk compute ------------------------
// xs: the q8 plane staged in shared memory, or null to read it from global
// memory (coherent loads: under programmatic dependent launch the plane may
// have been written by the kernel this one overlaps, and the non-coherent
// path may be hoisted above the grid-dependency wait).  With SUBDOTS the
// integer sub-block dots are written to a.isums instead of being combined.
// ---- q6_K ------------------------------------------------------------------
struct Q6kRegs : Q6kW {
    uint4 xa, xb;        // activation codes 0..15, 16..31 of the unit
    unsigned short dh;   // activation fp16 scale
};

__device__ __forceinline__ void load_x(const GemvLaunch &a, const uint8_t *xs, const Unit &x,
                                       int lane, Q6kRegs &R)
{
    if (x.active) {
        const int U = 32 * x.c + lane;
        if (!xs) {  // split plans: straight from L2, coherent (see the file comment)
            const uint4 *qs = reinterpret_cast<const uint4 *>(a.q8 + (size_t)U * 32);
            R.xa = __ldcg(qs);
            R.xb = __ldcg(qs + 1);
            R.dh = __ldcg(reinterpret_cast<const unsigned short *>(a.q8 + a.q8_d_off) + U);
            return;
        }
        const uint4 *qs = reinterpret_cast<const uint4 *>(xs + (size_t)U * 32);
        R.xa = qs[0];
        R.xb = qs[1];
        R.dh = reinterpret_cast<const unsigned short *>(xs + a.q8_d_off)[U];
    } else {
        R.xa = R.xb = make_uint4(0, 0, 0, 0);
        R.dh = 0;
    }
}

template <bool SUBDOTS>
__device__ __forceinline__ void compute(const GemvLaunch &a, const GemvPart &P, const Q6kRegs &R,
                                        const Unit &x, int lane, float (&acc)[8])
{
    const float d8 = __half2float(__ushort_as_half(R.dh));
    const int xs0 = sum16(R.xa), xs1 = sum16(R.xb);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        int dot0 = 0, dot1 = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t q0, q1;
            q6k_codes(R, r, m, q0, q1);
            dot0 = __dp4a((int)q0, (int)word(R.xa, m), dot0);
            dot1 = __dp4a((int)q1, (int)word(R.xb, m), dot1);
        }
        const int isum0 = dot0 - 32 * xs0;
        const int isum1 = dot1 - 32 * xs1;
        int sc0, sc1;
        float d;
        q6k_scales(R, r, sc0, sc1, d);
        if (SUBDOTS) {
            const int row = x.t * kTileRows + r;
            if (x.active && row < P.rows) {
                const int blk = kChunkBlocks * x.c + (lane >> 3), p = lane & 7;
                int32_t *o = a.isums + ((size_t)row * a.nb + blk) * 16 + 2 * p;
                o[0] = isum0;
                o[1] = isum1;
            }
        } else {
            acc[r] = fmaf(d * d8, (float)(sc0 * isum0 + sc1 * isum1), acc[r]);
        }
    }
}

// ---- q4_K and q5_K -----------------------------------------------------------
struct XSum {                    // the unit's activation codes, scale and code sum
    uint4 xa, xb;
    unsigned short dh;
    int qsum;
};
struct Q4kRegs : Q4kW, XSum {};
struct Q5kRegs : Q5kW, XSum {};

__device__ __forceinline__ void load_x(const GemvLaunch &a, const uint8_t *xs, const Unit &x,
                                       int lane, XSum &R)
{
    if (x.active) {
        const int U = 32 * x.c + lane;
        if (!xs) {  // split plans: straight from L2, coherent (see the file comment)
            const uint4 *qs = reinterpret_cast<const uint4 *>(a.q8 + (size_t)U * 32);
            R.xa = __ldcg(qs);
            R.xb = __ldcg(qs + 1);
            R.dh = __ldcg(reinterpret_cast<const unsigned short *>(a.q8 + a.q8_d_off) + U);
            R.qsum = __ldcg(reinterpret_cast<const int *>(a.q8 + a.q8_sum_off) + U);
            return;
        }
        const uint4 *qs = reinterpret_cast<const uint4 *>(xs + (size_t)U * 32);
        R.xa = qs[0];
        R.xb = qs[1];
        R.dh = reinterpret_cast<const unsigned short *>(xs + a.q8_d_off)[U];
        R.qsum = reinterpret_cast<const int *>(xs + a.q8_sum_off)[U];
    } else {
        R.xa = R.xb = make_uint4(0, 0, 0, 0);
        R.dh = 0;
        R.qsum = 0;
    }
}

// q4_K / q5_K: the unit is one 32-weight sub-block; term = d*sc*isum -
// dmin*m*qsum (qsum = the q8 block's code sum).
template <bool SUBDOTS, class Regs>
__device__ __forceinline__ void compute_q4like(const GemvLaunch &a, const GemvPart &P,
                                               const Regs &R, const Unit &x, int lane,
                                               float (&acc)[8])
{
    const float d8 = __half2float(__ushort_as_half(R.dh));
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        int dot = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t lo, hi;
            codes(R, r, m, lo, hi);
            dot = __dp4a((int)lo, (int)word(R.xa, m), dot);
            dot = __dp4a((int)hi, (int)word(R.xb, m), dot);
        }
        if (SUBDOTS) {
            const int row = x.t * kTileRows + r;
            if (x.active && row < P.rows) {
                const int blk = kChunkBlocks * x.c + (lane >> 3), k = lane & 7;
                a.isums[((size_t)row * a.nb + blk) * 8 + k] = dot;
            }
        } else {
            int sc, mn;
            float d, dmin;
            q4k_scales(R, r, sc, mn, d, dmin);
            const float term = fmaf(d, (float)(sc * dot), -dmin * (float)(mn * R.qsum));
            acc[r] = fmaf(d8, term, acc[r]);
        }
    }
}

template <bool SUBDOTS>
__device__ __forceinline__ void compute(const GemvLaunch &a, const GemvPart &P, const Q4kRegs &R,
                                        const Unit &x, int lane, float (&acc)[8])
{
    compute_q4like<SUBDOTS>(a, P, R, x, lane, acc);
}

template <bool SUBDOTS>
__device__ __forceinline__ void compute(const GemvLaunch &a, const GemvPart &P, const Q5kRegs &R,
                                        const Unit &x, int lane, float (&acc)[8])
{
    compute_q4like<SUBDOTS>(a, P, R, x, lane, acc);
}

// Per format code (6, 4, 5): the register set of one chunk and the bytes of
// a full chunk.
template <int FMT>
struct Fmt;
template <>
struct Fmt<6> {
    using Regs = Q6kRegs;
    using W = Q6kW;
    static constexpr int kChunkBytes = kQ6kChunkPerBlock * kChunkBlocks;
};
template <>
struct Fmt<4> {
    using Regs = Q4kRegs;
    using W = Q4kW;
    static constexpr int kChunkBytes = kQ4kChunkPerBlock * kChunkBlocks;
};
template <>
struct Fmt<5> {
    using Regs = Q5kRegs;
    using W = Q5kW;
    static constexpr int kChunkBytes = kQ5kChunkPerBlock * kChunkBlocks;
};

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

}  // namespace gemv_detail
}  // namespace mq
