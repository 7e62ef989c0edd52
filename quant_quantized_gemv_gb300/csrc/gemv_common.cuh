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

#include <type_traits>

#include "kernels.h"
#include "layout.h"

namespace mq {
namespace gemv_detail {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kLo4 = 0x0f0f0f0fu;
constexpr uint32_t kOnes = 0x01010101u;

// L2 policy of the weight stream: evict first.  Every weight byte is read
// once per decode step and a step streams far more than L2 holds, so the
// weights are the lines to drop first; the kernels' code, the q8 planes, the
// outputs and the producers' data then stay in L2 across the launches of a
// step.
__device__ __forceinline__ uint64_t stream_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte streaming load: read-only path, no L1 allocation (each weight
// byte is used once), evict-first in L2.
__device__ __forceinline__ uint4 ld_stream16(const uint8_t *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const uint8_t *p, uint64_t pol)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                 : "=r"(v)
                 : "l"(p), "l"(pol));
    return v;
}

// Shared-memory loads by 32-bit shared address.
__device__ __forceinline__ uint4 ld_smem16(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t ld_smem4(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Asynchronous 16-byte global -> shared copies (L1 bypassed), grouped per
// thread: a thread's copies become visible to it after cp.async.wait_group,
// to the other lanes of its warp after that and a __syncwarp.
__device__ __forceinline__ void cp_async16(uint32_t dst, const uint8_t *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Where a chunk's bytes are read from: global memory (streaming loads) or a
// verbatim copy of the chunk in shared memory (same offsets).
struct GlobalChunk {
    const uint8_t *base;
    uint64_t pol = stream_policy();
    __device__ __forceinline__ uint4 v16(size_t off) const { return ld_stream16(base + off, pol); }
    __device__ __forceinline__ uint32_t v4(size_t off) const { return ld_stream4(base + off, pol); }
};
struct SharedChunk {
    uint32_t base;
    __device__ __forceinline__ uint4 v16(size_t off) const { return ld_smem16(base + (uint32_t)off); }
    __device__ __forceinline__ uint32_t v4(size_t off) const { return ld_smem4(base + (uint32_t)off); }
};

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

// Staging of q8 planes (and the f32 row) into shared memory: 16-byte
// asynchronous copies through L2 (cp.async.cg: coherent with what the
// preceding kernel wrote before its completion released the grid-dependency
// wait), all of a thread's copies in flight at once with no registers held;
// then the thread waits for its own copies, and a CTA barrier publishes them
// to the others.
__device__ __forceinline__ void copy16_async(void *smem_dst, const void *gmem_src)
{
    cp_async16(smem_addr(smem_dst), static_cast<const uint8_t *>(gmem_src));
}
__device__ __forceinline__ void copy_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
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

template <class Src>
__device__ __forceinline__ void load_w_from(const Src &src, const Unit &x, int lane, Q6kW &R)
{
    const int nu = 8 * x.cb, cb = x.cb;
    if (x.active) {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.ql[r] = src.v16(((size_t)r * nu + lane) * 16);
#pragma unroll
        for (int p = 0; p < 4; ++p) R.qh[p] = src.v16((size_t)kQ6kQH * cb + ((size_t)p * nu + lane) * 16);
        R.sc = src.v16((size_t)kQ6kSC * cb + (size_t)lane * 16);
        R.dd = src.v16((size_t)kQ6kD * cb + (size_t)(lane >> 3) * 16);
    } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.ql[r] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int p = 0; p < 4; ++p) R.qh[p] = make_uint4(0, 0, 0, 0);
        R.sc = R.dd = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void load_w(const Unit &x, int lane, Q6kW &R)
{
    load_w_from(GlobalChunk{x.seg}, x, lane, R);
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
    uint4 qs[8];  // nibbles of 8 rows
    uint4 meta;   // the unit's META entry (layout.h)
};

// The QS and META planes (q4_K, and q5_K at another META offset).
template <int META, class Src>
__device__ __forceinline__ void load_w_q4like(const Src &src, const Unit &x, int lane, Q4kW &R)
{
    const int nu = 8 * x.cb, cb = x.cb;
    if (x.active) {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.qs[r] = src.v16(((size_t)r * nu + lane) * 16);
        R.meta = src.v16((size_t)META * cb + (size_t)lane * 16);
    } else {
#pragma unroll
        for (int r = 0; r < 8; ++r) R.qs[r] = make_uint4(0, 0, 0, 0);
        R.meta = make_uint4(0, 0, 0, 0);
    }
}

template <class Src>
__device__ __forceinline__ void load_w_from(const Src &src, const Unit &x, int lane, Q4kW &R)
{
    load_w_q4like<kQ4kMeta>(src, x, lane, R);
}
__device__ __forceinline__ void load_w(const Unit &x, int lane, Q4kW &R)
{
    load_w_from(GlobalChunk{x.seg}, x, lane, R);
}

// Row r's codes for words m of the unit: weights 4m..4m+3 (lo, against the
// activation codes xa) and 16+4m..16+4m+3 (hi, against xb), one per byte.
__device__ __forceinline__ void codes(const Q4kW &R, int r, int m, uint32_t &lo, uint32_t &hi)
{
    const uint32_t w = word(R.qs[r], m);
    lo = w & kLo4;
    hi = (w >> 4) & kLo4;
}

// The scales of a unit for its 8 rows, decoded once per chunk: the 6-bit
// scales and mins one per byte (rows 0, 2, 4, 6 and rows 1, 3, 5, 7), and
// each row's (d, dmin) taken from the META entry of the block's unit with
// that row's index.  Every lane of the warp must call this (shuffles).
struct Q4kDec {
    uint32_t sce, sco, me, mo;
    uint32_t dm[8];
};

__device__ __forceinline__ void decode_q4k(const Q4kW &R, int lane, Q4kDec &D)
{
    const uint32_t s0 = R.meta.x, s1 = R.meta.y, s2 = R.meta.z;
    D.sce = (s0 & kLo4) | ((s2 << 4) & 0x30303030u);
    D.sco = ((s0 >> 4) & kLo4) | (s2 & 0x30303030u);
    D.me = (s1 & kLo4) | ((s2 << 2) & 0x30303030u);
    D.mo = ((s1 >> 4) & kLo4) | ((s2 >> 2) & 0x30303030u);
    const int base = lane & ~7;
#pragma unroll
    for (int r = 0; r < 8; ++r) D.dm[r] = __shfl_sync(kFull, R.meta.w, base + r);
}

// Row r's 6-bit scale and min and fp16 d, dmin.
__device__ __forceinline__ void q4k_scales(const Q4kDec &D, int r, int &sc, int &mn, float &d,
                                           float &dmin)
{
    const int sh = 8 * (r >> 1);
    sc = (int)((((r & 1) ? D.sco : D.sce) >> sh) & 0xffu);
    mn = (int)((((r & 1) ? D.mo : D.me) >> sh) & 0xffu);
    d = half_lo(D.dm[r]);
    dmin = half_hi(D.dm[r]);
}

// dp4a with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ---- q5_K: q4_K's fields plus each code's fifth bit -------------------------
struct Q5kW : Q4kW {
    uint4 qh[2];  // fifth-bit words H of rows 0..3 and 4..7
};

template <class Src>
__device__ __forceinline__ void load_w_from(const Src &src, const Unit &x, int lane, Q5kW &R)
{
    load_w_q4like<kQ5kMeta>(src, x, lane, R);
    if (x.active) {
        const size_t hp = (size_t)kQ5kQH * x.cb + (size_t)lane * 32;
        R.qh[0] = src.v16(hp);
        R.qh[1] = src.v16(hp + 16);
    } else {
        R.qh[0] = R.qh[1] = make_uint4(0, 0, 0, 0);
    }
}
__device__ __forceinline__ void load_w(const Unit &x, int lane, Q5kW &R)
{
    load_w_from(GlobalChunk{x.seg}, x, lane, R);
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
struct X6 {               // the unit's activation codes and scale
    uint4 xa, xb;        // activation codes 0..15, 16..31 of the unit
    unsigned short dh;   // activation fp16 scale
};
struct Q6kRegs : Q6kW, X6 {};

__device__ __forceinline__ void load_x(const GemvLaunch &a, const uint8_t *xs, const Unit &x,
                                       int lane, X6 &R)
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
// dmin*m*qsum (qsum = the q8 block's code sum).  q4_K's high nibbles go to
// dp4a in place (16 x the code, bytes read unsigned), the sum shifted back
// once per row: the same integer isum as nibble by nibble.
template <bool SUBDOTS, class Regs>
__device__ __forceinline__ void compute_q4like(const GemvLaunch &a, const GemvPart &P,
                                               const Regs &R, const Unit &x, int lane,
                                               float (&acc)[8])
{
    constexpr bool kQ5 = std::is_base_of<Q5kW, Regs>::value;
    const float d8 = __half2float(__ushort_as_half(R.dh));
    Q4kDec D;
    if (!SUBDOTS) decode_q4k(R, lane, D);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        int dot = 0;
        if constexpr (kQ5) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t lo, hi;
                codes(R, r, m, lo, hi);
                dot = __dp4a((int)lo, (int)word(R.xa, m), dot);
                dot = __dp4a((int)hi, (int)word(R.xb, m), dot);
            }
        } else {
            int hi16 = 0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t w = word(R.qs[r], m);
                dot = __dp4a((int)(w & kLo4), (int)word(R.xa, m), dot);
                hi16 = dp4a_us(w & ~kLo4, word(R.xb, m), hi16);
            }
            dot += hi16 >> 4;  // exact: hi16 is a multiple of 16
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
            q4k_scales(D, r, sc, mn, d, dmin);
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
    using X = X6;
    static constexpr int kChunkBytes = kQ6kChunkPerBlock * kChunkBlocks;
};
template <>
struct Fmt<4> {
    using Regs = Q4kRegs;
    using W = Q4kW;
    using X = XSum;
    static constexpr int kChunkBytes = kQ4kChunkPerBlock * kChunkBlocks;
};
template <>
struct Fmt<5> {
    using Regs = Q5kRegs;
    using W = Q5kW;
    using X = XSum;
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
