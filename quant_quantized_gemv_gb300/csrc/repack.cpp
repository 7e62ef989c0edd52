// repack.cpp -- host repack of GGUF q6_K / q4_K / q5_K rows into the tile/chunk/plane
// layout of layout.h, and its exact inverse.  Runs once per weight at load
// (page "76 · D4-4 — dpl dense split-plane q6_K decode MMVQ", §3.1: the plane
// is built once at registration, so decode pays nothing for it).
#include <string.h>

#include "layout.h"
#include "mq.h"

namespace {

using namespace mq;

// ---- q6_K source decode (GGUF block: ql 128 | qh 64 | sc 16 | d 2) --------
// Unit p (0..7) of a block covers weights 32p..32p+31: half = p >> 2,
// g = p & 3; weight l of the unit has its low 4 bits in the low (g < 2) or
// high (g >= 2) nibble of ql[64*half + 32*(g&1) + l] and its high 2 bits at
// bit 2g of qh[32*half + l] (page "74 · D4-2", §3.2 Excerpt C addressing).
inline int q6k_lo(const uint8_t *blk, int p, int l)
{
    const int half = p >> 2, g = p & 3;
    const uint8_t b = blk[64 * half + 32 * (g & 1) + l];
    return g < 2 ? (b & 15) : (b >> 4);
}
inline int q6k_hi(const uint8_t *blk, int p, int l)
{
    const int half = p >> 2, g = p & 3;
    return (blk[128 + 32 * half + l] >> (2 * g)) & 3;
}
inline void q6k_put(uint8_t *blk, int p, int l, int lo, int hi)
{
    const int half = p >> 2, g = p & 3;
    uint8_t &b = blk[64 * half + 32 * (g & 1) + l];
    b |= (uint8_t)(g < 2 ? lo : lo << 4);
    blk[128 + 32 * half + l] |= (uint8_t)(hi << (2 * g));
}

// ---- q4_K source decode (GGUF block: d 2 | dmin 2 | scales 12 | qs 128) ---
// Weight l of sub-block k is the low (k even) or high (k odd) nibble of
// qs[32 * (k/2) + l]; the 6-bit scale and min of k are packed in 12 bytes.
inline void q4k_get_sm(const uint8_t *s, int k, int *sc, int *m)
{
    if (k < 4) {
        *sc = s[k] & 63;
        *m = s[k + 4] & 63;
    } else {
        *sc = (s[k + 4] & 15) | ((s[k - 4] >> 6) << 4);
        *m = (s[k + 4] >> 4) | ((s[k] >> 6) << 4);
    }
}
inline void q4k_put_sm(uint8_t *s, int k, int sc, int m)
{
    if (k < 4) {
        s[k] |= (uint8_t)(sc & 63);
        s[k + 4] |= (uint8_t)(m & 63);
    } else {
        s[k + 4] |= (uint8_t)((sc & 15) | ((m & 15) << 4));
        s[k - 4] |= (uint8_t)((sc >> 4) << 6);
        s[k] |= (uint8_t)((m >> 4) << 6);
    }
}
// ---- q5_K source decode (GGUF block: d 2 | dmin 2 | scales 12 | qh 32 | qs 128)
// Weight l of sub-block k: low 4 bits as q4_K (nibbles from qs @48), fifth
// bit = bit k of qh[l].
inline int q5k_bit(const uint8_t *blk, int k, int l) { return (blk[16 + l] >> k) & 1; }

// Bit position, in the fifth-bit word H of a unit and row, of weight l
// (= 16h + 4m + b) of the unit: 8b + 4h + m (layout.h).
inline int q5k_hpos(int l) { return 8 * (l & 3) + 4 * (l >> 4) + ((l >> 2) & 3); }

// The QS and META planes of a q4_K or q5_K unit i for tile row r (meta_off:
// the META plane's offset per block of the chunk; layout.h).
void put_q4like(uint8_t *out, size_t seg, int cb, int r, int i, const uint8_t *blk, int meta_off,
                int nib_off)
{
    const int nu = 8 * cb, k = i & 7;
    uint8_t *qs = out + seg + ((size_t)r * nu + i) * 16;
    for (int t = 0; t < 16; ++t) {
        const uint8_t lo = blk[nib_off + 32 * (k >> 1) + t], hi = blk[nib_off + 32 * (k >> 1) + 16 + t];
        qs[t] = (uint8_t)(((k & 1) ? lo >> 4 : lo & 15) | (((k & 1) ? hi >> 4 : hi & 15) << 4));
    }
    int sc, m;
    q4k_get_sm(blk + 4, k, &sc, &m);
    uint8_t *meta = out + seg + (size_t)meta_off * cb + (size_t)i * 16;
    uint32_t w[3];
    memcpy(w, meta, 12);
    w[0] |= (uint32_t)(sc & 15) << (4 * r);
    w[1] |= (uint32_t)(m & 15) << (4 * r);
    w[2] |= (uint32_t)((sc >> 4) | ((m >> 4) << 2)) << (4 * r);
    memcpy(meta, w, 12);
    if (r == k) memcpy(meta + 12, blk, 4);  // (d, dmin) of row k of the block
}

void get_q4like(const uint8_t *in, size_t seg, int cb, int r, int i, uint8_t *blk, int meta_off,
                int nib_off)
{
    const int nu = 8 * cb, k = i & 7;
    const uint8_t *qs = in + seg + ((size_t)r * nu + i) * 16;
    for (int l = 0; l < 32; ++l) {
        const int v = l < 16 ? (qs[l] & 15) : (qs[l - 16] >> 4);
        blk[nib_off + 32 * (k >> 1) + l] |= (uint8_t)((k & 1) ? v << 4 : v);
    }
    const uint8_t *meta = in + seg + (size_t)meta_off * cb + (size_t)i * 16;
    uint32_t w[3];
    memcpy(w, meta, 12);
    const int hi = (w[2] >> (4 * r)) & 15;
    const int sc = (int)((w[0] >> (4 * r)) & 15) | ((hi & 3) << 4);
    const int m = (int)((w[1] >> (4 * r)) & 15) | ((hi >> 2) << 4);
    q4k_put_sm(blk + 4, k, sc, m);
    if (r == k) memcpy(blk, meta + 12, 4);
}

bool shape_ok(int rows, int cols)
{
    return rows >= 1 && cols >= kQK && cols % kQK == 0 &&
           (long long)rows * cols < (1LL << 40);
}

// Visit every (row, block) of a tile-chunk with the destination pointers.
template <class F>
void for_each_unit(const Geom &g, int block_bytes, F f)
{
    for (int t = 0; t < g.ntiles; ++t)
        for (int c = 0; c < g.nchunks; ++c) {
            const int cb = (g.nb - kChunkBlocks * c) < kChunkBlocks ? g.nb - kChunkBlocks * c
                                                                  : kChunkBlocks;
            const size_t seg = (size_t)t * g.tile_bytes + (size_t)c * g.chunk_stride;
            for (int r = 0; r < kTileRows; ++r) {
                const int row = t * kTileRows + r;
                if (row >= g.rows) continue;  // padded rows stay zero
                for (int i = 0; i < 8 * cb; ++i)
                    f(seg, cb, r, row, kChunkBlocks * c + (i >> 3), i);
            }
        }
    (void)block_bytes;
}

}  // namespace

extern "C" {

size_t mq_repacked_bytes_q6k(int rows, int cols)
{
    if (!shape_ok(rows, cols)) return 0;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    return (size_t)g.ntiles * g.tile_bytes;
}

size_t mq_repacked_bytes_q4k(int rows, int cols)
{
    if (!shape_ok(rows, cols)) return 0;
    const Geom g = make_geom(rows, cols, kQ4kBytes);
    return (size_t)g.ntiles * g.tile_bytes;
}

int mq_repack_q6k(const void *gguf, void *dst, int rows, int cols)
{
    if (!gguf || !dst) return MQ_ERR_NULL;
    if (!shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const uint8_t *src = (const uint8_t *)gguf;
    uint8_t *out = (uint8_t *)dst;
    memset(out, 0, (size_t)g.ntiles * g.tile_bytes);
    for_each_unit(g, kQ6kBytes, [&](size_t seg, int cb, int r, int row, int b, int i) {
        const uint8_t *blk = src + ((size_t)row * g.nb + b) * kQ6kBytes;
        const int nu = 8 * cb, p = i & 7;
        uint8_t *ql = out + seg + ((size_t)r * nu + i) * 16;
        uint8_t *qh = out + seg + (size_t)kQ6kQH * cb + ((size_t)(r >> 1) * nu + i) * 16 + (r & 1) * 8;
        uint8_t *sc = out + seg + (size_t)kQ6kSC * cb + (size_t)i * 16 + r * 2;
        for (int k = 0; k < 16; ++k)
            ql[k] = (uint8_t)(q6k_lo(blk, p, k) | (q6k_lo(blk, p, 16 + k) << 4));
        for (int h = 0; h < 2; ++h)
            for (int k = 0; k < 4; ++k) {
                int v = 0;
                for (int m = 0; m < 4; ++m) v |= q6k_hi(blk, p, 16 * h + 4 * m + k) << (2 * m);
                qh[4 * h + k] = (uint8_t)v;
            }
        sc[0] = blk[192 + 2 * p];
        sc[1] = blk[192 + 2 * p + 1];
        if (p == 0) {
            uint8_t *d = out + seg + (size_t)kQ6kD * cb + (size_t)(i >> 3) * 16 + r * 2;
            d[0] = blk[208];
            d[1] = blk[209];
        }
    });
    return MQ_OK;
}

int mq_unrepack_q6k(const void *packed, void *gguf, int rows, int cols)
{
    if (!gguf || !packed) return MQ_ERR_NULL;
    if (!shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const uint8_t *in = (const uint8_t *)packed;
    uint8_t *dst = (uint8_t *)gguf;
    memset(dst, 0, (size_t)rows * g.nb * kQ6kBytes);
    for_each_unit(g, kQ6kBytes, [&](size_t seg, int cb, int r, int row, int b, int i) {
        uint8_t *blk = dst + ((size_t)row * g.nb + b) * kQ6kBytes;
        const int nu = 8 * cb, p = i & 7;
        const uint8_t *ql = in + seg + ((size_t)r * nu + i) * 16;
        const uint8_t *qh = in + seg + (size_t)kQ6kQH * cb + ((size_t)(r >> 1) * nu + i) * 16 + (r & 1) * 8;
        const uint8_t *sc = in + seg + (size_t)kQ6kSC * cb + (size_t)i * 16 + r * 2;
        for (int l = 0; l < 32; ++l) {
            const int lo = l < 16 ? (ql[l] & 15) : (ql[l - 16] >> 4);
            const int h = l >> 4, m = (l & 15) >> 2, k = l & 3;
            const int hi = (qh[4 * h + k] >> (2 * m)) & 3;
            q6k_put(blk, p, l, lo, hi);
        }
        blk[192 + 2 * p] = sc[0];
        blk[192 + 2 * p + 1] = sc[1];
        if (p == 0) {
            const uint8_t *d = in + seg + (size_t)kQ6kD * cb + (size_t)(i >> 3) * 16 + r * 2;
            blk[208] = d[0];
            blk[209] = d[1];
        }
    });
    return MQ_OK;
}

int mq_repack_q4k(const void *gguf, void *dst, int rows, int cols)
{
    if (!gguf || !dst) return MQ_ERR_NULL;
    if (!shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ4kBytes);
    const uint8_t *src = (const uint8_t *)gguf;
    uint8_t *out = (uint8_t *)dst;
    memset(out, 0, (size_t)g.ntiles * g.tile_bytes);
    for_each_unit(g, kQ4kBytes, [&](size_t seg, int cb, int r, int row, int b, int i) {
        const uint8_t *blk = src + ((size_t)row * g.nb + b) * kQ4kBytes;
        put_q4like(out, seg, cb, r, i, blk, kQ4kMeta, 16);
    });
    return MQ_OK;
}

int mq_unrepack_q4k(const void *packed, void *gguf, int rows, int cols)
{
    if (!gguf || !packed) return MQ_ERR_NULL;
    if (!shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ4kBytes);
    const uint8_t *in = (const uint8_t *)packed;
    uint8_t *dst = (uint8_t *)gguf;
    memset(dst, 0, (size_t)rows * g.nb * kQ4kBytes);
    for_each_unit(g, kQ4kBytes, [&](size_t seg, int cb, int r, int row, int b, int i) {
        uint8_t *blk = dst + ((size_t)row * g.nb + b) * kQ4kBytes;
        get_q4like(in, seg, cb, r, i, blk, kQ4kMeta, 16);
    });
    return MQ_OK;
}

size_t mq_repacked_bytes_q5k(int rows, int cols)
{
    if (!shape_ok(rows, cols)) return 0;
    const Geom g = make_geom(rows, cols, kQ5kBytes);
    return (size_t)g.ntiles * g.tile_bytes;
}

int mq_repack_q5k(const void *gguf, void *dst, int rows, int cols)
{
    if (!gguf || !dst) return MQ_ERR_NULL;
    if (!shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ5kBytes);
    const uint8_t *src = (const uint8_t *)gguf;
    uint8_t *out = (uint8_t *)dst;
    memset(out, 0, (size_t)g.ntiles * g.tile_bytes);
    for_each_unit(g, kQ5kBytes, [&](size_t seg, int cb, int r, int row, int b, int i) {
        const uint8_t *blk = src + ((size_t)row * g.nb + b) * kQ5kBytes;
        put_q4like(out, seg, cb, r, i, blk, kQ5kMeta, 48);
        const int k = i & 7;
        uint32_t H = 0;
        for (int l = 0; l < 32; ++l) H |= (uint32_t)q5k_bit(blk, k, l) << q5k_hpos(l);
        memcpy(out + seg + (size_t)kQ5kQH * cb + ((size_t)i * 8 + r) * 4, &H, 4);
    });
    return MQ_OK;
}

int mq_unrepack_q5k(const void *packed, void *gguf, int rows, int cols)
{
    if (!gguf || !packed) return MQ_ERR_NULL;
    if (!shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ5kBytes);
    const uint8_t *in = (const uint8_t *)packed;
    uint8_t *dst = (uint8_t *)gguf;
    memset(dst, 0, (size_t)rows * g.nb * kQ5kBytes);
    for_each_unit(g, kQ5kBytes, [&](size_t seg, int cb, int r, int row, int b, int i) {
        uint8_t *blk = dst + ((size_t)row * g.nb + b) * kQ5kBytes;
        get_q4like(in, seg, cb, r, i, blk, kQ5kMeta, 48);
        const int k = i & 7;
        uint32_t H;
        memcpy(&H, in + seg + (size_t)kQ5kQH * cb + ((size_t)i * 8 + r) * 4, 4);
        for (int l = 0; l < 32; ++l) blk[16 + l] |= (uint8_t)(((H >> q5k_hpos(l)) & 1) << k);
    });
    return MQ_OK;
}

}  // extern "C"
