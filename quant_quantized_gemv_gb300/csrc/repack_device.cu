// repack_device.cu -- the repack of repack.cpp done on the GPU, for weights
// that are already in device memory in GGUF order (the pages build their
// dense plane once at weight registration, page "76 · D4-4 — dpl dense
// split-plane q6_K decode MMVQ", §3.1; the page notes the repack is a few
// byte moves, here it is a kernel so that multi-GB weight sets are repacked
// at HBM speed instead of by one host thread).  The bytes written are
// exactly those of the host repack, padding rows included (zero).
//
// One thread per (tile, chunk, unit): it reads the unit's bytes of the 8
// rows of the tile from the GGUF blocks (byte loads: GGUF blocks of 210,
// 144 and 176 bytes are only 2-byte aligned) and writes every byte of the
// unit's planes, so no two threads write the same word (the 6-bit q4_K /
// q5_K scales of 8 rows share one word per unit).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "layout.h"

namespace mq {
namespace {

struct RepackArgs {
    const uint8_t *src;  // GGUF rows: rows x nb blocks
    uint8_t *dst;        // repacked, zero-filled before the launch
    int rows, nb, nchunks;
    unsigned long long tile_bytes;
    long long units;     // ntiles * nchunks * 32
};

__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return a | (b << 8) | (c << 16) | (d << 24);
}

// q6_K: GGUF block ql 128 | qh 64 | sc 16 | d 2.  Unit p covers weights
// 32p .. 32p+31: half = p >> 2, g = p & 3; weight l has its low 4 bits in
// the low (g < 2) or high (g >= 2) nibble of ql[64 half + 32 (g&1) + l] and
// its high 2 bits at bit 2g of qh[32 half + l].
__device__ void repack_unit_q6k(const RepackArgs &A, int t, int c, int i)
{
    const int cb = min(kChunkBlocks, A.nb - kChunkBlocks * c);
    if (i >= 8 * cb) return;
    const int nu = 8 * cb, p = i & 7, b = kChunkBlocks * c + (i >> 3);
    const int half = p >> 2, g = p & 3;
    uint8_t *seg = A.dst + (size_t)t * A.tile_bytes + (size_t)c * (kQ6kChunkPerBlock * kChunkBlocks);
    for (int r = 0; r < kTileRows; ++r) {
        const int row = t * kTileRows + r;
        if (row >= A.rows) break;  // padded rows stay zero
        const uint8_t *blk = A.src + ((size_t)row * A.nb + b) * kQ6kBytes;
        const uint8_t *qlp = blk + 64 * half + 32 * (g & 1);
        const uint8_t *qhp = blk + 128 + 32 * half;
        uint32_t lo[32], hi[32];
#pragma unroll
        for (int l = 0; l < 32; ++l) {
            const uint32_t v = qlp[l];
            lo[l] = g < 2 ? (v & 15u) : (v >> 4);
            hi[l] = (qhp[l] >> (2 * g)) & 3u;
        }
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)  // byte k: low nibble weight k, high nibble weight 16 + k
            w[j] = pack4(lo[4 * j] | (lo[16 + 4 * j] << 4), lo[4 * j + 1] | (lo[16 + 4 * j + 1] << 4),
                         lo[4 * j + 2] | (lo[16 + 4 * j + 2] << 4), lo[4 * j + 3] | (lo[16 + 4 * j + 3] << 4));
        *reinterpret_cast<uint4 *>(seg + ((size_t)r * nu + i) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        uint32_t h[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // word hh, byte k bits 2m: high bits of weight 16hh + 4m + k
            uint32_t by[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t v = 0;
#pragma unroll
                for (int m = 0; m < 4; ++m) v |= hi[16 * hh + 4 * m + k] << (2 * m);
                by[k] = v;
            }
            h[hh] = pack4(by[0], by[1], by[2], by[3]);
        }
        *reinterpret_cast<uint2 *>(seg + (size_t)kQ6kQH * cb + ((size_t)(r >> 1) * nu + i) * 16 +
                                   (r & 1) * 8) = make_uint2(h[0], h[1]);
        uint8_t *sc = seg + (size_t)kQ6kSC * cb + (size_t)i * 16 + r * 2;
        sc[0] = blk[192 + 2 * p];
        sc[1] = blk[192 + 2 * p + 1];
        if (p == 0) {
            uint8_t *d = seg + (size_t)kQ6kD * cb + (size_t)(i >> 3) * 16 + r * 2;
            d[0] = blk[208];
            d[1] = blk[209];
        }
    }
}

// q4_K (nib_off 16) and q5_K (nib_off 48): GGUF d 2 | dmin 2 | scales 12 |
// [qh 32 |] qs 128.  Unit i is sub-block k = i & 7 of block b: weight l is
// the low (k even) or high (k odd) nibble of qs[32 (k/2) + l]; q5_K adds the
// fifth bit, bit k of qh[l].
template <int META, int QH, int NIB, int BLOCK, int CHUNK>
__device__ void repack_unit_q4like(const RepackArgs &A, int t, int c, int i)
{
    const int cb = min(kChunkBlocks, A.nb - kChunkBlocks * c);
    if (i >= 8 * cb) return;
    const int nu = 8 * cb, k = i & 7, b = kChunkBlocks * c + (i >> 3);
    uint8_t *seg = A.dst + (size_t)t * A.tile_bytes + (size_t)c * CHUNK;
    uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    for (int r = 0; r < kTileRows; ++r) {
        const int row = t * kTileRows + r;
        if (row >= A.rows) break;  // padded rows stay zero
        const uint8_t *blk = A.src + ((size_t)row * A.nb + b) * BLOCK;
        const uint8_t *qs = blk + NIB + 32 * (k >> 1);
        uint32_t by[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) {  // byte l: low nibble weight l, high nibble weight 16 + l
            const uint32_t a = qs[l], bb = qs[16 + l];
            by[l] = ((k & 1) ? a >> 4 : a & 15u) | (((k & 1) ? bb >> 4 : bb & 15u) << 4);
        }
        *reinterpret_cast<uint4 *>(seg + ((size_t)r * nu + i) * 16) =
            make_uint4(pack4(by[0], by[1], by[2], by[3]), pack4(by[4], by[5], by[6], by[7]),
                       pack4(by[8], by[9], by[10], by[11]), pack4(by[12], by[13], by[14], by[15]));
        const uint8_t *s = blk + 4;  // 6-bit scale and min of sub-block k
        int sc, m;
        if (k < 4) {
            sc = s[k] & 63;
            m = s[k + 4] & 63;
        } else {
            sc = (s[k + 4] & 15) | ((s[k - 4] >> 6) << 4);
            m = (s[k + 4] >> 4) | ((s[k] >> 6) << 4);
        }
        w0 |= (uint32_t)(sc & 15) << (4 * r);
        w1 |= (uint32_t)(m & 15) << (4 * r);
        w2 |= (uint32_t)((sc >> 4) | ((m >> 4) << 2)) << (4 * r);
        if (r == k)  // (d, dmin) of row k of the block
            w3 = pack4(blk[0], blk[1], blk[2], blk[3]);
        if (QH > 0) {  // fifth bits: bit 8b + 4h + m of H = weight 16h + 4m + b
            uint32_t H = 0;
#pragma unroll
            for (int l = 0; l < 32; ++l)
                H |= (uint32_t)((blk[16 + l] >> k) & 1) << (8 * (l & 3) + 4 * (l >> 4) + ((l >> 2) & 3));
            *reinterpret_cast<uint32_t *>(seg + (size_t)QH * cb + ((size_t)i * 8 + r) * 4) = H;
        }
    }
    *reinterpret_cast<uint4 *>(seg + (size_t)META * cb + (size_t)i * 16) = make_uint4(w0, w1, w2, w3);
}

template <int FMT>
__global__ void __launch_bounds__(256) repack_kernel(const RepackArgs A)
{
    const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= A.units) return;
    const int i = (int)(u & 31);
    const long long tc = u >> 5;
    const int t = (int)(tc / A.nchunks), c = (int)(tc - (long long)t * A.nchunks);
    if (FMT == 6)
        repack_unit_q6k(A, t, c, i);
    else if (FMT == 4)
        repack_unit_q4like<kQ4kMeta, 0, 16, kQ4kBytes, kQ4kChunkPerBlock * kChunkBlocks>(A, t, c, i);
    else
        repack_unit_q4like<kQ5kMeta, kQ5kQH, 48, kQ5kBytes, kQ5kChunkPerBlock * kChunkBlocks>(A, t, c, i);
}

}  // namespace

cudaError_t launch_repack(int fmt, const void *src, void *dst, int rows, int cols, cudaStream_t st)
{
    const Geom g = make_geom(rows, cols, block_bytes(fmt));
    cudaError_t e = cudaMemsetAsync(dst, 0, (size_t)g.ntiles * g.tile_bytes, st);
    if (e != cudaSuccess) return e;
    RepackArgs A;
    A.src = (const uint8_t *)src;
    A.dst = (uint8_t *)dst;
    A.rows = rows;
    A.nb = g.nb;
    A.nchunks = g.nchunks;
    A.tile_bytes = g.tile_bytes;
    A.units = (long long)g.ntiles * g.nchunks * 32;
    const unsigned blocks = (unsigned)((A.units + 255) / 256);
    if (fmt == 6)
        repack_kernel<6><<<blocks, 256, 0, st>>>(A);
    else if (fmt == 4)
        repack_kernel<4><<<blocks, 256, 0, st>>>(A);
    else
        repack_kernel<5><<<blocks, 256, 0, st>>>(A);
    return cudaGetLastError();
}

}  // namespace mq
