// layout.h -- the repacked weight layout and the q8 plane layout, shared by
// the host repack (repack.cpp) and the GEMV kernels.  Internal to
// the library; callers see only sizes (include/mq.h).
//
// Why a new layout.  The minfer pages (page "76 · D4-4 — dpl dense
// split-plane q6_K decode MMVQ", §2) show that a decode GEMV is a pure weight
// stream and that every byte of the stream that is not content is paid in
// full; their dense split-plane row [ql|qh|sc|d] removed the 14 dead bytes of
// the 224 B padded block.  This layout keeps that property (exactly 210 B or
// 144 B per super-block, no padding for rows % 8 == 0) and additionally
// orders the bytes so that each warp-wide 16-byte vector load reads 512
// contiguous bytes and every byte is requested once.  (The pages' per-thread
// unit loads read each ql byte twice and each qh byte four times, because two
// units share a ql byte and four share a qh byte: page "74 · D4-2", §3.2
// Excerpt C.)  To get there the repack is a permutation of bits, not bytes:
// each 32-weight unit owns exactly 16 B of low nibbles and 8 B of 2-bit highs.
//
// Geometry.  A tile is 8 consecutive rows (the last tile is padded with zero
// rows).  A tile's columns are cut into chunks of 4 super-blocks (the last
// chunk may hold 1..3).  A chunk of cb blocks carries nu = 8*cb units of 32
// weights; lane i of a warp owns unit i for all 8 rows of the tile.  Tiles
// are stored one after the other; within a tile, chunks in column order;
// within a chunk, planes:
//
// q6_K chunk (1680*cb bytes):
//   QL  @0        [row 8][unit nu][16 B]  byte k: low nibble = 4-bit low part
//                 of weight l=k, high nibble = weight l=16+k of the unit
//   QH  @1024*cb  [row/2 4][unit nu][2 rows x 8 B]  word h (bytes 4h..4h+3):
//                 byte k bits 2m..2m+1 = 2-bit high part of weight 16h+4m+k
//   SC  @1536*cb  [unit nu][row 8][2 B]  the unit's two int8 sub-block scales
//   D   @1664*cb  [block cb][row 8][2 B] the block's fp16 d
// q4_K chunk (1152*cb bytes):
//   QS   @0        [row 8][unit nu][16 B]  unit = one 32-weight sub-block;
//                  byte k: low nibble = weight k, high nibble = weight 16+k
//   META @1024*cb  [unit nu][16 B]  the unit's scales and one row's block
//                  scales, so that a lane gets all it reads besides its
//                  codes with one 16-byte load:
//                  word0 bits 4r..4r+3 = sc_r & 15, word1 bits 4r.. = m_r & 15,
//                  word2 bits 4r,4r+1 = sc_r >> 4 and bits 4r+2,4r+3 = m_r >> 4
//                  (r = row within the tile); word3 = (d, dmin) fp16 of row
//                  (unit & 7) of the unit's block (unit >> 3): the 8 units of
//                  a block hold its 8 rows' (d, dmin), which the kernels pass
//                  between the block's 8 lanes with shuffles
// q5_K chunk (1408*cb bytes): q4_K's planes plus the fifth bits
//   QS   @0        as q4_K (low 4 bits of each code)
//   QH   @1024*cb  [unit nu][row 8][4 B]  word H of (unit, row): bit
//                  8b + 4h + m = fifth bit of weight 16h + 4m + b, so that
//                  ((H >> m) & 0x01010101) << 4 lines up with the low-nibble
//                  word m and ((H >> (m+4)) & 0x01010101) << 4 with the high
//   META @1280*cb  as q4_K
// Every plane offset and every per-lane load address is 16-byte aligned,
// because 8 rows x 210 B, 8 rows x 144 B and 8 rows x 176 B are all
// multiples of 16.
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace mq {

constexpr int kQK = 256;           // weights per super-block
constexpr int kTileRows = 8;       // rows per tile
constexpr int kChunkBlocks = 4;    // super-blocks per chunk (32 units)
constexpr int kQ6kBytes = 210;
constexpr int kQ4kBytes = 144;
constexpr int kQ5kBytes = 176;

// q6_K chunk plane offsets, per block of the chunk (multiply by cb)
constexpr int kQ6kQH = 1024, kQ6kSC = 1536, kQ6kD = 1664, kQ6kChunkPerBlock = 1680;
// q4_K chunk plane offsets, per block of the chunk (multiply by cb)
constexpr int kQ4kMeta = 1024, kQ4kChunkPerBlock = 1152;
// q5_K chunk plane offsets, per block of the chunk (multiply by cb)
constexpr int kQ5kQH = 1024, kQ5kMeta = 1280, kQ5kChunkPerBlock = 1408;

// Bytes of one super-block (= per block of a chunk / 8 rows) by format code
// (6 = q6_K, 4 = q4_K, 5 = q5_K); 0 for an unknown code.
constexpr int block_bytes(int fmt)
{
    return fmt == 6 ? kQ6kBytes : fmt == 4 ? kQ4kBytes : fmt == 5 ? kQ5kBytes : 0;
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct Geom {
    int rows, cols, nb, ntiles, nchunks;
    size_t tile_bytes;    // bytes of one 8-row tile
    size_t chunk_stride;  // bytes of one full (4-block) chunk
};

inline Geom make_geom(int rows, int cols, int block_bytes)
{
    Geom g;
    g.rows = rows;
    g.cols = cols;
    g.nb = cols / kQK;
    g.ntiles = ceil_div(rows, kTileRows);
    g.nchunks = ceil_div(g.nb, kChunkBlocks);
    g.tile_bytes = (size_t)kTileRows * g.nb * block_bytes;
    g.chunk_stride = (size_t)kTileRows * kChunkBlocks * block_bytes;
    return g;
}

// q8 plane for n values (n % 32 == 0): [qs n B][d nq*2 B][sum nq*4 B], each
// section starting on a 16-byte boundary.
inline size_t round16(size_t x) { return (x + 15) & ~(size_t)15; }
inline size_t q8_d_offset(int n) { return round16((size_t)n); }
inline size_t q8_sum_offset(int n) { return q8_d_offset(n) + round16((size_t)(n / 32) * 2); }
inline size_t q8_plane_bytes(int n) { return q8_sum_offset(n) + round16((size_t)(n / 32) * 4); }

}  // namespace mq
