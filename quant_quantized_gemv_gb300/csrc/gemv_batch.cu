// gemv_batch.cu -- small-batch decode GEMV: nt = 1..8 activation rows (the
// tokens of a speculative or batched decode step) against one pass over the
// repacked q6_K / q4_K weights.  The minfer pages' MMVQ kernels already carry
// a token index for this (page "74 · D4-2 — B0 latent correctness fix", §2:
// the launch takes nt and each token is a grid row); here every streamed
// weight byte is used for all nt tokens instead of being read nt times.
//
// Per token the arithmetic is the single-token GEMV's (gemv.cu): the same
// integer sub-block dots with dp4a, then the f32 combine with the block and
// sub-block scales and the token's fp16 activation scale, reduced with the
// same fixed butterfly and combined across splits in ascending split order.
// Up to 4 tokens the f32 order is the single-token kernel's; beyond that the
// butterfly runs once per chunk instead of once per tile (a different but
// equally fixed order).
//
// What changes with nt:
//   * All nt q8 planes are staged in shared memory once per CTA (after the
//     grid-dependency wait), whatever the plan; each chunk's codes for a
//     group of tokens (all of them up to 4, else groups of 2-4, see
//     group_size and compute) are then read from there into registers.
//   * A weight row's codes are decoded once per token group and used for
//     every token of the group: the decode, not the dp4a, dominates the ALU
//     work of a chunk.
//   * One CTA per SM stages the planes once for all its warps: as many as
//     the register file holds at the instance's register cap (16 warps at
//     128 registers for 2 tokens, 14-15 for 3-4 tokens of most formats, 12
//     at 168 otherwise).
//   * With one register buffer per warp, lane 0 prefetches the warp's next
//     chunk into L2 while the current one computes (kPrefetchNext).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "gemv_common.cuh"
#include "kernels.h"
#include "layout.h"
#include "prefetch.cuh"

namespace mq {
namespace {

using namespace gemv_detail;

// Tokens whose activation codes are held in registers at once: all of them
// up to kGroup.  Beyond that the groups run one at a time in a rolled loop,
// and every group decodes the 8 rows again: q6_K and q5_K take two groups of
// 3 or 4 at 6 and 8 tokens (spill-free at 168 registers; 8 tokens: 7B
// 36.3 -> 33.9 us, head 267 -> 243 us), q4_K, whose decode is cheap, pairs
// (its 8-token gate 25.7 against 26.5 us with groups of 4).  5 and 7 tokens
// are arranged in compute().
constexpr int kGroup = 4;
__host__ __device__ constexpr int group_size(int nt, int fmt)
{
    return nt <= kGroup ? nt : fmt != 4 && (nt == 6 || nt == 8) ? nt / 2 : 2;
}

// Running sums of a work item.  Up to kGroup tokens each lane keeps its own
// partial sums of the 8 rows (reduced across lanes when a tile is flushed,
// as in the single-token kernel).  With more tokens that would take 8 x nt
// registers, so each token group's chunk partials are reduced across lanes
// at once and each lane keeps only the sum of its row (lane >> 2) per token.
template <int NT>
struct Acc {
    static constexpr bool kEach = NT > kGroup;  // reduce every chunk
    float v[kEach ? 1 : NT][8];                 // per-lane partials (not kEach)
    float s[kEach ? NT : 1];                    // row (lane >> 2) sums (kEach)
};

// Activation codes of one unit for the tokens [t0, t0 + G) of a group.
template <int G>
struct XCodes {
    static constexpr int kG = G;
    uint4 xa[G], xb[G];  // codes 0..15 and 16..31 of the unit's q8 block
    float d8[G];         // fp16 activation scale
    int k0[G], k1[G];    // q6_K: -32 * sum(xa), -32 * sum(xb); q4_K: k0 = the block's sum
    float kf[G];         // q4_K / q5_K: the block's sum as f32
};

template <int FMT, int G>
__device__ __forceinline__ void load_x_group(const GemvLaunch &a, const uint8_t *xs, int t0, int nt,
                                             const Unit &x, int lane, XCodes<G> &X)
{
    const int U = 32 * x.c + lane;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        if (x.active && t0 + j < nt) {
            const uint8_t *pl = xs + (size_t)(t0 + j) * a.q8_bytes;
            const uint4 *qs = reinterpret_cast<const uint4 *>(pl + (size_t)U * 32);
            X.xa[j] = qs[0];
            X.xb[j] = qs[1];
            X.d8[j] = __half2float(
                __ushort_as_half(reinterpret_cast<const unsigned short *>(pl + a.q8_d_off)[U]));
            if (FMT == 6) {
                X.k0[j] = -32 * sum16(X.xa[j]);
                X.k1[j] = -32 * sum16(X.xb[j]);
            } else {
                X.k0[j] = reinterpret_cast<const int *>(pl + a.q8_sum_off)[U];
                X.k1[j] = 0;
                X.kf[j] = (float)X.k0[j];
            }
        } else {
            X.xa[j] = X.xb[j] = make_uint4(0, 0, 0, 0);
            X.d8[j] = 0.0f;
            X.k0[j] = X.k1[j] = 0;
            X.kf[j] = 0.0f;
        }
    }
}

// q6_K: sub-block 0 of the unit is weights 0..15 against codes xa, sub-block
// 1 is weights 16..31 against xb; isum_s = dot(q, x) - 32 * sum(x), the
// -32 * sum(x) term seeding each dp4a chain.  The two sums are kept apart so
// each sub-block's integer is the single-token one.  (LEAN has no effect.)
template <int NT, int G, bool LEAN>
__device__ __forceinline__ void compute_group(const Q6kW &W, const XCodes<G> &X, int t0,
                                              float (&out)[G][8])
{
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        uint32_t q0[4], q1[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) q6k_codes(W, r, m, q0[m], q1[m]);
        int sc0, sc1;
        float d;
        q6k_scales(W, r, sc0, sc1, d);
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if (t0 + j >= NT) break;
            int isum0 = X.k0[j], isum1 = X.k1[j];  // the -32 * sum(x) terms seed the chains
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                isum0 = __dp4a((int)q0[m], (int)word(X.xa[j], m), isum0);
                isum1 = __dp4a((int)q1[m], (int)word(X.xb[j], m), isum1);
            }
            out[j][r] = fmaf(d * X.d8[j], (float)(sc0 * isum0 + sc1 * isum1), out[j][r]);
        }
    }
}

// q4_K / q5_K: the unit is one 32-weight sub-block; term = d*sc*isum -
// dmin*m*qsum.  LEAN forms d*sc and dmin*m once per row for all the group's
// tokens (4 instead of 7 per row and token after the dp4a chain; 7B-shape
// q4_K gate at 5 tokens 19.9 -> 18.1 us); q5_K up to 4 tokens keeps the
// per-token form, which spills less there (at 4 tokens 22.2 against 21.9 us).
template <int NT, int G, bool LEAN, class Q4like>
__device__ __forceinline__ void compute_group(const Q4like &W, const Q4kDec &D, const XCodes<G> &X,
                                              int t0, float (&out)[G][8])
{
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) codes(W, r, m, lo[m], hi[m]);
        int sc, mn;
        float d, dmin;
        q4k_scales(D, r, sc, mn, d, dmin);
        const float dsc = d * (float)sc, dmm = dmin * (float)mn;  // LEAN: shared by the tokens
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if (t0 + j >= NT) break;
            int dot = 0;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                dot = __dp4a((int)lo[m], (int)word(X.xa[j], m), dot);
                dot = __dp4a((int)hi[m], (int)word(X.xb[j], m), dot);
            }
            if constexpr (LEAN) {
                out[j][r] = fmaf(X.d8[j], fmaf(dsc, (float)dot, -dmm * X.kf[j]), out[j][r]);
            } else {
                const float term = fmaf(d, (float)(sc * dot), -dmin * (float)(mn * X.k0[j]));
                out[j][r] = fmaf(X.d8[j], term, out[j][r]);
            }
        }
    }
}

template <int FMT, int NT>
__device__ __forceinline__ void compute(const GemvLaunch &a, const uint8_t *xs, const Unit &x,
                                        int lane, const typename Fmt<FMT>::W &W, Acc<NT> &acc)
{
    constexpr int G = group_size(NT, FMT);
    constexpr bool kLean = !(FMT == 5 && NT <= kGroup);
    // q4_K / q5_K: the unit's scales for its 8 rows, decoded once per chunk
    // (every lane takes part: the block scales move by shuffles)
    Q4kDec D;
    if constexpr (FMT != 6) decode_q4k(W, lane, D);
    auto run_group = [&](const auto &X, int t0, auto &out) {
        if constexpr (FMT == 6)
            compute_group<NT, std::remove_reference_t<decltype(X)>::kG, kLean>(W, X, t0, out);
        else
            compute_group<NT, std::remove_reference_t<decltype(X)>::kG, kLean>(W, D, X, t0, out);
    };
    if constexpr (!Acc<NT>::kEach) {  // one group: accumulate straight into the per-lane partials
        XCodes<G> X;
        load_x_group<FMT, G>(a, xs, 0, NT, x, lane, X);
        run_group(X, 0, reinterpret_cast<float(&)[G][8]>(acc.v));
    } else {
        // one group of GS tokens starting at t0 (GS is a compile-time size)
        auto group = [&](auto gs, int t0) {
            constexpr int GS = decltype(gs)::value;
            XCodes<GS> X;
            load_x_group<FMT, GS>(a, xs, t0, NT, x, lane, X);
            float part[GS][8];
#pragma unroll
            for (int j = 0; j < GS; ++j)
#pragma unroll
                for (int r = 0; r < 8; ++r) part[j][r] = 0.0f;
            run_group(X, t0, part);
#pragma unroll
            for (int j = 0; j < GS; ++j)
                if (t0 + j < NT) acc.s[t0 + j] += reduce8(part[j], lane);
        };
        using GroupG = std::integral_constant<int, G>;
        if constexpr (NT == 6 || NT == 8) {
            // one token group at a time: unrolled, the groups' live ranges
            // overlap and spill 190-360 bytes; rolled, only the row sums go
            // to (L1-resident) local memory (7B at 8 tokens in pairs 40.4 ->
            // 36.3 us)
#pragma unroll 1
            for (int t0 = 0; t0 < NT; t0 += G) group(GroupG{}, t0);
        } else if constexpr (NT == 7) {
            // 3 + 2 + 2: a group of three, then the pairs rolled -- spill-free
            // at 168 registers (7B at 7 tokens 34.7 -> 31.8 us); four pairs
            // with a masked last token spilled 120-290 bytes, and two rolled
            // groups of four with a masked token were slower (34.0 us)
            group(std::integral_constant<int, 3>{}, 0);
#pragma unroll 1
            for (int t0 = 3; t0 < NT; t0 += 2) group(std::integral_constant<int, 2>{}, t0);
        } else {
            // 5 tokens: unrolled pairs 2 + 2 + 1 (the last token of the last
            // pair masked).  They spill 4-164 bytes, but rolled (spill-free)
            // the 7B shape took 29.2 against 26.3 us, and 3 + 2 spilled more.
#pragma unroll
            for (int t0 = 0; t0 < NT; t0 += G) group(GroupG{}, t0);
        }
    }
}

// Tile t is finished for this warp: reduce (or take) its nt x 8 sums and
// write them, or -- with S > 1 -- leave them in shared memory, meet the
// tile's other split warps at one barrier and let split 0 add the S
// partials in ascending split order.  The exchange buffer alternates with the
// tile iteration, so one barrier per tile suffices: a buffer is rewritten two
// iterations later, after every warp of the group has passed the barrier in
// between.
static_assert(2 + kBatchMaxCtaWarps / 2 <= 16, "a named barrier per tile group");

template <int NT, int FMT>
__device__ __forceinline__ void flush_tile(const GemvLaunch &a, const GemvPart &P, int t, bool valid,
                                           int iter, Acc<NT> &acc, int lane)
{
    constexpr int kWarps = batch_warp_budget_max(NT, FMT);
    __shared__ float xchg[2][kWarps][NT][8];
    float v[NT];
#pragma unroll
    for (int k = 0; k < NT; ++k) {
        if (Acc<NT>::kEach) {
            v[k] = acc.s[k];
            acc.s[k] = 0.0f;
        } else {
            v[k] = reduce8(acc.v[k], lane);
#pragma unroll
            for (int r = 0; r < 8; ++r) acc.v[k][r] = 0.0f;
        }
    }
    const int row0 = t * kTileRows;
    if (a.splits == 1) {
        if (valid && (lane & 3) == 0 && row0 + (lane >> 2) < P.rows) {
#pragma unroll
            for (int k = 0; k < NT; ++k) P.y[(size_t)k * P.rows + row0 + (lane >> 2)] = v[k];
        }
        return;
    }
    const int w = threadIdx.x >> 5, sp = w % a.splits;
    float(&buf)[kWarps][NT][8] = xchg[iter & 1];
#pragma unroll
    for (int k = 0; k < NT; ++k) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float pr = __shfl_sync(kFull, v[k], 4 * r);
            if (lane == r) buf[w][k][r] = pr;
        }
    }
    // only the tile's S warps meet (named barrier 2 + its group; at most
    // kBatchMaxCtaWarps / 2 groups): the CTA's other groups run on.  Bitwise
    // the same; 7B nt=4 17.97 -> 17.85 us, nt=8 32.55 -> 32.33 us.
    asm volatile("bar.sync %0, %1;" ::"r"(2 + w / a.splits), "r"(32 * a.splits) : "memory");
    if (sp == 0 && valid && lane < 8 && row0 + lane < P.rows) {
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            float sum = 0.0f;
            for (int j = 0; j < a.splits; ++j) sum += buf[w + j][k][lane];
            P.y[(size_t)k * P.rows + row0 + lane] = sum;
        }
    }
}

// Wait for the producer, then stage the nt q8 planes in shared memory
// (16-byte cp.async copies through L2, every copy of a thread in flight at
// once: one round trip, where a token at a time took nt; 7B at 4 tokens
// 18.47 -> 16.17 us) and meet at named barrier 1.  Every warp of the CTA
// calls this exactly once.
__device__ __forceinline__ void stage_planes(const GemvLaunch &a, uint8_t *xs)
{
    griddep_wait();
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q8);
    uint4 *dst = reinterpret_cast<uint4 *>(xs);
    const int per = (int)(a.q8_bytes >> 4), stride = (int)(a.q8_stride >> 4);
    for (int t = 0; t < a.nt; ++t)
        for (int i = threadIdx.x; i < per; i += blockDim.x)
            copy16_async(dst + (size_t)t * per + i, src + (size_t)t * stride + i);
    copy_async_wait_all();
    asm volatile("bar.sync 1, %0;" ::"r"(blockDim.x) : "memory");
}

// Work decomposition.  A CTA has S * G warps (S = a.splits, G = a.wpc / S tiles
// per group): warp w takes split w % S of tile w / S of each group.  The CTA
// runs a.tpi consecutive groups, so the staged planes serve a.tpi * G tiles.
// Split s covers chunks [s * cps, min((s + 1) * cps, nchunks)) of a row.  A
// warp streams its (group, chunk) units in order with two register buffers,
// loading unit u + 1 (possibly the next group's first chunk) while unit u
// is computed (one token), or right after it (more tokens).  Warps of a
// group past the last tile compute nothing but still meet their CTA at
// every tile's barrier.
struct Cursor {
    int i, c;  // group iteration and chunk of the next unit to load
};

// Two register buffers of weights for one token (chunk u + 1 in flight while
// chunk u is computed); with more tokens one buffer, issued as soon as the
// previous chunk's compute is done: the SM's other warps (12 to 16,
// batch_reg_cap) hide each other's load latency better than 8 warps with
// two buffers (which would need more than 168 registers and spill).
template <int NT>
constexpr bool kTwoBuffers = NT == 1;

// With one buffer, lane 0 asks L2 for chunk u + 1 (one bulk prefetch of its
// contiguous bytes) before chunk u computes, so that the register loads
// issued after the compute find it there: 7B at 2 and 4 tokens 14.8 -> 13.9
// and 19.5 -> 18.6 us, the q4_K gate 7-9% faster.  q5_K at 4 tokens was
// slower with it (22.6 against 22.0 us) and goes without.
template <int NT, int FMT>
constexpr bool kPrefetchNext = !kTwoBuffers<NT> && !(FMT == 5 && NT == 4);

template <int FMT, int NT>
__device__ __forceinline__ void run_batch(const GemvLaunch &a, const GemvPart &P, uint8_t *xs, int lane)
{
    using W = typename Fmt<FMT>::W;
    constexpr int kChunkBytes = Fmt<FMT>::kChunkBytes;
    const int S = a.splits, G = a.wpc / S;
    const int w = threadIdx.x >> 5, sp = w % S, o = w / S;
    const int c_lo = sp * a.cps, c_hi = min(c_lo + a.cps, a.nchunks);
    const int group0 = blockIdx.x * a.tpi;
    const int n_units = a.tpi * (c_hi - c_lo);
    auto tile_of = [&](int i) { return (group0 + i) * G + o; };
    auto unit_at = [&](const Cursor &k) {
        const int t = tile_of(k.i);
        Unit x = locate(a, P, t < P.ntiles ? t : 0, k.c, lane, kChunkBytes);
        x.t = t;
        x.active = x.active && t < P.ntiles;
        return x;
    };
    auto advance = [&](Cursor &k) {
        if (++k.c == c_hi) { k.c = c_lo; ++k.i; }
    };

    W A, B;
    Cursor next{0, c_lo};
    Unit xa = unit_at(next), xb;
    load_w(xa, lane, A);  // weights do not depend on the preceding kernel
    stage_planes(a, xs);  // the planes and y do
    advance(next);

    Acc<NT> acc;
#pragma unroll
    for (int k = 0; k < (Acc<NT>::kEach ? 1 : NT); ++k)
#pragma unroll
        for (int r = 0; r < 8; ++r) acc.v[k][r] = 0.0f;
#pragma unroll
    for (int k = 0; k < (Acc<NT>::kEach ? NT : 1); ++k) acc.s[k] = 0.0f;

    int done = 0;  // tiles flushed so far
    if constexpr (!kTwoBuffers<NT>) {  // one buffer: the next chunk's loads follow its compute
        for (int u = 0; u < n_units; ++u) {
            if (kPrefetchNext<NT, FMT> && lane == 0 && u + 1 < n_units) {
                const Unit nx = unit_at(next);
                if (nx.t < P.ntiles) prefetch_l2(nx.seg, (unsigned)(kChunkBytes / kChunkBlocks * nx.cb));
            }
            compute<FMT, NT>(a, xs, xa, lane, A, acc);
            const int t = xa.t;
            const bool last = xa.c == c_hi - 1;
            if (u + 1 < n_units) {
                xa = unit_at(next);
                load_w(xa, lane, A);
                advance(next);
            }
            if (last) {
                flush_tile<NT, FMT>(a, P, t, t < P.ntiles, done, acc, lane);
                ++done;
            }
        }
    } else {
        for (int u = 0; u < n_units; u += 2) {
            const bool has_b = u + 1 < n_units;
            if (has_b) {
                xb = unit_at(next);
                load_w(xb, lane, B);
                advance(next);
            }
            compute<FMT, NT>(a, xs, xa, lane, A, acc);
            if (xa.c == c_hi - 1) {
                flush_tile<NT, FMT>(a, P, xa.t, xa.t < P.ntiles, done, acc, lane);
                ++done;
            }
            if (!has_b) break;
            const bool has_a = u + 2 < n_units;
            if (has_a) {
                xa = unit_at(next);
                load_w(xa, lane, A);
                advance(next);
            }
            compute<FMT, NT>(a, xs, xb, lane, B, acc);
            if (xb.c == c_hi - 1) {
                flush_tile<NT, FMT>(a, P, xb.t, xb.t < P.ntiles, done, acc, lane);
                ++done;
            }
        }
    }
}

// One kernel per (tokens, format): each gets its own register allocation.
template <int NT, int FMT>
__global__ void __maxnreg__(batch_reg_cap(NT, FMT))
    gemv_batch_kernel(const __grid_constant__ GemvLaunch a)
{
    extern __shared__ __align__(16) uint8_t xs[];  // the nt q8 planes
    const int lane = threadIdx.x & 31;
    griddep_launch_dependents();
    run_batch<FMT, NT>(a, a.part[0], xs, lane);
}

using KernelFn = void (*)(GemvLaunch);

template <int NT>
KernelFn kernel_of_fmt(int fmt)
{
    return fmt == 6 ? gemv_batch_kernel<NT, 6> : fmt == 5 ? gemv_batch_kernel<NT, 5>
         : fmt == 4 ? gemv_batch_kernel<NT, 4> : nullptr;
}

KernelFn kernel_for(int nt, int fmt)
{
    switch (nt) {
    case 1: return kernel_of_fmt<1>(fmt);
    case 2: return kernel_of_fmt<2>(fmt);
    case 3: return kernel_of_fmt<3>(fmt);
    case 4: return kernel_of_fmt<4>(fmt);
    case 5: return kernel_of_fmt<5>(fmt);
    case 6: return kernel_of_fmt<6>(fmt);
    case 7: return kernel_of_fmt<7>(fmt);
    case 8: return kernel_of_fmt<8>(fmt);
    default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_gemv_batch(const GemvLaunch &a, cudaStream_t st)
{
    const KernelFn k = kernel_for(a.nt, a.part[0].fmt);
    if (!k) return cudaErrorInvalidValue;
    const int warps = gemv_batch_cta_warps(a.splits, a.wpc);
    return launch_maybe_pdl(k, dim3((unsigned)a.n_items), dim3(32 * warps),
                            (size_t)a.nt * a.q8_bytes, a.pdl, st, a);
}

int gemv_batch_ctas_per_sm(int nt, int fmt, int warps_per_cta, size_t smem)
{
    const KernelFn k = kernel_for(nt, fmt);
    int blocks = 0;
    if (!k) return 0;
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, 32 * warps_per_cta, smem);
    if (e != cudaSuccess) cuda_fail("small-batch GEMV occupancy", e);
    return e == cudaSuccess ? blocks : -1;
}

size_t gemv_batch_max_smem()
{
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int limit = optin - 8192;  // room for the split-exchange buffers
    for (int nt = 1; nt <= kMaxTokens && e == cudaSuccess; ++nt)
        for (int fmt : {6, 4, 5})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kernel_for(nt, fmt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         limit);
    if (e != cudaSuccess) {
        cuda_fail("small-batch GEMV shared-memory opt-in", e);
        return 0;
    }
    return (size_t)limit & ~(size_t)15;
}

}  // namespace mq
