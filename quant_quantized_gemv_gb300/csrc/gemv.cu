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
//     kernel time is weight streaming), so there are no tensor cores and the
//     weights go straight to registers: each lane issues 14 (q6_K), 9 (q4_K)
//     or 11 (q5_K) independent 16-byte loads per chunk, every warp-wide load
//     of a plane covers 512 contiguous bytes (q4_K's scales and block scales
//     included: one META entry per lane), and the weight loads bypass L1
//     (ld.global.nc.L1::no_allocate) because each byte is used once.
//   * One register buffer per lane and a 128-register cap, so 16 warps fit
//     an SM: a warp issues chunk u+1's loads (~7 KB per warp) as soon as
//     chunk u is computed, and the other warps of the SM hide the latency.
//     Two buffers at 168 registers (12 warps per SM, each with a chunk in
//     flight while it computes the other) measured slower on GB300: 14B
//     decode sweep 2.383 against 2.298 ms per step, 5120 x 13824 13.7
//     against 12.4 us, 3584 x 18944 12.38 against 11.71 us, the 152064 x
//     5120 head equal (93.4 against 93.0 us).
//   * One resident wave of warps: the host sizes the grid to the number of
//     warps the SMs can hold.  A warp's work item is a contiguous run of
//     chunk units: whole 8-row tiles when there are more tiles than warps,
//     else one of `splits` tile-aligned column ranges of a tile ("split-K",
//     the tall-row case of page "74 · D4-2", §2).  Lane i owns unit i of each
//     chunk for the tile's 8 rows, so its activation codes are loaded once
//     per chunk and reused 8 times.
//   * A whole tile is reduced (fixed 9-shuffle butterfly) and written
//     directly.  With 2..12 splits the splits of a tile are the warps of one
//     CTA and meet in shared memory (one __syncthreads, ascending split
//     order).  With more splits (very few tiles, very long rows) each split
//     leaves its 8 partial sums in the workspace and the split that arrives
//     last (atomic ticket, no waiting) loads all of them at once and adds
//     them in ascending split order.  Either way the result does not depend
//     on arrival order, and the host proves before launch that the splits
//     cover every chunk exactly once (the page's §6 lesson).
//   * With whole-tile plans the q8 plane (a few KB to ~25 KB) is copied once
//     per CTA into shared memory and every lane reads its activation codes
//     from there: each plane byte leaves L2 once per CTA instead of once per
//     warp and tile.  Split plans read each activation chunk from L2 with
//     its weights, one chunk ahead (a CTA there reads each byte once).
//   * Opt-in (mq_set_gemv_ring): a ring of 1..3 shared-memory slots per warp
//     filled with 16-byte cp.async copies, so that the next chunks stream
//     while one is computed from registers.  Bitwise the same results; off
//     by default because it measured slower on every matrix of the 14B
//     decode step on GB300 (faster only for whole-tile q4_K shapes with few
//     warps per SM).
//   * With programmatic dependent launch the first chunk's weight loads are
//     issued before griddepcontrol.wait, so the weight stream starts while
//     the preceding kernel (the q8 producer) drains; the q8 plane, the
//     output and the workspace are touched only after the wait.  The plane
//     is read through L2 (ld.global.cg, or cp.async.cg copies into shared
//     memory), never the non-coherent path: the compiler treats
//     non-coherent loads as invariant and may hoist them above the wait,
//     and under PDL the plane is still being written then.
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

// Tile t of part P is finished for this warp (work item `item`, covering the
// part's units [u0, u1)): write it, or combine it with the tile's other splits.
// WS: the workspace combine (splits > kMaxCtaSplits) is compiled in.
template <bool WS>
__device__ __forceinline__ void flush_tile(const GemvLaunch &a, const GemvPart &P, int t,
                                           float (&acc)[8], int item, int u0, int u1, int lane)
{
    __shared__ float cta_part[kMaxCtaSplits][8];
    const float v = reduce8(acc, lane);
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    const int row0 = t * kTileRows;
    const int tu0 = t * a.nchunks, tu1 = tu0 + a.nchunks;
    if (tu0 >= u0 && tu1 <= u1) {  // whole tile in this range
        if ((lane & 3) == 0 && row0 + (lane >> 2) < P.rows) P.y[row0 + (lane >> 2)] = v;
        return;
    }
    if (a.splits <= kMaxCtaSplits) {
        // the splits of tile t are the warps of this CTA (one flush each):
        // combine through shared memory in ascending split order
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
        return;
    }
    if constexpr (!WS) return;  // the launch never gives this instance such a plan
    // more splits than a CTA holds: lane 0 publishes the 8 partials to the
    // workspace, fences them and takes a ticket (writer and ticket holder are
    // one thread); the last of the tile's splits adds them all
    float *dst = a.ws_part + (size_t)item * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float pk = __shfl_sync(kFull, v, 4 * k);
        if (lane == 0) dst[k] = pk;
    }
    const int gt = P.tile0 + t;  // global tile
    int last = 0;
    if (lane == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(a.ws_cnt + gt, 1u);
        last = prev == (unsigned)(a.splits - 1);
    }
    last = __shfl_sync(kFull, last, 0);
    if (!last) return;
    __threadfence();
    // last arriver: lane (8g + r) loads split base+g of row r, four splits
    // per round trip; lanes 0..7 add them in ascending split order
    const float *base_ptr = a.ws_part + ((size_t)P.item0 + (size_t)t * a.splits) * 8;
    float sum = 0.0f;
    for (int base = 0; base < a.splits; base += 4) {
        const int s = base + (lane >> 3);
        const float p = s < a.splits ? __ldcg(base_ptr + (size_t)s * 8 + (lane & 7)) : 0.0f;
        const float p1 = __shfl_down_sync(kFull, p, 8);
        const float p2 = __shfl_down_sync(kFull, p, 16);
        const float p3 = __shfl_down_sync(kFull, p, 24);
        sum = (((sum + p) + p1) + p2) + p3;
    }
    if (lane < 8 && row0 + lane < P.rows) P.y[row0 + lane] = sum;
    if (lane == 0) a.ws_cnt[gt] = 0u;  // ready for the next call
}

// Wait for the producer.  Whole-tile plans (splits == 1) then copy the whole
// q8 plane into shared memory once per CTA (16-byte cp.async copies through
// L2, all in flight at once) and meet at named barrier 1: every warp of such a CTA calls this
// exactly once, from whichever code path it is on (a named barrier counts
// arrivals, not call sites).  Returns where the activation is read from:
// the shared copy, or null for the global plane (split plans, whose CTAs
// read each plane byte once anyway).
__device__ __forceinline__ const uint8_t *stage_plane(const GemvLaunch &a, uint8_t *xs)
{
    griddep_wait();  // the q8 plane, y and the workspace depend on it
    if (a.splits != 1) return nullptr;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q8);
    uint4 *dst = reinterpret_cast<uint4 *>(xs);
    const int n16 = (int)(a.q8_bytes >> 4);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) copy16_async(dst + i, src + i);
    copy_async_wait_all();
    asm volatile("bar.sync 1, %0;" ::"r"(blockDim.x) : "memory");
    return xs;
}

// Kernel modes: the GEMV; its integer sub-dots; the GEMV that also counts,
// per (tile, chunk) unit, how many times a warp processed it (a debug and
// test aid that checks the work decomposition on the device).
constexpr int kModeGemv = 0, kModeSubdots = 1, kModeCover = 2;

// Stream the part's units [u0, u1) through one register buffer: compute a
// chunk, issue the next chunk's loads into the same registers, then finish
// the tile if the chunk was its last.
template <int FMT, int MODE, bool WS = true>
__device__ __forceinline__ void run_range(const GemvLaunch &a, const GemvPart &P, uint8_t *smem,
                                          int item, int u0, int u1, int lane)
{
    using Regs = typename Fmt<FMT>::Regs;
    constexpr int kChunkBytes = Fmt<FMT>::kChunkBytes;
    const int nch = a.nchunks;
    Regs A;
    int t = u0 / nch, c = u0 - t * nch;  // position of the next chunk to load
    Unit xa = locate(a, P, t, c, lane, kChunkBytes);
    load_w(xa, lane, A);   // weights do not depend on the preceding kernel
    const uint8_t *xs = stage_plane(a, smem);  // the q8 plane, y and the workspace do
    load_x(a, xs, xa, lane, A);
    if (++c == nch) { c = 0; ++t; }

    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    for (int u = u0; u < u1; ++u) {
        const int tcur = xa.t;
        constexpr bool SUBDOTS = MODE == kModeSubdots;
        if constexpr (MODE == kModeCover) {
            if (lane == 0) atomicAdd(a.cover + ((size_t)(P.tile0 + xa.t) * nch + xa.c), 1u);
        }
        compute<SUBDOTS>(a, P, A, xa, lane, acc);
        const bool more = u + 1 < u1;
        if (more) {
            xa = locate(a, P, t, c, lane, kChunkBytes);
            load_w(xa, lane, A);
            load_x(a, xs, xa, lane, A);
            if (++c == nch) { c = 0; ++t; }
        }
        if (!SUBDOTS && (!more || xa.t != tcur)) flush_tile<WS>(a, P, tcur, acc, item, u0, u1, lane);
    }
}

// The same through the warp's ring of S shared-memory slots.  Every lane
// copies 16-byte words lane, lane + 32, ... of each upcoming chunk (the chunk
// verbatim, so the layout's offsets hold in the slot) with asynchronous
// copies, one copy group per chunk.  Chunk u's group is complete when at most
// S - 1 newer groups are pending; a __syncwarp then makes every lane's words
// visible to the warp.  The warp moves the chunk into its registers, meets
// again (every lane has read the slot), refills the slot with the chunk S
// ahead -- before computing, so the next chunks stream while this one is
// computed -- and computes.  Cursors advance incrementally (no division).
template <int FMT, int MODE, int S>
__device__ __forceinline__ void run_range_ring(const GemvLaunch &a, const GemvPart &P,
                                               uint8_t *smem, int item, int u0, int u1, int lane)
{
    using Regs = typename Fmt<FMT>::Regs;
    using X = typename Fmt<FMT>::X;
    constexpr int kChunkBytes = Fmt<FMT>::kChunkBytes;
    constexpr int kWords = kChunkBytes / 16;           // 16-byte words of a full chunk
    constexpr int kPerLane = (kWords + 31) / 32;       // copies per lane of a full chunk
    constexpr bool SUBDOTS = MODE == kModeSubdots;
    const int nch = a.nchunks;
    const int last_words = (a.nb - kChunkBlocks * (nch - 1)) * (kWords / kChunkBlocks);
    const size_t tile_bytes = (size_t)P.tile_bytes_div16 * 16;
    const uint32_t ring =
        smem_addr(smem) + a.ring_off + (uint32_t)(threadIdx.x >> 5) * (uint32_t)(S * a.slot_bytes);
    // issue cursor: the next chunk to copy, its slot, how many remain
    int it = u0 / nch, ic = u0 - it * nch, is = 0, left = u1 - u0;
    const uint8_t *isrc = P.W + (size_t)it * tile_bytes + (size_t)ic * kChunkBytes;
    auto issue = [&]() {
        if (left > 0) {
            const int words = ic == nch - 1 ? last_words : kWords;
            const uint32_t dst = ring + (uint32_t)is * a.slot_bytes + 16u * (uint32_t)lane;
            const uint8_t *src = isrc + 16 * lane;
#pragma unroll
            for (int k = 0; k < kPerLane; ++k)
                if (lane + 32 * k < words) cp_async16(dst + 512u * k, src + 512 * k);
            --left;
            is = is + 1 == S ? 0 : is + 1;
            if (++ic == nch) {
                ic = 0;
                ++it;
                isrc = P.W + (size_t)it * tile_bytes;
            } else {
                isrc += kChunkBytes;
            }
        }
        cp_async_commit();
    };
    const int npre = min(a.pre, S);
    for (int j = 0; j < npre; ++j) issue();     // weights do not depend on the preceding kernel
    const uint8_t *xs = stage_plane(a, smem);  // the q8 plane, y and the workspace do
    for (int j = npre; j < S; ++j) issue();
    int t = u0 / nch, c = u0 - t * nch, rs = 0;  // compute cursor and its slot
    Unit x = locate(a, P, t, c, lane, kChunkBytes);
    X xn;  // the activation of chunk x, loaded a chunk ahead
    load_x(a, xs, x, lane, xn);

    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    Regs A;
    for (int u = u0; u < u1; ++u) {
        if (S == 1)
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        else if (S == 2)
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        else
            asm volatile("cp.async.wait_group 2;" ::: "memory");
        __syncwarp();  // every lane's words of chunk u are visible
        load_w_from(SharedChunk{ring + (uint32_t)rs * a.slot_bytes}, x, lane, A);
        static_cast<X &>(A) = xn;
        rs = rs + 1 == S ? 0 : rs + 1;
        __syncwarp();  // every lane has read the slot: refill it
        issue();
        const Unit xc = x;
        if (u + 1 < u1) {
            if (++c == nch) { c = 0; ++t; }
            x = locate(a, P, t, c, lane, kChunkBytes);
            load_x(a, xs, x, lane, xn);
        }
        if constexpr (MODE == kModeCover) {
            if (lane == 0) atomicAdd(a.cover + ((size_t)(P.tile0 + xc.t) * nch + xc.c), 1u);
        }
        compute<SUBDOTS>(a, P, A, xc, lane, acc);
        if (!SUBDOTS && (u + 1 == u1 || x.t != xc.t)) flush_tile<true>(a, P, xc.t, acc, item, u0, u1, lane);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // only empty groups remain
}

template <int FMT, int MODE>
__device__ __forceinline__ void run_ring(const GemvLaunch &a, const GemvPart &P, uint8_t *smem,
                                         int item, int u0, int u1, int lane)
{
    if (a.stages == 1)
        run_range_ring<FMT, MODE, 1>(a, P, smem, item, u0, u1, lane);
    else if (a.stages == 2)
        run_range_ring<FMT, MODE, 2>(a, P, smem, item, u0, u1, lane);
    else
        run_range_ring<FMT, MODE, 3>(a, P, smem, item, u0, u1, lane);
}

// CTA shapes: splits == 1 (whole tiles) and splits > kMaxCtaSplits use CTAs
// of kGemvWarpsPerBlock independent warps; 2..kMaxCtaSplits splits use one
// CTA per tile whose warps are its splits.  The part of a work item is found
// with constant indices (the part table stays in parameter space).
// One kernel serves every format (the part's format picks the code path):
// in a decode chain with programmatic dependent launch, switching between
// kernel functions from one GEMV to the next costs more than the branch.
// Measured on the 14B sweep: 2.39 ms with one kernel for all formats
// against 2.49 ms with a kernel per format set (qkv, o, down alternating).
// Code a launch never runs still costs it on GB300, so the kernel comes in
// three instances (KIND): q6_K and q4_K parts with at most kMaxCtaSplits
// splits (no workspace combine), every format and plan, and the weight ring
// (every format; launched only when a.stages > 0).  With the ring's code
// compiled into the default kernel the 14B sweep's GEMVs took 2174 against
// 2114 us per step and its PDL step 2219 against 2178 us (single shapes
// 1-2%); without the q5_K path as well the step took 2161 against 2171 us;
// without the workspace combine as well the GEMVs took 2105 against 2114 us
// (5120 x 5120 q4_K 5.48 against 5.59 us).  Every launch of the sweep uses
// the first instance, so its chain never switches kernel functions.
// A fourth instance (kKindQ46Lo), the first one compiled at kGemvGroupRegs
// registers, serves grouped launches: 21 warps per SM let the 14B q/k/v group (896 tiles
// of 5 chunks) run 3 splits per tile (at most 2 chunks per warp) in one
// wave, and its CTAs become resident sooner behind the previous kernel of a
// PDL chain.  The 14B sweep's PDL step took 2091.6 against 2115.9 us with
// it (q/k/v 7.33 against 8.38 us); its GEMVs back to back 2099.7 against
// 2093.6 us, the cost of switching kernel functions between q/k/v and the
// other launches.  At 96 registers for every launch the single shapes were
// slower (5120 x 5120 q4_K 5.90 against 5.60 us, the head 98.7 against
// 95.8 us).
constexpr int kKindQ46 = 0, kKindAll = 1, kKindRing = 2, kKindQ46Lo = 3;
template <int MODE, int KIND>
__global__ void __maxnreg__(MODE == kModeSubdots ? 168
                            : KIND == kKindQ46Lo ? kGemvGroupRegs
                                                 : kGemvMaxRegs)
    gemv_kernel(const __grid_constant__ GemvLaunch a)
{
    extern __shared__ __align__(16) uint8_t xs[];  // the q8 plane, staged per CTA
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    griddep_launch_dependents();
    if (item >= a.n_items) {
        // no work item (only in the last CTA of a whole-tile or workspace
        // grid): still help stage the plane, then leave.  CTAs that combine
        // splits in shared memory are launched exact.
        stage_plane(a, xs);
        return;
    }
    int pi = 0;
#pragma unroll
    for (int k = 1; k < kMaxParts; ++k)
        if (k < a.nparts && item >= a.part[k].item0) pi = k;
    const GemvPart &P = a.part[pi];  // stays in the kernel's constant parameter space
    const int li = item - P.item0;
    const int nch = a.nchunks;
    int u0, u1;
    if (a.splits > 1) {
        const int tt = li / a.splits, s = li - tt * a.splits;
        u0 = tt * nch + s * a.cps;
        u1 = tt * nch + min(s * a.cps + a.cps, nch);
    } else {
        u0 = li * a.tpi * nch;
        u1 = min(u0 + a.tpi * nch, P.ntiles * nch);
    }
    if constexpr (KIND == kKindRing) {
        if (P.fmt == 6)
            run_ring<6, MODE>(a, P, xs, item, u0, u1, lane);
        else if (P.fmt == 5)
            run_ring<5, MODE>(a, P, xs, item, u0, u1, lane);
        else
            run_ring<4, MODE>(a, P, xs, item, u0, u1, lane);
    } else if constexpr (KIND == kKindQ46 || KIND == kKindQ46Lo) {
        if (P.fmt == 6)
            run_range<6, MODE, false>(a, P, xs, item, u0, u1, lane);
        else
            run_range<4, MODE, false>(a, P, xs, item, u0, u1, lane);
    } else {
        if (P.fmt == 6)
            run_range<6, MODE>(a, P, xs, item, u0, u1, lane);
        else if (P.fmt == 5)
            run_range<5, MODE>(a, P, xs, item, u0, u1, lane);
        else
            run_range<4, MODE>(a, P, xs, item, u0, u1, lane);
    }
}

template <int MODE>
cudaError_t launch(const GemvLaunch &a, cudaStream_t st)
{
    const int warps = gemv_cta_warps(a.splits, MODE == kModeSubdots);
    const long long blocks = (a.n_items + warps - 1) / warps;
    const size_t smem = gemv_dyn_smem(warps, a.splits == 1, a.q8_bytes, a.stages, a.slot_bytes);
    const dim3 grid((unsigned)blocks), block(32 * warps);
    if (a.stages > 0) return launch_maybe_pdl(gemv_kernel<MODE, kKindRing>, grid, block, smem, a.pdl, st, a);
    bool q5 = false;
    for (int p = 0; p < a.nparts; ++p) q5 = q5 || a.part[p].fmt == 5;
    if constexpr (MODE == kModeGemv) {  // (no q6_K/q4_K instance of the other modes is built)
        if (!q5 && a.splits <= kMaxCtaSplits && a.lo)
            return launch_maybe_pdl(gemv_kernel<MODE, kKindQ46Lo>, grid, block, smem, a.pdl, st, a);
        if (!q5 && a.splits <= kMaxCtaSplits)
            return launch_maybe_pdl(gemv_kernel<MODE, kKindQ46>, grid, block, smem, a.pdl, st, a);
    }
    return launch_maybe_pdl(gemv_kernel<MODE, kKindAll>, grid, block, smem, a.pdl, st, a);
}

using KernelFn = void (*)(GemvLaunch);
const KernelFn kAllKernels[] = {
    gemv_kernel<kModeGemv, kKindQ46>,    gemv_kernel<kModeGemv, kKindAll>,
    gemv_kernel<kModeGemv, kKindRing>,   gemv_kernel<kModeSubdots, kKindAll>,
    gemv_kernel<kModeSubdots, kKindRing>, gemv_kernel<kModeCover, kKindAll>,
    gemv_kernel<kModeCover, kKindRing>,   gemv_kernel<kModeGemv, kKindQ46Lo>};

}  // namespace

cudaError_t launch_gemv(const GemvLaunch &a, cudaStream_t st) { return launch<kModeGemv>(a, st); }
cudaError_t launch_subdots(const GemvLaunch &a, cudaStream_t st) { return launch<kModeSubdots>(a, st); }
cudaError_t launch_cover(const GemvLaunch &a, cudaStream_t st) { return launch<kModeCover>(a, st); }

int gemv_ctas_per_sm(int warps_per_cta, size_t smem)
{
    int blocks = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &blocks, gemv_kernel<kModeGemv, kKindAll>, 32 * warps_per_cta, smem);  // the others: the same
    if (e != cudaSuccess) cuda_fail("GEMV occupancy", e);
    return e == cudaSuccess ? blocks : 0;
}

int gemv_ctas_per_sm_lo(int warps_per_cta, size_t smem)
{
    int blocks = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &blocks, gemv_kernel<kModeGemv, kKindQ46Lo>, 32 * warps_per_cta, smem);
    if (e != cudaSuccess) cuda_fail("GEMV occupancy", e);
    return e == cudaSuccess ? blocks : 0;
}

size_t gemv_max_plane_bytes()
{
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int limit = optin - 1024;  // room for the kernel's static shared memory
    for (KernelFn k : kAllKernels)
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (e != cudaSuccess) {
        cuda_fail("GEMV shared-memory opt-in", e);
        return 0;
    }
    return (size_t)limit & ~(size_t)15;
}

}  // namespace mq
