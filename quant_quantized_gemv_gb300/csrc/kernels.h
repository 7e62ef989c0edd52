// kernels.h -- launch interface between the C ABI (api.cpp) and the CUDA
// kernels (gemv.cu, producers.cu).  Internal to the library.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mq {

// One GEMV launch over a group of 1..kMaxParts matrices ("parts") that
// share one q8 activation plane (the same cols): q, k, v of a layer, or its
// gate and up.  Each part is cut into ntiles tiles of 8 rows x nchunks chunk
// units (chunk = 4 super-blocks).  A work item (one warp) streams a
// contiguous range of one part's units:
//   splits == 1: whole tiles, tpi per item (a part's last item may hold fewer);
//   splits > 1 (tall rows): one of `splits` tile-aligned column ranges of a
//     tile, chunks [s*cps, min((s+1)*cps, nchunks)).  Up to kMaxCtaSplits the
//     splits of a tile are the warps of one CTA and combine in shared memory;
//     beyond that they combine through the workspace, where the last one to
//     finish adds the partials in ascending split order.
// Items are numbered part by part; part p owns items [item0, item0 + items)
// and global tiles [tile0, tile0 + ntiles).
constexpr int kMaxParts = 8;

struct GemvPart {
    const uint8_t *W;       // repacked weights (layout.h)
    float *y;               // rows outputs
    int rows, ntiles;
    int fmt;                // 6 = q6_K, 4 = q4_K
    int item0, tile0;       // first work item and first global tile of the part
    int tile_bytes_div16;   // bytes of one 8-row tile / 16
};

struct GemvLaunch {
    GemvPart part[kMaxParts];
    int nparts;
    const uint8_t *q8;      // q8 plane of cols values
    int32_t *isums;         // sub-dot mode (one part): rows * nb * {16 | 8} int32, else null
    unsigned *ws_cnt;       // arrival counters [total tiles] (splits > kMaxCtaSplits)
    float *ws_part;         // partials [n_items][8 rows] (splits > kMaxCtaSplits)
    int nb, nchunks;        // super-blocks and chunks per row (all parts)
    int splits, cps, tpi;   // the plan (see above)
    int n_items;
    unsigned q8_d_off, q8_sum_off;
    unsigned q8_bytes;      // bytes of the q8 plane (multiple of 16), staged in shared memory
    int pdl;                // launch with programmatic stream serialization
    int nt;                 // activation rows (tokens) of the small-batch kernel
    unsigned q8_stride;     // bytes from one token's plane to the next (small batch)
    unsigned *cover;        // coverage mode: a count per (global tile, chunk), else null
    int wpc;                // small batch: warps a CTA may hold (its plan's G = wpc / splits)
    // single-token GEMV weight ring: each warp keeps `stages` chunks in
    // flight in its own shared-memory slots of slot_bytes (the largest chunk
    // of the launch's formats), after the staged plane (ring_off bytes, 0 on
    // split plans); `pre` of them are requested before the grid-dependency
    // wait.  stages == 0: chunks go straight to registers.
    int stages, pre;
    unsigned slot_bytes, ring_off;
    // grouped launches (q6_K/q4_K parts, default plan, no ring): the
    // kGemvGroupRegs instance, planned with its own occupancy
    int lo;
};

cudaError_t launch_gemv(const GemvLaunch &a, cudaStream_t st);
cudaError_t launch_subdots(const GemvLaunch &a, cudaStream_t st);
// The GEMV that also adds 1 to a.cover[global tile * nchunks + chunk] for
// every unit a warp processes (a device-side check of the decomposition).
cudaError_t launch_cover(const GemvLaunch &a, cudaStream_t st);
// Gate||up GEMV with the SwiGLU -> q8 epilogue (gemv_gateup.cu): g.part[0]
// is gate, g.part[1] is up (same rows and format), g.q8 the input plane.
// Rows come in q8 blocks of 32 (rows % 32 == 0); a CTA of wpb warps (1..8)
// takes whole blocks, grid-stride over nblk blocks.
struct GateUpLaunch {
    GemvLaunch g;
    float *act;                   // rows outputs: silu(gate) * up
    uint8_t *q8o;                 // act's q8 plane (rows values)
    unsigned o_d_off, o_sum_off;  // its fp16-scale and sum sections
    int nblk;                     // rows / 32
    int wpb;                      // warps per CTA
};
cudaError_t launch_gateup(const GateUpLaunch &L, int ctas, cudaStream_t st);
int gateup_ctas_per_sm(int fmt, int warps_per_cta, size_t smem);
bool gateup_opt_in(size_t max_plane);  // accept a staged plane of max_plane bytes

// Small-batch GEMV (gemv_batch.cu), 1 <= a.nt <= kMaxTokens, one part whose
// y holds nt x rows outputs, token-major.  Its plan reads differently: each
// CTA holds `splits` warps for each of wpc / splits tiles (a
// group) and runs tpi consecutive groups; n_items is the number of CTAs.
cudaError_t launch_gemv_batch(const GemvLaunch &a, cudaStream_t st);

// q6_K GEMV against an f32 activation row (gemv_f32.cu): one part; q8 is
// the row (cols floats) and q8_bytes its size; whole-tile plans or 2..12
// splits per tile (no workspace).  Every CTA stages the row.
cudaError_t launch_gemv_f32(const GemvLaunch &a, cudaStream_t st);
int gemv_f32_ctas_per_sm(int warps_per_cta, size_t smem);
size_t gemv_f32_max_x_bytes();  // largest row it stages; opts the kernel in

constexpr int kGemvWarpsPerBlock = 4;   // CTA of independent warps
constexpr int kGemvMaxRegs = 128;       // single-token GEMV registers per thread: 16 warps per SM
constexpr int kGemvGroupRegs = 96;      // its grouped launches' instance: 21 warps per SM
// Resident CTAs per SM of that instance (0 on error).
int gemv_ctas_per_sm_lo(int warps_per_cta, size_t smem);
constexpr int kMaxCtaSplits = 12;       // largest CTA whose warps are one tile's splits
constexpr int kGemvStaticSmem = kMaxCtaSplits * 8 * 4;  // the split-combine buffer
constexpr int kMaxTokens = 8;           // activation rows of the small-batch GEMV
constexpr int kBatchMaxCtaSplits = 12;  // most splits of a tile (warps of one tile in a CTA)
constexpr int kBatchMaxCtaWarps = 16;   // most warps of a CTA (a whole SM at 128 registers)
constexpr int kBatchStaticSmem = 2 * kBatchMaxCtaSplits * kMaxTokens * 8 * 4;  // split exchange (max)

// Register cap of the small-batch kernel for nt tokens of format fmt: for
// q6_K and q5_K the smallest that compiles without spilling, so that as
// many warps as possible fit an SM; one token keeps two weight buffers and
// 5..8 tokens take 168.  At 5 tokens 168 still spills (q6_K 164 bytes,
// q5_K 16), but 176 or 184 registers (11 warps) measured far slower (7B
// 22.4 -> 28.8 us).  3 tokens of q6_K spilled 24 bytes at 136 and are
// faster spill-free at 144 with a warp less (head 108.9 -> 103.0 us), 4 of
// q5_K spilled 8 at 152 (22.59 -> 22.44 us at 160).  q4_K keeps 168 (12
// warps): more warps measured slower there (14B gate at 2 tokens 13.2
// against 12.6 us).
__host__ __device__ constexpr int batch_reg_cap(int nt, int fmt)
{
    return fmt == 4 ? 168
         : nt == 2 ? 128
         : nt == 3 ? (fmt == 6 ? 144 : 136)
         : nt == 4 ? (fmt == 6 ? 168 : 160)
         : 168;
}
// Most warps a CTA can hold at that cap (at most 16): sizes the kernel's
// split-exchange buffer.  The warps a CTA actually holds (GemvLaunch::wpc)
// come from the device's occupancy query and never exceed this.
__host__ __device__ constexpr int batch_warp_budget_max(int nt, int fmt)
{
    return 65536 / (32 * batch_reg_cap(nt, fmt)) < kBatchMaxCtaWarps
               ? 65536 / (32 * batch_reg_cap(nt, fmt))
               : kBatchMaxCtaWarps;
}

// Single-token GEMV weight ring (GemvLaunch::stages): most stages a warp
// may keep, and the dynamic shared memory of a CTA of `warps` warps.
constexpr int kGemvMaxStages = 3;
inline size_t gemv_ring_off(bool whole_tiles, size_t plane)
{
    return whole_tiles ? (plane + 127) & ~(size_t)127 : 0;
}
inline size_t gemv_dyn_smem(int warps, bool whole_tiles, size_t plane, int stages, size_t slot)
{
    return gemv_ring_off(whole_tiles, plane) + (size_t)warps * stages * slot;
}

// Warps per CTA for a plan with `splits` splits.
inline int gemv_cta_warps(int splits, bool subdots = false)
{
    return (!subdots && splits > 1 && splits <= kMaxCtaSplits) ? splits : kGemvWarpsPerBlock;
}

// Warps per CTA of the small-batch kernel: `splits` warps per tile times
// budget / splits tiles per group.
inline int gemv_batch_cta_warps(int splits, int budget)
{
    return splits * (budget / splits);
}

// Resident CTAs per SM of the small-batch kernel for nt tokens of format
// fmt (0 if such a CTA does not fit, -1 on error), and the largest dynamic
// shared memory (all nt planes) the small-batch kernels accept.
int gemv_batch_ctas_per_sm(int nt, int fmt, int warps_per_cta, size_t smem);
size_t gemv_batch_max_smem();

// Resident CTAs per SM of the GEMV kernel with `warps_per_cta` warps and
// `smem` bytes of dynamic shared memory, on the current device (0 on error).
int gemv_ctas_per_sm(int warps_per_cta, size_t smem);

// Largest q8 plane (bytes) the GEMV can stage in shared memory; makes the
// kernels accept that much dynamic shared memory on the current device.
size_t gemv_max_plane_bytes();

// Producers over `rows` rows of n values (row-major), writing one q8 plane
// per row, planes `stride` bytes apart.  d_off / sum_off locate a plane's
// fp16-scale and sum sections (layout.h q8_d_offset / q8_sum_offset).
cudaError_t launch_quantize_q8(const float *x, uint8_t *q8, int n, int rows, unsigned stride,
                               unsigned d_off, unsigned sum_off, int pdl, cudaStream_t st);
cudaError_t launch_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y,
                                    uint8_t *q8, int n, int rows, unsigned stride, unsigned d_off,
                                    unsigned sum_off, int pdl, cudaStream_t st);
cudaError_t launch_swiglu_quant_q8(const float *g, const float *u, float *y, uint8_t *q8, int n,
                                   int rows, unsigned stride, unsigned d_off, unsigned sum_off,
                                   int pdl, cudaStream_t st);

// A plain one-launch read of `bytes` (multiple of 16) from src: the floor for
// any kernel that streams those bytes once (readfloor.cu).  sink may be null.
cudaError_t launch_read_floor(const void *src, size_t bytes, unsigned *sink, int sms, cudaStream_t st);

// The host repack of repack.cpp on the device (repack_device.cu): zero-fills
// dst, then writes every unit's planes (fmt 6, 4 or 5; shape already checked).
cudaError_t launch_repack(int fmt, const void *src, void *dst, int rows, int cols, cudaStream_t st);

// Copy `bytes` (multiple of 16) from src to dst, both device-addressable
// (copy.cu), as a kernel that takes part in the launch chain.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int pdl, cudaStream_t st);

// The process-wide programmatic-dependent-launch setting (mq_set_pdl).
int pdl_setting();

// Record the library's last CUDA failure on this thread (`where` and the CUDA
// error, readable with mq_last_error); returns MQ_ERR_CUDA.
int cuda_fail(const char *where, cudaError_t e);

// Launch `kernel` on `st`, with programmatic stream serialization when pdl
// is set (the kernel then may start before its predecessor in the stream
// finishes and must call griddep_wait() before touching dependent data).
template <class... KArgs, class... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int pdl,
                             cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace mq

#ifdef __CUDACC__
// Programmatic dependent launch controls (no-ops without the attribute).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif
