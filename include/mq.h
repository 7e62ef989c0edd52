/*
 * mq.h -- C ABI of the GB300 (sm_103a) k-quant batch-1 decode GEMV library.
 *
 * What it computes (the minfer engineering log, cited by page and section):
 *   "76 · D4-4 — dpl dense split-plane q6_K decode MMVQ"      [D4-4]
 *   "74 · D4-2 — B0 latent correctness fix"                   [D4-2]
 *   "67 · D3 — 14B decode attribution / bitwise MMVQ"         [D3]
 *   "70 · D3-5 — fused-producer decode A-quantize"            [D3-5]
 * y = W x_hat, W a k-quantized matrix (GGUF q6_K or q4_K super-blocks of 256
 * weights), x_hat an activation row quantized to int8 in 32-value blocks
 * (the q8 plane), computed with integer sub-block dot products and an f32
 * scale combine.  The q8 plane is written by one of three producers.
 *
 * Conventions for every entry point:
 *   - All pointers are owned by the caller.  The library allocates and frees
 *     nothing.  "device" pointers must be CUDA device (or managed) memory of
 *     the current device; "host" pointers are ordinary host memory.
 *   - GPU entry points are asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and return after the launch.
 *   - Every call validates its arguments before launching anything and
 *     returns an mq_status: MQ_OK, or an error with nothing launched, or
 *     MQ_ERR_CUDA when the launch itself failed (cudaGetLastError()).
 *   - Shapes: cols % 256 == 0 (whole super-blocks, the gate of [D4-4] §3.1),
 *     n % 32 == 0 for the producers ([D3-5] §3.1), rows >= 1, all sizes
 *     below 2^31 elements.
 *   - Alignment: every device pointer must be 16-byte aligned (the vector
 *     loads of [D4-4] §3.3 "the dpl row base is not naturally 16B aligned").
 *   - Host-resident activations: the inputs x, g, u of the producers (single
 *     and batched) and the output rows y of the GEMVs may instead be pinned
 *     host memory, passed by the address mq_device_address gives for it (on
 *     GB300, with unified addressing, the host pointer of cudaHostAlloc
 *     memory itself).  The kernels then read or write it over NVLink-C2C,
 *     so a decode step needs no separate copy in or out.  Quantize and
 *     SwiGLU read each input element once; rms_norm reads its row once per
 *     CTA (the sum of squares), so a wide row is better copied in first
 *     (mq_copy).  The host must not touch such a buffer while a kernel that
 *     uses it may run.  Weights, q8 planes and workspaces stay in device
 *     memory.
 *   - Not thread-safe for the same workspace: calls that share a workspace
 *     must be ordered on one stream.
 */
#ifndef MQ_H
#define MQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MQ_OK = 0,
    MQ_ERR_SHAPE = 1,      /* a size breaks the shape rules above            */
    MQ_ERR_ALIGN = 2,      /* a device pointer is not 16-byte aligned         */
    MQ_ERR_NULL = 3,       /* a required pointer is NULL                      */
    MQ_ERR_COVERAGE = 4,   /* a dispatch plan would leave work uncovered or
                              cover it twice; nothing was launched ([D4-2] §6
                              lesson 1: a gate must bound both sides)         */
    MQ_ERR_WORKSPACE = 5,  /* split-K needs a larger workspace               */
    MQ_ERR_CUDA = 6,       /* a CUDA call failed (mq_last_error says which)   */
    MQ_ERR_ACCESS = 7      /* a pointer the GPU cannot address (pageable host
                              memory, or not an allocation CUDA knows)         */
} mq_status;

/* Static message for a status code. */
const char *mq_strerror(int status);

/* Library version string. */
const char *mq_version(void);

/* What the last MQ_ERR_CUDA on the calling thread came from: the library
 * step and CUDA's error text (empty before any).  The buffer is the
 * thread's own and is overwritten by its next failure. */
const char *mq_last_error(void);

/* ------------------------------------------------------------------------
 * Weight repack (host, once at load).  [D4-4] §2-§3.1: the GGUF q6_K block
 * (210 B: ql 128 | qh 64 | sc 16 | d 2) is rearranged once so that every byte
 * a decode GEMV streams from HBM is content.  The repacked form here groups
 * rows in tiles of 8 and columns in chunks of 4 super-blocks and stores each
 * tile-chunk as planes in the order the kernel's lanes read them; it is a
 * lossless permutation of the block's bits (exactly rows*cols/256 * 210 B of
 * content; rows are padded to a multiple of 8 with zero rows, which decode to
 * zero).  q4_K (144 B: d | dmin | scales 12 | qs 128, the GGUF q4_K block)
 * and q5_K (176 B: d | dmin | scales 12 | qh 32 | qs 128, the GGUF q5_K
 * block; the pages only name it, [D3-5] §4) are treated the same way.  The
 * repacked layout is private to this library.
 *
 * mq_repacked_bytes_*: bytes of the repacked matrix (0 on a bad shape).
 * mq_repack_*:   gguf (host, rows x cols/256 blocks, row-major, GGUF order)
 *                -> dst (host, mq_repacked_bytes_* bytes).  Overwrites dst.
 * mq_unrepack_*: the exact inverse: dst -> gguf.  Used to prove the repack is
 *                a permutation (round trip is the identity).
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE.  Host only, synchronous, thread-safe.
 * ------------------------------------------------------------------------ */
size_t mq_repacked_bytes_q6k(int rows, int cols);
size_t mq_repacked_bytes_q4k(int rows, int cols);
size_t mq_repacked_bytes_q5k(int rows, int cols);
int mq_repack_q6k(const void *gguf, void *dst, int rows, int cols);
int mq_repack_q4k(const void *gguf, void *dst, int rows, int cols);
int mq_repack_q5k(const void *gguf, void *dst, int rows, int cols);
int mq_unrepack_q6k(const void *packed, void *gguf, int rows, int cols);
int mq_unrepack_q4k(const void *packed, void *gguf, int rows, int cols);
int mq_unrepack_q5k(const void *packed, void *gguf, int rows, int cols);

/* ------------------------------------------------------------------------
 * The q8 activation plane ([D3-5] §3.2, the pad40 block's fields): for each
 * block of 32 values an fp16 scale d, 32 int8 values and their int32 sum.
 * The plane is stored split by field (qs | d | sum, each 16-byte aligned); it
 * is opaque to callers, who size it with mq_q8_bytes and read it (for tests)
 * with mq_q8_unpack_host.
 *
 * mq_q8_bytes(n): bytes of the plane for n values (0 unless n % 32 == 0).
 * mq_q8_unpack_host: plane (host copy) -> d[n/32] (fp16 bits), qs[n],
 *                    sum[n/32].  Any output pointer may be NULL.
 * ------------------------------------------------------------------------ */
size_t mq_q8_bytes(int n);
int mq_q8_unpack_host(const void *plane, int n, uint16_t *d, int8_t *qs, int32_t *sum);

/* ------------------------------------------------------------------------
 * Producers (device).  Each writes the q8 plane of n values, quantized per
 * 32-value block exactly as [D3-5] §3.2 prints it: am = max|v|, d = am/127,
 * di = d != 0 ? 1/d : 0 (IEEE f32), q = clamp(rint(v * di), -128, 127)
 * (rint rounds half to even), d stored as fp16 (round to nearest even), sum =
 * sum of q.  The q8 bytes are a per-element function of the f32 values that
 * were quantized ([D3-5] §2.3), so a fused producer's plane equals the
 * standalone quantizer applied to the f32 output it wrote.
 *
 * mq_quantize_q8:      x[n] (device f32) -> q8.
 * mq_rmsnorm_quant_q8: y = x / sqrt(mean(x^2) + eps) * gain (f32; the rms arm
 *                      of [D3-5] §3.2, body not printed there), writes y[n]
 *                      (device f32) and q8.  One row; y must not alias x or
 *                      gain.
 * mq_swiglu_quant_q8:  y = (g / (1 + exp(-g))) * u ([D3-5] §3.2), writes y[n]
 *                      and q8.  g, u, y device f32; y may alias g or u.
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE (n <= 0 or n % 32), MQ_ERR_ALIGN,
 *         MQ_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int mq_quantize_q8(const float *x, void *q8, int n, void *stream);
int mq_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y, void *q8,
                        int n, void *stream);
int mq_swiglu_quant_q8(const float *g, const float *u, float *y, void *q8, int n, void *stream);

/* ------------------------------------------------------------------------
 * Decode GEMV (device): y[rows] = W x_hat.
 *   q6_K ([D4-2] §3.2 Excerpt C): y_r = sum over blocks b and 16-weight
 *        sub-blocks s of f16(d_b) * sc_s * f16(d8) * isum_s,
 *        isum_s = sum (q - 32) * q8 (int32).
 *   q4_K: y_r = sum over 32-weight sub-blocks k of
 *        f16(d8_k) * (f16(d) * sc_k * isum_k - f16(dmin) * m_k * qsum_k),
 *        isum_k = sum q * q8, qsum_k = the q8 block's sum.
 *   q5_K: as q4_K with 5-bit codes q = nibble + 16 * fifth bit (0..31).
 * Wp: repacked weights (device, mq_repack_* output).  q8: plane of cols
 * values (device).  y: rows f32 (device).  The f32 combine order is fixed
 * (ascending chunks within a work item, a fixed butterfly across lanes,
 * splits summed in ascending order), so results are deterministic run to run.
 *
 * Work decomposition.  Rows are cut into tiles of 8 and each tile's columns
 * into nchunks = ceil(cols/1024) chunks of 4 super-blocks.  A plan is
 * (splits, chunks_per_split, tiles_per_item); one warp per work item:
 *   splits == 1: every item covers tiles_per_item whole tiles;
 *     chunks_per_split must still cover a row (>= nchunks).
 *   splits > 1 ("split-K", the tall-row case of [D4-2] §2): every tile is cut
 *     into `splits` tile-aligned ranges of chunks_per_split chunks (the last
 *     may be shorter); tiles_per_item must be 1.  With splits <= 12 the
 *     splits of a tile are the warps of one CTA and add their partial row
 *     sums in shared memory in ascending split order.  With splits > 12 each
 *     split leaves its partials in `ws` and the split that finishes last adds
 *     all of them in ascending split order (an atomic ticket; nothing waits
 *     or spins).
 * Before any launch the host checks the plan: splits * chunks_per_split >=
 * nchunks (no chunk dropped) and (splits - 1) * chunks_per_split < nchunks
 * (no empty split), else MQ_ERR_COVERAGE ([D4-2] §6 lesson 1: a gate must
 * bound both sides).  The default plan fills one resident wave of the GPU:
 * whole tiles when there are more tiles than warps, else the largest CTA
 * split count whose one-CTA-per-tile grid fits the wave, and workspace splits
 * only when that still leaves the wave less than half full (very few tiles,
 * rows longer than 12 chunks).
 *
 * Whole-tile CTAs stage the q8 plane in shared memory, so for every plan
 * mq_q8_bytes(cols) rounded up to 128 bytes must fit one CTA's opt-in shared
 * memory less 1 KiB (cols <= 194816 on GB300), else MQ_ERR_SHAPE.
 *
 * mq_gemv_workspace_bytes(rows, cols): workspace the default plans (q6_K,
 *   q4_K and q5_K) need on the current device (0 unless splits > 12).  ws must be
 *   device memory, zero-filled before its first use; every completed call
 *   leaves it zero-filled again.  ws may be NULL when 0 bytes are needed.
 * mq_gemv_workspace_bytes_for: the same for an explicit plan (0 if invalid).
 * mq_gemv_plan: the default plan for format 6 (q6_K), 4 (q4_K) or 5 (q5_K)
 *   on the current device (from the kernel's measured occupancy).
 * mq_gemv_plan_for: the default plan for a device with `sms` SMs and a
 *   kernel using regs_per_thread registers (64K registers per SM), from the
 *   register limit alone (the weight ring's shared memory is not modelled).
 *   Host only.
 * mq_gemv_*_q8_plan: the GEMV with an explicit plan.
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_WORKSPACE,
 *         MQ_ERR_COVERAGE, MQ_ERR_CUDA.
 * ------------------------------------------------------------------------ */
size_t mq_gemv_workspace_bytes(int rows, int cols);
size_t mq_gemv_workspace_bytes_for(int rows, int cols, int splits, int chunks_per_split,
                                   int tiles_per_item);
int mq_gemv_plan(int rows, int cols, int fmt, int *splits, int *chunks_per_split,
                 int *tiles_per_item);
int mq_gemv_plan_for(int rows, int cols, int sms, int regs_per_thread, int *splits,
                     int *chunks_per_split, int *tiles_per_item);
int mq_gemv_q6k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream);
int mq_gemv_q4k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream);
int mq_gemv_q6k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream);
int mq_gemv_q4k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream);
int mq_gemv_q5k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream);
int mq_gemv_q5k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream);

/* q6_K GEMV for callers that cannot allocate device memory (no counterpart
 * on the pages; it exists for integration).  Some callers only receive
 * input and output pointers: a plugin or callback inside a host framework
 * that owns every allocation, a real-time loop that may not allocate once
 * running, code in a region where cudaMalloc is forbidden or would stall the
 * device.  They cannot provide the split-K workspace of mq_gemv_q6k_q8.
 * This entry point computes the same y with the same kernel and default
 * plan; when that plan needs scratch (more than 12 splits per tile) it is
 * kept in a static device array inside the library (128 KiB per GPU, held
 * until the process exits).  It allocates nothing.
 *   - Limit: if the default plan on this device needs more than 128 KiB of
 *     scratch the call returns MQ_ERR_WORKSPACE and launches nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any CUDA graph capture.
 *   - Every call uses the same array.  Each call clears the counters it
 *     needs (an async memset on `stream`) before its kernel; calls whose
 *     work overlaps on the GPU (other streams, other threads) race on the
 *     array and give wrong results: order them on one stream.
 * Arguments and other errors as mq_gemv_q6k_q8. */
int mq_gemv_q6k_q8_noalloc(const void *Wp, const void *q8, float *y, int rows, int cols,
                           void *stream);

/* ------------------------------------------------------------------------
 * q6_K GEMV against an f32 activation row (device): the dequantize-and-FMA
 * family the pages keep beside the q8 MMVQ ([D3] §2.3 and §3.3, the
 * "padded f32" kernels; on GB10 they won below od*id ~ 24M).  No q8
 * producer is needed: x is read as is.
 *   y_r = sum_e w_{r,e} x_e,   w = f16(d) * sc_{e/16} * (q_e - 32)
 * computed in f32: a fused multiply-add chain over each 16-weight
 * sub-block, then acc_r += (d * sc) * subsum, partial sums combined in the
 * fixed order of the q8 GEMV (deterministic run to run).
 *   Wp: repacked q6_K weights (device, mq_repack_q6k output; the same copy
 *       serves the q8 GEMV).  x: cols f32 (device).  y: rows f32 (device).
 *   Every CTA stages x in shared memory, so cols * 4 bytes must fit in one
 *   CTA's opt-in shared memory less 1 KB (cols <= 57856 on GB300), else
 *   MQ_ERR_SHAPE.
 *   Plans are those of mq_gemv_q6k_q8 without workspace splits: splits must
 *   be 1..12 (MQ_ERR_COVERAGE otherwise, with the same coverage checks);
 *   mq_gemv_q6k_f32_plan_of returns the default plan on the current device.
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_COVERAGE,
 *         MQ_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int mq_gemv_q6k_f32(const void *Wp, const float *x, float *y, int rows, int cols, void *stream);
int mq_gemv_q6k_f32_plan(const void *Wp, const float *x, float *y, int rows, int cols, int splits,
                         int chunks_per_split, int tiles_per_item, void *stream);
int mq_gemv_q6k_f32_plan_of(int rows, int cols, int *splits, int *chunks_per_split,
                            int *tiles_per_item);

/* ------------------------------------------------------------------------
 * Grouped GEMV (device): up to MQ_MAX_GROUP matrices that read the same q8
 * plane (same cols) in ONE launch, e.g. the q, k, v projections of a layer
 * (q4_K, q4_K, q6_K) after one rms_norm->q8, or its gate and up (the
 * gate||up pair of [D4-4] §2, L3).  Each part may be q6_K or q4_K and gets
 * its own y; the arithmetic per part is exactly that of mq_gemv_q6k_q8 /
 * mq_gemv_q4k_q8, and a group of one is that call.  One launch means one
 * wave, one ramp and one tail for the group instead of one per matrix.
 * The plan (and the workspace, when it needs one) is sized on the group's
 * total tile count; work items never straddle two parts.
 *   parts: host array of nparts descriptors (read during the call only).
 *   mq_gemv_group_workspace_bytes: workspace for the default plan
 *     (splits == 0) or an explicit one; the Wp / y fields may be NULL here.
 * Errors: as mq_gemv_q6k_q8; MQ_ERR_SHAPE also for nparts outside
 *         1..MQ_MAX_GROUP or a format other than 6 / 4 / 5.
 * ------------------------------------------------------------------------ */
#define MQ_MAX_GROUP 8

typedef struct {
    int fmt;            /* 6 = q6_K, 4 = q4_K, 5 = q5_K               */
    int rows;           /* rows of this matrix (>= 1)                  */
    const void *Wp;     /* its repacked weights (device)               */
    float *y;           /* its rows f32 outputs (device)               */
} mq_gemv_part;

size_t mq_gemv_group_workspace_bytes(const mq_gemv_part *parts, int nparts, int cols, int splits,
                                     int chunks_per_split, int tiles_per_item);
int mq_gemv_group_q8(const mq_gemv_part *parts, int nparts, const void *q8, int cols, void *ws,
                     size_t ws_bytes, void *stream);
int mq_gemv_group_q8_plan(const mq_gemv_part *parts, int nparts, const void *q8, int cols,
                          int splits, int chunks_per_split, int tiles_per_item, void *ws,
                          size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Small-batch GEMV (device): nt = 1..MQ_MAX_TOKENS activation rows (the
 * tokens of a batched or speculative decode step) against ONE pass over the
 * weights.  The pages' MMVQ launch already takes a token count and gives
 * each token a grid row, reading the weights once per token ([D4-2] §2);
 * here every streamed weight byte is used for all nt tokens.  Per token the
 * integer sub-block dots and the f32 combine are those of mq_gemv_q6k_q8 /
 * mq_gemv_q4k_q8; the f32 reduction order is fixed (deterministic) but not
 * the single-token kernel's, so results agree with it to rounding.
 *   q8: nt planes of cols values, back to back: token t's plane starts at
 *       q8 + t * mq_q8_bytes(cols) (what the _batch producers write).
 *   y:  nt x rows f32, token-major: y[t * rows + r].
 *   nt == 1 (default plan) runs the single-token GEMV of the format when
 *   its default plan needs no workspace, else this kernel for one token;
 *   either way no workspace is taken (mq_gemv_q6k_q8's long-row plans may
 *   need one).  The _plan forms always run this kernel.  So at nt == 1 the
 *   default form's y equals mq_gemv_*_q8's bit for bit whenever that
 *   kernel ran, and may differ in the last bits from the _plan form's y and
 *   from token 0 of an nt >= 2 call (another f32 reduction order).
 *   Every CTA stages all nt planes in shared memory: nt * mq_q8_bytes(cols)
 *   must not exceed the device's per-CTA limit less 8 KiB (about 219 KiB on
 *   GB300, i.e. cols <= 23552 at nt = 8 and 188672 at nt = 1), else
 *   MQ_ERR_SHAPE.
 * Plans read differently from the single-token ones: splits S
 * (1..12) cuts every row into S ranges of chunks_per_split chunks (coverage
 * checked as above, no empty range); a CTA holds S warps for each of B / S
 * tiles (a "group") and runs tiles_per_item consecutive groups, so the
 * staged planes serve tiles_per_item * (B / S) tiles.  B, the warps one CTA
 * holds, is 12 to 16: the most that fit an SM at the register count of the
 * kernel for nt tokens of that format (asked of the device once).  A tile's S splits
 * add their partial sums in shared memory in ascending split order; there
 * is no workspace.  The default plan picks S and tiles_per_item so that the
 * busiest warp streams the fewest chunks, scaled up when the grid leaves SMs
 * idle.
 * mq_gemv_batch_plan: the default plan for nt tokens of q6_K on the current
 *   device (other formats may hold a different B).
 * mq_gemv_batch_plan_for: the same for a device with `sms` SMs and a kernel
 *   of regs_per_thread registers (B = the warps that fit, at most 16).
 *   Host only.
 * mq_gemv_*_q8_batch_plan: the GEMV with an explicit plan.
 * Errors: as mq_gemv_q6k_q8; MQ_ERR_SHAPE also for nt outside
 *         1..MQ_MAX_TOKENS; MQ_ERR_COVERAGE for a bad plan.
 * ------------------------------------------------------------------------ */
#define MQ_MAX_TOKENS 8

int mq_gemv_batch_plan(int rows, int cols, int nt, int *splits, int *chunks_per_split,
                       int *tiles_per_item);
int mq_gemv_batch_plan_for(int rows, int cols, int nt, int sms, int regs_per_thread, int *splits,
                           int *chunks_per_split, int *tiles_per_item);
int mq_gemv_q6k_q8_batch(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                         void *stream);
int mq_gemv_q4k_q8_batch(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                         void *stream);
int mq_gemv_q5k_q8_batch(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                         void *stream);
int mq_gemv_q6k_q8_batch_plan(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *stream);
int mq_gemv_q4k_q8_batch_plan(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *stream);
int mq_gemv_q5k_q8_batch_plan(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *stream);

/* Producers over nt rows (1..MQ_MAX_TOKENS) of n values each: x, g, u and y
 * are nt x n row-major (device f32); q8 receives nt planes, token t's at
 * q8 + t * mq_q8_bytes(n).  Each row is exactly what the single-row call
 * computes on that row; rms_norm normalizes every row by its own mean
 * square, with the one gain vector of n values.  Errors: as the single-row
 * producers; MQ_ERR_SHAPE also for nt outside 1..MQ_MAX_TOKENS. */
int mq_quantize_q8_batch(const float *x, void *q8, int n, int nt, void *stream);
int mq_rmsnorm_quant_q8_batch(const float *x, const float *gain, float eps, float *y, void *q8,
                              int n, int nt, void *stream);
int mq_swiglu_quant_q8_batch(const float *g, const float *u, float *y, void *q8, int n, int nt,
                             void *stream);

/* ------------------------------------------------------------------------
 * FFN gate||up GEMV with the SwiGLU -> q8 producer fused in (device).
 * One launch computes, for r < rows,
 *     act[r] = silu(g_r) * u_r = (g_r / (1 + exp(-g_r))) * u_r,
 *     g = Wg x_hat, u = Wu x_hat  (each exactly as mq_gemv_q6k_q8 /
 *                                  mq_gemv_q4k_q8 with a whole-tile plan),
 * writes act (f32) and act's q8 plane (rows values, quantized as by
 * mq_quantize_q8), i.e. what GEMV(gate), GEMV(up) and mq_swiglu_quant_q8
 * produce in three launches, bit for bit.  This is the concatenated
 * gate||up launch with a SwiGLU epilogue that [D4-4] §2 and §5 closed on
 * GB10 for running 1.5 waves; here the grid is one resident wave.
 *   fmt: 6 (q6_K), 4 (q4_K) or 5 (q5_K), for both matrices.  Wg, Wu: repacked
 *   weights, rows x cols each (device).  q8: plane of cols values (device).
 *   act: rows f32 (device).  q8_out: mq_q8_bytes(rows) bytes (device).
 *   rows must be a multiple of 32 (q8 blocks of act are whole).
 * Plan: CTAs of warps_per_cta warps (1..8) each take whole 32-row blocks,
 * the block's 4 gate and 4 up tiles shared among the warps; `ctas` CTAs
 * (1..rows/32) stride over the blocks.  The default takes the most warps per
 * CTA whose one-CTA-per-block grid fits one resident wave.
 * mq_gemv_gateup_plan_for: that plan for `sms` SMs and regs_per_thread
 *   registers (host only).
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE (fmt, cols % 256, rows % 32, a plane too
 *   large for shared memory), MQ_ERR_ALIGN, MQ_ERR_COVERAGE (a plan outside
 *   the ranges above), MQ_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int mq_gemv_gateup_swiglu_q8(int fmt, const void *Wg, const void *Wu, const void *q8, int rows,
                             int cols, float *act, void *q8_out, void *stream);
int mq_gemv_gateup_swiglu_q8_plan(int fmt, const void *Wg, const void *Wu, const void *q8, int rows,
                                  int cols, float *act, void *q8_out, int warps_per_cta, int ctas,
                                  void *stream);
int mq_gemv_gateup_plan_for(int rows, int sms, int regs_per_thread, int *warps_per_cta, int *ctas);

/* Coverage check used by every GEMV dispatch, exposed for tests: MQ_OK iff
 * all arguments are >= 1, splits * chunks_per_split >= nchunks (nothing
 * dropped) and (splits - 1) * chunks_per_split < nchunks (no empty split);
 * else MQ_ERR_COVERAGE. */
int mq_check_coverage(int nchunks, int splits, int chunks_per_split);

/* ------------------------------------------------------------------------
 * Programmatic dependent launch (process-wide switch, default off; returns
 * the previous setting).  When on, every kernel is launched with CUDA's
 * programmatic stream serialization, so it may start while the previous
 * kernel in the stream drains: producers then wait (griddepcontrol.wait)
 * before reading their activations (the rms producer reads its first slice
 * of gain before waiting), and a GEMV issues its first weight loads BEFORE
 * waiting and touches the q8 plane, y and ws only after.  This hides launch
 * and ramp latency in a producer -> GEMV -> producer chain (the retry
 * condition of [D4-4] §5 for PDL: a purely bandwidth-bound chain).  Turn it
 * on only when the kernel that directly precedes a GEMV in the stream does
 * not write that GEMV's weight matrix, nor the kernel before an rms
 * producer its gain (both are weights in a decode step).
 * ------------------------------------------------------------------------ */
int mq_set_pdl(int enable);

/* ------------------------------------------------------------------------
 * Weight ring of the single-token GEMV (process-wide tuning control; no
 * counterpart on the pages, whose kernels read each unit straight into
 * registers).  Each warp of mq_gemv_*_q8 / mq_gemv_group_q8 keeps `stages`
 * chunks of its weight range in flight in its own shared-memory slots
 * (16-byte asynchronous copies) while it computes the previous chunk from
 * registers; `pre_wait` of them are requested before the kernel waits for
 * its predecessor under programmatic dependent launch (mq_set_pdl).
 *   stages: 0 = no ring (each chunk is loaded straight into registers, one
 *           chunk per warp in flight), 1..3, or -1 = the default (0: on
 *           GB300 the ring measured slower on every matrix of the 14B decode
 *           step and faster only on whole-tile q4_K shapes with few warps,
 *           e.g. a 13824 x 5120 q4_K GEMV at 2 stages).  Clamped so that the
 *           largest CTA fits the device's shared memory.
 *   pre_wait: 0..stages, or -1 = all of them.
 * Plans chosen after a change account for the ring's shared memory (it can
 * lower the resident CTAs per SM, and so change a default plan).  Results
 * do not depend on the setting: the same sub-dots in the same order.
 * Returns the previous stages value.
 * ------------------------------------------------------------------------ */
int mq_set_gemv_ring(int stages, int pre_wait);

/* ------------------------------------------------------------------------
 * Integer sub-block dots (device), for bit-exact testing of the GEMV's
 * integer path: the same kernel and lane mapping as the GEMV, writing
 * isums[r][b][s] (int32) instead of accumulating: 16 per block (q6_K,
 * isum_s = sum (q - 32) * q8) or 8 per block (q4_K and q5_K,
 * isum_k = sum q * q8).
 * isums: rows * cols/256 * {16, 8} int32 (device).
 * ------------------------------------------------------------------------ */
int mq_gemv_q6k_q8_subdots(const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                           void *stream);
int mq_gemv_q4k_q8_subdots(const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                           void *stream);
int mq_gemv_q5k_q8_subdots(const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                           void *stream);

/* Device-side coverage check of a plan (test and debug aid): the grouped
 * GEMV of mq_gemv_group_q8_plan (splits == 0: the default plan), same
 * arguments and the same outputs, which also adds 1 to
 * counts[global tile * nchunks + chunk] for every chunk unit a warp
 * processes.  Global tiles number the parts' 8-row tiles in part order;
 * nchunks = ceil(cols / 1024).  counts: device, 16-byte aligned, one uint32
 * per unit, zero-filled by the caller.  The plan covers the work exactly
 * once iff every count is 1 afterwards (the host check of the plan runs
 * first, as for every GEMV).
 * Errors: as mq_gemv_group_q8_plan. */
int mq_gemv_group_q8_coverage(const mq_gemv_part *parts, int nparts, const void *q8, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *ws,
                              size_t ws_bytes, unsigned *counts, void *stream);

/* Repack on the device: the same bytes as mq_repack_q6k / _q4k / _q5k (host)
 * for GGUF rows that are already in device memory, written by a kernel
 * (the pages build the dense plane once at weight registration, [D4-4]
 * §3.1; on the GPU a multi-GB weight set repacks at memory speed).
 *   fmt: 6 (q6_K), 4 (q4_K) or 5 (q5_K).
 *   gguf: device, rows x cols/256 GGUF blocks (2-byte aligned or better).
 *   dst: device, mq_repacked_bytes_*(rows, cols) bytes, 16-byte aligned;
 *        zero-filled, then written (padding rows stay zero), on `stream`.
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE (fmt or shape), MQ_ERR_ALIGN, MQ_ERR_CUDA. */
int mq_repack_device(int fmt, const void *gguf, void *dst, int rows, int cols, void *stream);

/* Copy for the ends of a decode step (no counterpart on the pages): moves
 * `bytes` from src to dst with a kernel, so that the host-to-device copy of
 * a step's input and the device-to-host copy of its result join the launch
 * chain of the producers and GEMVs (programmatic dependent launch, graph
 * capture) instead of handing the stream to a copy engine and back.
 *   src, dst: device memory of the current device, or pinned host memory
 *     (cudaHostAlloc / cudaMallocHost / cudaHostRegister) that the device
 *     can address; the library looks each pointer up (cudaPointerGetAttributes)
 *     and uses the device-side address of pinned host memory.  Pageable host
 *     memory and unknown pointers give MQ_ERR_ACCESS and nothing runs.
 *   bytes: a multiple of 16 (> 0); both pointers 16-byte aligned.
 *   Ordering: the kernel waits for the preceding kernel in the stream
 *   before it reads or writes, so it may follow a GEMV (its output) or
 *   precede a producer (its input).  The host must not touch a pinned buffer
 *   while a copy that uses it may run (synchronize first).
 * Errors: MQ_ERR_NULL, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_ACCESS, MQ_ERR_CUDA. */
int mq_copy(void *dst, const void *src, size_t bytes, void *stream);

/* The address a kernel on the current device uses for p: p itself for
 * device or managed memory of the current device, the device-side address of
 * pinned host memory (cudaHostAlloc / cudaMallocHost / cudaHostRegister).
 * Look a buffer up once and pass the result to the entry points above that
 * take host-resident activations.
 *   p: any pointer; *out: written on MQ_OK only.
 * Errors: MQ_ERR_NULL (p or out NULL), MQ_ERR_ACCESS (pageable host memory,
 * another device's memory, or a pointer CUDA does not know). */
int mq_device_address(const void *p, void **out);

/* Measurement aid: read `bytes` (a multiple of 16) at src (device, 16-byte
 * aligned) once, in one launch, and do nothing with them.  Its time is the
 * floor for any single launch that streams that many bytes on this GPU,
 * ramp and tail included, so a GEMV's time can be judged against it as well
 * as against the sustained copy peak.  Errors: MQ_ERR_NULL, MQ_ERR_SHAPE,
 * MQ_ERR_ALIGN, MQ_ERR_CUDA. */
int mq_read_floor(const void *src, size_t bytes, void *stream);

/* Number of streaming multiprocessors of the current device (0 on error);
 * the dispatch plan sizes its grid from it. */
int mq_device_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* MQ_H */
