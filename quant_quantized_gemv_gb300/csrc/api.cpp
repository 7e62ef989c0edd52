// api.cpp -- the C ABI of include/mq.h: argument validation, the GEMV dispatch
// plan and its coverage check, then the launch.  Nothing here allocates.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "kernels.h"
#include "layout.h"
#include "mq.h"

namespace {

using namespace mq;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
// resident GEMV CTAs per SM: [device][q6_K, q4_K][warps per CTA]
std::atomic<int> g_ctas[kMaxDevices][2][kMaxCtaSplits + 1];
std::atomic<int> g_pdl{0};

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool gemv_shape_ok(int rows, int cols)
{
    return rows >= 1 && cols >= kQK && cols % kQK == 0 && (long long)rows * cols < (1LL << 40);
}

bool vec_shape_ok(int n) { return n > 0 && n % 32 == 0; }

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int device_sms()
{
    const int dev = current_device();
    if (dev < 0) return 0;
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev].store(v, std::memory_order_relaxed);
    return v;
}

// ctas[w], w = 1..kMaxCtaSplits: resident GEMV CTAs per SM with w warps each.
struct Occupancy {
    int ctas[kMaxCtaSplits + 1];
};

bool device_occupancy(int fmt, Occupancy *o)
{
    const int dev = current_device();
    if (dev < 0) return false;
    for (int w = 1; w <= kMaxCtaSplits; ++w) {
        std::atomic<int> &slot = g_ctas[dev][fmt == 6 ? 0 : 1][w];
        int v = slot.load(std::memory_order_relaxed);
        if (v <= 0) {
            v = gemv_ctas_per_sm(fmt, w);
            if (v <= 0) return false;
            slot.store(v, std::memory_order_relaxed);
        }
        o->ctas[w] = v;
    }
    return true;
}

// The same from a register count (host-only planning, tests): 64K registers
// per SM, at most 2048 threads and 32 CTAs.
Occupancy model_occupancy(int regs_per_thread)
{
    Occupancy o;
    const int regs = ((regs_per_thread + 7) / 8) * 8;
    for (int w = 1; w <= kMaxCtaSplits; ++w) {
        int c = 65536 / (w * 32 * regs);
        if (c > 2048 / (32 * w)) c = 2048 / (32 * w);
        if (c > 32) c = 32;
        o.ctas[w] = c;
    }
    return o;
}

struct Plan {
    int splits, cps, tpi;
};

// One resident wave.  Enough tiles: whole tiles per warp.  Fewer: one CTA
// per tile whose warps are the tile's splits (the largest split count whose
// grid still fits one wave).  Very few tiles with long rows: warp splits
// that meet in the workspace, as many as the wave holds.
Plan plan_for(int ntiles, int nchunks, int sms, const Occupancy &o)
{
    if (sms <= 0) sms = 1;
    const long long wave = (long long)sms * (o.ctas[kGemvWarpsPerBlock] > 0 ? o.ctas[kGemvWarpsPerBlock] : 1) *
                           kGemvWarpsPerBlock;  // warps in one wave of 4-warp CTAs
    if (ntiles >= wave || nchunks == 1)
        return Plan{1, nchunks, (int)((ntiles + wave - 1) / wave)};
    int best = 1;
    for (int sp = 2; sp <= kMaxCtaSplits && sp <= nchunks; ++sp)
        if ((long long)ntiles <= (long long)sms * o.ctas[sp]) best = sp;
    Plan p{1, nchunks, 1};
    if (best > 1) {
        p.cps = ceil_div(nchunks, best);
        p.splits = ceil_div(nchunks, p.cps);
        if (p.splits == 1) p.cps = nchunks;
    }
    if (nchunks > kMaxCtaSplits && (long long)ntiles * p.splits * 2 < wave) {
        long long s2 = wave / ntiles;
        if (s2 > nchunks) s2 = nchunks;
        const int cps2 = ceil_div(nchunks, (int)s2);
        const int sp2 = ceil_div(nchunks, cps2);
        if (sp2 > kMaxCtaSplits) return Plan{sp2, cps2, 1};
    }
    return p;
}

long long plan_items(int ntiles, const Plan &p)
{
    return p.splits > 1 ? (long long)ntiles * p.splits : (ntiles + p.tpi - 1) / p.tpi;
}

size_t ws_bytes_for(int ntiles, const Plan &p)
{
    if (p.splits <= kMaxCtaSplits) return 0;  // splits meet in shared memory (or none)
    return round16((size_t)ntiles * 4) + (size_t)plan_items(ntiles, p) * 8 * sizeof(float);
}

int check_coverage(int nchunks, int splits, int cps)
{
    if (nchunks < 1 || splits < 1 || cps < 1) return MQ_ERR_COVERAGE;
    // every chunk lies in some split:  splits * cps >= nchunks
    if ((long long)splits * cps < nchunks) return MQ_ERR_COVERAGE;
    // every split owns at least one chunk (no empty or duplicated work item)
    if ((long long)(splits - 1) * cps >= nchunks) return MQ_ERR_COVERAGE;
    return MQ_OK;
}

int check_plan(const Geom &g, const Plan &p)
{
    if (p.tpi < 1 || (p.splits > 1 && p.tpi != 1)) return MQ_ERR_COVERAGE;
    const int cov = check_coverage(g.nchunks, p.splits, p.cps);
    if (cov != MQ_OK) return cov;
    if (plan_items(g.ntiles, p) >= (1LL << 31)) return MQ_ERR_SHAPE;
    return MQ_OK;
}

int gemv_common(int fmt, const void *Wp, const void *q8, float *y, int rows, int cols,
                const Plan *explicit_plan, void *ws, size_t ws_bytes, void *stream)
{
    if (!Wp || !q8 || !y) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    if (!aligned16(Wp) || !aligned16(q8) || !aligned16(y)) return MQ_ERR_ALIGN;
    const Geom g = make_geom(rows, cols, fmt == 6 ? kQ6kBytes : kQ4kBytes);
    Plan p;
    if (explicit_plan) {
        p = *explicit_plan;
    } else {
        Occupancy o;
        if (!device_occupancy(fmt, &o)) return MQ_ERR_CUDA;
        p = plan_for(g.ntiles, g.nchunks, device_sms(), o);
    }
    const int cov = check_plan(g, p);
    if (cov != MQ_OK) return cov;
    GemvLaunch a;
    memset(&a, 0, sizeof a);
    const size_t need = ws_bytes_for(g.ntiles, p);
    if (need > 0) {
        if (!ws) return MQ_ERR_NULL;
        if (!aligned16(ws)) return MQ_ERR_ALIGN;
        if (ws_bytes < need) return MQ_ERR_WORKSPACE;
        a.ws_cnt = (unsigned *)ws;
        a.ws_part = (float *)((uint8_t *)ws + round16((size_t)g.ntiles * 4));
    }
    a.W = (const uint8_t *)Wp;
    a.q8 = (const uint8_t *)q8;
    a.y = y;
    a.rows = rows;
    a.nb = g.nb;
    a.ntiles = g.ntiles;
    a.nchunks = g.nchunks;
    a.splits = p.splits;
    a.cps = p.cps;
    a.tpi = p.tpi;
    a.n_items = (int)plan_items(g.ntiles, p);
    a.tile_bytes = g.tile_bytes;
    a.q8_d_off = (unsigned)q8_d_offset(cols);
    a.q8_sum_off = (unsigned)q8_sum_offset(cols);
    a.pdl = g_pdl.load(std::memory_order_relaxed);
    const cudaError_t e = fmt == 6 ? launch_gemv_q6k(a, (cudaStream_t)stream)
                                   : launch_gemv_q4k(a, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

int subdots_common(int fmt, const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                   void *stream)
{
    if (!Wp || !q8 || !isums) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    if (!aligned16(Wp) || !aligned16(q8) || !aligned16(isums)) return MQ_ERR_ALIGN;
    const Geom g = make_geom(rows, cols, fmt == 6 ? kQ6kBytes : kQ4kBytes);
    GemvLaunch a;
    memset(&a, 0, sizeof a);
    a.W = (const uint8_t *)Wp;
    a.q8 = (const uint8_t *)q8;
    a.isums = isums;
    a.rows = rows;
    a.nb = g.nb;
    a.ntiles = g.ntiles;
    a.nchunks = g.nchunks;
    if ((long long)g.ntiles * g.nchunks >= (1LL << 31)) return MQ_ERR_SHAPE;
    a.splits = g.nchunks;  // one chunk per work item
    a.cps = 1;
    a.tpi = 1;
    a.n_items = g.ntiles * g.nchunks;
    a.tile_bytes = g.tile_bytes;
    a.q8_d_off = (unsigned)q8_d_offset(cols);
    a.q8_sum_off = (unsigned)q8_sum_offset(cols);
    a.pdl = g_pdl.load(std::memory_order_relaxed);
    const cudaError_t e = fmt == 6 ? launch_subdots_q6k(a, (cudaStream_t)stream)
                                   : launch_subdots_q4k(a, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *mq_strerror(int status)
{
    switch (status) {
    case MQ_OK: return "ok";
    case MQ_ERR_SHAPE: return "bad shape (cols % 256, n % 32, sizes >= 1)";
    case MQ_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case MQ_ERR_NULL: return "required pointer is NULL";
    case MQ_ERR_COVERAGE: return "dispatch plan does not cover every chunk exactly once";
    case MQ_ERR_WORKSPACE: return "split-K workspace too small";
    case MQ_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
    }
}

const char *mq_version(void) { return "mq 0.1 sm_103a"; }

int mq_device_sms(void) { return device_sms(); }

size_t mq_q8_bytes(int n) { return vec_shape_ok(n) ? q8_plane_bytes(n) : 0; }

int mq_q8_unpack_host(const void *plane, int n, uint16_t *d, int8_t *qs, int32_t *sum)
{
    if (!plane) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    const uint8_t *p = (const uint8_t *)plane;
    if (qs) memcpy(qs, p, (size_t)n);
    if (d) memcpy(d, p + q8_d_offset(n), (size_t)(n / 32) * 2);
    if (sum) memcpy(sum, p + q8_sum_offset(n), (size_t)(n / 32) * 4);
    return MQ_OK;
}

int mq_quantize_q8(const float *x, void *q8, int n, void *stream)
{
    if (!x || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_quantize_q8(x, (uint8_t *)q8, n, (unsigned)q8_d_offset(n),
                                             (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed),
                                             (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

int mq_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y, void *q8, int n,
                        void *stream)
{
    if (!x || !gain || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gain) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_rmsnorm_quant_q8(x, gain, eps, y, (uint8_t *)q8, n,
                                                  (unsigned)q8_d_offset(n),
                                                  (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed),
                                             (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

int mq_swiglu_quant_q8(const float *g, const float *u, float *y, void *q8, int n, void *stream)
{
    if (!g || !u || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    if (!aligned16(g) || !aligned16(u) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_swiglu_quant_q8(g, u, y, (uint8_t *)q8, n,
                                                 (unsigned)q8_d_offset(n),
                                                 (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed),
                                             (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

int mq_check_coverage(int nchunks, int splits, int chunks_per_split)
{
    return check_coverage(nchunks, splits, chunks_per_split);
}

int mq_gemv_plan_for(int rows, int cols, int sms, int regs_per_thread, int *splits,
                     int *chunks_per_split, int *tiles_per_item)
{
    if (!splits || !chunks_per_split || !tiles_per_item) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols) || regs_per_thread < 1 || regs_per_thread > 255) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const Plan p = plan_for(g.ntiles, g.nchunks, sms, model_occupancy(regs_per_thread));
    *splits = p.splits;
    *chunks_per_split = p.cps;
    *tiles_per_item = p.tpi;
    return MQ_OK;
}

int mq_gemv_plan(int rows, int cols, int fmt, int *splits, int *chunks_per_split,
                 int *tiles_per_item)
{
    if (!splits || !chunks_per_split || !tiles_per_item) return MQ_ERR_NULL;
    if (fmt != 6 && fmt != 4) return MQ_ERR_SHAPE;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    Occupancy o;
    if (!device_occupancy(fmt, &o)) return MQ_ERR_CUDA;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const Plan p = plan_for(g.ntiles, g.nchunks, device_sms(), o);
    *splits = p.splits;
    *chunks_per_split = p.cps;
    *tiles_per_item = p.tpi;
    return MQ_OK;
}

size_t mq_gemv_workspace_bytes_for(int rows, int cols, int splits, int chunks_per_split,
                                   int tiles_per_item)
{
    if (!gemv_shape_ok(rows, cols)) return 0;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const Plan p{splits, chunks_per_split, tiles_per_item};
    if (check_plan(g, p) != MQ_OK) return 0;
    return ws_bytes_for(g.ntiles, p);
}

size_t mq_gemv_workspace_bytes(int rows, int cols)
{
    size_t need = 0;
    for (int fmt : {6, 4}) {
        int s = 0, c = 0, t = 0;
        if (mq_gemv_plan(rows, cols, fmt, &s, &c, &t) != MQ_OK) return 0;
        const size_t b = mq_gemv_workspace_bytes_for(rows, cols, s, c, t);
        if (b > need) need = b;
    }
    return need;
}

int mq_set_pdl(int enable)
{
    return g_pdl.exchange(enable ? 1 : 0);
}

int mq_gemv_q6k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream)
{
    return gemv_common(6, Wp, q8, y, rows, cols, nullptr, ws, ws_bytes, stream);
}

int mq_gemv_q4k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream)
{
    return gemv_common(4, Wp, q8, y, rows, cols, nullptr, ws, ws_bytes, stream);
}

int mq_gemv_q6k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream)
{
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(6, Wp, q8, y, rows, cols, &p, ws, ws_bytes, stream);
}

int mq_gemv_q4k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream)
{
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(4, Wp, q8, y, rows, cols, &p, ws, ws_bytes, stream);
}

int mq_gemv_q6k_q8_subdots(const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                           void *stream)
{
    return subdots_common(6, Wp, q8, isums, rows, cols, stream);
}

int mq_gemv_q4k_q8_subdots(const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                           void *stream)
{
    return subdots_common(4, Wp, q8, isums, rows, cols, stream);
}

}  // extern "C"
