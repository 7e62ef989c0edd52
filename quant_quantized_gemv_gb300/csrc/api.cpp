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

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool gemv_shape_ok(int rows, int cols)
{
    return rows >= 1 && cols >= kQK && cols % kQK == 0 && (long long)rows * cols < (1LL << 40);
}

bool vec_shape_ok(int n) { return n > 0 && n % 32 == 0; }

int device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev].store(v, std::memory_order_relaxed);
    return v;
}

// Split count for a (rows, cols) GEMV: enough warps in flight to keep HBM
// busy, and no more splits than that (each split adds a partial write and a
// share of a combine).  A warp streams ~6.7 KB (q6_K) per chunk; about 16
// resident warp-items per SM keep >= 20 MB of loads queued GPU-wide.
int plan_splits(int ntiles, int nchunks, int sms)
{
    if (sms <= 0) sms = 1;
    const long long target = (long long)sms * 16;
    if (ntiles >= target) return 1;
    long long s = (target + ntiles - 1) / ntiles;
    if (s > nchunks) s = nchunks;
    const int cps = ceil_div(nchunks, (int)s);
    return ceil_div(nchunks, cps);
}

size_t ws_bytes_for(int ntiles, int splits)
{
    if (splits <= 1) return 0;
    return round16((size_t)ntiles * 4) + (size_t)splits * ntiles * 8 * sizeof(float);
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

int gemv_common(int fmt, const void *Wp, const void *q8, float *y, int rows, int cols,
                int splits, int cps, void *ws, size_t ws_bytes, void *stream)
{
    if (!Wp || !q8 || !y) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    if (!aligned16(Wp) || !aligned16(q8) || !aligned16(y)) return MQ_ERR_ALIGN;
    const Geom g = make_geom(rows, cols, fmt == 6 ? kQ6kBytes : kQ4kBytes);
    if (splits <= 0) {
        splits = plan_splits(g.ntiles, g.nchunks, device_sms());
        cps = ceil_div(g.nchunks, splits);
    }
    const int cov = check_coverage(g.nchunks, splits, cps);
    if (cov != MQ_OK) return cov;
    GemvLaunch a;
    memset(&a, 0, sizeof a);
    if (splits > 1) {
        if (!ws) return MQ_ERR_NULL;
        if (!aligned16(ws)) return MQ_ERR_ALIGN;
        if (ws_bytes < ws_bytes_for(g.ntiles, splits)) return MQ_ERR_WORKSPACE;
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
    a.splits = splits;
    a.cps = cps;
    a.n_items = (long long)g.ntiles * splits;
    a.tile_bytes = g.tile_bytes;
    a.q8_d_off = (unsigned)q8_d_offset(cols);
    a.q8_sum_off = (unsigned)q8_sum_offset(cols);
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
    a.splits = g.nchunks;  // one chunk per work item
    a.cps = 1;
    a.n_items = (long long)g.ntiles * g.nchunks;
    a.tile_bytes = g.tile_bytes;
    a.q8_d_off = (unsigned)q8_d_offset(cols);
    a.q8_sum_off = (unsigned)q8_sum_offset(cols);
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
                                             (unsigned)q8_sum_offset(n), (cudaStream_t)stream);
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
                                                  (unsigned)q8_sum_offset(n), (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

int mq_swiglu_quant_q8(const float *g, const float *u, float *y, void *q8, int n, void *stream)
{
    if (!g || !u || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    if (!aligned16(g) || !aligned16(u) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_swiglu_quant_q8(g, u, y, (uint8_t *)q8, n,
                                                 (unsigned)q8_d_offset(n),
                                                 (unsigned)q8_sum_offset(n), (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : MQ_ERR_CUDA;
}

int mq_check_coverage(int nchunks, int splits, int chunks_per_split)
{
    return check_coverage(nchunks, splits, chunks_per_split);
}

int mq_gemv_plan_for(int rows, int cols, int sms, int *splits, int *chunks_per_split)
{
    if (!splits || !chunks_per_split) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    *splits = plan_splits(g.ntiles, g.nchunks, sms);
    *chunks_per_split = ceil_div(g.nchunks, *splits);
    return MQ_OK;
}

int mq_gemv_splits(int rows, int cols)
{
    if (!gemv_shape_ok(rows, cols)) return 0;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    return plan_splits(g.ntiles, g.nchunks, device_sms());
}

size_t mq_gemv_workspace_bytes(int rows, int cols)
{
    if (!gemv_shape_ok(rows, cols)) return 0;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    return ws_bytes_for(g.ntiles, plan_splits(g.ntiles, g.nchunks, device_sms()));
}

size_t mq_gemv_workspace_bytes_for(int rows, int splits)
{
    if (rows < 1) return 0;
    return ws_bytes_for(ceil_div(rows, kTileRows), splits);
}

int mq_gemv_q6k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream)
{
    return gemv_common(6, Wp, q8, y, rows, cols, 0, 0, ws, ws_bytes, stream);
}

int mq_gemv_q4k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream)
{
    return gemv_common(4, Wp, q8, y, rows, cols, 0, 0, ws, ws_bytes, stream);
}

int mq_gemv_q6k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, void *ws, size_t ws_bytes, void *stream)
{
    if (splits < 1 || chunks_per_split < 1) return MQ_ERR_COVERAGE;
    return gemv_common(6, Wp, q8, y, rows, cols, splits, chunks_per_split, ws, ws_bytes, stream);
}

int mq_gemv_q4k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, void *ws, size_t ws_bytes, void *stream)
{
    if (splits < 1 || chunks_per_split < 1) return MQ_ERR_COVERAGE;
    return gemv_common(4, Wp, q8, y, rows, cols, splits, chunks_per_split, ws, ws_bytes, stream);
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
