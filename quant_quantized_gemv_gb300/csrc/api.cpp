// api.cpp -- the C ABI of include/mq.h: argument validation, the GEMV dispatch
// plan and its coverage check, then the launch.  Nothing here allocates.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "layout.h"
#include "mq.h"

namespace mq {

thread_local char g_last_error[256];

int cuda_fail(const char *where, cudaError_t e)
{
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorString(e),
             cudaGetErrorName(e));
    return MQ_ERR_CUDA;
}

}  // namespace mq

namespace {

using namespace mq;

static_assert(kMaxParts == MQ_MAX_GROUP, "kernel part table and public group size differ");

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
// resident GEMV CTAs per SM: [device][warps per CTA]
std::atomic<int> g_ctas[kMaxDevices][kMaxCtaSplits + 1];
std::atomic<int> g_pdl{0};
// single-token GEMV weight ring (mq_set_gemv_ring): stages per warp and how
// many of them are requested before the grid-dependency wait; -1 = default
std::atomic<int> g_ring_stages{-1};
std::atomic<int> g_ring_pre{-1};
// resident small-batch CTAs per SM (register limit): [device][nt][warps per CTA]
std::atomic<int> g_batch_ctas[kMaxDevices][kMaxTokens + 1][7][kBatchMaxCtaWarps + 1];  // [..][fmt]
// resident gate||up CTAs per SM (register limit): [device][warps per CTA]
constexpr int kGateUpMaxWarps = 8;
std::atomic<int> g_gateup_ctas[kMaxDevices][7][kGateUpMaxWarps + 1];  // [device][fmt][warps]
// resident f32-activation GEMV CTAs per SM (register limit): [device][warps per CTA]
std::atomic<int> g_f32_ctas[kMaxDevices][kMaxCtaSplits + 1];

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool gemv_shape_ok(int rows, int cols)
{
    return rows >= 1 && cols >= kQK && cols % kQK == 0 && (long long)rows * cols < (1LL << 40);
}

bool vec_shape_ok(int n) { return n > 0 && n % 32 == 0; }

int current_device()
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_fail("cudaGetDevice", e);
        return -1;
    }
    if (dev < 0 || dev >= kMaxDevices) return -1;
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
    int ctas[kBatchMaxCtaWarps + 1];  // CTAs with w warps, no dynamic shared memory
    int ctas_tiles;               // 4-warp whole-tile CTAs holding the staged plane
};

struct DeviceLimits {
    int smem_per_sm, smem_reserved;  // shared memory per SM, reserved per CTA
    size_t max_plane;                // largest q8 plane the GEMV stages
    size_t max_batch_planes;         // largest nt planes the small-batch GEMV stages
    size_t max_x_f32;                // largest f32 row the f32-activation GEMV stages
};
std::atomic<bool> g_limits_ok[kMaxDevices];
DeviceLimits g_limits[kMaxDevices];
std::mutex g_limits_mutex;

bool device_limits(DeviceLimits *out)
{
    const int dev = current_device();
    if (dev < 0) return false;
    if (!g_limits_ok[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_limits_mutex);
        if (!g_limits_ok[dev].load(std::memory_order_relaxed)) {
            DeviceLimits l;
            cudaError_t e = cudaDeviceGetAttribute(&l.smem_per_sm,
                                                   cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&l.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock,
                                           dev);
            if (e != cudaSuccess) {
                cuda_fail("shared-memory attributes", e);
                return false;
            }
            l.max_plane = gemv_max_plane_bytes();  // also opts the kernels in
            l.max_batch_planes = gemv_batch_max_smem();
            l.max_x_f32 = gemv_f32_max_x_bytes();
            if (l.max_plane == 0 || l.max_batch_planes == 0 || l.max_x_f32 == 0 ||
                !gateup_opt_in(l.max_plane))
                return false;
            g_limits[dev] = l;
            g_limits_ok[dev].store(true, std::memory_order_release);
        }
    }
    *out = g_limits[dev];
    return true;
}

// The single-token GEMV's weight ring for a launch over parts of the given
// formats (mq_set_gemv_ring; off unless set): one slot holds the largest
// full chunk among them; the depth is clamped so that the largest CTA
// (kMaxCtaSplits warps, or 4 warps beside the staged plane) fits the
// device's shared memory.
struct Ring {
    int stages, pre;
    size_t slot;
};

Ring ring_for(const int *fmts, int n, size_t plane, const DeviceLimits &lim)
{
    Ring r{0, 0, 0};
    for (int i = 0; i < n; ++i) {
        const size_t c = (size_t)kTileRows * kChunkBlocks * block_bytes(fmts[i]);
        if (c > r.slot) r.slot = c;
    }
    int st = g_ring_stages.load(std::memory_order_relaxed);
    if (st < 0) st = 0;  // default: no ring (measured slower on the decode shapes)
    if (st > kGemvMaxStages) st = kGemvMaxStages;
    while (st > 0 && r.slot > 0 &&
           ((size_t)kMaxCtaSplits * st * r.slot > lim.max_plane ||
            gemv_dyn_smem(kGemvWarpsPerBlock, true, plane, st, r.slot) > lim.max_plane))
        --st;
    r.stages = r.slot > 0 ? st : 0;
    if (r.stages == 0) {
        r.slot = 0;
        return r;
    }
    const int pre = g_ring_pre.load(std::memory_order_relaxed);
    r.pre = pre < 0 || pre > r.stages ? r.stages : pre;
    return r;
}

// Resident GEMV CTAs per SM with w warps and dyn bytes of dynamic shared
// memory, asked of the device once per (device, w, dyn).
struct OccEntry {
    int w;
    size_t dyn;
    int ctas;
};
std::vector<OccEntry> g_occ[kMaxDevices][2];  // [device][lo]
std::atomic<int> g_ctas_lo[kMaxDevices][kMaxCtaSplits + 1];
std::mutex g_occ_mutex;

// lo: the grouped launches' instance (kGemvGroupRegs registers).
int gemv_ctas(int dev, int w, size_t dyn, bool lo = false)
{
    auto query = [&](size_t d) { return lo ? gemv_ctas_per_sm_lo(w, d) : gemv_ctas_per_sm(w, d); };
    if (dyn == 0) {  // register limit only: lock-free cache
        std::atomic<int> &slot = lo ? g_ctas_lo[dev][w] : g_ctas[dev][w];
        int v = slot.load(std::memory_order_relaxed);
        if (v <= 0) {
            v = query(0);
            if (v > 0) slot.store(v, std::memory_order_relaxed);
        }
        return v;
    }
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (const OccEntry &e : g_occ[dev][lo])
        if (e.w == w && e.dyn == dyn) return e.ctas;
    const int v = query(dyn);
    if (v > 0) g_occ[dev][lo].push_back(OccEntry{w, dyn, v});
    return v;
}

// CTAs per SM of the single-token GEMV: split CTAs of w warps hold their
// warps' ring slots; whole-tile CTAs (kGemvWarpsPerBlock warps) also the
// staged plane of `plane` bytes.
bool device_occupancy(Occupancy *o, size_t plane, const Ring &ring, bool lo = false)
{
    const int dev = current_device();
    DeviceLimits lim;
    if (dev < 0 || !device_limits(&lim)) return false;
    for (int w = 1; w <= kMaxCtaSplits; ++w) {
        const int v = gemv_ctas(dev, w, gemv_dyn_smem(w, false, plane, ring.stages, ring.slot), lo);
        if (v < 0) return false;
        o->ctas[w] = v;
    }
    o->ctas_tiles = gemv_ctas(dev, kGemvWarpsPerBlock,
                              gemv_dyn_smem(kGemvWarpsPerBlock, true, plane, ring.stages, ring.slot), lo);
    return o->ctas_tiles > 0;
}

// The ring of a launch over the given formats on the current device.
bool device_ring(const int *fmts, int n, size_t plane, Ring *r)
{
    DeviceLimits lim;
    if (!device_limits(&lim)) return false;
    *r = ring_for(fmts, n, plane, lim);
    return true;
}

// Resident CTAs per SM of the small-batch kernel for nt tokens of format fmt
// with w warps (register limit, measured once per device and shape); 0
// when such a CTA does not fit, -1 on a CUDA error.
int batch_ctas_regs(int nt, int fmt, int w)
{
    const int dev = current_device();
    if (dev < 0) return -1;
    std::atomic<int> &slot = g_batch_ctas[dev][nt][fmt][w];
    int v = slot.load(std::memory_order_relaxed);
    if (v == 0) {
        v = gemv_batch_ctas_per_sm(nt, fmt, w, 0);
        if (v < 0) return -1;
        slot.store(v > 0 ? v : -2, std::memory_order_relaxed);  // -2: does not fit
    }
    return v > 0 ? v : (v == -2 ? 0 : v);
}

// Warps a CTA of the small-batch kernel holds on this device: the most (up
// to the kernel's compile-time bound) for which one CTA fits an SM; 0 on
// error.
int batch_budget(int nt, int fmt)
{
    int best = 0;
    for (int w = 1; w <= batch_warp_budget_max(nt, fmt); ++w) {
        const int v = batch_ctas_regs(nt, fmt, w);
        if (v < 0) return 0;
        if (v == 0) break;
        best = w;
    }
    return best;
}

// The small-batch kernel for nt tokens: every CTA stages all nt planes.
// CTA shapes up to the device's warp budget (batch_budget).
bool batch_occupancy(Occupancy *o, int nt, int fmt, size_t planes, int *budget_out)
{
    DeviceLimits lim;
    if (!device_limits(&lim)) return false;
    const long long per_cta = (long long)planes + kBatchStaticSmem + lim.smem_reserved;
    const int by_smem = (int)(lim.smem_per_sm / per_cta);
    const int budget = batch_budget(nt, fmt);
    if (budget < 1) return false;
    for (int w = 1; w <= kBatchMaxCtaWarps; ++w) {
        const int v = w <= budget ? batch_ctas_regs(nt, fmt, w) : 0;
        o->ctas[w] = v < by_smem ? v : by_smem;
    }
    o->ctas_tiles = 0;  // unused by the small-batch plans
    *budget_out = budget;
    return o->ctas[budget] > 0;
}

// The same from a register count (host-only planning, tests): 64K registers
// per SM, at most 2048 threads and 32 CTAs.
Occupancy model_occupancy(int regs_per_thread, size_t plane)
{
    Occupancy o;
    const int regs = ((regs_per_thread + 7) / 8) * 8;
    const int by_smem = (int)(233472 / ((long long)plane + kGemvStaticSmem + 1024));
    for (int w = 1; w <= kBatchMaxCtaWarps; ++w) {
        int c = 65536 / (w * 32 * regs);
        if (c > 2048 / (32 * w)) c = 2048 / (32 * w);
        if (c > 32) c = 32;
        o.ctas[w] = c;
    }
    o.ctas_tiles = o.ctas[kGemvWarpsPerBlock] < by_smem ? o.ctas[kGemvWarpsPerBlock] : by_smem;
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
    const long long wave = (long long)sms * (o.ctas_tiles > 0 ? o.ctas_tiles : 1) *
                           kGemvWarpsPerBlock;  // warps in one wave of 4-warp whole-tile CTAs
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

// Small-batch plan: S splits per tile (1..12, none empty), CTAs of S warps
// per tile x budget / S tiles, each CTA running tpi tile groups.  Every CTA
// stages all nt planes, so the resident CTAs per SM come from the
// occupancy with that much shared memory.  Choose the S whose busiest warp
// streams the fewest chunks, scaled up when the grid leaves SMs idle.
Plan batch_plan_for(int ntiles, int nchunks, int sms, const Occupancy &o, int budget)
{
    if (sms <= 0) sms = 1;
    Plan best{1, nchunks, 1};
    double best_score = -1.0;
    for (int S = 1; S <= kBatchMaxCtaSplits && S <= nchunks; ++S) {
        const int cps = ceil_div(nchunks, S);
        if ((long long)(S - 1) * cps >= nchunks) continue;  // an empty split
        const int G = budget / S, W = S * G;
        const long long resident = (long long)sms * o.ctas[W];
        if (resident <= 0) continue;
        const long long groups = (ntiles + G - 1) / G;
        const long long tpc = (groups + resident - 1) / resident;
        const long long ctas = (groups + tpc - 1) / tpc;
        const double busy = ctas >= sms ? 1.0 : (double)ctas / sms;
        const double score = (double)(tpc * cps) / busy;
        if (best_score < 0 || score < best_score) {
            best_score = score;
            best = Plan{S, cps, (int)tpc};
        }
    }
    return best;
}

long long batch_ctas(int ntiles, const Plan &p, int budget)
{
    const int G = budget / p.splits;
    const long long groups = (ntiles + G - 1) / G;
    return (groups + p.tpi - 1) / p.tpi;
}

long long plan_items(int ntiles, const Plan &p)
{
    return p.splits > 1 ? (long long)ntiles * p.splits : (ntiles + p.tpi - 1) / p.tpi;
}

// Workspace of a plan: arrival counters and 8 partials per work item, only
// when the splits are too many to meet in one CTA.
size_t ws_bytes_for(long long total_tiles, long long n_items, const Plan &p)
{
    if (p.splits <= kMaxCtaSplits) return 0;  // splits meet in shared memory (or none)
    return round16((size_t)total_tiles * 4) + (size_t)n_items * 8 * sizeof(float);
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

int check_batch_plan(int nchunks, const Plan &p)
{
    if (p.splits < 1 || p.splits > kBatchMaxCtaSplits || p.tpi < 1) return MQ_ERR_COVERAGE;
    return check_coverage(nchunks, p.splits, p.cps);
}

int check_plan(int nchunks, const Plan &p)
{
    if (p.tpi < 1 || (p.splits > 1 && p.tpi != 1)) return MQ_ERR_COVERAGE;
    return check_coverage(nchunks, p.splits, p.cps);
}

struct Part {
    int fmt, rows;
    const void *Wp;
    float *y;
};

// Validate a group, pick or check its plan, size the workspace.  On MQ_OK,
// `a` holds everything but the workspace pointers, and *need the bytes.
// nt == 0: the single-token GEMV; nt >= 1: the small-batch kernel for nt tokens.
int prepare_group(const Part *parts, int nparts, const void *q8, int cols, const Plan *explicit_plan,
                  GemvLaunch *a, size_t *need, bool sizes_only = false, int nt = 0)
{
    if (nparts < 1 || nparts > kMaxParts) return MQ_ERR_SHAPE;
    if (nt < 0 || nt > kMaxTokens) return MQ_ERR_SHAPE;
    const bool batch = nt > 0;
    if (!parts || (!q8 && !sizes_only)) return MQ_ERR_NULL;
    if (cols < kQK || cols % kQK != 0) return MQ_ERR_SHAPE;
    if (!aligned16(q8)) return MQ_ERR_ALIGN;
    memset(a, 0, sizeof *a);
    const int nb = cols / kQK, nchunks = ceil_div(nb, kChunkBlocks);
    long long total_tiles = 0;
    for (int p = 0; p < nparts; ++p) {
        const Part &x = parts[p];
        if (block_bytes(x.fmt) == 0) return MQ_ERR_SHAPE;
        if ((!x.Wp || !x.y) && !sizes_only) return MQ_ERR_NULL;
        if (!gemv_shape_ok(x.rows, cols)) return MQ_ERR_SHAPE;
        if (!aligned16(x.Wp) || !aligned16(x.y)) return MQ_ERR_ALIGN;
        total_tiles += ceil_div(x.rows, kTileRows);
    }
    if (total_tiles * nchunks >= (1LL << 31)) return MQ_ERR_SHAPE;
    const size_t plane = q8_plane_bytes(cols);
    if (batch && nparts != 1) return MQ_ERR_SHAPE;  // the small-batch kernel takes one matrix
    if (explicit_plan) {  // a wrong plan is refused before anything touches the device
        const int cov = batch ? check_batch_plan(nchunks, *explicit_plan)
                              : check_plan(nchunks, *explicit_plan);
        if (cov != MQ_OK) return cov;
    }
    // small batch: the warps one CTA holds (the device's, or the compile-time
    // bound when only sizes are asked for: then nothing is launched)
    int wpc = batch ? batch_warp_budget_max(nt, parts[0].fmt) : 0;
    if (!sizes_only) {
        DeviceLimits lim;
        if (!device_limits(&lim)) return MQ_ERR_CUDA;
        // the plane(s) must fit in shared memory (a whole-tile CTA stages its
        // plane rounded up to 128 bytes)
        if (!batch ? gemv_dyn_smem(kGemvWarpsPerBlock, true, plane, 0, 0) > lim.max_plane
                   : (size_t)nt * plane > lim.max_batch_planes)
            return MQ_ERR_SHAPE;
        if (batch && (wpc = batch_budget(nt, parts[0].fmt)) < 1) return MQ_ERR_CUDA;
    }
    Ring ring{0, 0, 0};  // asked of the device only when a launch or a default plan needs it
    if (!batch && (!sizes_only || !explicit_plan)) {
        int fmts[kMaxParts];
        for (int p = 0; p < nparts; ++p) fmts[p] = parts[p].fmt;
        if (!device_ring(fmts, nparts, plane, &ring)) return MQ_ERR_CUDA;
    }
    Plan pl;
    bool lo = false;
    if (explicit_plan) {
        pl = *explicit_plan;
    } else {
        Occupancy o;
        if (!batch) {
            // a group of q6_K/q4_K parts without a ring runs the kernel's
            // kGemvGroupRegs instance (gemv.cu), planned with its occupancy
            bool q5 = false;
            for (int p = 0; p < nparts; ++p) q5 = q5 || parts[p].fmt == 5;
            lo = nparts >= 2 && !q5 && ring.stages == 0;
            if (!device_occupancy(&o, plane, ring, lo)) return MQ_ERR_CUDA;
            pl = plan_for((int)total_tiles, nchunks, device_sms(), o);
        } else {
            if (!batch_occupancy(&o, nt, parts[0].fmt, (size_t)nt * plane, &wpc)) return MQ_ERR_CUDA;
            pl = batch_plan_for((int)total_tiles, nchunks, device_sms(), o, wpc);
        }
    }
    const int cov = batch ? check_batch_plan(nchunks, pl) : check_plan(nchunks, pl);
    if (cov != MQ_OK) return cov;
    long long items = 0, tiles = 0;
    for (int p = 0; p < nparts; ++p) {
        const Part &x = parts[p];
        const Geom g = make_geom(x.rows, cols, block_bytes(x.fmt));
        GemvPart &gp = a->part[p];
        gp.W = (const uint8_t *)x.Wp;
        gp.y = x.y;
        gp.rows = x.rows;
        gp.ntiles = g.ntiles;
        gp.fmt = x.fmt;
        gp.item0 = (int)items;
        gp.tile0 = (int)tiles;
        gp.tile_bytes_div16 = (int)(g.tile_bytes / 16);
        items += batch ? batch_ctas(g.ntiles, pl, wpc) : plan_items(g.ntiles, pl);
        tiles += g.ntiles;
    }
    if (items >= (1LL << 31)) return MQ_ERR_SHAPE;
    a->nparts = nparts;
    a->q8 = (const uint8_t *)q8;
    a->nb = nb;
    a->nchunks = nchunks;
    a->splits = pl.splits;
    a->cps = pl.cps;
    a->tpi = pl.tpi;
    a->n_items = (int)items;
    a->q8_d_off = (unsigned)q8_d_offset(cols);
    a->q8_sum_off = (unsigned)q8_sum_offset(cols);
    a->q8_bytes = (unsigned)plane;
    a->pdl = g_pdl.load(std::memory_order_relaxed);
    a->nt = batch ? nt : 1;
    a->q8_stride = (unsigned)plane;
    a->wpc = wpc;
    a->stages = ring.stages;
    a->pre = ring.pre;
    a->slot_bytes = (unsigned)ring.slot;
    a->ring_off = (unsigned)gemv_ring_off(pl.splits == 1, plane);
    a->lo = lo ? 1 : 0;
    *need = batch ? 0 : ws_bytes_for(total_tiles, items, pl);  // small batch: splits meet in the CTA
    return MQ_OK;
}

int gemv_group(const Part *parts, int nparts, const void *q8, int cols, const Plan *explicit_plan,
               void *ws, size_t ws_bytes, void *stream, int nt = 0, unsigned *cover = nullptr)
{
    GemvLaunch a;
    size_t need = 0;
    if (explicit_plan) {  // argument errors first, before anything asks the device
        const int st0 = prepare_group(parts, nparts, q8, cols, explicit_plan, &a, &need, true, nt);
        if (st0 != MQ_OK) return st0;
        if (need > 0 && !ws) return MQ_ERR_NULL;
        if (need > 0 && ws_bytes < need) return MQ_ERR_WORKSPACE;
    }
    const int st = prepare_group(parts, nparts, q8, cols, explicit_plan, &a, &need, false, nt);
    if (st != MQ_OK) return st;
    if (need > 0) {
        if (!ws) return MQ_ERR_NULL;
        if (!aligned16(ws)) return MQ_ERR_ALIGN;
        if (ws_bytes < need) return MQ_ERR_WORKSPACE;
        long long total_tiles = 0;
        for (int p = 0; p < nparts; ++p) total_tiles += a.part[p].ntiles;
        a.ws_cnt = (unsigned *)ws;
        a.ws_part = (float *)((uint8_t *)ws + round16((size_t)total_tiles * 4));
    }
    a.cover = cover;
    const cudaError_t e = nt > 0 ? launch_gemv_batch(a, (cudaStream_t)stream)
                          : cover ? launch_cover(a, (cudaStream_t)stream)
                                  : launch_gemv(a, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail(nt > 0 ? "small-batch GEMV launch" : "GEMV launch", e);
}

int gemv_common(int fmt, const void *Wp, const void *q8, float *y, int rows, int cols,
                const Plan *explicit_plan, void *ws, size_t ws_bytes, void *stream, int nt = 0)
{
    if (!Wp || !q8 || !y) return MQ_ERR_NULL;
    const Part part{fmt, rows, Wp, y};
    return gemv_group(&part, 1, q8, cols, explicit_plan, ws, ws_bytes, stream, nt);
}

// The small-batch entry points (default plan).  One token goes to the
// single-token GEMV when that kernel's default plan needs no workspace (the
// batch entry points take none): it streams one token faster (7B ffn_down
// 11.2 against 12.8 us).  Otherwise, and for 2..8 tokens, the batch kernel.
int batch_entry(int fmt, const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                void *stream)
{
    if (nt < 1) return MQ_ERR_SHAPE;
    if (nt == 1) {
        // the single-token plan is worked out once and launched as checked
        if (!Wp || !q8 || !y) return MQ_ERR_NULL;
        const Part part{fmt, rows, Wp, y};
        GemvLaunch a;
        size_t need = 0;
        const int st = prepare_group(&part, 1, q8, cols, nullptr, &a, &need, false, 0);
        if (st == MQ_OK && need == 0) {
            const cudaError_t e = launch_gemv(a, (cudaStream_t)stream);
            return e == cudaSuccess ? MQ_OK : cuda_fail("GEMV launch", e);
        }
        // a shape the single-token kernel refuses is the batch kernel's to
        // judge; any other failure is the caller's answer
        if (st != MQ_OK && st != MQ_ERR_SHAPE) return st;
    }
    return gemv_common(fmt, Wp, q8, y, rows, cols, nullptr, nullptr, 0, stream, nt);
}

int batch_plan_of(int rows, int cols, int nt, Plan *p)
{
    if (!gemv_shape_ok(rows, cols) || nt < 1 || nt > kMaxTokens) return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const size_t plane = q8_plane_bytes(cols);
    Occupancy o;
    DeviceLimits lim;
    if (!device_limits(&lim)) return MQ_ERR_CUDA;
    if ((size_t)nt * plane > lim.max_batch_planes) return MQ_ERR_SHAPE;
    int wpc = 0;
    if (!batch_occupancy(&o, nt, 6, (size_t)nt * plane, &wpc)) return MQ_ERR_CUDA;
    *p = batch_plan_for(g.ntiles, g.nchunks, device_sms(), o, wpc);
    return MQ_OK;
}

// Gate||up + SwiGLU -> q8 plan: W warps per CTA (1..8) and the grid.  The
// largest W whose one-CTA-per-block grid fits one resident wave; failing
// that (very many blocks) 4 warps and a one-wave grid that strides over the
// blocks.  sms/ctas_of give the machine.
struct GateUpPlan {
    int wpb, ctas;
};

template <class CtasOf>
GateUpPlan gateup_plan_for(int nblk, int sms, CtasOf ctas_of)
{
    if (sms <= 0) sms = 1;
    for (int w = kGateUpMaxWarps; w >= 1; --w) {
        const long long resident = (long long)sms * ctas_of(w);
        if (resident > 0 && nblk <= resident) return GateUpPlan{w, nblk};
    }
    long long resident = (long long)sms * ctas_of(4);
    if (resident < 1) resident = 1;
    return GateUpPlan{4, (int)(nblk < resident ? nblk : resident)};
}

int gateup_device_ctas(int fmt, int w, size_t plane)
{
    const int dev = current_device();
    DeviceLimits lim;
    if (dev < 0 || !device_limits(&lim)) return 0;
    std::atomic<int> &slot = g_gateup_ctas[dev][fmt][w];
    int v = slot.load(std::memory_order_relaxed);
    if (v <= 0) {
        v = gateup_ctas_per_sm(fmt, w, 0);
        if (v <= 0) return 0;
        slot.store(v, std::memory_order_relaxed);
    }
    const long long per_cta = (long long)plane + 2 * 8 * 8 * 4 + lim.smem_reserved;
    const int by_smem = (int)(lim.smem_per_sm / per_cta);
    return v < by_smem ? v : by_smem;
}

int gateup_common(int fmt, const void *Wg, const void *Wu, const void *q8, int rows, int cols,
                  float *act, void *q8o, const GateUpPlan *explicit_plan, void *stream)
{
    if (!Wg || !Wu || !q8 || !act || !q8o) return MQ_ERR_NULL;
    if (block_bytes(fmt) == 0) return MQ_ERR_SHAPE;
    if (!gemv_shape_ok(rows, cols) || rows % 32 != 0) return MQ_ERR_SHAPE;
    if (!aligned16(act) || !aligned16(q8o)) return MQ_ERR_ALIGN;
    const int nblk = rows / 32;
    if (explicit_plan && (explicit_plan->wpb < 1 || explicit_plan->wpb > kGateUpMaxWarps ||
                          explicit_plan->ctas < 1 || explicit_plan->ctas > nblk))
        return MQ_ERR_COVERAGE;
    const Part parts[2] = {Part{fmt, rows, Wg, nullptr}, Part{fmt, rows, Wu, nullptr}};
    GateUpLaunch L;
    memset(&L, 0, sizeof L);
    size_t need = 0;
    const int nchunks = ceil_div(cols / kQK, kChunkBlocks);
    const Plan whole{1, nchunks, 1};  // fills the geometry; the gate||up kernel has its own plan
    Part checked[2] = {parts[0], parts[1]};
    checked[0].y = checked[1].y = act;  // stand-ins: prepare_group requires an output pointer
    const int st = prepare_group(checked, 2, q8, cols, &whole, &L.g, &need);
    if (st != MQ_OK) return st;
    GateUpPlan pl;
    if (explicit_plan) {
        pl = *explicit_plan;
    } else {
        bool ok = true;
        const size_t plane = q8_plane_bytes(cols);
        pl = gateup_plan_for(nblk, device_sms(), [&](int w) {
            const int c = gateup_device_ctas(fmt, w, plane);
            if (c <= 0) ok = false;
            return c;
        });
        if (!ok) return MQ_ERR_CUDA;
    }
    L.act = act;
    L.q8o = (uint8_t *)q8o;
    L.o_d_off = (unsigned)q8_d_offset(rows);
    L.o_sum_off = (unsigned)q8_sum_offset(rows);
    L.nblk = nblk;
    L.wpb = pl.wpb;
    const cudaError_t e = launch_gateup(L, pl.ctas, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("gate||up launch", e);
}

int subdots_common(int fmt, const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                   void *stream)
{
    if (!Wp || !q8 || !isums) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    if (!aligned16(Wp) || !aligned16(q8) || !aligned16(isums)) return MQ_ERR_ALIGN;
    const Geom g = make_geom(rows, cols, block_bytes(fmt));
    const Plan pl{g.nchunks, 1, 1};  // one chunk per work item
    const Part part{fmt, rows, Wp, (float *)isums};
    GemvLaunch a;
    size_t need = 0;
    const int st = prepare_group(&part, 1, q8, cols, &pl, &a, &need);
    if (st != MQ_OK) return st;
    a.part[0].y = nullptr;
    a.isums = isums;
    const cudaError_t e = launch_subdots(a, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("sub-dot launch", e);
}

// ---- q6_K against an f32 activation row --------------------------------
// CTAs per SM of the f32 kernel: its register limit and the shared memory
// of a staged row of `xbytes` (every CTA stages it, split CTAs included).
bool f32_occupancy(Occupancy *o, size_t xbytes)
{
    const int dev = current_device();
    DeviceLimits lim;
    if (dev < 0 || !device_limits(&lim)) return false;
    const long long per_cta = (long long)xbytes + kGemvStaticSmem + lim.smem_reserved;
    const int by_smem = (int)(lim.smem_per_sm / per_cta);
    for (int w = 1; w <= kMaxCtaSplits; ++w) {
        std::atomic<int> &slot = g_f32_ctas[dev][w];
        int v = slot.load(std::memory_order_relaxed);
        if (v <= 0) {
            v = gemv_f32_ctas_per_sm(w, 0);
            if (v <= 0) return false;
            slot.store(v, std::memory_order_relaxed);
        }
        o->ctas[w] = v < by_smem ? v : by_smem;
    }
    o->ctas_tiles = o->ctas[kGemvWarpsPerBlock];
    return o->ctas_tiles > 0;
}

// The q8 GEMV's plan with the split count capped at one CTA's warps.
Plan f32_plan_for(int ntiles, int nchunks, int sms, const Occupancy &o)
{
    Plan p = plan_for(ntiles, nchunks, sms, o);
    if (p.splits > kMaxCtaSplits) {
        p.cps = ceil_div(nchunks, kMaxCtaSplits);
        p.splits = ceil_div(nchunks, p.cps);
        p.tpi = 1;
    }
    return p;
}

int f32_plan_of(int rows, int cols, Plan *p)
{
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    DeviceLimits lim;
    if (!device_limits(&lim)) return MQ_ERR_CUDA;
    const size_t xbytes = (size_t)cols * 4;
    if (xbytes > lim.max_x_f32) return MQ_ERR_SHAPE;
    Occupancy o;
    if (!f32_occupancy(&o, xbytes)) return MQ_ERR_CUDA;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    *p = f32_plan_for(g.ntiles, g.nchunks, device_sms(), o);
    return MQ_OK;
}

int gemv_f32_common(const void *Wp, const float *x, float *y, int rows, int cols,
                    const Plan *explicit_plan, void *stream)
{
    if (!Wp || !x || !y) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    if (!aligned16(Wp) || !aligned16(x) || !aligned16(y)) return MQ_ERR_ALIGN;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    if ((long long)g.ntiles * g.nchunks >= (1LL << 31)) return MQ_ERR_SHAPE;
    if (explicit_plan) {  // refused before anything touches the device
        if (explicit_plan->splits > kMaxCtaSplits) return MQ_ERR_COVERAGE;
        const int cov = check_plan(g.nchunks, *explicit_plan);
        if (cov != MQ_OK) return cov;
    }
    Plan pl;
    if (explicit_plan) {
        DeviceLimits lim;
        if (!device_limits(&lim)) return MQ_ERR_CUDA;
        if ((size_t)cols * 4 > lim.max_x_f32) return MQ_ERR_SHAPE;
        pl = *explicit_plan;
    } else {
        const int st = f32_plan_of(rows, cols, &pl);
        if (st != MQ_OK) return st;
    }
    GemvLaunch a;
    memset(&a, 0, sizeof a);
    GemvPart &gp = a.part[0];
    gp.W = (const uint8_t *)Wp;
    gp.y = y;
    gp.rows = rows;
    gp.ntiles = g.ntiles;
    gp.fmt = 6;
    gp.tile_bytes_div16 = (int)(g.tile_bytes / 16);
    const long long items = plan_items(g.ntiles, pl);
    if (items >= (1LL << 31)) return MQ_ERR_SHAPE;
    a.nparts = 1;
    a.q8 = (const uint8_t *)x;
    a.nb = g.nb;
    a.nchunks = g.nchunks;
    a.splits = pl.splits;
    a.cps = pl.cps;
    a.tpi = pl.tpi;
    a.n_items = (int)items;
    a.q8_bytes = (unsigned)((size_t)cols * 4);
    a.pdl = g_pdl.load(std::memory_order_relaxed);
    a.nt = 1;
    const cudaError_t e = launch_gemv_f32(a, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("f32 GEMV launch", e);
}

// The address a kernel on the current device uses for p: p itself for
// device or managed memory, the mapped device address for pinned host
// memory; MQ_ERR_ACCESS for pageable host memory or unknown pointers.
int device_address(const void *p, void **out)
{
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of a failed lookup
        return MQ_ERR_ACCESS;
    }
    const int dev = current_device();
    switch (at.type) {
    case cudaMemoryTypeDevice:
        if (at.device != dev) return MQ_ERR_ACCESS;
        *out = const_cast<void *>(p);
        return MQ_OK;
    case cudaMemoryTypeManaged:
        *out = const_cast<void *>(p);
        return MQ_OK;
    case cudaMemoryTypeHost:
        if (!at.devicePointer) return MQ_ERR_ACCESS;
        *out = at.devicePointer;
        return MQ_OK;
    default:
        return MQ_ERR_ACCESS;
    }
}

}  // namespace

namespace mq {
int pdl_setting() { return g_pdl.load(std::memory_order_relaxed); }
}  // namespace mq

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
    case MQ_ERR_CUDA: return "a CUDA call failed (mq_last_error names it)";
    case MQ_ERR_ACCESS: return "pointer not addressable by the GPU (pageable host memory?)";
    default: return "unknown status";
    }
}

const char *mq_version(void) { return "mq 0.1 sm_103a"; }

const char *mq_last_error(void) { return g_last_error; }

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
    const cudaError_t e = launch_quantize_q8(x, (uint8_t *)q8, n, 1, 0, (unsigned)q8_d_offset(n),
                                             (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed),
                                             (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("producer launch", e);
}

int mq_rmsnorm_quant_q8(const float *x, const float *gain, float eps, float *y, void *q8, int n,
                        void *stream)
{
    if (!x || !gain || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gain) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_rmsnorm_quant_q8(x, gain, eps, y, (uint8_t *)q8, n, 1, 0,
                                                  (unsigned)q8_d_offset(n),
                                                  (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed),
                                             (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("producer launch", e);
}

int mq_swiglu_quant_q8(const float *g, const float *u, float *y, void *q8, int n, void *stream)
{
    if (!g || !u || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n)) return MQ_ERR_SHAPE;
    if (!aligned16(g) || !aligned16(u) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_swiglu_quant_q8(g, u, y, (uint8_t *)q8, n, 1, 0,
                                                 (unsigned)q8_d_offset(n),
                                                 (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed),
                                             (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("producer launch", e);
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
    const Plan p = plan_for(g.ntiles, g.nchunks, sms, model_occupancy(regs_per_thread, q8_plane_bytes(cols)));
    *splits = p.splits;
    *chunks_per_split = p.cps;
    *tiles_per_item = p.tpi;
    return MQ_OK;
}

int mq_gemv_plan(int rows, int cols, int fmt, int *splits, int *chunks_per_split,
                 int *tiles_per_item)
{
    if (!splits || !chunks_per_split || !tiles_per_item) return MQ_ERR_NULL;
    if (block_bytes(fmt) == 0) return MQ_ERR_SHAPE;
    if (!gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    const size_t plane = q8_plane_bytes(cols);
    Ring ring;
    if (!device_ring(&fmt, 1, plane, &ring)) return MQ_ERR_CUDA;
    Occupancy o;
    if (!device_occupancy(&o, plane, ring)) return MQ_ERR_CUDA;
    const Geom g = make_geom(rows, cols, block_bytes(fmt));
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
    if (check_plan(g.nchunks, p) != MQ_OK) return 0;
    return ws_bytes_for(g.ntiles, plan_items(g.ntiles, p), p);
}

size_t mq_gemv_workspace_bytes(int rows, int cols)
{
    // the default plan can depend on the format (its ring slots change the
    // occupancy): enough for the default plan of any format
    size_t most = 0;
    for (int fmt : {6, 4, 5}) {
        int s = 0, c = 0, t = 0;
        if (mq_gemv_plan(rows, cols, fmt, &s, &c, &t) != MQ_OK) return 0;
        const size_t b = mq_gemv_workspace_bytes_for(rows, cols, s, c, t);
        if (b > most) most = b;
    }
    return most;
}

size_t mq_gemv_group_workspace_bytes(const mq_gemv_part *parts, int nparts, int cols, int splits,
                                     int chunks_per_split, int tiles_per_item)
{
    if (!parts || nparts < 1 || nparts > kMaxParts) return 0;
    Part ps[kMaxParts];
    for (int p = 0; p < nparts; ++p) ps[p] = Part{parts[p].fmt, parts[p].rows, parts[p].Wp, parts[p].y};
    const Plan pl{splits, chunks_per_split, tiles_per_item};
    GemvLaunch a;
    size_t need = 0;
    if (prepare_group(ps, nparts, nullptr, cols, splits > 0 ? &pl : nullptr, &a, &need, true) != MQ_OK)
        return 0;
    return need;
}

int mq_gemv_group_q8(const mq_gemv_part *parts, int nparts, const void *q8, int cols, void *ws,
                     size_t ws_bytes, void *stream)
{
    return mq_gemv_group_q8_plan(parts, nparts, q8, cols, 0, 0, 0, ws, ws_bytes, stream);
}

int mq_gemv_group_q8_coverage(const mq_gemv_part *parts, int nparts, const void *q8, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *ws,
                              size_t ws_bytes, unsigned *counts, void *stream)
{
    if (!parts || !counts) return MQ_ERR_NULL;
    if (nparts < 1 || nparts > kMaxParts) return MQ_ERR_SHAPE;
    if (!aligned16(counts)) return MQ_ERR_ALIGN;
    Part ps[kMaxParts];
    for (int p = 0; p < nparts; ++p) ps[p] = Part{parts[p].fmt, parts[p].rows, parts[p].Wp, parts[p].y};
    const Plan pl{splits, chunks_per_split, tiles_per_item};
    return gemv_group(ps, nparts, q8, cols, splits > 0 ? &pl : nullptr, ws, ws_bytes, stream, 0, counts);
}

int mq_gemv_group_q8_plan(const mq_gemv_part *parts, int nparts, const void *q8, int cols,
                          int splits, int chunks_per_split, int tiles_per_item, void *ws,
                          size_t ws_bytes, void *stream)
{
    if (!parts) return MQ_ERR_NULL;
    if (nparts < 1 || nparts > kMaxParts) return MQ_ERR_SHAPE;
    Part ps[kMaxParts];
    for (int p = 0; p < nparts; ++p) ps[p] = Part{parts[p].fmt, parts[p].rows, parts[p].Wp, parts[p].y};
    const Plan pl{splits, chunks_per_split, tiles_per_item};
    return gemv_group(ps, nparts, q8, cols, splits > 0 ? &pl : nullptr, ws, ws_bytes, stream);
}

int mq_quantize_q8_batch(const float *x, void *q8, int n, int nt, void *stream)
{
    if (!x || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n) || nt < 1 || nt > kMaxTokens) return MQ_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_quantize_q8(x, (uint8_t *)q8, n, nt, (unsigned)q8_plane_bytes(n),
                                             (unsigned)q8_d_offset(n), (unsigned)q8_sum_offset(n),
                                             g_pdl.load(std::memory_order_relaxed), (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("producer launch", e);
}

int mq_rmsnorm_quant_q8_batch(const float *x, const float *gain, float eps, float *y, void *q8,
                              int n, int nt, void *stream)
{
    if (!x || !gain || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n) || nt < 1 || nt > kMaxTokens) return MQ_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gain) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_rmsnorm_quant_q8(
        x, gain, eps, y, (uint8_t *)q8, n, nt, (unsigned)q8_plane_bytes(n), (unsigned)q8_d_offset(n),
        (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed), (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("producer launch", e);
}

int mq_swiglu_quant_q8_batch(const float *g, const float *u, float *y, void *q8, int n, int nt,
                             void *stream)
{
    if (!g || !u || !y || !q8) return MQ_ERR_NULL;
    if (!vec_shape_ok(n) || nt < 1 || nt > kMaxTokens) return MQ_ERR_SHAPE;
    if (!aligned16(g) || !aligned16(u) || !aligned16(y) || !aligned16(q8)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_swiglu_quant_q8(
        g, u, y, (uint8_t *)q8, n, nt, (unsigned)q8_plane_bytes(n), (unsigned)q8_d_offset(n),
        (unsigned)q8_sum_offset(n), g_pdl.load(std::memory_order_relaxed), (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("producer launch", e);
}

int mq_gemv_batch_plan(int rows, int cols, int nt, int *splits, int *chunks_per_split,
                       int *tiles_per_item)
{
    if (!splits || !chunks_per_split || !tiles_per_item) return MQ_ERR_NULL;
    Plan p;
    const int st = batch_plan_of(rows, cols, nt, &p);
    if (st != MQ_OK) return st;
    *splits = p.splits;
    *chunks_per_split = p.cps;
    *tiles_per_item = p.tpi;
    return MQ_OK;
}

int mq_gemv_batch_plan_for(int rows, int cols, int nt, int sms, int regs_per_thread, int *splits,
                           int *chunks_per_split, int *tiles_per_item)
{
    if (!splits || !chunks_per_split || !tiles_per_item) return MQ_ERR_NULL;
    if (!gemv_shape_ok(rows, cols) || nt < 1 || nt > kMaxTokens || regs_per_thread < 1 ||
        regs_per_thread > 255)
        return MQ_ERR_SHAPE;
    const Geom g = make_geom(rows, cols, kQ6kBytes);
    const size_t planes = (size_t)nt * q8_plane_bytes(cols);
    Occupancy o = model_occupancy(regs_per_thread, 0);
    const int by_smem = (int)(233472 / ((long long)planes + kBatchStaticSmem + 1024));
    for (int w = 1; w <= kBatchMaxCtaWarps; ++w)
        if (o.ctas[w] > by_smem) o.ctas[w] = by_smem;
    // the kernel's budget follows its register cap: the warps the register
    // file holds at that count, at most 16
    const int fit = 65536 / (32 * regs_per_thread);
    const int budget = fit < kBatchMaxCtaWarps ? (fit > 0 ? fit : 1) : kBatchMaxCtaWarps;
    const Plan p = batch_plan_for(g.ntiles, g.nchunks, sms, o, budget);
    *splits = p.splits;
    *chunks_per_split = p.cps;
    *tiles_per_item = p.tpi;
    return MQ_OK;
}

int mq_gemv_q6k_q8_batch(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                         void *stream)
{
    return batch_entry(6, Wp, q8, nt, y, rows, cols, stream);
}

int mq_gemv_q4k_q8_batch(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                         void *stream)
{
    return batch_entry(4, Wp, q8, nt, y, rows, cols, stream);
}

int mq_gemv_q5k_q8_batch(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                         void *stream)
{
    return batch_entry(5, Wp, q8, nt, y, rows, cols, stream);
}

int mq_gemv_q5k_q8_batch_plan(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *stream)
{
    if (nt < 1) return MQ_ERR_SHAPE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(5, Wp, q8, y, rows, cols, &p, nullptr, 0, stream, nt);
}

int mq_gemv_q6k_q8_batch_plan(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *stream)
{
    if (nt < 1) return MQ_ERR_SHAPE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(6, Wp, q8, y, rows, cols, &p, nullptr, 0, stream, nt);
}

int mq_gemv_q4k_q8_batch_plan(const void *Wp, const void *q8, int nt, float *y, int rows, int cols,
                              int splits, int chunks_per_split, int tiles_per_item, void *stream)
{
    if (nt < 1) return MQ_ERR_SHAPE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(4, Wp, q8, y, rows, cols, &p, nullptr, 0, stream, nt);
}

int mq_gemv_gateup_swiglu_q8(int fmt, const void *Wg, const void *Wu, const void *q8, int rows,
                             int cols, float *act, void *q8_out, void *stream)
{
    return gateup_common(fmt, Wg, Wu, q8, rows, cols, act, q8_out, nullptr, stream);
}

int mq_gemv_gateup_swiglu_q8_plan(int fmt, const void *Wg, const void *Wu, const void *q8, int rows,
                                  int cols, float *act, void *q8_out, int warps_per_cta, int ctas,
                                  void *stream)
{
    const GateUpPlan p{warps_per_cta, ctas};
    return gateup_common(fmt, Wg, Wu, q8, rows, cols, act, q8_out, &p, stream);
}

int mq_gemv_gateup_plan_for(int rows, int sms, int regs_per_thread, int *warps_per_cta, int *ctas)
{
    if (!warps_per_cta || !ctas) return MQ_ERR_NULL;
    if (rows < 32 || rows % 32 != 0 || regs_per_thread < 1 || regs_per_thread > 255) return MQ_ERR_SHAPE;
    const Occupancy o = model_occupancy(regs_per_thread, 0);
    const GateUpPlan p = gateup_plan_for(rows / 32, sms, [&](int w) { return o.ctas[w]; });
    *warps_per_cta = p.wpb;
    *ctas = p.ctas;
    return MQ_OK;
}

int mq_repack_device(int fmt, const void *gguf, void *dst, int rows, int cols, void *stream)
{
    if (!gguf || !dst) return MQ_ERR_NULL;
    if (block_bytes(fmt) == 0 || !gemv_shape_ok(rows, cols)) return MQ_ERR_SHAPE;
    if (!aligned16(dst) || ((uintptr_t)gguf & 1u) != 0) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_repack(fmt, gguf, dst, rows, cols, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("device repack launch", e);
}

int mq_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (!dst || !src) return MQ_ERR_NULL;
    if (bytes == 0 || bytes % 16 != 0) return MQ_ERR_SHAPE;
    if (!aligned16(dst) || !aligned16(src)) return MQ_ERR_ALIGN;
    void *d = nullptr;
    const void *sp = nullptr;
    int st = device_address(dst, &d);
    if (st == MQ_OK) st = device_address(src, const_cast<void **>(&sp));
    if (st != MQ_OK) return st;
    if (!aligned16(d) || !aligned16(sp)) return MQ_ERR_ALIGN;
    const cudaError_t e = launch_copy(d, sp, bytes, g_pdl.load(std::memory_order_relaxed),
                                      (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("copy launch", e);
}

int mq_device_address(const void *p, void **out)
{
    if (!p || !out) return MQ_ERR_NULL;
    return device_address(p, out);
}

int mq_read_floor(const void *src, size_t bytes, void *stream)
{
    if (!src) return MQ_ERR_NULL;
    if (bytes == 0 || bytes % 16 != 0) return MQ_ERR_SHAPE;
    if (!aligned16(src)) return MQ_ERR_ALIGN;
    const int sms = device_sms();
    if (sms <= 0) return MQ_ERR_CUDA;
    const cudaError_t e = launch_read_floor(src, bytes, nullptr, sms, (cudaStream_t)stream);
    return e == cudaSuccess ? MQ_OK : cuda_fail("read-floor launch", e);
}

int mq_set_pdl(int enable)
{
    return g_pdl.exchange(enable ? 1 : 0);
}

int mq_set_gemv_ring(int stages, int pre_wait)
{
    if (stages < -1) stages = -1;
    if (stages > kGemvMaxStages) stages = kGemvMaxStages;
    g_ring_pre.store(pre_wait < -1 ? -1 : pre_wait, std::memory_order_relaxed);
    return g_ring_stages.exchange(stages);
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
    if (splits < 1) return MQ_ERR_COVERAGE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(6, Wp, q8, y, rows, cols, &p, ws, ws_bytes, stream);
}

int mq_gemv_q4k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream)
{
    if (splits < 1) return MQ_ERR_COVERAGE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(4, Wp, q8, y, rows, cols, &p, ws, ws_bytes, stream);
}

int mq_gemv_q5k_q8(const void *Wp, const void *q8, float *y, int rows, int cols, void *ws,
                   size_t ws_bytes, void *stream)
{
    return gemv_common(5, Wp, q8, y, rows, cols, nullptr, ws, ws_bytes, stream);
}

int mq_gemv_q5k_q8_plan(const void *Wp, const void *q8, float *y, int rows, int cols, int splits,
                        int chunks_per_split, int tiles_per_item, void *ws, size_t ws_bytes,
                        void *stream)
{
    if (splits < 1) return MQ_ERR_COVERAGE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_common(5, Wp, q8, y, rows, cols, &p, ws, ws_bytes, stream);
}

int mq_gemv_q5k_q8_subdots(const void *Wp, const void *q8, int32_t *isums, int rows, int cols,
                           void *stream)
{
    return subdots_common(5, Wp, q8, isums, rows, cols, stream);
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

int mq_gemv_q6k_f32(const void *Wp, const float *x, float *y, int rows, int cols, void *stream)
{
    return gemv_f32_common(Wp, x, y, rows, cols, nullptr, stream);
}

int mq_gemv_q6k_f32_plan(const void *Wp, const float *x, float *y, int rows, int cols, int splits,
                         int chunks_per_split, int tiles_per_item, void *stream)
{
    if (splits < 1) return MQ_ERR_COVERAGE;
    const Plan p{splits, chunks_per_split, tiles_per_item};
    return gemv_f32_common(Wp, x, y, rows, cols, &p, stream);
}

int mq_gemv_q6k_f32_plan_of(int rows, int cols, int *splits, int *chunks_per_split,
                            int *tiles_per_item)
{
    if (!splits || !chunks_per_split || !tiles_per_item) return MQ_ERR_NULL;
    Plan p;
    const int st = f32_plan_of(rows, cols, &p);
    if (st != MQ_OK) return st;
    *splits = p.splits;
    *chunks_per_split = p.cps;
    *tiles_per_item = p.tpi;
    return MQ_OK;
}

}  // extern "C"
