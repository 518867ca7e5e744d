// api.cu -- the C ABI declared in include/rmsnorm.h: argument validation, the
// dispatch table over (rows, D, dtype, alignment, SM count), gw scratch, and
// the device status word.
//
// Dispatch (a pure function of its inputs, so the VJP's summation order and
// hence gw's bits are fixed for a given device):
//   * unaligned pointers or D*2 not a multiple of 16 -> generic tier;
//   * rows <= DECODE_ROWS (decode: one token per sequence)  -> direct tier;
//   * D <= 16384 -> staged tier (TMA bulk ring): sub-warp/warp per row for
//     D <= 1024, CTA per row above;
//   * longer rows -> direct tier (forward up to 32768, VJP up to 16384), then
//     generic.
#include "rmsnorm.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "plan.h"

using namespace rmsn;

namespace {

constexpr int64_t DECODE_ROWS = 8;
constexpr int MAX_DEVICES = 64;
// Shared-memory budget of one CTA when two share an SM (228 KB per SM, 1 KB
// reserved per CTA), and when one CTA has the SM to itself (227 KB opt-in).
constexpr size_t SMEM_TWO_PER_SM = 110 * 1024;
constexpr size_t SMEM_THREE_PER_SM = 72 * 1024;
constexpr size_t SMEM_ONE_PER_SM = 225 * 1024;
// Target bytes of one tensor's tile in the sub-warp/warp-per-row shape.
constexpr size_t SMALL_TILE_BYTES = 16 * 1024;
// Bytes of tiles in flight per SM the ring is sized for.  Measured on GB300
// (rows 16384, D 4096 and 8192): more read-ahead than this starves the
// kernel's own writes and lowers the bandwidth, less leaves HBM idle.  The
// forward writes as much as it reads and wants ~64 KB; the VJP (two bytes
// read per byte written) ~96 KB.
constexpr size_t INFLIGHT_FWD = 64 * 1024;
constexpr size_t INFLIGHT_VJP = 96 * 1024;

__device__ unsigned int g_devstatus;  // RMSNORM_DEVSTATUS_* bits, per device

thread_local int t_last_cuda_error = 0;

struct DevInfo {
    bool ready = false;
    int sm_count = 0;
    unsigned int *status = nullptr;  // device address of g_devstatus
    cudaMemPool_t pool = nullptr;    // gw scratch of rmsnorm_vjp; keeps its memory
};
std::mutex g_dev_mu;
DevInfo g_dev[MAX_DEVICES];

std::atomic<int64_t> g_drop_tile{-1};
std::atomic<long long> g_wait_budget{DEFAULT_WAIT_BUDGET};

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return RMSNORM_ERR_CUDA;
}

int current_device(DevInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= MAX_DEVICES) return RMSNORM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_devstatus);
        if (e != cudaSuccess) return cuda_fail(e);
        d.status = static_cast<unsigned int *>(p);
        d.ready = true;
    }
    *out = d;
    return RMSNORM_OK;
}

// The memory pool rmsnorm_vjp takes its gw scratch from, created on the
// first rmsnorm_vjp call on the current device (no other entry point needs
// one).
int scratch_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= MAX_DEVICES) return RMSNORM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.pool) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return cuda_fail(e);
        // Keep freed scratch in the pool: the next call reuses it without
        // going back to the driver.
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return cuda_fail(e);
        }
        d.pool = pool;
    }
    *out = d.pool;
    return RMSNORM_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Scalar and shape checks common to both operations.
int check_common(int64_t rows, int64_t D, int dtype, float eps, float weight_bias) {
    if (dtype != RMSNORM_F16 && dtype != RMSNORM_BF16) return RMSNORM_ERR_INVALID_ARG;
    if (rows < 0 || D <= 0) return RMSNORM_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return RMSNORM_ERR_INVALID_ARG;
    if (!std::isfinite(weight_bias)) return RMSNORM_ERR_INVALID_ARG;
    if (D > RMSNORM_MAX_D) return RMSNORM_ERR_UNSUPPORTED;
    if (rows > INT64_MAX / (2 * D)) return RMSNORM_ERR_UNSUPPORTED;
    return RMSNORM_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

// An output may coincide exactly with a same-sized input, or be disjoint.
bool bad_alias(const void *out, size_t nout, const void *in, size_t nin) {
    if (!overlaps(out, nout, in, nin)) return false;
    return !(out == in && nout == nin);
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// ---- dispatch planning ----------------------------------------------------

// Overrides of the staged tier's choices, read once from RMSNORM_TUNE
// ("cfg=N,cps=N,stages=N", any subset) for tuning sweeps.  Unset, the plan
// is a pure function of the problem and the device.
struct Tuning {
    int cfg = -1;    // staged configuration index
    int cps = 0;     // CTAs per SM (capped by what the registers allow)
    int stages = 0;  // maximum ring depth
};

Tuning parse_tuning() {
    Tuning t;
    const char *env = std::getenv("RMSNORM_TUNE");
    if (!env) return t;
    char buf[128];
    std::snprintf(buf, sizeof(buf), "%s", env);
    for (char *tok = std::strtok(buf, ","); tok; tok = std::strtok(nullptr, ",")) {
        int v = 0;
        if (std::sscanf(tok, "cfg=%d", &v) == 1 && v >= 0 && v < N_STAGED_CFG) t.cfg = v;
        else if (std::sscanf(tok, "cps=%d", &v) == 1 && v >= 1 && v <= 3) t.cps = v;
        else if (std::sscanf(tok, "stages=%d", &v) == 1 && v >= 2 && v <= MAX_STAGES) t.stages = v;
    }
    return t;
}

const Tuning &tuning() {
    static const Tuning t = parse_tuning();
    return t;
}

// Ring depth for a stage of `per_stage` bytes with `cps` CTAs per SM: one
// stage being consumed plus enough in flight to reach the mode's target
// (at least one).  An explicit RMSNORM_TUNE stages= wins.
int ring_stages(int mode, size_t per_stage, int cps) {
    if (tuning().stages) return tuning().stages;
    const size_t target = is_vjp(mode) ? INFLIGHT_VJP : INFLIGHT_FWD;
    const size_t per_sm_stage = per_stage * (size_t)cps;
    const int ahead = (int)std::max<size_t>(1, (target + per_sm_stage / 2) / per_sm_stage);
    return std::min(MAX_STAGES, 1 + ahead);
}

bool plan_staged(int mode, int64_t rows, int D, int sm_count, int ci, Plan *p) {
    const StagedCfg &c = STAGED_CFGS[ci];
    const Tuning &tu = tuning();
    const int ntens = input_tensors(mode);
    const size_t row_bytes = (size_t)D * 2;
    const int max_stages = tu.stages ? tu.stages : MAX_STAGES;
    const int cps_max = staged_max_ctas_per_sm(mode, c.nt, c.g, c.v);
    int cps = tu.cps ? std::min(tu.cps, cps_max) : staged_ctas_per_sm(mode, c.nt, c.g, c.v);
    p->tier = TIER_STAGED;
    p->cfg = ci;
    p->nt = c.nt;
    p->g = c.g;
    p->v = c.v;
    if (c.g < c.nt) {
        // Several rows per tile; shuffle-only reductions.
        const int ng = c.nt / c.g;
        const int64_t rpg_max =
            std::max<int64_t>(1, (int64_t)(SMALL_TILE_BYTES / (ng * row_bytes)));
        const int64_t want_tiles = (int64_t)sm_count * cps * 2;
        const int64_t rpg =
            std::min(rpg_max, std::max<int64_t>(1, ceil_div(rows, ng * want_tiles)));
        p->tile_rows = (int)(ng * rpg);
        p->stage_bytes = (uint32_t)(p->tile_rows * row_bytes);
        const size_t per_stage = (size_t)ntens * p->stage_bytes;
        cps = std::min(cps, 2);
        const size_t cap = cps == 2 ? SMEM_TWO_PER_SM : SMEM_ONE_PER_SM;
        p->stages = (int)std::min<size_t>(std::min<size_t>(max_stages, cap / per_stage),
                                          ring_stages(mode, per_stage, cps));
        if (p->stages < 2) return false;
        p->smem = STAGED_HEADER_BYTES + (size_t)p->stages * per_stage;
        if (is_vjp(mode))  // the cross-group gw sum reuses the ring
            p->smem = std::max(p->smem, (size_t)STAGED_HEADER_BYTES + (size_t)ng * D * 4);
    } else {
        // One row per tile, the whole CTA on it.  Two CTAs per SM when the
        // registers allow it and each can hold three stages, else one CTA
        // with at least two; the depth then follows the in-flight target.
        p->tile_rows = 1;
        p->stage_bytes = (uint32_t)row_bytes;
        const size_t per_stage = (size_t)ntens * row_bytes;
        const int64_t s3 = (int64_t)(SMEM_THREE_PER_SM / per_stage);
        const int64_t s2 = (int64_t)(SMEM_TWO_PER_SM / per_stage);
        const int64_t s1 = (int64_t)(SMEM_ONE_PER_SM / per_stage);
        if (cps == 3 && s3 >= 2) {
            p->stages = (int)std::min<int64_t>(std::min<int64_t>(max_stages, s3),
                                               ring_stages(mode, per_stage, 3));
        } else if (cps >= 2 && s2 >= 3) {
            cps = 2;
            p->stages = (int)std::min<int64_t>(std::min<int64_t>(max_stages, s2),
                                               ring_stages(mode, per_stage, 2));
        } else if (s1 >= 2) {
            cps = 1;
            p->stages = (int)std::min<int64_t>(std::min<int64_t>(max_stages, s1),
                                               ring_stages(mode, per_stage, 1));
        } else {
            return false;
        }
        p->smem = STAGED_HEADER_BYTES + (size_t)p->stages * per_stage;
    }
    p->num_tiles = ceil_div(rows, p->tile_rows);
    p->grid = (int)std::min<int64_t>(p->num_tiles, (int64_t)sm_count * cps);
    return true;
}

Plan make_plan(int mode, int64_t rows, int D, bool aligned, int sm_count) {
    Plan p{};
    const int nv = D / 8;
    if (aligned && rows > DECODE_ROWS) {
        const int forced = tuning().cfg;
        if (forced >= 0 && nv <= STAGED_CFGS[forced].max_nv &&
            !(is_vjp(mode) && forced == STAGED_CFG_WIDE) &&
            plan_staged(mode, rows, D, sm_count, forced, &p))
            return p;
        for (int ci = 0; ci < STAGED_CFG_WIDE; ++ci) {
            if (nv <= STAGED_CFGS[ci].max_nv) {
                if (plan_staged(mode, rows, D, sm_count, ci, &p)) return p;
                break;
            }
        }
    }
    if (aligned) {
        for (int ci = 0; ci < N_DIRECT_CFG; ++ci) {
            const DirectCfg &c = DIRECT_CFGS[ci];
            if (nv <= c.max_nv && !(is_vjp(mode) && c.v > 2)) {
                p = Plan{};
                p.tier = TIER_DIRECT;
                p.cfg = ci;
                p.nt = c.nt;
                p.g = c.nt;
                p.v = c.v;
                p.tile_rows = 1;
                p.num_tiles = rows;
                const int64_t resident = std::max(1, 2048 / c.nt);
                p.grid = (int)std::min<int64_t>(rows, (int64_t)sm_count * resident);
                return p;
            }
        }
    }
    p = Plan{};
    p.tier = TIER_GENERIC;
    p.nt = GENERIC_NT;
    p.g = GENERIC_NT;
    p.tile_rows = 1;
    p.num_tiles = rows;
    p.grid = (int)std::min<int64_t>(rows, (int64_t)sm_count * 8);
    return p;
}

size_t partials_bytes(const Plan &p, int64_t D) {
    const size_t b = (size_t)p.grid * (size_t)D * sizeof(float);
    return (b + 255) & ~(size_t)255;
}

cudaError_t launch_plan(int dtype, int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (p.tier) {
        case TIER_STAGED: return launch_staged(dtype, mode, p, a, s);
        case TIER_DIRECT: return launch_direct(dtype, mode, p, a, s);
        default: return launch_generic(dtype, mode, p, a, s);
    }
}

KernelArgs base_args(const DevInfo &dev, const Plan &p, float eps, float wb, int64_t rows,
                     int64_t D) {
    KernelArgs a{};
    a.status = dev.status;
    a.eps = eps;
    a.weight_bias = wb;
    a.rows = rows;
    a.D = (int)D;
    a.tile_rows = p.tile_rows;
    a.stages = p.stages;
    a.num_tiles = p.num_tiles;
    a.stage_bytes = p.stage_bytes;
    a.wait_budget = g_wait_budget.load(std::memory_order_relaxed);
    a.drop_tile = g_drop_tile.load(std::memory_order_relaxed);
    return a;
}

// Validation shared by the VJP entry points; *plan is filled on success when
// rows > 0.  g_res (the gradient reaching new_residual of the fused op) is
// null for the plain VJP.
int vjp_prepare(const void *x, const void *w, const void *g, const void *g_res, float eps,
                float weight_bias, void *gx, float *gw, int64_t rows, int64_t D, int dtype,
                DevInfo *dev, Plan *plan) {
    int st = check_common(rows, D, dtype, eps, weight_bias);
    if (st != RMSNORM_OK) return st;
    if (!w || !gw) return RMSNORM_ERR_INVALID_ARG;
    const size_t nw = (size_t)D * 2, ngw = (size_t)D * 4;
    if (rows > 0) {
        if (!x || !g || !gx) return RMSNORM_ERR_INVALID_ARG;
        const size_t n = (size_t)rows * (size_t)D * 2;
        if (overlaps(gx, n, gw, ngw)) return RMSNORM_ERR_INVALID_ARG;
        if (bad_alias(gx, n, x, n) || bad_alias(gx, n, g, n) || bad_alias(gx, n, g_res, n) ||
            overlaps(gx, n, w, nw))
            return RMSNORM_ERR_INVALID_ARG;
        if (overlaps(gw, ngw, x, n) || overlaps(gw, ngw, g, n) || overlaps(gw, ngw, g_res, n))
            return RMSNORM_ERR_INVALID_ARG;
    }
    if (overlaps(gw, ngw, w, nw)) return RMSNORM_ERR_INVALID_ARG;
    st = current_device(dev);
    if (st != RMSNORM_OK) return st;
    if (rows > 0) {
        const bool aligned = (D * 2) % 16 == 0 && aligned16(x) && aligned16(g) && aligned16(gx) &&
                             aligned16(w) && (!g_res || aligned16(g_res));
        *plan = make_plan(g_res ? MODE_VJP_ADD : MODE_VJP, rows, (int)D, aligned, dev->sm_count);
    }
    return RMSNORM_OK;
}

int vjp_run(const void *x, const void *w, const void *g, const void *g_res, float eps,
            float weight_bias, void *gx, float *gw, int64_t rows, int64_t D, int dtype,
            const DevInfo &dev, const Plan &p, float *partials, cudaStream_t s) {
    KernelArgs a = base_args(dev, p, eps, weight_bias, rows, D);
    a.in0 = x;
    a.in1 = g;
    a.in2 = g_res;
    a.w = w;
    a.out0 = gx;
    a.out1 = nullptr;
    a.partials = partials;
    cudaError_t e = launch_plan(dtype, g_res ? MODE_VJP_ADD : MODE_VJP, p, a, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_gw_reduce(partials, gw, p.grid, (int)D, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return RMSNORM_OK;
}

// The VJP with scratch from the library's stream-ordered pool.
int vjp_pooled(const void *x, const void *w, const void *g, const void *g_res, float eps,
               float weight_bias, void *gx, float *gw, int64_t rows, int64_t D, int dtype,
               void *stream) {
    DevInfo dev;
    Plan p{};
    int st = vjp_prepare(x, w, g, g_res, eps, weight_bias, gx, gw, rows, D, dtype, &dev, &p);
    if (st != RMSNORM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0) {
        cudaError_t e = cudaMemsetAsync(gw, 0, (size_t)D * sizeof(float), s);
        return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
    }
    cudaMemPool_t pool = nullptr;
    st = scratch_pool(&pool);
    if (st != RMSNORM_OK) return st;
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, partials_bytes(p, D), pool, s);
    if (e == cudaErrorMemoryAllocation) {
        (void)cudaGetLastError();
        return RMSNORM_ERR_NO_MEMORY;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    st = vjp_run(x, w, g, g_res, eps, weight_bias, gx, gw, rows, D, dtype, dev, p,
                 static_cast<float *>(ws), s);
    e = cudaFreeAsync(ws, s);
    if (st == RMSNORM_OK && e != cudaSuccess) st = cuda_fail(e);
    return st;
}

const char *tier_name(int t) {
    return t == TIER_STAGED ? "staged" : t == TIER_DIRECT ? "direct" : "generic";
}

}  // namespace

extern "C" {

int rmsnorm_fwd(const void *x, const void *residual, const void *w, float eps, float weight_bias,
                void *out, void *new_residual, int64_t rows, int64_t D, int dtype, void *stream) {
    int st = check_common(rows, D, dtype, eps, weight_bias);
    if (st != RMSNORM_OK) return st;
    if (!w) return RMSNORM_ERR_INVALID_ARG;
    if (rows == 0) return RMSNORM_OK;
    if (!x || !out) return RMSNORM_ERR_INVALID_ARG;
    if ((residual == nullptr) != (new_residual == nullptr)) return RMSNORM_ERR_INVALID_ARG;
    const size_t n = (size_t)rows * (size_t)D * 2, nw = (size_t)D * 2;
    if (overlaps(out, n, new_residual, n)) return RMSNORM_ERR_INVALID_ARG;
    if (bad_alias(out, n, x, n) || bad_alias(out, n, residual, n) || overlaps(out, n, w, nw))
        return RMSNORM_ERR_INVALID_ARG;
    if (bad_alias(new_residual, n, x, n) || bad_alias(new_residual, n, residual, n) ||
        overlaps(new_residual, n, w, nw))
        return RMSNORM_ERR_INVALID_ARG;

    DevInfo dev;
    st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    const int mode = residual ? MODE_FWD_RES : MODE_FWD_NORES;
    const bool aligned = (D * 2) % 16 == 0 && aligned16(x) && aligned16(w) && aligned16(out) &&
                         (!residual || (aligned16(residual) && aligned16(new_residual)));
    const Plan p = make_plan(mode, rows, (int)D, aligned, dev.sm_count);
    KernelArgs a = base_args(dev, p, eps, weight_bias, rows, D);
    a.in0 = x;
    a.in1 = residual;
    a.w = w;
    a.out0 = out;
    a.out1 = new_residual;
    a.partials = nullptr;
    cudaError_t e = launch_plan(dtype, mode, p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return RMSNORM_OK;
}

size_t rmsnorm_vjp_workspace_size(int64_t rows, int64_t D, int dtype) {
    if (check_common(rows, D, dtype, 0.f, 0.f) != RMSNORM_OK || rows == 0) return 0;
    DevInfo dev;
    if (current_device(&dev) != RMSNORM_OK) return 0;
    // The plan depends on pointer alignment; cover both outcomes.
    const Plan pa = make_plan(MODE_VJP, rows, (int)D, (D * 2) % 16 == 0, dev.sm_count);
    const Plan pu = make_plan(MODE_VJP, rows, (int)D, false, dev.sm_count);
    return std::max(partials_bytes(pa, D), partials_bytes(pu, D));
}

int rmsnorm_vjp_ws(const void *x, const void *w, const void *g, float eps, float weight_bias,
                   void *gx, float *gw, int64_t rows, int64_t D, int dtype, void *workspace,
                   size_t workspace_bytes, void *stream) {
    DevInfo dev;
    Plan p{};
    int st = vjp_prepare(x, w, g, nullptr, eps, weight_bias, gx, gw, rows, D, dtype, &dev, &p);
    if (st != RMSNORM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0) {
        cudaError_t e = cudaMemsetAsync(gw, 0, (size_t)D * sizeof(float), s);
        return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
    }
    const size_t need = partials_bytes(p, D);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u) != 0)
        return RMSNORM_ERR_INVALID_ARG;
    const size_t n = (size_t)rows * (size_t)D * 2;
    if (overlaps(workspace, need, x, n) || overlaps(workspace, need, g, n) ||
        overlaps(workspace, need, gx, n) || overlaps(workspace, need, w, (size_t)D * 2) ||
        overlaps(workspace, need, gw, (size_t)D * 4))
        return RMSNORM_ERR_INVALID_ARG;
    return vjp_run(x, w, g, nullptr, eps, weight_bias, gx, gw, rows, D, dtype, dev, p,
                   static_cast<float *>(workspace), s);
}

int rmsnorm_vjp(const void *x, const void *w, const void *g, float eps, float weight_bias,
                void *gx, float *gw, int64_t rows, int64_t D, int dtype, void *stream) {
    return vjp_pooled(x, w, g, nullptr, eps, weight_bias, gx, gw, rows, D, dtype, stream);
}

int rmsnorm_fused_vjp(const void *h, const void *w, const void *g_out, const void *g_residual,
                      float eps, float weight_bias, void *g_h, float *gw, int64_t rows, int64_t D,
                      int dtype, void *stream) {
    return vjp_pooled(h, w, g_out, g_residual, eps, weight_bias, g_h, gw, rows, D, dtype, stream);
}

const char *rmsnorm_status_string(int status) {
    switch (status) {
        case RMSNORM_OK: return "ok";
        case RMSNORM_ERR_INVALID_ARG: return "invalid argument";
        case RMSNORM_ERR_UNSUPPORTED: return "unsupported problem size";
        case RMSNORM_ERR_CUDA: return "CUDA error";
        case RMSNORM_ERR_NO_MEMORY: return "out of device memory";
        case RMSNORM_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

int rmsnorm_last_cuda_error(void) { return t_last_cuda_error; }

int rmsnorm_device_status(unsigned int *bits, int clear) {
    if (!bits) return RMSNORM_ERR_INVALID_ARG;
    DevInfo dev;
    int st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemcpy(bits, dev.status, sizeof(unsigned int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (clear) {
        e = cudaMemset(dev.status, 0, sizeof(unsigned int));
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return (*bits & RMSNORM_DEVSTATUS_WAIT_TIMEOUT) ? RMSNORM_ERR_TIMEOUT : RMSNORM_OK;
}

int rmsnorm_debug_inject(int64_t drop_tile, int64_t budget_cycles) {
    g_drop_tile.store(drop_tile < 0 ? -1 : drop_tile);
    g_wait_budget.store(budget_cycles > 0 ? (long long)budget_cycles : DEFAULT_WAIT_BUDGET);
    return RMSNORM_OK;
}

const char *rmsnorm_describe_dispatch(int op, int64_t rows, int64_t D, int dtype,
                                      int has_residual, int aligned) {
    thread_local char buf[160];
    if (check_common(rows, D, dtype, 0.f, 0.f) != RMSNORM_OK || rows == 0 || (op != 0 && op != 1))
        return "invalid";
    DevInfo dev;
    if (current_device(&dev) != RMSNORM_OK) return "no-device";
    const int mode = op == 1 ? (has_residual ? MODE_VJP_ADD : MODE_VJP)
                             : (has_residual ? MODE_FWD_RES : MODE_FWD_NORES);
    const Plan p = make_plan(mode, rows, (int)D, aligned && (D * 2) % 16 == 0, dev.sm_count);
    std::snprintf(buf, sizeof(buf), "%s:cfg%d:nt%d:g%d:v%d:s%d:tr%d:grid%d:smem%zu",
                  tier_name(p.tier), p.cfg, p.nt, p.g, p.v, p.stages, p.tile_rows, p.grid,
                  p.smem);
    return buf;
}

}  // extern "C"

// ---- helpers for the entry points of noalloc.cu and gated.cu -----------------
namespace rmsn {

// Bytes of gw scratch rmsnorm_vjp_ws needs for exactly these pointers on the
// current device (0 when rows == 0 or the arguments are invalid).
size_t vjp_partials_bytes_for(const void *x, const void *w, const void *g, const void *gx,
                              int64_t rows, int64_t D, int dtype) {
    if (check_common(rows, D, dtype, 0.f, 0.f) != RMSNORM_OK || rows == 0) return 0;
    DevInfo dev;
    if (current_device(&dev) != RMSNORM_OK) return 0;
    const bool aligned =
        (D * 2) % 16 == 0 && aligned16(x) && aligned16(g) && aligned16(gx) && aligned16(w);
    return partials_bytes(make_plan(MODE_VJP, rows, (int)D, aligned, dev.sm_count), D);
}

// Records a failed CUDA call for rmsnorm_last_cuda_error().
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

// SM count of the current device (cached with the device's other set-up).
int current_sm_count(int *sm) {
    DevInfo dev;
    const int st = current_device(&dev);
    if (st == RMSNORM_OK) *sm = dev.sm_count;
    return st;
}

}  // namespace rmsn
