// api.cu -- the C ABI declared in include/rmsnorm.h: argument validation, the
// dispatch table over (rows, D, dtype, alignment, SM count), gw scratch, and
// the device status word.
//
// The dispatch table itself is in planner.h.
#include "rmsnorm.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "common.cuh"
#include "plan.h"
#include "planner.h"

using namespace rmsn;
using rmsn::planner::make_plan;

namespace {

constexpr int MAX_DEVICES = 64;

__device__ unsigned int g_devstatus;  // RMSNORM_DEVSTATUS_* bits, per device

// Claim counters of the staged forwards that take their tiles at run time:
// sets of CLAIM_WORDS words (group counters and a finished-CTA count), zero
// from module load on and put back to zero by each launch's last CTA.
// Launches outside a graph capture take the sets in turn (CTR_DIRECT of
// them, so two launches share one only with CTR_DIRECT launches between
// them, both still running); each launch recorded into a graph keeps one of
// its own (CTR_CAPTURE per device, then the static round robin).
constexpr uint32_t CTR_DIRECT = 16384;
constexpr size_t CLAIM_MIN_ROW_TRAFFIC = 96 * 1024;
constexpr uint32_t CTR_CAPTURE = 2048;
__device__ unsigned long long g_tile_ctrs[(size_t)CLAIM_WORDS * (CTR_DIRECT + CTR_CAPTURE)];

thread_local int t_last_cuda_error = 0;

struct DevInfo {
    bool ready = false;
    int sm_count = 0;
    unsigned int *status = nullptr;  // device address of g_devstatus
    cudaMemPool_t pool = nullptr;    // gw scratch of rmsnorm_vjp; keeps its memory
    int cluster_cap[9] = {};         // clusters of 2, 4, 8 CTAs the device holds at once
    int index = 0;                   // device ordinal
    unsigned long long *tile_ctrs = nullptr;  // device address of g_tile_ctrs
};
std::mutex g_dev_mu;
DevInfo g_dev[MAX_DEVICES];

std::atomic<int64_t> g_drop_tile{-1};
std::atomic<long long> g_wait_budget{DEFAULT_WAIT_BUDGET};
std::atomic<int> g_fail_allocs{0};  // scratch allocations still to report as failed
std::atomic<uint64_t> g_ctr_next[MAX_DEVICES];  // next direct-launch counter pair
std::atomic<uint32_t> g_ctr_captured[MAX_DEVICES];  // counter pairs kept by captured launches
std::atomic<uint32_t> g_ctr_cycle{CTR_DIRECT};        // direct-launch pairs in use (test hook)

// Takes one injected allocation failure if any is pending.
bool take_injected_alloc_failure() {
    int n = g_fail_allocs.load();
    while (n > 0 && !g_fail_allocs.compare_exchange_weak(n, n - 1)) {
    }
    return n > 0;
}

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
        e = cudaGetSymbolAddress(&p, g_tile_ctrs);
        if (e != cudaSuccess) return cuda_fail(e);
        d.tile_ctrs = static_cast<unsigned long long *>(p);
        d.index = dev;
        for (int cl : {2, 4, 8}) d.cluster_cap[cl] = cluster_capacity(cl);
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

int esize_of(int dtype) { return dtype == RMSNORM_F32 ? 4 : 2; }

// Scalar and shape checks common to every norm entry point.
int check_common(int64_t rows, int64_t D, int dtype, float eps, float weight_bias) {
    if (dtype != RMSNORM_F16 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F32)
        return RMSNORM_ERR_INVALID_ARG;
    if (rows < 0 || D <= 0) return RMSNORM_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return RMSNORM_ERR_INVALID_ARG;
    if (!std::isfinite(weight_bias)) return RMSNORM_ERR_INVALID_ARG;
    if (D > RMSNORM_MAX_D) return RMSNORM_ERR_UNSUPPORTED;
    if (rows > INT64_MAX / (4 * D)) return RMSNORM_ERR_UNSUPPORTED;
    return RMSNORM_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// A [rows, D] tensor of `es`-byte elements whose rows start `ld` elements
// apart (ld >= D).  A single row has no stride; it is normalised to D so
// that the same row under two strides compares equal.
struct Mat {
    const void *p;
    int64_t ld;
};

Mat mat(const void *p, int64_t ld, int64_t rows, int64_t D) { return Mat{p, rows <= 1 ? D : ld}; }

// Checks a stride and that the tensor's extent fits in the address space.
int check_ld(int64_t ld, int64_t rows, int64_t D, int es) {
    if (ld < D) return RMSNORM_ERR_INVALID_ARG;
    if (rows > 1 && (rows - 1) > (INT64_MAX / es - D) / ld) return RMSNORM_ERR_UNSUPPORTED;
    return RMSNORM_OK;
}

size_t extent(const Mat &m, int64_t rows, int64_t D, int es) {
    return (!m.p || rows == 0) ? 0 : (size_t)((rows - 1) * m.ld + D) * (size_t)es;
}

int64_t floor_div(int64_t a, int64_t b) {
    const int64_t q = a / b;
    return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

// Whether two [rows, D] tensors share a byte.  With equal strides the test is
// exact (rows i of a and j of b meet iff |(b - a) - (i - j) * ld| < the row's
// bytes for some i - j in [-(rows - 1), rows - 1]), so interleaved tensors
// such as the two halves of a [rows, 2D] buffer count as disjoint; with
// different strides the whole extents are compared.
bool mats_overlap(const Mat &a, const Mat &b, int64_t rows, int64_t D, int es) {
    const size_t na = extent(a, rows, D, es), nb = extent(b, rows, D, es);
    if (!overlaps(a.p, na, b.p, nb)) return false;
    if (a.ld != b.ld) return true;
    const int64_t L = a.ld * es, R = D * es;
    const int64_t d = (int64_t)((uintptr_t)b.p - (uintptr_t)a.p);
    const int64_t k0 = floor_div(d, L);
    for (int64_t k : {k0, k0 + 1}) {
        k = std::min<int64_t>(std::max<int64_t>(k, -(rows - 1)), rows - 1);
        const int64_t off = d - k * L;
        if (off > -R && off < R) return true;
    }
    return false;
}

// An output may be exactly an input (same pointer and stride: every element
// is read before the thread that owns it writes it), or share no byte with it.
bool bad_alias(const Mat &out, const Mat &in, int64_t rows, int64_t D, int es) {
    if (!mats_overlap(out, in, rows, D, es)) return false;
    return !(out.p == in.p && out.ld == in.ld);
}

// Whether a [rows, D] tensor overlaps a plain buffer of n bytes.
bool mat_hits(const Mat &m, int64_t rows, int64_t D, int es, const void *p, size_t n) {
    return overlaps(m.p, extent(m, rows, D, es), p, n);
}

// The vectorised tiers need 16-byte aligned rows: base and stride.
bool rows_aligned(const Mat &m, int es) {
    return !m.p || (aligned16(m.p) && (m.ld * es) % 16 == 0);
}

// Every element of every operand must sit at a multiple of its size.
bool elem_aligned(const void *p, int es) { return ((uintptr_t)p % (uintptr_t)es) == 0; }

// How the row tensors of one call (null entries ignored) and w sit relative
// to 16-byte boundaries (planner Align): every row aligned -> ALIGN_VEC
// (dense rows, no rstd) or ALIGN_VEC_GEN (rows a stride apart, or rstd);
// dense rows (stride D) whose tensors all start at the same offset from a
// boundary, with no rstd -> ALIGN_SHIFT; anything else -> ALIGN_NONE.
int align_of(std::initializer_list<const Mat *> ms, const void *w, const void *rstd, int64_t D,
             int es) {
    bool vec = (D * es) % 16 == 0 && aligned16(w);
    bool dense = rstd == nullptr;
    for (const Mat *m : ms) {
        vec = vec && rows_aligned(*m, es);
        dense = dense && (!m->p || m->ld == D);
    }
    if (vec) return dense ? ALIGN_VEC : ALIGN_VEC_GEN;
    if (rstd) return ALIGN_NONE;
    int off = -1;
    for (const Mat *m : ms) {
        if (!m->p) continue;
        if (m->ld != D) return ALIGN_NONE;
        const int o = (int)((uintptr_t)m->p & 15u);
        if (off >= 0 && o != off) return ALIGN_NONE;
        off = o;
    }
    return ALIGN_SHIFT;
}

// Whether a forward plan takes its tiles from counters: the CTA-per-row
// staged forwards of CLAIM_MIN_NT threads or more on dense aligned rows whose
// rows take long enough.  A claim is an L2 atomic whose round trip, with HBM saturated,
// outlasts a short row: claims lost time wherever a CTA's row moved less than
// ~96 KB per SM (GB300, bf16 with residual, rows 16384: D = 4096 (two CTAs an
// SM) -3 %, 8192 +-0; 8192 x 4096 fp16 without residual -20 %) and won it
// above (D = 16384 with residual, 128 KB: 6310 -> 6677 GB/s).
bool claims_tiles(const Plan &p, int mode, int64_t D, int es, int align, int sm_count) {
    if (p.tier != TIER_STAGED || p.shift || p.g != p.nt || is_vjp(mode) || align != ALIGN_VEC ||
        p.nt < CLAIM_MIN_NT)
        return false;
    const size_t row_traffic = (size_t)D * es * (mode == MODE_FWD_RES ? 4 : 2);
    const size_t per_sm = row_traffic * (size_t)std::max(1, p.grid / std::max(1, sm_count));
    return per_sm >= CLAIM_MIN_ROW_TRAFFIC;
}

// The counter set a staged forward on stream s claims its tiles from, or
// null for the static round robin (tuned off, capture state unknown, or
// every capture set taken).
unsigned long long *tile_counter(const DevInfo &d, cudaStream_t s) {
    if (!d.tile_ctrs || !planner::tuning().claim) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) {
        const uint32_t i = g_ctr_captured[d.index].fetch_add(1);
        return i < CTR_CAPTURE ? d.tile_ctrs + (size_t)CLAIM_WORDS * ((size_t)CTR_DIRECT + i)
                               : nullptr;
    }
    return d.tile_ctrs +
           (size_t)CLAIM_WORDS * (size_t)(g_ctr_next[d.index].fetch_add(1) % g_ctr_cycle.load());
}

// gw partial rows of a VJP plan: one per CTA, or one per cluster.
int partial_rows(const Plan &p) {
    return p.tier == TIER_CLUSTER                ? p.grid / p.cl
           : (p.tier == TIER_DIRECT && p.cl > 1) ? 1  // the cluster sums its rows itself
                                                   : p.grid;
}

size_t partials_bytes(const Plan &p, int64_t D) {
    const size_t b = (size_t)partial_rows(p) * (size_t)D * sizeof(float);
    return (b + 255) & ~(size_t)255;
}

cudaError_t launch_plan(int dtype, int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (p.tier) {
        case TIER_STAGED: return launch_staged(dtype, mode, p, a, s);
        case TIER_DIRECT: return launch_direct(dtype, mode, p, a, s);
        case TIER_CLUSTER: return launch_cluster(dtype, mode, p, a, s);
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
    a.cl_cols = p.cl_cols;
    a.drop_tile = g_drop_tile.load(std::memory_order_relaxed);
    return a;
}

// The operands of one VJP call: x (the normalised tensor), g (the gradient of
// out), g_res (the gradient reaching new_residual of the fused op; null for
// the plain VJP), gx, each with its row stride; w, gw; and the forward's
// per-row rstd (null: recomputed from x).
struct VjpOperands {
    Mat x, g, g_res, gx;
    const void *w;
    float *gw;
    const float *rstd;
};

VjpOperands dense_vjp(const void *x, const void *w, const void *g, const void *g_res, void *gx,
                      float *gw, int64_t D) {
    return VjpOperands{Mat{x, D}, Mat{g, D}, Mat{g_res, D}, Mat{gx, D}, w, gw, nullptr};
}

// Validation shared by the VJP entry points; *plan is filled on success when
// rows > 0.
int vjp_prepare(const VjpOperands &o, float eps, float weight_bias, int64_t rows, int64_t D,
                int dtype, DevInfo *dev, Plan *plan) {
    int st = check_common(rows, D, dtype, eps, weight_bias);
    if (st != RMSNORM_OK) return st;
    if (!o.w || !o.gw) return RMSNORM_ERR_INVALID_ARG;
    const int es = esize_of(dtype);
    if (!elem_aligned(o.w, es) || !elem_aligned(o.gw, 4) || !elem_aligned(o.rstd, 4))
        return RMSNORM_ERR_INVALID_ARG;
    for (const Mat *m : {&o.x, &o.g, &o.g_res, &o.gx})
        if (!elem_aligned(m->p, es)) return RMSNORM_ERR_INVALID_ARG;
    const size_t nw = (size_t)D * es, ngw = (size_t)D * 4, nr = (size_t)rows * 4;
    if (rows > 0) {
        if (!o.x.p || !o.g.p || !o.gx.p) return RMSNORM_ERR_INVALID_ARG;
        for (const Mat *m : {&o.x, &o.g, &o.g_res, &o.gx}) {
            if (!m->p) continue;
            st = check_ld(m->ld, rows, D, es);
            if (st != RMSNORM_OK) return st;
        }
        const Mat x = mat(o.x.p, o.x.ld, rows, D), g = mat(o.g.p, o.g.ld, rows, D);
        const Mat gr = mat(o.g_res.p, o.g_res.ld, rows, D), gx = mat(o.gx.p, o.gx.ld, rows, D);
        if (bad_alias(gx, x, rows, D, es) || bad_alias(gx, g, rows, D, es) ||
            bad_alias(gx, gr, rows, D, es))
            return RMSNORM_ERR_INVALID_ARG;
        if (mat_hits(gx, rows, D, es, o.gw, ngw) || mat_hits(gx, rows, D, es, o.w, nw) ||
            mat_hits(gx, rows, D, es, o.rstd, nr))
            return RMSNORM_ERR_INVALID_ARG;
        for (const Mat *m : {&x, &g, &gr})
            if (mat_hits(*m, rows, D, es, o.gw, ngw)) return RMSNORM_ERR_INVALID_ARG;
        if (overlaps(o.gw, ngw, o.rstd, nr)) return RMSNORM_ERR_INVALID_ARG;
    }
    if (overlaps(o.gw, ngw, o.w, nw)) return RMSNORM_ERR_INVALID_ARG;
    st = current_device(dev);
    if (st != RMSNORM_OK) return st;
    if (rows > 0) {
        const Mat x = mat(o.x.p, o.x.ld, rows, D), g = mat(o.g.p, o.g.ld, rows, D);
        const Mat gr = mat(o.g_res.p, o.g_res.ld, rows, D), gx = mat(o.gx.p, o.gx.ld, rows, D);
        const int align = align_of({&x, &g, &gr, &gx}, o.w, o.rstd, D, es);
        *plan = make_plan(o.g_res.p ? MODE_VJP_ADD : MODE_VJP, rows, (int)D, es, align,
                          dev->sm_count, dev->cluster_cap);
    }
    return RMSNORM_OK;
}

// A VJP launched as a single CTA (decode: one row) has one partial row, which
// is gw itself: the kernel writes it in place, with no scratch and no second
// kernel (the fixed-order sum of one row is that row, so the bits are the
// same).  The tiers store partial rows as 16-byte vectors, so gw must be
// 16-byte aligned for this; otherwise the two-stage path runs.
bool gw_in_place(const Plan &p, const float *gw) { return partial_rows(p) == 1 && aligned16(gw); }

int vjp_run(const VjpOperands &o, float eps, float weight_bias, int64_t rows, int64_t D,
            int dtype, const DevInfo &dev, const Plan &p, float *partials, cudaStream_t s) {
    const bool in_place = gw_in_place(p, o.gw);
    KernelArgs a = base_args(dev, p, eps, weight_bias, rows, D);
    a.in0 = o.x.p;
    a.ld_in0 = o.x.ld;
    a.in1 = o.g.p;
    a.ld_in1 = o.g.ld;
    a.in2 = o.g_res.p;
    a.ld_in2 = o.g_res.p ? o.g_res.ld : 0;
    a.w = o.w;
    a.out0 = const_cast<void *>(o.gx.p);
    a.ld_out0 = o.gx.ld;
    a.out1 = nullptr;
    a.partials = in_place ? o.gw : partials;
    a.rstd = const_cast<float *>(o.rstd);  // read only in the VJP kernels
    cudaError_t e = launch_plan(dtype, o.g_res.p ? MODE_VJP_ADD : MODE_VJP, p, a, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if (in_place) return RMSNORM_OK;
    e = launch_gw_reduce(partials, o.gw, partial_rows(p), (int)D, s);
    if (e != cudaSuccess) return cuda_fail(e);
    return RMSNORM_OK;
}

// The VJP with scratch from the library's stream-ordered pool.
int vjp_pooled(const VjpOperands &o, float eps, float weight_bias, int64_t rows, int64_t D,
               int dtype, void *stream) {
    DevInfo dev;
    Plan p{};
    int st = vjp_prepare(o, eps, weight_bias, rows, D, dtype, &dev, &p);
    if (st != RMSNORM_OK) return st;
    float *gw = o.gw;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0) {
        cudaError_t e = cudaMemsetAsync(gw, 0, (size_t)D * sizeof(float), s);
        return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
    }
    if (gw_in_place(p, gw))
        return vjp_run(o, eps, weight_bias, rows, D, dtype, dev, p, nullptr, s);
    if (take_injected_alloc_failure()) return RMSNORM_ERR_NO_MEMORY;  // test hook
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
    st = vjp_run(o, eps, weight_bias, rows, D, dtype, dev, p, static_cast<float *>(ws), s);
    e = cudaFreeAsync(ws, s);
    if (st == RMSNORM_OK && e != cudaSuccess) st = cuda_fail(e);
    return st;
}

const char *tier_name(int t) {
    return t == TIER_STAGED ? "staged" : t == TIER_DIRECT ? "direct" : t == TIER_CLUSTER ? "cluster"
                                                                                    : "generic";
}

}  // namespace

extern "C" {

int rmsnorm_fwd_ex(const void *x, int64_t ld_x, const void *residual, int64_t ld_residual,
                   const void *w, float eps, float weight_bias, void *out, int64_t ld_out,
                   void *new_residual, int64_t ld_new_residual, float *rstd, int64_t rows,
                   int64_t D, int dtype, void *stream) {
    int st = check_common(rows, D, dtype, eps, weight_bias);
    if (st != RMSNORM_OK) return st;
    if (!w) return RMSNORM_ERR_INVALID_ARG;
    if (rows == 0) return RMSNORM_OK;
    if (!x || !out) return RMSNORM_ERR_INVALID_ARG;
    if ((residual == nullptr) != (new_residual == nullptr)) return RMSNORM_ERR_INVALID_ARG;
    const int es = esize_of(dtype);
    st = check_ld(ld_x, rows, D, es);
    if (st == RMSNORM_OK) st = check_ld(ld_out, rows, D, es);
    if (st == RMSNORM_OK && residual) st = check_ld(ld_residual, rows, D, es);
    if (st == RMSNORM_OK && residual) st = check_ld(ld_new_residual, rows, D, es);
    if (st != RMSNORM_OK) return st;
    const Mat mx = mat(x, ld_x, rows, D), mo = mat(out, ld_out, rows, D);
    const Mat mr = mat(residual, ld_residual, rows, D);
    const Mat mn = mat(new_residual, ld_new_residual, rows, D);
    for (const void *q : {x, residual, w, (const void *)out, (const void *)new_residual})
        if (!elem_aligned(q, es)) return RMSNORM_ERR_INVALID_ARG;
    if (!elem_aligned(rstd, 4)) return RMSNORM_ERR_INVALID_ARG;
    const size_t nw = (size_t)D * es, nr = (size_t)rows * 4;
    if (mats_overlap(mo, mn, rows, D, es)) return RMSNORM_ERR_INVALID_ARG;
    for (const Mat *o : {&mo, &mn}) {
        if (bad_alias(*o, mx, rows, D, es) || bad_alias(*o, mr, rows, D, es) ||
            mat_hits(*o, rows, D, es, w, nw) || mat_hits(*o, rows, D, es, rstd, nr))
            return RMSNORM_ERR_INVALID_ARG;
    }
    if (mat_hits(mx, rows, D, es, rstd, nr) || mat_hits(mr, rows, D, es, rstd, nr) ||
        overlaps(rstd, nr, w, nw))
        return RMSNORM_ERR_INVALID_ARG;

    DevInfo dev;
    st = current_device(&dev);
    if (st != RMSNORM_OK) return st;
    const int mode = residual ? MODE_FWD_RES : MODE_FWD_NORES;
    const int align = align_of({&mx, &mr, &mo, &mn}, w, rstd, D, es);
    const Plan p = make_plan(mode, rows, (int)D, es, align, dev.sm_count, dev.cluster_cap);
    KernelArgs a = base_args(dev, p, eps, weight_bias, rows, D);
    a.in0 = x;
    a.ld_in0 = mx.ld;
    a.in1 = residual;
    a.ld_in1 = residual ? mr.ld : 0;
    a.w = w;
    a.out0 = out;
    a.ld_out0 = mo.ld;
    a.out1 = new_residual;
    a.ld_out1 = new_residual ? mn.ld : 0;
    a.partials = nullptr;
    a.rstd = rstd;
    if (claims_tiles(p, mode, D, es, align, dev.sm_count)) {
        a.tile_ctr = tile_counter(dev, static_cast<cudaStream_t>(stream));
        // as many groups as divide the grid, up to the tuned or default number
        int k = planner::tuning().claim_k;
        while (p.grid % k) k /= 2;
        a.claim_k = k;
    }
    cudaError_t e = launch_plan(dtype, mode, p, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return RMSNORM_OK;
}

int rmsnorm_fwd(const void *x, const void *residual, const void *w, float eps, float weight_bias,
                void *out, void *new_residual, int64_t rows, int64_t D, int dtype, void *stream) {
    return rmsnorm_fwd_ex(x, D, residual, D, w, eps, weight_bias, out, D, new_residual, D, nullptr,
                          rows, D, dtype, stream);
}

size_t rmsnorm_vjp_workspace_size(int64_t rows, int64_t D, int dtype) {
    if (check_common(rows, D, dtype, 0.f, 0.f) != RMSNORM_OK || rows == 0) return 0;
    DevInfo dev;
    if (current_device(&dev) != RMSNORM_OK) return 0;
    // The plan depends on pointer alignment; cover every outcome.
    const int es = esize_of(dtype);
    size_t most = 0;
    for (int align : {ALIGN_VEC, ALIGN_SHIFT, ALIGN_NONE})
        most = std::max(most, partials_bytes(make_plan(MODE_VJP, rows, (int)D, es, align,
                                                       dev.sm_count, dev.cluster_cap), D));
    return most;
}

int rmsnorm_vjp_ws(const void *x, const void *w, const void *g, float eps, float weight_bias,
                   void *gx, float *gw, int64_t rows, int64_t D, int dtype, void *workspace,
                   size_t workspace_bytes, void *stream) {
    DevInfo dev;
    Plan p{};
    const VjpOperands o = dense_vjp(x, w, g, nullptr, gx, gw, D);
    int st = vjp_prepare(o, eps, weight_bias, rows, D, dtype, &dev, &p);
    if (st != RMSNORM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0) {
        cudaError_t e = cudaMemsetAsync(gw, 0, (size_t)D * sizeof(float), s);
        return e == cudaSuccess ? RMSNORM_OK : cuda_fail(e);
    }
    const size_t need = partials_bytes(p, D);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u) != 0)
        return RMSNORM_ERR_INVALID_ARG;
    const int es = esize_of(dtype);
    const size_t n = (size_t)rows * (size_t)D * es;
    if (overlaps(workspace, need, x, n) || overlaps(workspace, need, g, n) ||
        overlaps(workspace, need, gx, n) || overlaps(workspace, need, w, (size_t)D * es) ||
        overlaps(workspace, need, gw, (size_t)D * 4))
        return RMSNORM_ERR_INVALID_ARG;
    return vjp_run(o, eps, weight_bias, rows, D, dtype, dev, p, static_cast<float *>(workspace), s);
}

int rmsnorm_vjp(const void *x, const void *w, const void *g, float eps, float weight_bias,
                void *gx, float *gw, int64_t rows, int64_t D, int dtype, void *stream) {
    return vjp_pooled(dense_vjp(x, w, g, nullptr, gx, gw, D), eps, weight_bias, rows, D, dtype,
                      stream);
}

int rmsnorm_fused_vjp(const void *h, const void *w, const void *g_out, const void *g_residual,
                      float eps, float weight_bias, void *g_h, float *gw, int64_t rows, int64_t D,
                      int dtype, void *stream) {
    return vjp_pooled(dense_vjp(h, w, g_out, g_residual, g_h, gw, D), eps, weight_bias, rows, D,
                      dtype, stream);
}

int rmsnorm_vjp_ex(const void *x, int64_t ld_x, const void *w, const void *g, int64_t ld_g,
                   const void *g_residual, int64_t ld_g_residual, const float *rstd, float eps,
                   float weight_bias, void *gx, int64_t ld_gx, float *gw, int64_t rows, int64_t D,
                   int dtype, void *stream) {
    const VjpOperands o{Mat{x, ld_x}, Mat{g, ld_g}, Mat{g_residual, ld_g_residual}, Mat{gx, ld_gx},
                        w, gw, rstd};
    return vjp_pooled(o, eps, weight_bias, rows, D, dtype, stream);
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
    if (*bits & RMSNORM_DEVSTATUS_WAIT_TIMEOUT) return RMSNORM_ERR_TIMEOUT;
    if (*bits & RMSNORM_DEVSTATUS_BAD_INDEX) return RMSNORM_ERR_INVALID_ARG;
    return RMSNORM_OK;
}

int rmsnorm_debug_inject(int64_t drop_tile, int64_t budget_cycles) {
    g_drop_tile.store(drop_tile < 0 ? -1 : drop_tile);
    g_wait_budget.store(budget_cycles > 0 ? (long long)budget_cycles : DEFAULT_WAIT_BUDGET);
    return RMSNORM_OK;
}

int rmsnorm_debug_fail_allocs(int count) {
    if (count < 0) return RMSNORM_ERR_INVALID_ARG;
    g_fail_allocs.store(count);
    return RMSNORM_OK;
}

int rmsnorm_debug_claim_counters(int count) {
    if (count < 0 || count > (int)CTR_DIRECT) return RMSNORM_ERR_INVALID_ARG;
    g_ctr_cycle.store(count == 0 ? CTR_DIRECT : (uint32_t)count);
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
    const int es = esize_of(dtype);
    const int align = aligned == 2               ? ALIGN_SHIFT
                      : !aligned                  ? ALIGN_NONE
                      : (D * es) % 16 == 0        ? ALIGN_VEC
                                                  : ALIGN_SHIFT;
    const Plan p = make_plan(mode, rows, (int)D, es, align, dev.sm_count, dev.cluster_cap);
    std::snprintf(buf, sizeof(buf), "%s%s:cfg%d:nt%d:g%d:v%d:s%d:tr%d:grid%d:smem%zu:cl%d%s",
                  tier_name(p.tier), p.shift ? "-shift" : "", p.cfg, p.nt, p.g, p.v, p.stages,
                  p.tile_rows, p.grid, p.smem, p.cl,
                  claims_tiles(p, mode, D, es, align, dev.sm_count) && planner::tuning().claim
                      ? ":claim"
                      : "");
    return buf;
}

}  // extern "C"

// ---- helpers for the entry points of noalloc.cu, gated.cu and rope.cu --------
namespace rmsn {

// Bytes of gw scratch rmsnorm_vjp_ws needs for exactly these pointers on the
// current device (0 when rows == 0 or the arguments are invalid).
size_t vjp_partials_bytes_for(const void *x, const void *w, const void *g, const void *gx,
                              int64_t rows, int64_t D, int dtype) {
    if (check_common(rows, D, dtype, 0.f, 0.f) != RMSNORM_OK || rows == 0) return 0;
    DevInfo dev;
    if (current_device(&dev) != RMSNORM_OK) return 0;
    const int es = esize_of(dtype);
    const Mat mx{x, D}, mg{g, D}, mgx{gx, D};
    const int align = align_of({&mx, &mg, &mgx}, w, nullptr, D, es);
    return partials_bytes(make_plan(MODE_VJP, rows, (int)D, es, align, dev.sm_count, dev.cluster_cap), D);
}

// Records a failed CUDA call for rmsnorm_last_cuda_error().
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

// Device address of the current device's status word.
int current_status_word(unsigned int **status) {
    DevInfo dev;
    const int st = current_device(&dev);
    if (st == RMSNORM_OK) *status = dev.status;
    return st;
}

// SM count of the current device (cached with the device's other set-up).
int current_sm_count(int *sm) {
    DevInfo dev;
    const int st = current_device(&dev);
    if (st == RMSNORM_OK) *sm = dev.sm_count;
    return st;
}

}  // namespace rmsn
