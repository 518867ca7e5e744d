// planner.h -- the dispatch table: which kernel, launch shape and ring depth
// a problem gets.  A pure function of (mode, rows, D, element size,
// alignment, SM count) plus the RMSNORM_TUNE override, so the VJP's summation
// order, and with it gw's bits, is fixed for a given device.  The tiers work
// in 16-byte vectors, so the thresholds below are in vectors (nv = D * esize
// / 16) and bytes; the D figures quoted are for 2-byte elements (fp32 rows
// reach each threshold at half the D).
//   * rows off 16-byte boundaries: dense rows whose tensors share one offset
//     take the staged tier's shifted-rows instances (more than DECODE_ROWS
//     rows), anything else -> generic tier;
//   * rows <= DECODE_ROWS (decode: one token per sequence)  -> direct tier;
//   * D <= 16384 -> staged tier (TMA bulk ring): sub-warp/warp per row for
//     D <= 1024, CTA per row above;
//   * longer aligned rows -> the cluster tier (2-8 CTAs per row, one per SM,
//     each streaming a slice of up to 2048 vectors through a ring of three to
//     eight stages), then generic;
//   * rows <= DECODE_ROWS of up to 4096 (forward) / 2048 (VJP) vectors ->
//     direct tier.
#pragma once

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "plan.h"

namespace rmsn {
namespace planner {

constexpr int64_t DECODE_ROWS = 8;
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
// read per byte written) ~96 KB.  Sub-warp tiles (sweeps at D = 128-1024,
// 32768-262144 rows) want less: ~48 KB for the forward (D = 640: 6313 GB/s
// against 5945 with 80 KB) and ~64 KB for the VJP with two or more vectors
// per lane (D = 1024: 5431 against 5121 with 128 KB); the one-vector VJP
// keeps ~96 KB (D = 256: 5417 against 4614 with 64 KB).
constexpr size_t INFLIGHT_FWD = 64 * 1024;
constexpr size_t INFLIGHT_VJP = 96 * 1024;
constexpr size_t INFLIGHT_FWD_SUBWARP = 48 * 1024;
constexpr size_t INFLIGHT_VJP_SUBWARP = 64 * 1024;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shared memory one CTA may take when `cps` CTAs share an SM.
inline size_t smem_per_cta(int cps) {
    return cps <= 1 ? SMEM_ONE_PER_SM
           : cps == 2 ? SMEM_TWO_PER_SM
           : cps == 3 ? SMEM_THREE_PER_SM
                      : (size_t)(224 * 1024) / (size_t)cps - 2048;
}


// Overrides of the staged tier's choices, read once from RMSNORM_TUNE
// ("cfg=N,cps=N,stages=N,tmap=0,claim=0,claimk=N,cl=N", any subset) for tuning sweeps and for
// testing the per-row copy path that strided sub-warp tiles take where no
// tensor map can be made.  Unset, the plan is a pure function of the problem
// and the device.
struct Tuning {
    int cfg = -1;     // staged configuration index
    int cps = 0;      // CTAs per SM (capped by what the registers allow)
    int stages = 0;   // maximum ring depth
    bool tmap = true; // tensor maps for strided sub-warp tiles
    bool claim = true; // staged forwards: tiles claimed at run time
    int claim_k = 1;  // claim groups (a power of two up to CLAIM_MAX_K)
    int cl = 0;       // cluster tier: CTAs per cluster (2, 4 or 8)
};

inline Tuning parse_tuning() {
    Tuning t;
    const char *env = std::getenv("RMSNORM_TUNE");
    if (!env) return t;
    char buf[128];
    std::snprintf(buf, sizeof(buf), "%s", env);
    for (char *tok = std::strtok(buf, ","); tok; tok = std::strtok(nullptr, ",")) {
        int v = 0;
        if (std::sscanf(tok, "cfg=%d", &v) == 1 && v >= 0 && v < N_STAGED_CFG) t.cfg = v;
        else if (std::sscanf(tok, "cps=%d", &v) == 1 && v >= 1 && v <= 6) t.cps = v;
        else if (std::sscanf(tok, "stages=%d", &v) == 1 && v >= 2 && v <= MAX_STAGES) t.stages = v;
        else if (std::sscanf(tok, "tmap=%d", &v) == 1) t.tmap = v != 0;
        else if (std::sscanf(tok, "claim=%d", &v) == 1) t.claim = v != 0;
        else if (std::sscanf(tok, "cl=%d", &v) == 1 && (v == 2 || v == 4 || v == 8)) t.cl = v;
        else if (std::sscanf(tok, "claimk=%d", &v) == 1 && v >= 1 && v <= CLAIM_MAX_K &&
                 (v & (v - 1)) == 0)
            t.claim_k = v;
    }
    return t;
}

inline const Tuning &tuning() {
    static const Tuning t = parse_tuning();
    return t;
}

// Ring depth for a stage of `per_stage` bytes with `cps` CTAs per SM: one
// stage being consumed plus enough in flight to reach `target` bytes per SM
// (at least one).  An explicit RMSNORM_TUNE stages= wins.
inline int ring_stages(size_t target, size_t per_stage, int cps) {
    if (tuning().stages) return tuning().stages;
    const size_t per_sm_stage = per_stage * (size_t)cps;
    const int ahead = (int)std::max<size_t>(1, (target + per_sm_stage / 2) / per_sm_stage);
    return std::min(MAX_STAGES, 1 + ahead);
}

// Whole 16-byte vectors a row holds at most (shifted rows: a row off a
// boundary holds one fewer or as many, its edge elements handled apart).
inline int64_t row_vectors(int64_t D, int esize) { return D * esize / 16; }

// Bytes of one tensor's stage for `tr` rows (shifted rows: their aligned
// superset at the worst offset).
inline size_t stage_bytes_for(int64_t tr, int64_t D, int esize, bool shift) {
    return shift ? (size_t)(((int64_t)(16 - esize) + tr * D * esize + 15) / 16 * 16)
                 : (size_t)(tr * D * esize);
}

// Rows after which a row's offset from a 16-byte boundary repeats.
inline int shift_period(int64_t D, int esize) {
    const int64_t rb = (D * esize) % 16;
    return rb == 0 ? 1 : rb % 8 == 0 ? 2 : rb % 4 == 0 ? 4 : 8;
}

inline bool plan_staged(int mode, int64_t rows, int D, int esize, int sm_count, int ci, bool shift,
                        Plan *p) {
    const StagedCfg &c = STAGED_CFGS[ci];
    const Tuning &tu = tuning();
    const int ntens = input_tensors(mode);
    const size_t row_bytes = (size_t)D * esize;
    p->shift = shift;
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
        p->tile_rows = (int)(ng * rpg);  // a multiple of 8 rows (shifted rows rely on it)
        p->stage_bytes = (uint32_t)stage_bytes_for(p->tile_rows, D, esize, shift);
        const size_t per_stage = (size_t)ntens * p->stage_bytes;
        cps = std::min(cps, 2);
        const size_t cap = cps == 2 ? SMEM_TWO_PER_SM : SMEM_ONE_PER_SM;
        p->stages = (int)std::min<size_t>(std::min<size_t>(max_stages, cap / per_stage),
                                          ring_stages(!is_vjp(mode) ? INFLIGHT_FWD_SUBWARP
                                                      : c.v >= 2 ? INFLIGHT_VJP_SUBWARP
                                                                 : INFLIGHT_VJP,
                                                      per_stage, cps));
        if (p->stages < 2) return false;
        p->smem = STAGED_HEADER_BYTES + (size_t)p->stages * per_stage;
        if (is_vjp(mode))  // the cross-group gw sum reuses the ring
            p->smem = std::max(p->smem, (size_t)STAGED_HEADER_BYTES + (size_t)ng * D * 4);
    } else {
        // One row per tile, the whole CTA on it.  The requested CTAs per SM
        // when each CTA's share of shared memory holds its stages (two with
        // three or more CTAs, three with two), fewer otherwise, down to one
        // CTA with at least two; the depth then follows the in-flight target,
        // but is at least three stages, where they fit, with one CTA per SM
        // and for the VJP.  A stage is refilled only after the next row's
        // barrier, so two stages leave nothing in flight while a row is read
        // and reduced (bf16, rotating: forward D = 12288 5781 -> 6251 GB/s,
        // 16384 5907 -> 6168; fused VJP D = 12288 5700 -> 6264, and with two
        // CTAs per SM D = 6144 6045 -> 6231).  The forwards with two or more
        // CTAs per SM keep two (D = 7168: 6230 against 6081 with three).
        p->tile_rows = 1;
        p->stage_bytes = (uint32_t)stage_bytes_for(1, D, esize, shift);
        const size_t per_stage = (size_t)ntens * p->stage_bytes;
        int chosen = 0;
        for (int c = cps; c >= 1 && !chosen; --c) {
            const int64_t sc = (int64_t)(smem_per_cta(c) / per_stage);
            if (sc >= (c >= 3 ? 2 : c == 2 ? 3 : 2)) {
                chosen = c;
                const int floor = tu.stages ? 0 : (c == 1 || is_vjp(mode)) ? 3 : 2;
                p->stages = (int)std::min<int64_t>(
                    std::min<int64_t>(max_stages, sc),
                    std::max(floor, ring_stages(is_vjp(mode) ? INFLIGHT_VJP : INFLIGHT_FWD,
                                                per_stage, c)));
            }
        }
        if (!chosen) return false;
        cps = chosen;
        p->smem = STAGED_HEADER_BYTES + (size_t)p->stages * per_stage;
    }
    p->num_tiles = ceil_div(rows, p->tile_rows);
    p->grid = (int)std::min<int64_t>(p->num_tiles, (int64_t)sm_count * cps);
    // Shifted rows, one per tile: a CTA that takes several rows sees the
    // same offset on all of them when the grid is a multiple of its period.
    const int period = shift && c.g == c.nt ? shift_period(D, esize) : 1;
    if (p->grid < p->num_tiles && p->grid % period != 0)
        p->grid = std::max(period, p->grid - p->grid % period);
    return true;
}

// Cluster plan for aligned rows longer than the staged and direct tiers take
// (more than 2048 vectors): clusters of 2, 4 or
// 8 CTAs, one per SM, each CTA's slice a whole number of vectors (at most
// 2048) and each CTA sized to its slice, threads rounded up to a warp: two
// vectors a thread up to CLUSTER_NT_V2 threads, else four.  A CTA of 512
// threads for every slice left half its warps a vector short of the rest at
// each row's barrier (2000 x 40000 bf16 VJP, slices of 1250 vectors: 3652 ->
// 3721 GB/s with 640 threads of two).  The ring takes at
// least three slices (four or more: the row loop overlaps a row's exchange
// with the next row, which measured faster wherever they fit: 2000 x 40000
// bf16 VJP 2815 -> 3276 GB/s, D = 24576 3431 -> 4051; three: one row at a
// time, which lets the longest slices fit: D = 32768 3210 -> 4063, 65536
// 2198 -> 2741).  Of the fitting sizes, the one with the most SMs busy
// (clusters the device holds at once, cap[cl], times CTAs per cluster); but a
// forward whose busiest size leaves the ring three slices deep takes a size
// with four or more if that keeps at least 94 % as many SMs busy and gives
// each cluster at least 32 rows (GB/s, with a residual, clusters of two on
// 152 SMs with three stages against four on 144 with five: bf16 4096 x 32768
// 5994 -> 6475, fp32 2048 x 16384 6001 -> 6212; with fewer rows a cluster
// the longer row chain loses: bf16 1024 x 30720 5675 -> 5609, 300 x 32768
// 5214 -> 4250).  The VJP keeps the busiest size (bf16 4096 x 32768: 5972
// against 4286).
inline bool plan_cluster(int mode, int64_t rows, int D, int esize, const int *cap, int sm_count,
                         Plan *p) {
    const int64_t nv = (int64_t)D * esize / 16;
    const int ntens = input_tensors(mode);
    int best_cl = 0;
    int64_t best = 0;
    int64_t busy_of[9] = {}, depth_of[9] = {}, clusters_of[9] = {};
    for (int cl : {2, 4, 8}) {
        if (tuning().cl && cl != tuning().cl) continue;
        const int64_t slice = ceil_div(nv, cl);  // vectors of one CTA's slice
        if (slice > 4 * CLUSTER_NT_V4) continue;
        const int64_t depth = (int64_t)SMEM_ONE_PER_SM / ((int64_t)ntens * slice * 16);
        if (depth < 3) continue;
        const int64_t clusters = cap ? cap[cl] : sm_count / cl;
        if (clusters <= 0) continue;
        const int64_t busy = std::min<int64_t>(clusters, rows) * cl;
        busy_of[cl] = busy;
        depth_of[cl] = depth;
        clusters_of[cl] = clusters;
        if (busy > best) {
            best = busy;
            best_cl = cl;
        }
    }
    if (!best_cl) return false;
    if (!is_vjp(mode) && depth_of[best_cl] < 4) {
        int alt = 0;
        for (int cl : {2, 4, 8})
            if (depth_of[cl] >= 4 && busy_of[cl] * 100 >= best * 94 &&
                rows >= 32 * clusters_of[cl] && (!alt || busy_of[cl] > busy_of[alt]))
                alt = cl;
        if (alt) best_cl = alt;
    }
    const int64_t per_cta_vec = ceil_div(nv, best_cl);
    *p = Plan{};
    p->tier = TIER_CLUSTER;
    p->v = per_cta_vec <= 2 * CLUSTER_NT_V2 ? 2 : 4;
    p->nt = (int)(ceil_div(ceil_div(per_cta_vec, p->v), 32) * 32);
    p->g = p->nt;
    p->cl = best_cl;
    p->cl_cols = (int)(per_cta_vec * 16 / esize);
    p->tile_rows = 1;
    p->stage_bytes = (uint32_t)(per_cta_vec * 16);
    const size_t per_stage = (size_t)ntens * p->stage_bytes;
    // Four stages or more: the kernel overlaps a row's exchange with the next
    // row (two rows held, the rest in flight); three: one row at a time.
    const int64_t sc = (int64_t)(SMEM_ONE_PER_SM / per_stage);
    p->stages = sc >= 4 ? (int)std::min<int64_t>(
                              std::min<int64_t>(MAX_STAGES, sc),
                              std::max(4, 2 + ring_stages(is_vjp(mode) ? INFLIGHT_VJP : INFLIGHT_FWD,
                                                          per_stage, 1)))
                        : 3;
    p->smem = 1024 + (size_t)p->stages * per_stage;  // header of the cluster kernel
    p->num_tiles = rows;
    const int64_t clusters = cap ? cap[best_cl] : sm_count / best_cl;
    p->grid = (int)(std::min<int64_t>(clusters, rows) * best_cl);
    return true;
}

inline Plan make_plan(int mode, int64_t rows, int D, int esize, int align, int sm_count,
                      const int *cluster_cap = nullptr) {
    Plan p{};
    const bool aligned = align == ALIGN_VEC || align == ALIGN_VEC_GEN;
    const bool shift = align == ALIGN_SHIFT;
    const int64_t nv = row_vectors(D, esize);
    if ((aligned || shift) && rows > DECODE_ROWS) {
        const int forced = tuning().cfg;
        if (forced >= 0 && nv <= STAGED_CFGS[forced].max_nv &&
            !(is_vjp(mode) && forced == STAGED_CFG_WIDE) &&
            plan_staged(mode, rows, D, esize, sm_count, forced, shift, &p))
            return p;
        // the configuration that fits the row most tightly (the wide one
        // only when tuned)
        int best = -1;
        for (int ci = 0; ci < N_STAGED_CFG; ++ci)
            if (ci != STAGED_CFG_WIDE && nv <= STAGED_CFGS[ci].max_nv &&
                (best < 0 || STAGED_CFGS[ci].max_nv < STAGED_CFGS[best].max_nv))
                best = ci;
        if (best >= 0 && plan_staged(mode, rows, D, esize, sm_count, best, shift, &p)) return p;
    }
    // Rows of more than 2048 vectors: the cluster tier, forward and VJP.  The
    // forwards of 2049-4096 vectors ran 17-40 % slower on the direct tier
    // (a row in one CTA's registers; GB300, same buffers back to back, bf16
    // 4096 x 24576 with residual 5218 -> 6114 GB/s, without 4156 -> 5624, fp16
    // 8192 x 20480 without 3930 -> 5517, fp32 4096 x 12288 5125 -> 6163).
    if (align == ALIGN_VEC && rows > DECODE_ROWS && nv > 2048 &&
        plan_cluster(mode, rows, D, esize, cluster_cap, sm_count, &p))
        return p;
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
                // A decode VJP of 2-8 rows runs as one cluster of its rows,
                // which sums gw itself: no partial rows, no second kernel.
                if (is_vjp(mode) && rows >= 2 && rows <= DECODE_ROWS) {
                    p.cl = (int)rows;
                    p.smem = (size_t)D * sizeof(float);
                }
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
    // The VJP's partial rows (one per CTA) stay within 10 % of its bytes
    // (P * 4 <= 0.1 * 3 * esize * rows) and within two CTAs per SM, but a
    // decode-sized VJP keeps a CTA per row (at most 8 partial rows).
    p.grid = is_vjp(mode)
                 ? (int)std::max<int64_t>(std::min<int64_t>(rows, DECODE_ROWS),
                                          std::min<int64_t>((int64_t)sm_count * 2,
                                                            rows * 3 * esize / 40))
                 : (int)std::min<int64_t>(rows, (int64_t)sm_count * 8);
    return p;
}

}  // namespace planner
}  // namespace rmsn
