// plan.h -- launch plans and kernel parameters shared by the host dispatcher
// (api.cu) and the per-tier launchers.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rmsn {

enum Tier : int { TIER_STAGED = 0, TIER_DIRECT = 1, TIER_GENERIC = 2, TIER_CLUSTER = 3 };

// Kernel arguments.  in0 = x; in1 = residual (forward) or g (VJP);
// in2 = the gradient of new_residual (fused-op VJP); out0 = out (forward), gx
// (VJP) or gx + in2 (fused-op VJP); out1 = new_residual (forward).
struct KernelArgs {
    const void *in0;
    const void *in1;
    const void *in2;
    const void *w;
    void *out0;
    void *out1;
    float *partials;          // VJP: [grid, D] fp32 gw partials, one row per CTA
    unsigned int *status;     // device status word
    float eps;
    float weight_bias;
    int64_t rows;
    int D;
    // staged tier
    int tile_rows;            // rows per tile (one bulk copy per tensor)
    int stages;               // shared-memory ring depth
    int64_t num_tiles;
    uint32_t stage_bytes;     // bytes of one full tile of one tensor
    long long wait_budget;    // SM cycles per bounded wait
    int64_t drop_tile;        // test hook: tile whose copy is never issued (-1: none)
    // Row strides in elements (D for dense rows).
    int64_t ld_in0, ld_in1, ld_in2, ld_out0, ld_out1;
    // Per-row 1/sqrt(ms + eps), fp32 [rows] or null: written by the forward,
    // read (instead of summing h^2) by the VJP.
    float *rstd;
    // General sub-warp instance: tiles land in shared memory as column boxes
    // [D / box_cols][tile_rows][box_cols] (box_cols == D: plain rows).  With
    // use_tmap the inputs in0..in2 come through the 2-D tensor maps tmap[],
    // one copy per box; without, one bulk copy per row.
    int box_cols;
    int use_tmap;
    CUtensorMap tmap[3];
    // Cluster tier: columns of each CTA's slice of a row (a whole number of
    // 16-byte vectors).
    int cl_cols;
    // Staged forwards that claim their tiles at run time: claim_k group
    // counters (CLAIM_STRIDE apart) and then the count of finished CTAs, all
    // zero at launch and put back to zero by the launch's last CTA; null for
    // the static round robin.  claim_k divides the grid.
    unsigned long long *tile_ctr;
    int claim_k;
};

// Layout of one set of claim counters (in 8-byte words): group counter j at
// j * CLAIM_STRIDE (a 32-byte sector each), the finished-CTA count after the
// CLAIM_MAX_K group counters.
constexpr int CLAIM_MAX_K = 8;
constexpr int CLAIM_STRIDE = 4;
constexpr int CLAIM_WORDS = CLAIM_STRIDE * (CLAIM_MAX_K + 1);
// Staged configurations that can claim tiles: CTA per row, this many
// threads or more (the rows long enough for a claim to pay).
constexpr int CLAIM_MIN_NT = 768;

struct Plan {
    int tier;
    int cfg;           // index into the tier's configuration table
    int nt;            // threads per CTA
    int g;             // threads per row
    int v;             // 16-byte vectors per thread per row (8 fp16/bf16 or 4 fp32 elements)
    int stages;
    int tile_rows;
    int64_t num_tiles;
    int grid;          // CTAs; for the VJP also the number of gw partial rows
    size_t smem;       // dynamic shared memory bytes
    uint32_t stage_bytes;
    bool shift;        // staged tier: shifted-rows instance (rows off a 16-byte boundary)
    int cl;            // cluster tier: CTAs per cluster (per row)
    int cl_cols;       // cluster tier: columns of one CTA's slice
};

// How a problem's row tensors sit relative to 16-byte boundaries.
//   ALIGN_VEC:   every row of every tensor (and w) starts on a boundary;
//   ALIGN_SHIFT: dense rows whose tensors all start at the same offset from a
//                boundary (an unaligned base, or D * size not a multiple of
//                16), elements naturally aligned;
//   ALIGN_VEC_GEN: every row aligned, but rows a stride apart or a per-row
//                rstd given (the general instances; not the cluster tier);
//   ALIGN_NONE:  anything else (the element-at-a-time tier).
enum Align : int { ALIGN_NONE = 0, ALIGN_VEC = 1, ALIGN_SHIFT = 2, ALIGN_VEC_GEN = 3 };

// Configuration tables (index = Plan::cfg).
struct StagedCfg { int nt, g, v, max_nv; };
struct DirectCfg { int nt, v, max_nv; };

constexpr int N_STAGED_CFG = 19;
constexpr StagedCfg STAGED_CFGS[N_STAGED_CFG] = {
    // sub-warp / warp per row (shuffle-only reductions), 256 threads
    {256, 8, 1, 8}, {256, 16, 1, 16}, {256, 32, 1, 32},
    {256, 32, 2, 64}, {256, 32, 3, 96}, {256, 32, 4, 128},
    // CTA per row
    {128, 128, 2, 256}, {256, 256, 2, 512}, {512, 512, 2, 1024}, {1024, 1024, 2, 2048},
    // CTA per row, four vectors per thread: two 256-thread CTAs per SM for
    // rows of up to 8192 (forward only: the VJP would need too many registers)
    {256, 256, 4, 1024},
    // CTA per row for rows of 3 * 2^k vectors (D = 1536, 3072, 6144, 12288 in
    // bf16), which the power-of-two CTAs above fit with a quarter of their
    // threads idle
    {96, 96, 2, 192}, {192, 192, 2, 384}, {384, 384, 2, 768}, {768, 768, 2, 1536},
    // and for rows of 5 * 2^k and 7 * 2^k vectors (D = 2560, 5120; 3584, 7168)
    {160, 160, 2, 320}, {224, 224, 2, 448}, {320, 320, 2, 640}, {448, 448, 2, 896},
};
constexpr int STAGED_CFG_WIDE = 10;

constexpr int N_DIRECT_CFG = 6;
constexpr DirectCfg DIRECT_CFGS[N_DIRECT_CFG] = {
    {128, 1, 128}, {256, 1, 256}, {512, 1, 512}, {512, 2, 1024}, {1024, 2, 2048}, {1024, 4, 4096},
};

// Whether a VJP instance re-reads its rows from the stage for its outputs
// instead of holding them in registers across the reduction (the stage stays
// resident until the tile is done).  That is a second pass over shared memory
// for fewer registers, and it pays where it buys CTAs or removes spills
// (bf16 VJP, rotating buffers, GB300):
//   * sub-warp tiles with three or four vectors per lane: 128 registers, two
//     CTAs per SM instead of one (D = 640: 4370 -> 5484 GB/s);
//   * CTAs of 384 and 448 threads: about 80 registers, two CTAs per SM
//     instead of one (D = 6144: 5341 -> 5983, D = 7168: 5297 -> 5527);
//   * CTAs of 768 and 1024 threads, whose register cap (80, 64) spilled
//     (D = 12288: 4641 -> 5978, D = 16384: 3670 -> 6010).
// Elsewhere it loses: 224-320 threads with three CTAs per SM instead of two
// (D = 4096: 5746 against 5902), 512 threads with two instead of one (D =
// 8192: 5882 against 6229).
__host__ __device__ constexpr bool staged_reload(int mode, int nt, int g, int v) {
    return mode >= 2 && (g != nt ? v >= 3 : (nt == 384 || nt == 448 || nt >= 768));
}

// Most CTAs of a staged configuration that can share one SM, as the kernels'
// __launch_bounds__ promise it (registers per thread capped to fit).
// CTA-per-row forwards with two vectors per thread (about 80 registers):
// 6 of up to 128 threads, 3 of up to 256, 2 of up to 448.  CTA-per-row VJPs
// with two vectors (about 110 registers): 6 of 96 threads, 4 of 128, 3 of up
// to 192, 2 of up to 320, and 2 of 384 or 448 threads, which re-read their
// rows.  Other CTAs of up to 256 threads 2 (128 registers; the sub-warp VJP
// with three or four vectors per lane fits by re-reading rows from shared
// memory); larger CTAs 1.
constexpr int staged_max_ctas_per_sm(int mode, int nt, int g, int v) {
    return (g == nt && mode < 2 && nt <= 128 && v <= 2)    ? 6
           : (g == nt && mode < 2 && nt <= 256 && v <= 2)  ? 3
           : (g == nt && mode < 2 && nt <= 448 && v <= 2)  ? 2
           : (g == nt && mode >= 2 && nt <= 96 && v <= 2)  ? 6
           : (g == nt && mode >= 2 && nt <= 128 && v <= 2) ? 4
           : (g == nt && mode >= 2 && nt <= 192 && v <= 2) ? 3
           : (nt <= 256)                                   ? 2
           : (g == nt && mode >= 2 && nt <= 320 && v <= 2) ? 2
           : (g == nt && staged_reload(mode, nt, g, v) && nt <= 448) ? 2
                                                            : 1;
}
// CTAs per SM the plan uses unless tuned otherwise, from sweeps of 1-6 on
// GB300 (bf16, rotating buffers, 8192-32768 rows).  CTA-per-row shapes:
//   * up to 128 threads: as many as fit (D = 2048 forward 5697 -> 6442 GB/s,
//     VJP 3522 -> 5814 against two);
//   * the forward without a residual (mode 1): three of up to 256 threads
//     (D = 3072: 4486 -> 5622), two of up to 448 (D = 7168: 4197 -> 5853);
//   * the forward with a residual (mode 0): three of up to 192 threads, two
//     of 224-320 (D = 4096: 6394 against 6221 with three) and of 448 (D =
//     7168: 6259 against 6152), one of 384 (D = 6144: 6566 against 6144 with
//     two, whose rings are then only two stages deep) and of 512 or more;
//   * the VJP: as many as fit up to 192 threads (D = 3072: 5032 -> 5294
//     against two), two of up to 448 (D = 5120: 3714 -> 5767), one above.
// Sub-warp shapes: two, or one where only one fits.
constexpr int staged_ctas_per_sm(int mode, int nt, int g, int v) {
    const int most = staged_max_ctas_per_sm(mode, nt, g, v);
    const int want = (g != nt)    ? 2
                     : (nt <= 128) ? most
                     : (mode == 1) ? (nt <= 256 ? 3 : nt <= 448 ? 2 : 1)
                     : (mode == 0) ? (nt <= 192 ? 3 : (nt <= 320 || nt == 448) ? 2 : 1)
                                   : (nt <= 192 ? most : nt <= 448 ? 2 : 1);
    return want < most ? want : most;
}

constexpr int GENERIC_NT = 256;
constexpr int STAGED_HEADER_BYTES = 640;  // 16 mbarriers (128 B) + reduction scratch (512 B)
constexpr int MAX_STAGES = 8;
// Threads of a cluster CTA at two vectors a thread (the VJP's 92 registers
// fit 640 threads) and at four (512).
constexpr int CLUSTER_NT_V2 = 640;
constexpr int CLUSTER_NT_V4 = 512;

// Launchers (one translation unit per tier / dtype).  dtype: 0 fp16, 1 bf16,
// 2 fp32.
cudaError_t launch_staged(int dtype, int mode, const Plan &plan, const KernelArgs &a,
                          cudaStream_t stream);
cudaError_t launch_direct(int dtype, int mode, const Plan &plan, const KernelArgs &a,
                          cudaStream_t stream);
cudaError_t launch_generic(int dtype, int mode, const Plan &plan, const KernelArgs &a,
                           cudaStream_t stream);
cudaError_t launch_gw_reduce(const float *partials, float *gw, int P, int D, cudaStream_t stream);
cudaError_t launch_cluster(int dtype, int mode, const Plan &plan, const KernelArgs &a,
                           cudaStream_t stream);
// Clusters of `cl` CTAs (2..8), one CTA per SM, that the current device can
// hold at once (0 if clusters are unavailable).
int cluster_capacity(int cl);

// A 2-D tensor map of a [rows, D] tensor with row stride ld elements and
// boxes of box_cols x box_rows elements, counted in 8-byte units (box rows of
// up to 2 KB; no swizzle, zero fill past the last row; the x coordinate of a
// copy is in 8-byte units too).  False if the driver refuses it or the entry
// point is missing.
bool encode_rows_tmap(CUtensorMap *map, const void *base, int64_t rows, int64_t D, int64_t ld,
                      int dtype, int box_cols, int box_rows);

}  // namespace rmsn
