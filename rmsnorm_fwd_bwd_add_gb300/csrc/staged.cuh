// staged.cuh -- persistent RMSNorm kernels that stage rows through a shared
// memory ring with the 1-D TMA bulk copy (cp.async.bulk + mbarrier).
//
// Work unit: a tile of `tile_rows` consecutive rows.  Rows are contiguous, so
// one tile of one tensor is ONE bulk copy.  CTA b owns tiles b, b + grid,
// b + 2*grid, ... (a static assignment, so the VJP's gw partials are summed in
// the same order on every run).  Thread 0 keeps `stages` tiles in flight;
// every thread waits on the tile's mbarrier, reads its vectors from shared
// memory, and writes its outputs straight to global memory.
//
// Two shapes of work inside a tile:
//   * G == NT ("CTA per row", D > 1024): one row per tile; each thread owns
//     V vectors of 8 elements; sum of squares = warp shuffle tree, then the
//     warp totals in shared memory added in warp order (the warp-then-block
//     reduction of the fused-norm design), one CTA barrier per row.
//   * G <= 32 ("sub-warp / warp per row", D <= 1024): NT/G rows at a time,
//     each reduced by a G-lane shuffle tree only; no shared-memory reduction,
//     so no multi-warp band exists to get wrong.
// The weight vectors a thread multiplies by are the same for every row it
// touches (fixed column ownership), so w is read once per CTA and, in the VJP,
// the gw contribution of every row stays in the owning thread's registers.
//
// Sources: "Fused residual-add RMSNorm and fused RoPE + KV-append decode
// kernels", Background (FusedAddRMSNorm: one pass, fp32 sum kept once,
// warp-then-block sum of squares, weight_bias, two outputs); "RMSNormVJP
// backward writes a full {n_rows, D} gw_temp intermediate", Proposed changes
// (reduce gw across rows inside the kernel, no {n_rows, D} temporary).
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rmsn {

template <typename T, int MODE, int NT, int G, int V, int MINB>
__global__ void __launch_bounds__(NT, MINB) staged_kernel(const KernelArgs a) {
    constexpr int NWARPS = NT / 32;
    constexpr int NG = NT / G;  // rows processed side by side
    constexpr bool CTA_ROW = (G == NT);
    constexpr int NTENS = (MODE == MODE_FWD_NORES) ? 1 : 2;
    constexpr bool VJP = (MODE == MODE_VJP);
    static_assert(G <= 32 || G == NT, "a row belongs to at most one warp, or to the whole CTA");
    static_assert(NWARPS <= 32, "reduction scratch holds 32 warps");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [MAX_STAGES]
    float *red = reinterpret_cast<float *>(smem + 128);   // [2][NWARPS][2]
    unsigned char *ring = smem + STAGED_HEADER_BYTES;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gid = tid / G;
    const int gl = tid % G;
    const int D = a.D;
    const int NV = D >> 3;
    const int S = a.stages;
    const int TR = a.tile_rows;
    const int64_t rows = a.rows;
    const uint32_t SB = a.stage_bytes;
    const int64_t grid = gridDim.x;
    const int64_t nk = (a.num_tiles - (int64_t)blockIdx.x + grid - 1) / grid;  // >= 1
    const float eps = a.eps;
    const float wb = a.weight_bias;
    const float Df = (float)D;  // exact: D <= 2^24

    const T *in0 = static_cast<const T *>(a.in0);
    const T *in1 = static_cast<const T *>(a.in1);
    uint4 *out0 = static_cast<uint4 *>(a.out0);
    uint4 *out1 = static_cast<uint4 *>(a.out1);

    auto stage_ptr = [&](int64_t k, int tensor) -> unsigned char * {
        return ring + ((size_t)(k % S) * NTENS + tensor) * SB;
    };

    // ---- producer state (thread 0 only) ----
    int64_t issued = 0;
    const uint64_t policy = l2_evict_first_policy();
    auto issue = [&](int64_t k) {
        const int64_t t = (int64_t)blockIdx.x + k * grid;
        if (t != a.drop_tile) {
            const int64_t row0 = t * TR;
            const int64_t nr = min((int64_t)TR, rows - row0);
            const uint32_t bytes = (uint32_t)(nr * D * (int64_t)sizeof(T));
            uint64_t *bar = &full[k % S];
            mbar_arrive_expect_tx(bar, bytes * NTENS);
            bulk_g2s(stage_ptr(k, 0), in0 + row0 * D, bytes, bar, policy);
            if constexpr (NTENS == 2) bulk_g2s(stage_ptr(k, 1), in1 + row0 * D, bytes, bar, policy);
        }
        issued = k + 1;
    };
    // Timeout exit: flag it, then wait (bounded) for this CTA's copies that
    // may still be landing in shared memory before the CTA retires.
    auto fail = [&](int64_t k) {
        if (tid == 0) {
            atomicOr(a.status, DEVSTATUS_WAIT_TIMEOUT);
            for (int64_t kk = k; kk < issued; ++kk) {
                if ((int64_t)blockIdx.x + kk * grid == a.drop_tile) continue;
                mbar_wait_bounded(&full[kk % S], (uint32_t)((kk / S) & 1), DEFAULT_WAIT_BUDGET);
            }
        }
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const int64_t n0 = min((int64_t)S, nk);
        for (int64_t k = 0; k < n0; ++k) issue(k);
    }

    // Weight vectors owned by this thread, packed (converted at use).
    uint4 wv[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int vi = gl + j * G;
        wv[j] = vi < NV ? reinterpret_cast<const uint4 *>(a.w)[vi] : make_uint4(0, 0, 0, 0);
    }
    float acc[VJP ? V : 1][8];
#pragma unroll
    for (int j = 0; j < (VJP ? V : 1); ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;

    // Phase 1: this thread's share of sum(h^2) and, for the VJP, of
    // dot = sum(g * w' * x).
    auto partial_sums = [&](const uint4 *r0, const uint4 *r1, float &sa, float &sb) {
        sa = 0.f;
        sb = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = gl + j * G;
            if (vi < NV) {
                float f0[8];
                unpack8<T>(r0[vi], f0);
                if constexpr (MODE == MODE_FWD_RES) {
                    float f1[8];
                    unpack8<T>(r1[vi], f1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float h = f0[e] + f1[e];
                        sa += h * h;
                    }
                } else if constexpr (MODE == MODE_FWD_NORES) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) sa += f0[e] * f0[e];
                } else {
                    float f1[8], wf[8];
                    unpack8<T>(r1[vi], f1);
                    unpack8<T>(wv[j], wf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sa += f0[e] * f0[e];
                        sb += (f1[e] * (wb + wf[e])) * f0[e];
                    }
                }
            }
        }
    };

    // Phase 2: outputs of one row (re-reading the staged row).
    auto row_outputs = [&](const uint4 *r0, const uint4 *r1, int64_t row, float r, float dot) {
        const size_t base = (size_t)row * NV;
        const float c = (r * r) * (dot / Df);  // r^2 * dot / D
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = gl + j * G;
            if (vi < NV) {
                float f0[8], wf[8], o[8];
                unpack8<T>(r0[vi], f0);
                unpack8<T>(wv[j], wf);
                if constexpr (MODE == MODE_FWD_RES) {
                    float f1[8];
                    unpack8<T>(r1[vi], f1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        f0[e] = f0[e] + f1[e];  // h, unrounded
                        o[e] = (f0[e] * r) * (wb + wf[e]);
                    }
                    st_global(out1 + base + vi, pack8<T>(f0));
                } else if constexpr (MODE == MODE_FWD_NORES) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = (f0[e] * r) * (wb + wf[e]);
                } else {
                    float f1[8];
                    unpack8<T>(r1[vi], f1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float gwp = f1[e] * (wb + wf[e]);
                        o[e] = r * (gwp - f0[e] * c);
                        acc[j][e] += (f1[e] * f0[e]) * r;
                    }
                }
                st_global(out0 + base + vi, pack8<T>(o));
            }
        }
    };

    if constexpr (CTA_ROW) {
        for (int64_t k = 0; k < nk; ++k) {
            const int64_t row = (int64_t)blockIdx.x + k * grid;  // tile_rows == 1
            const bool ok = mbar_wait_bounded(&full[k % S], (uint32_t)((k / S) & 1), a.wait_budget);
            const uint4 *r0 = reinterpret_cast<const uint4 *>(stage_ptr(k, 0));
            const uint4 *r1 = reinterpret_cast<const uint4 *>(stage_ptr(k, NTENS - 1));
            float sa, sb;
            partial_sums(r0, r1, sa, sb);
            sa = group_sum<32>(sa);
            if constexpr (VJP) sb = group_sum<32>(sb);
            float *rb = red + (k & 1) * (NWARPS * 2);
            if (lane == 0) {
                rb[warp * 2] = sa;
                rb[warp * 2 + 1] = sb;
            }
            // Everyone has finished row k-1 (so its stage is free) and has
            // published row k's warp totals.
            if (__syncthreads_or(!ok)) {
                fail(k);
                return;
            }
            if (tid == 0 && k >= 1 && k - 1 + S < nk) issue(k - 1 + S);
            float ss = 0.f, dot = 0.f;
#pragma unroll
            for (int w = 0; w < NWARPS; ++w) {
                ss += rb[w * 2];
                if constexpr (VJP) dot += rb[w * 2 + 1];
            }
            const float r = rsqrtf(ss / Df + eps);
            row_outputs(r0, r1, row, r, dot);
        }
    } else {
        for (int64_t k = 0; k < nk; ++k) {
            const int64_t row0 = ((int64_t)blockIdx.x + k * grid) * TR;
            const int nr = (int)min((int64_t)TR, rows - row0);
            const bool ok = mbar_wait_bounded(&full[k % S], (uint32_t)((k / S) & 1), a.wait_budget);
            const uint4 *t0 = reinterpret_cast<const uint4 *>(stage_ptr(k, 0));
            const uint4 *t1 = reinterpret_cast<const uint4 *>(stage_ptr(k, NTENS - 1));
            for (int qb = 0; qb < TR; qb += NG) {  // same trip count in every lane
                const int q = qb + gid;
                const bool valid = q < nr;
                const uint4 *r0 = t0 + (size_t)q * NV;
                const uint4 *r1 = t1 + (size_t)q * NV;
                float sa = 0.f, sb = 0.f;
                if (valid) partial_sums(r0, r1, sa, sb);
                sa = group_sum<G>(sa);
                if constexpr (VJP) sb = group_sum<G>(sb);
                if (valid && ok) row_outputs(r0, r1, row0 + q, rsqrtf(sa / Df + eps), sb);
            }
            if (__syncthreads_or(!ok)) {  // the whole tile is consumed
                fail(k);
                return;
            }
            if (tid == 0 && k + S < nk) issue(k + S);
        }
    }

    if constexpr (VJP) {
        float *prow = a.partials + (size_t)blockIdx.x * D;
        if constexpr (CTA_ROW) {
            // Each column is owned by exactly one thread of the CTA.
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = gl + j * G;
                if (vi < NV) {
                    float4 *dst = reinterpret_cast<float4 *>(prow + (size_t)vi * 8);
                    dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                    dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
                }
            }
        } else {
            // NG groups own the same columns: add their registers in group
            // order through shared memory (the ring is idle now).
            __syncthreads();
            float *buf = reinterpret_cast<float *>(ring);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = gl + j * G;
                if (vi < NV) {
                    float4 *dst = reinterpret_cast<float4 *>(buf + (size_t)gid * D + (size_t)vi * 8);
                    dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                    dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
                }
            }
            __syncthreads();
            for (int col = tid; col < D; col += NT) {
                float s = 0.f;
                for (int gg = 0; gg < NG; ++gg) s += buf[(size_t)gg * D + col];
                prow[col] = s;
            }
        }
    }
}

}  // namespace rmsn
