// cluster.cuh -- RMSNorm kernels for rows longer than one CTA's shared-memory
// ring holds (more than 2048 16-byte vectors: D > 16384 for fp16/bf16, D >
// 8192 for fp32).
//
// A thread-block cluster of CL CTAs takes one row at a time (cluster c owns
// rows c, c + clusters, ..., a static assignment).  CTA `rank` of the cluster
// owns the contiguous column slice [rank * C, rank * C + C) of every row and
// streams that slice through its own ring with the 1-D TMA bulk copy, exactly
// as the staged kernels stream whole rows; the CTA is sized to its slice.
// Per row, each CTA reduces its slice (warp shuffle tree, then warp 0 sums
// the warp totals in one fixed order) and warp 0 writes the slice's
// (sum h^2, dot) into its slot of every cluster CTA's shared memory with an
// asynchronous store (st.async) that completes 8 bytes on that CTA's slot
// mbarrier, which each CTA arms once per row for all CL slots.  (A release
// arrival instead would make the sender wait, every row, for its own earlier
// global stores to be acknowledged.)  Each CTA then adds the CL slots in rank
// order, so every CTA of the cluster forms the same row sums, bit for bit,
// whatever order the slots arrived in.  A CTA's columns never change, so its
// w' and its gw contributions stay in registers; the cluster writes one gw
// partial row (one per cluster), summed in a fixed order by the same stage-2
// kernel as the other tiers.
//
// Every wait is bounded.  On a timeout the CTA flags it, waits (bounded) for
// its own copies in flight, and before it exits arrives on every cluster
// CTA's exit mbarrier and waits (bounded) for theirs, so no CTA exits while
// another may still write into its shared memory.
//
// Sources: "Fused residual-add RMSNorm and fused RoPE + KV-append decode
// kernels", Background (FusedAddRMSNorm: one pass, fp32 sums, warp-then-block
// reduction, weight_bias, two outputs); "RMSNormVJP backward writes a full
// {n_rows, D} gw_temp intermediate", Proposed changes (gw reduced across rows
// inside the kernel, no {n_rows, D} temporary).
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rmsn {

constexpr int CLUSTER_HEADER_BYTES = 1024;
constexpr int CLUSTER_MAX = 8;  // portable cluster size
// blockDim.x = NT threads (a multiple of 32, at most NTMAX), up to V
// 16-byte vectors of the slice each (the slice is at most NT * V vectors;
// the plan sizes the CTA to its slice, so every warp has about the same share
// of a row); PIPE: the exchange of a row's sums overlaps the next row (four
// or more stages), else one row at a time (three).
template <typename T, int MODE, int NTMAX, int V, int CL, bool PIPE>
__global__ void __launch_bounds__(NTMAX, 1) cluster_kernel(const __grid_constant__ KernelArgs a) {
    const int NT = blockDim.x;
    const int NWARPS = NT >> 5;
    constexpr int VP = vec_pairs<T>();
    constexpr int EPV = vec_elems<T>();
    constexpr int NTENS = input_tensors(MODE);
    constexpr bool VJP = is_vjp(MODE);
    constexpr bool ADD = (MODE == MODE_VJP_ADD);
    static_assert(CL >= 2 && CL <= CLUSTER_MAX, "a cluster of 2 to 8 CTAs");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);        // [MAX_STAGES]: slice landed
    uint64_t *clbar = reinterpret_cast<uint64_t *>(smem + 64);  // [4]: every CTA's sums arrived
    uint64_t *xbar = reinterpret_cast<uint64_t *>(smem + 96);   // exit handshake
    float2 *cred = reinterpret_cast<float2 *>(smem + 128);      // [4][CL] the CTAs' slice sums
    float2 *red = reinterpret_cast<float2 *>(smem + 512);       // [2][NWARPS <= 32] warp totals
    unsigned char *ring = smem + CLUSTER_HEADER_BYTES;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    const int64_t cid = blockIdx.x / CL;   // this CTA's cluster
    const int64_t ncl = gridDim.x / CL;    // clusters
    const int D = a.D;
    const int c0 = (int)rank * a.cl_cols;  // first column of this CTA's slice
    const int nc = max(0, min(a.cl_cols, D - c0));
    const int NVS = nc / EPV;              // vectors of the slice
    const int vc0 = c0 / EPV;              // the slice's first vector in a row
    const int64_t NVR = D / EPV;           // vectors of a row
    const uint32_t slice_bytes = (uint32_t)nc * (uint32_t)sizeof(T);
    const int S = a.stages;
    const uint32_t SB = a.stage_bytes;
    const int64_t rows = a.rows;
    const int64_t nk = cid < rows ? (rows - cid + ncl - 1) / ncl : 0;
    const float eps = a.eps;
    const float inv_D = 1.0f / (float)D;

    const T *in0 = static_cast<const T *>(a.in0);
    const T *in1 = static_cast<const T *>(a.in1);
    const T *in2 = static_cast<const T *>(a.in2);
    uint4 *out0 = static_cast<uint4 *>(a.out0);
    uint4 *out1 = static_cast<uint4 *>(a.out1);

    auto stage_ptr = [&](int s, int tensor) -> unsigned char * {
        return ring + ((size_t)s * NTENS + tensor) * SB;
    };

    // ---- producer (thread 0): one copy of the slice per tensor per row ----
    int64_t issued = 0;
    int issue_stage = 0;
    const uint64_t policy = l2_evict_first_policy();
    auto issue_next = [&]() {
        const int64_t row = cid + issued * ncl;
        if (row * CL + rank != a.drop_tile) {  // test hook: a copy that never arrives
            uint64_t *bar = &full[issue_stage];
            mbar_arrive_expect_tx(bar, slice_bytes * NTENS);
            if (slice_bytes) {
                const int64_t off = row * D + c0;
                bulk_g2s(stage_ptr(issue_stage, 0), in0 + off, slice_bytes, bar, policy);
                if constexpr (NTENS >= 2)
                    bulk_g2s(stage_ptr(issue_stage, 1), in1 + off, slice_bytes, bar, policy);
                if constexpr (NTENS == 3)
                    bulk_g2s(stage_ptr(issue_stage, 2), in2 + off, slice_bytes, bar, policy);
            }
        }
        ++issued;
        issue_stage = issue_stage + 1 == S ? 0 : issue_stage + 1;
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&clbar[i], 1);  // armed once per row
        mbar_init(xbar, CL);
        fence_mbar_init();
    }
    // Every CTA of the cluster has initialised its barriers before any CTA
    // arrives on them remotely.
    cluster_sync_all();
    // Launched as a programmatic dependent: no global memory access before
    // the previous kernel on the stream has completed.
    griddep_wait();
    if (tid == 0)
        while (issued < min((int64_t)S, nk)) issue_next();

    // w' = weight_bias + w for this thread's columns of the slice, in fp32.
    float2 wp[V][VP];
    {
        const float2 wb2 = make_float2(a.weight_bias, a.weight_bias);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            const uint4 wv = vi < NVS ? reinterpret_cast<const uint4 *>(a.w)[vc0 + vi]
                                      : make_uint4(0, 0, 0, 0);
            float2 wf[VP];
            unpack_vec<T>(wv, wf);
#pragma unroll
            for (int q = 0; q < VP; ++q) wp[j][q] = f2add(wb2, wf[q]);
        }
    }
    float2 acc[VJP ? V : 1][VP];
#pragma unroll
    for (int j = 0; j < (VJP ? V : 1); ++j)
#pragma unroll
        for (int q = 0; q < VP; ++q) acc[j][q] = make_float2(0.f, 0.f);

    constexpr int RD = 4;  // slots of slice sums (and their barriers)
    // Iteration k: A(k) = row k's slice sums, reduced in the CTA and sent to
    // the cluster; B(k-1) = row k-1's outputs, once every CTA's sums of that
    // row have arrived, with the slice re-read from its stage.  The cluster
    // exchange of a row so overlaps the next row's loads and sums.  The CTA
    // barrier of iteration k follows every thread's B(k-2), so the stage of
    // row k-2 is refilled then: rows k-1 and k hold stages, S - 3 rows are in
    // flight ahead.  A CTA sends row k + 4 (slot k % RD again) only after
    // every CTA's sums of row k + 2, which this CTA sends after its B(k):
    // RD = 4 slots never overwrite sums still to be read, and no slot
    // barrier runs two phases ahead of a waiter.
    bool ok = true;
    // Stage and phase of row k, and stage of row k - 1, advanced one step per
    // row: no 64-bit division by the runtime ring depth in the row loop (a
    // few of those per row cost as many instructions as the row's arithmetic).
    int a_stage = 0, b_stage = 0;
    uint32_t a_phase = 0;
    auto next_a = [&]() {
        if (++a_stage == S) {
            a_stage = 0;
            a_phase ^= 1u;
        }
    };
    static_assert(RD == 4, "slot k & 3, slot phase (k >> 2) & 1");
    if constexpr (PIPE) {
    for (int64_t k = 0; k <= nk; ++k) {
        if (k < nk) {
            if (tid == 0) mbar_arrive_expect_tx(&clbar[k & 3], CL * 8);  // row k's CL pairs
            const int sk = a_stage;
            ok = ok && mbar_wait_bounded(&full[sk], a_phase, a.wait_budget);
            next_a();
            const uint4 *r0 = reinterpret_cast<const uint4 *>(stage_ptr(sk, 0));
            const uint4 *r1 = reinterpret_cast<const uint4 *>(stage_ptr(sk, NTENS >= 2 ? 1 : 0));
            float2 s2 = make_float2(0.f, 0.f), d2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = tid + j * NT;
                if (vi < NVS) {
                    float2 xa[VP], xb[VP];
                    unpack_vec<T>(r0[vi], xa);
                    if constexpr (NTENS >= 2) unpack_vec<T>(r1[vi], xb);
                    if constexpr (MODE == MODE_FWD_RES) {
#pragma unroll
                        for (int q = 0; q < VP; ++q) xa[q] = f2add(xa[q], xb[q]);  // h
                    }
#pragma unroll
                    for (int q = 0; q < VP; ++q) s2 = f2fma(xa[q], xa[q], s2);
                    if constexpr (VJP) {
#pragma unroll
                        for (int q = 0; q < VP; ++q) d2 = f2fma(f2mul(xb[q], wp[j][q]), xa[q], d2);
                    }
                }
            }
            const float sa = group_sum<32>(s2.x + s2.y);
            const float sb = VJP ? group_sum<32>(d2.x + d2.y) : 0.f;
            if (lane == 0) red[(k & 1) * NWARPS + warp] = make_float2(sa, sb);
        }
        // Row k's warp totals are published and every thread is done with
        // iteration k - 1; a failed wait anywhere is seen by all.
        if (__syncthreads_or(!ok)) break;
        if (tid == 0 && k >= 2 && issued < nk) issue_next();  // into row k-2's stage
        if (k < nk && warp == 0) {
            // warp 0 (the sender) sums the warp totals in one fixed order:
            // lane l holds warp l's, zeros past NWARPS
            const float2 *rb = red + (k & 1) * NWARPS;
            float2 tot = lane < NWARPS ? rb[lane] : make_float2(0.f, 0.f);
            tot.x = group_sum<32>(tot.x);
            if constexpr (VJP) tot.y = group_sum<32>(tot.y);
            // lane q writes CTA q's slot, completing 8 bytes on its barrier,
            // so the CL sends go out side by side
            const int p = (int)(k & 3);
            if (lane < CL)
                dsmem_store_async_f2(dsmem_addr(&cred[p * CL + rank], (uint32_t)lane), tot,
                                     dsmem_addr(&clbar[p], (uint32_t)lane));
        }
        if (k >= 1) {
            const int64_t kk = k - 1;
            const int64_t row = cid + kk * ncl;
            const int sk = b_stage;
            if (++b_stage == S) b_stage = 0;
            const int p = (int)(kk & 3);
            ok = ok && mbar_wait_cluster_bounded(&clbar[p], (uint32_t)((kk >> 2) & 1),
                                                 a.wait_budget);
            if (ok) {
                float ss = 0.f, dot = 0.f;
#pragma unroll
                for (int q = 0; q < CL; ++q) {  // rank order
                    const float2 c = cred[p * CL + q];
                    ss += c.x;
                    dot += c.y;
                }
                const float r = rsqrtf(ss * inv_D + eps);
                const float2 rr = make_float2(r, r);
                const float cc = (r * r) * (dot * inv_D);
                const float2 nc2 = make_float2(-cc, -cc);
                const size_t base = (size_t)row * (size_t)NVR + (size_t)vc0;
                const uint4 *r0 = reinterpret_cast<const uint4 *>(stage_ptr(sk, 0));
                const uint4 *r1 = reinterpret_cast<const uint4 *>(stage_ptr(sk, NTENS >= 2 ? 1 : 0));
                const uint4 *r2 = reinterpret_cast<const uint4 *>(stage_ptr(sk, NTENS - 1));
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int vi = tid + j * NT;
                    if (vi < NVS) {
                        float2 xj[VP], gj[VP], o[VP];
                        unpack_vec<T>(r0[vi], xj);
                        if constexpr (NTENS >= 2) unpack_vec<T>(r1[vi], gj);
                        if constexpr (VJP) {
#pragma unroll
                            for (int q = 0; q < VP; ++q) {
                                const float2 u = f2mul(gj[q], wp[j][q]);              // g w'
                                o[q] = f2mul(f2fma(xj[q], nc2, u), rr);                // r (g w' - x c)
                                acc[j][q] = f2fma(gj[q], f2mul(xj[q], rr), acc[j][q]);  // g x r
                            }
                            if constexpr (ADD) {
                                float2 gr[VP];
                                unpack_vec<T>(r2[vi], gr);
#pragma unroll
                                for (int q = 0; q < VP; ++q) o[q] = f2add(o[q], gr[q]);
                            }
                        } else {
                            if constexpr (MODE == MODE_FWD_RES) {
#pragma unroll
                                for (int q = 0; q < VP; ++q) xj[q] = f2add(xj[q], gj[q]);  // h
                                st_global(out1 + base + vi, pack_vec<T>(xj));
                            }
#pragma unroll
                            for (int q = 0; q < VP; ++q) o[q] = f2mul(f2mul(xj[q], rr), wp[j][q]);
                        }
                        st_global(out0 + base + vi, pack_vec<T>(o));
                    }
                }
            }
        }
    }
    } else {
    // PIPE = false: row k's sums, the exchange and its outputs in one
    // iteration; the stage of row k-1 is refilled after iteration k's
    // barrier, so three stages suffice (and slices of four vectors a thread
    // fit where four stages of them would not).  The row is held in
    // registers across the exchange, or re-read from its stage when four
    // vectors of x and g would not fit them (the VJP).
    for (int64_t k = 0; k < nk; ++k) {
        const int sk = a_stage;
        const int64_t row = cid + k * ncl;
        const uint4 *r0 = reinterpret_cast<const uint4 *>(stage_ptr(sk, 0));
        const uint4 *r1 = reinterpret_cast<const uint4 *>(stage_ptr(sk, NTENS >= 2 ? 1 : 0));
        const uint4 *r2 = reinterpret_cast<const uint4 *>(stage_ptr(sk, NTENS - 1));
        float2 xa[V][VP], xb[V][VP];
        if (tid == 0) mbar_arrive_expect_tx(&clbar[k & 3], CL * 8);  // row k's CL pairs
        ok = ok && mbar_wait_bounded(&full[sk], a_phase, a.wait_budget);
        next_a();
        float2 s2 = make_float2(0.f, 0.f), d2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            if (vi < NVS) {
                unpack_vec<T>(r0[vi], xa[j]);
                if constexpr (NTENS >= 2) unpack_vec<T>(r1[vi], xb[j]);
                if constexpr (MODE == MODE_FWD_RES) {
#pragma unroll
                    for (int q = 0; q < VP; ++q) xa[j][q] = f2add(xa[j][q], xb[j][q]);
                }
#pragma unroll
                for (int q = 0; q < VP; ++q) s2 = f2fma(xa[j][q], xa[j][q], s2);
                if constexpr (VJP) {
#pragma unroll
                    for (int q = 0; q < VP; ++q) d2 = f2fma(f2mul(xb[j][q], wp[j][q]), xa[j][q], d2);
                }
            }
        }
        const float sa = group_sum<32>(s2.x + s2.y);
        const float sb = VJP ? group_sum<32>(d2.x + d2.y) : 0.f;
        if (lane == 0) red[(k & 1) * NWARPS + warp] = make_float2(sa, sb);
        if (__syncthreads_or(!ok)) break;
        if (tid == 0 && k >= 1 && issued < nk) issue_next();  // into row k-1's stage
        const int p = (int)(k & 3);
        if (warp == 0) {  // the sender, as in the pipelined loop
            const float2 *rb = red + (k & 1) * NWARPS;
            float2 tot = lane < NWARPS ? rb[lane] : make_float2(0.f, 0.f);
            tot.x = group_sum<32>(tot.x);
            if constexpr (VJP) tot.y = group_sum<32>(tot.y);
            if (lane < CL)
                dsmem_store_async_f2(dsmem_addr(&cred[p * CL + rank], (uint32_t)lane), tot,
                                     dsmem_addr(&clbar[p], (uint32_t)lane));
        }
        ok = ok && mbar_wait_cluster_bounded(&clbar[p], (uint32_t)((k >> 2) & 1), a.wait_budget);
        if (ok) {
            float ss = 0.f, dot = 0.f;
#pragma unroll
            for (int q = 0; q < CL; ++q) {
                const float2 c = cred[p * CL + q];
                ss += c.x;
                dot += c.y;
            }
            const float r = rsqrtf(ss * inv_D + eps);
            const float2 rr = make_float2(r, r);
            const float cc = (r * r) * (dot * inv_D);
            const float2 nc2 = make_float2(-cc, -cc);
            const size_t base = (size_t)row * (size_t)NVR + (size_t)vc0;
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = tid + j * NT;
                if (vi < NVS) {
                    float2 o[VP];
                    constexpr bool RELOAD = VJP && V > 2;
                    float2 ra[VP], rbv[VP];
                    const float2 *xj = xa[j], *gj = xb[j];
                    if constexpr (RELOAD) {
                        unpack_vec<T>(r0[vi], ra);
                        unpack_vec<T>(r1[vi], rbv);
                        xj = ra;
                        gj = rbv;
                    }
                    if constexpr (VJP) {
#pragma unroll
                        for (int q = 0; q < VP; ++q) {
                            const float2 u = f2mul(gj[q], wp[j][q]);
                            o[q] = f2mul(f2fma(xj[q], nc2, u), rr);
                            acc[j][q] = f2fma(gj[q], f2mul(xj[q], rr), acc[j][q]);
                        }
                        if constexpr (ADD) {
                            float2 gr[VP];
                            unpack_vec<T>(r2[vi], gr);
#pragma unroll
                            for (int q = 0; q < VP; ++q) o[q] = f2add(o[q], gr[q]);
                        }
                    } else {
                        if constexpr (MODE == MODE_FWD_RES) st_global(out1 + base + vi, pack_vec<T>(xa[j]));
#pragma unroll
                        for (int q = 0; q < VP; ++q) o[q] = f2mul(f2mul(xa[j][q], rr), wp[j][q]);
                    }
                    st_global(out0 + base + vi, pack_vec<T>(o));
                }
            }
        }
    }
    }
    const bool failed = __syncthreads_or(!ok);
    if (failed) {
        // Timeout: flag it and drain this CTA's copies still in flight.
        if (tid == 0) {
            atomicOr(a.status, DEVSTATUS_WAIT_TIMEOUT);
            for (int64_t kk = max((int64_t)0, issued - S); kk < issued; ++kk) {
                if ((cid + kk * ncl) * CL + rank == a.drop_tile) continue;
                mbar_wait_bounded(&full[kk % S], (uint32_t)((kk / S) & 1), DEFAULT_WAIT_BUDGET);
            }
        }
    } else {
        griddep_launch_dependents();
        if constexpr (VJP) {
            float *prow = a.partials + (size_t)cid * D + c0;  // the cluster's partial row
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int vi = tid + j * NT;
                if (vi < NVS) {
                    float4 *dst = reinterpret_cast<float4 *>(prow + (size_t)vi * EPV);
#pragma unroll
                    for (int u = 0; u < VP / 2; ++u)
                        dst[u] = make_float4(acc[j][2 * u].x, acc[j][2 * u].y, acc[j][2 * u + 1].x,
                                             acc[j][2 * u + 1].y);
                }
            }
        }
    }
    // Leave only when every CTA of the cluster is leaving, so that no remote
    // write can still reach this CTA's shared memory (a bounded handshake on
    // an mbarrier, not the hardware cluster barrier: a CTA that gave up
    // early still lets the others go).
    __syncthreads();  // every thread is done with this CTA's part of the cluster's work
    if (tid < CL) mbar_arrive_remote(dsmem_addr(xbar, (uint32_t)tid));
    if (!mbar_wait_cluster_bounded(xbar, 0, a.wait_budget) && tid == 0)
        atomicOr(a.status, DEVSTATUS_WAIT_TIMEOUT);
}

}  // namespace rmsn
