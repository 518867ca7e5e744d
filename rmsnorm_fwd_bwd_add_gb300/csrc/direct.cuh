// direct.cuh -- RMSNorm kernels that load rows straight into registers, one
// CTA per row (grid-stride over rows).
//
// Used for decode-sized problems (a few rows, where a staging ring has
// nothing to overlap and latency is all that matters: every thread issues its
// 16-byte loads at once) and for aligned rows too long for the shared-memory
// ring.  Each thread owns V 16-byte vectors of the row (eight fp16/bf16 or
// four fp32 elements each, fixed across rows); the sum of squares is a warp shuffle tree plus the warp totals added
// in warp order through shared memory.  The VJP keeps its gw contributions in
// registers and writes one partial row per CTA -- or, launched as one
// thread-block cluster of a decode step's rows (CGW), sums the CTAs'
// contributions itself: each CTA leaves its row's contribution in its shared
// memory, and after the cluster barrier each CTA adds, for its share of the
// columns, every CTA's contribution in rank order (distributed shared memory)
// and writes gw; a second cluster barrier keeps every contribution in place
// until all are read.  One kernel per decode VJP, with no scratch.
//
// Sources: "Fused residual-add RMSNorm and fused RoPE + KV-append decode
// kernels", Background (FusedAddRMSNorm; the decode loop runs it once per
// token); "RMSNormVJP backward writes a full {n_rows, D} gw_temp
// intermediate", Proposed changes (gw reduced inside the kernel).
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rmsn {

template <typename T, int MODE, int NT, int V, bool CGW = false>
__global__ void __launch_bounds__(NT) direct_kernel(const KernelArgs a) {
    constexpr int NWARPS = NT / 32;
    constexpr int NTENS = input_tensors(MODE);
    constexpr bool VJP = is_vjp(MODE);
    constexpr bool ADD = (MODE == MODE_VJP_ADD);
    constexpr int E = vec_elems<T>();
    __shared__ float red[2][NWARPS][2];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int D = a.D;
    const int NV = D / E;
    const float eps = a.eps;
    const float wb = a.weight_bias;
    const float inv_D = 1.0f / (float)D;  // per-row means by product
    const uint4 *in0 = static_cast<const uint4 *>(a.in0);
    const uint4 *in1 = static_cast<const uint4 *>(a.in1);
    const uint4 *in2 = static_cast<const uint4 *>(a.in2);
    const uint4 *wg = static_cast<const uint4 *>(a.w);
    uint4 *out0 = static_cast<uint4 *>(a.out0);
    uint4 *out1 = static_cast<uint4 *>(a.out1);

    float acc[VJP ? V : 1][E];
#pragma unroll
    for (int j = 0; j < (VJP ? V : 1); ++j)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[j][e] = 0.f;
    // Row strides in vectors.
    const int64_t l0 = a.ld_in0 / E, l1 = a.ld_in1 / E, l2 = a.ld_in2 / E;
    const int64_t lo0 = a.ld_out0 / E, lo1 = a.ld_out1 / E;

    griddep_wait();  // programmatic dependent: no global access before this
    int it = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, ++it) {
        const float r_saved = (VJP && a.rstd) ? __ldg(a.rstd + row) : 0.f;
        uint4 v0[V], v1[V], v2[ADD ? V : 1];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            if (vi < NV) {
                v0[j] = ld_stream(in0 + row * l0 + vi);
                if constexpr (NTENS >= 2) v1[j] = ld_stream(in1 + row * l1 + vi);
                if constexpr (ADD) v2[j] = ld_stream(in2 + row * l2 + vi);
            }
        }
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            if (vi < NV) {
                float f0[E];
                unpack_vec<T>(v0[j], f0);
                if constexpr (MODE == MODE_FWD_RES) {
                    float f1[E];
                    unpack_vec<T>(v1[j], f1);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float h = f0[e] + f1[e];
                        sa += h * h;
                    }
                } else if constexpr (MODE == MODE_FWD_NORES) {
#pragma unroll
                    for (int e = 0; e < E; ++e) sa += f0[e] * f0[e];
                } else {
                    float f1[E], wf[E];
                    unpack_vec<T>(v1[j], f1);
                    unpack_vec<T>(__ldg(wg + vi), wf);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        sa += f0[e] * f0[e];
                        sb += (f1[e] * (wb + wf[e])) * f0[e];
                    }
                }
            }
        }
        sa = group_sum<32>(sa);
        if constexpr (VJP) sb = group_sum<32>(sb);
        if (lane == 0) {
            red[it & 1][warp][0] = sa;
            red[it & 1][warp][1] = sb;
        }
        __syncthreads();
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) {
            ss += red[it & 1][w][0];
            if constexpr (VJP) dot += red[it & 1][w][1];
        }
        float r = rsqrtf(ss * inv_D + eps);
        if constexpr (VJP) {
            if (a.rstd) r = r_saved;
        } else {
            if (a.rstd && tid == 0) a.rstd[row] = r;
        }
        const float c = (r * r) * (dot * inv_D);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            if (vi < NV) {
                float f0[E], wf[E], o[E];
                unpack_vec<T>(v0[j], f0);
                unpack_vec<T>(__ldg(wg + vi), wf);
                if constexpr (MODE == MODE_FWD_RES) {
                    float f1[E];
                    unpack_vec<T>(v1[j], f1);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        f0[e] = f0[e] + f1[e];
                        o[e] = (f0[e] * r) * (wb + wf[e]);
                    }
                    st_global(out1 + row * lo1 + vi, pack_vec<T>(f0));
                } else if constexpr (MODE == MODE_FWD_NORES) {
#pragma unroll
                    for (int e = 0; e < E; ++e) o[e] = (f0[e] * r) * (wb + wf[e]);
                } else {
                    float f1[E];
                    unpack_vec<T>(v1[j], f1);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float gwp = f1[e] * (wb + wf[e]);
                        o[e] = r * (gwp - f0[e] * c);
                        acc[j][e] += (f1[e] * f0[e]) * r;
                    }
                    if constexpr (ADD) {
                        float f2[E];
                        unpack_vec<T>(v2[j], f2);
#pragma unroll
                        for (int e = 0; e < E; ++e) o[e] = o[e] + f2[e];  // + g_new_residual
                    }
                }
                st_global(out0 + row * lo0 + vi, pack_vec<T>(o));
            }
        }
    }

    griddep_launch_dependents();
    if constexpr (VJP && CGW) {
        // One row per CTA, gridDim.x CTAs in one cluster: gw = the sum of the
        // CTAs' contributions, in rank order, written to a.partials (gw).
        extern __shared__ __align__(16) float part[];  // [D]
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            if (vi < NV) {
#pragma unroll
                for (int u = 0; u < E / 4; ++u)
                    reinterpret_cast<float4 *>(part + (size_t)vi * E)[u] = make_float4(
                        acc[j][4 * u], acc[j][4 * u + 1], acc[j][4 * u + 2], acc[j][4 * u + 3]);
            }
        }
        cluster_sync_all();  // every CTA's contribution is in place and visible
        const int ncta = (int)gridDim.x;
        const int rank = (int)cluster_rank();
        for (int q4 = rank * NT + tid; q4 < D / 4; q4 += ncta * NT) {
            float4 s = dsmem_load_f4(dsmem_addr(part + 4 * q4, 0u));
            for (int c = 1; c < ncta; ++c) {
                const float4 t = dsmem_load_f4(dsmem_addr(part + 4 * q4, (uint32_t)c));
                s = make_float4(s.x + t.x, s.y + t.y, s.z + t.z, s.w + t.w);
            }
            reinterpret_cast<float4 *>(a.partials)[q4] = s;
        }
        cluster_sync_all();  // no CTA leaves while another may still read its part[]
    } else if constexpr (VJP) {
        float *prow = a.partials + (size_t)blockIdx.x * D;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int vi = tid + j * NT;
            if (vi < NV) {
                float4 *dst = reinterpret_cast<float4 *>(prow + (size_t)vi * E);
#pragma unroll
                for (int u = 0; u < E / 4; ++u)
                    dst[u] = make_float4(acc[j][4 * u], acc[j][4 * u + 1], acc[j][4 * u + 2],
                                         acc[j][4 * u + 3]);
            }
        }
    }
}

}  // namespace rmsn
