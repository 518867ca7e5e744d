// generic.cuh -- element-at-a-time RMSNorm kernels for any D and any
// alignment (rows whose start is not 16-byte aligned, D not a multiple of 8,
// or rows longer than the vectorised tiers take), and the gw stage-2 sum.
//
// One CTA per row, grid-stride; pass 1 forms the sums, pass 2 re-reads the row
// (from L1/L2) and writes the outputs.  A thread's share of a row can be long
// (65536 elements at D = 2^24), so its sums are compensated (Neumaier): the
// error of r then stays at a few fp32 roundings at any D instead of growing
// with the row length (a plain running sum left r off by 2e-5 at D = 2^24).  The VJP accumulates each CTA's gw
// contributions in that CTA's own row of the partials buffer; thread t owns
// columns t, t + NT, ..., so no two threads ever touch the same partial and
// the order is fixed.
//
// Sources: as for the vectorised tiers ("Fused residual-add RMSNorm and fused
// RoPE + KV-append decode kernels", Background; "RMSNormVJP backward writes a
// full {n_rows, D} gw_temp intermediate", Proposed changes).
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rmsn {

// s + v into (s, c): s the running sum, c the running rounding error of it.
__device__ __forceinline__ void neumaier_add(float &s, float &c, float v) {
    const float t = __fadd_rn(s, v);
    c = __fadd_rn(c, fabsf(s) >= fabsf(v) ? __fadd_rn(__fsub_rn(s, t), v)
                                          : __fadd_rn(__fsub_rn(v, t), s));
    s = t;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(GENERIC_NT) generic_kernel(const KernelArgs a) {
    constexpr int NT = GENERIC_NT;
    constexpr int NWARPS = NT / 32;
    constexpr bool VJP = is_vjp(MODE);
    constexpr bool ADD = (MODE == MODE_VJP_ADD);
    __shared__ float red[2][NWARPS][2];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int D = a.D;
    const float eps = a.eps;
    const float wb = a.weight_bias;
    const float inv_D = 1.0f / (float)D;  // per-row means by product
    const T *in0 = static_cast<const T *>(a.in0);
    const T *in1 = static_cast<const T *>(a.in1);
    const T *in2 = static_cast<const T *>(a.in2);
    const T *w = static_cast<const T *>(a.w);
    T *out0 = static_cast<T *>(a.out0);
    T *out1 = static_cast<T *>(a.out1);
    float *prow = VJP ? a.partials + (size_t)blockIdx.x * D : nullptr;
    const int64_t l0 = a.ld_in0, l1 = a.ld_in1, l2 = a.ld_in2, lo0 = a.ld_out0, lo1 = a.ld_out1;

    griddep_wait();  // programmatic dependent: no global access before this
    if constexpr (VJP)
        for (int c = tid; c < D; c += NT) prow[c] = 0.f;

    int it = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, ++it) {
        const T *x_row = in0 + row * l0;
        const T *y_row = in1 + row * l1;  // residual or g
        float sa = 0.f, sb = 0.f, ca = 0.f, cb = 0.f;
        for (int c = tid; c < D; c += NT) {
            const float x = Cvt<T>::load1(x_row + c);
            if constexpr (MODE == MODE_FWD_RES) {
                const float h = x + Cvt<T>::load1(y_row + c);
                neumaier_add(sa, ca, __fmul_rn(h, h));
            } else if constexpr (MODE == MODE_FWD_NORES) {
                neumaier_add(sa, ca, __fmul_rn(x, x));
            } else {
                const float g = Cvt<T>::load1(y_row + c);
                neumaier_add(sa, ca, __fmul_rn(x, x));
                neumaier_add(sb, cb, __fmul_rn(__fmul_rn(g, wb + Cvt<T>::load1(w + c)), x));
            }
        }
        sa += ca;
        sb += cb;
        sa = group_sum<32>(sa);
        if constexpr (VJP) sb = group_sum<32>(sb);
        if (lane == 0) {
            red[it & 1][warp][0] = sa;
            red[it & 1][warp][1] = sb;
        }
        __syncthreads();
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int k = 0; k < NWARPS; ++k) {
            ss += red[it & 1][k][0];
            if constexpr (VJP) dot += red[it & 1][k][1];
        }
        float r = rsqrtf(ss * inv_D + eps);
        if constexpr (VJP) {
            if (a.rstd) r = a.rstd[row];
        } else {
            if (a.rstd && tid == 0) a.rstd[row] = r;
        }
        const float cc = (r * r) * (dot * inv_D);
        T *o_row = out0 + row * lo0;
        for (int c = tid; c < D; c += NT) {
            const float x = Cvt<T>::load1(x_row + c);
            const float wp = wb + Cvt<T>::load1(w + c);
            if constexpr (MODE == MODE_FWD_RES) {
                const float h = x + Cvt<T>::load1(y_row + c);
                Cvt<T>::store1(out1 + row * lo1 + c, h);
                Cvt<T>::store1(o_row + c, (h * r) * wp);
            } else if constexpr (MODE == MODE_FWD_NORES) {
                Cvt<T>::store1(o_row + c, (x * r) * wp);
            } else {
                const float g = Cvt<T>::load1(y_row + c);
                float o = r * (g * wp - x * cc);
                if constexpr (ADD) o = o + Cvt<T>::load1(in2 + row * l2 + c);  // + g_new_residual
                Cvt<T>::store1(o_row + c, o);
                prow[c] += (g * x) * r;
            }
        }
    }
    griddep_launch_dependents();
}

// Stage 2 of gw: gw[c] = sum over p of partials[p, c].  A CTA covers 32
// columns with GWR_CHUNKS warps; warp k adds the k-th contiguous chunk of the
// P partial rows in ascending order, then warp 0 adds the chunk sums in warp
// order.  The order depends only on (P, D), never on timing.  Each thread
// issues up to GWR_BATCH loads before its first add, so a chunk costs one
// L2 round trip.  Launched as a programmatic dependent of the VJP kernel that
// wrote the partials.
constexpr int GWR_CHUNKS = 32;
constexpr int GWR_BATCH = 16;

__global__ void __launch_bounds__(32 * GWR_CHUNKS) gw_reduce_kernel(
    const float *__restrict__ partials, float *__restrict__ gw, int P, int D) {
    __shared__ float part[GWR_CHUNKS][33];
    griddep_wait();
    griddep_launch_dependents();
    const int tx = threadIdx.x & 31;
    const int ty = threadIdx.x >> 5;
    const int64_t col = (int64_t)blockIdx.x * 32 + tx;
    const int per = (P + GWR_CHUNKS - 1) / GWR_CHUNKS;
    const int p0 = ty * per;
    const int p1 = min(P, p0 + per);
    float s = 0.f;
    if (col < D) {
        for (int b = p0; b < p1; b += GWR_BATCH) {
            float v[GWR_BATCH];
#pragma unroll
            for (int i = 0; i < GWR_BATCH; ++i)
                v[i] = b + i < p1 ? partials[(size_t)(b + i) * D + col] : 0.f;
#pragma unroll
            for (int i = 0; i < GWR_BATCH; ++i)
                if (b + i < p1) s += v[i];
        }
    }
    part[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && col < D) {
        float t = part[0][tx];
#pragma unroll
        for (int k = 1; k < GWR_CHUNKS; ++k) t += part[k][tx];
        gw[col] = t;
    }
}

}  // namespace rmsn
