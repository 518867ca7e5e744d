// gw_fused.cuh -- the gw stage-2 sum folded into the VJP kernel.
//
// Every CTA of a VJP launch writes one partial row partials[b, :].  With the
// two-kernel scheme a second kernel then sums the P rows; here the CTAs of the
// same (cooperative, hence co-resident) launch do it themselves:
//   1. CTA b publishes its row: all its threads have stored it, thread 0
//      fences and writes flags[b] = epoch, a 64-bit value unique to this
//      launch (so flags left over from earlier launches never match and the
//      flags need no clearing);
//   2. warp 0 waits, with a bounded spin, until flags[0..P) all equal epoch;
//   3. the CTA sums its share of 32-column strips: warp w adds a contiguous
//      chunk of the P rows in ascending order, then the chunk sums are added
//      in warp order -- an order fixed by (P, D, NT), never by timing.
// A wait that runs out sets RMSNORM_DEVSTATUS_WAIT_TIMEOUT and leaves gw
// unwritten; nothing hangs.
//
// Source: "RMSNormVJP backward writes a full {n_rows, D} gw_temp
// intermediate", Proposed changes (combine the rows' gw contributions inside
// the kernel instead of a second pass over a {n_rows, D} temporary).
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rmsn {

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_volatile_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Call with every thread of the CTA after the CTA's partial row is stored.
// `scratch` is shared memory for (NT/32) * 33 floats that no thread uses any
// more.
template <int NT>
__device__ __forceinline__ void fused_gw_finish(const KernelArgs &a, float *scratch) {
    constexpr int NWARPS = NT / 32;
    __shared__ int s_all_published;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int P = gridDim.x;
    const int D = a.D;

    __syncthreads();  // this CTA's partial row is written
    if (tid == 0) {
        __threadfence();
        st_volatile_u64(a.flags + blockIdx.x, a.epoch);
    }
    if (warp == 0) {
        bool ok = true;
        const long long t0 = clock64();
        for (int i = lane; i < P && ok; i += 32) {
            while (ld_volatile_u64(a.flags + i) != a.epoch) {
                if (clock64() - t0 > a.wait_budget) {
                    ok = false;
                    break;
                }
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        __threadfence();
        if (lane == 0) s_all_published = ok ? 1 : 0;
    }
    __syncthreads();
    if (!s_all_published) {
        if (tid == 0) atomicOr(a.status, DEVSTATUS_WAIT_TIMEOUT);
        return;
    }

    constexpr int BATCH = 16;
    const int units = (D + 31) / 32;
    const int per = (P + NWARPS - 1) / NWARPS;
    const int p0 = warp * per;
    const int p1 = min(P, p0 + per);
    for (int u = blockIdx.x; u < units; u += P) {
        const int col = u * 32 + lane;
        float s = 0.f;
        if (col < D) {
            for (int b = p0; b < p1; b += BATCH) {
                float v[BATCH];
#pragma unroll
                for (int i = 0; i < BATCH; ++i)  // L2 loads: the rows come from other SMs
                    v[i] = b + i < p1 ? __ldcg(a.partials + (size_t)(b + i) * D + col) : 0.f;
#pragma unroll
                for (int i = 0; i < BATCH; ++i)
                    if (b + i < p1) s += v[i];
            }
        }
        scratch[warp * 33 + lane] = s;
        __syncthreads();
        if (warp == 0 && col < D) {
            float t = scratch[lane];
#pragma unroll
            for (int w = 1; w < NWARPS; ++w) t += scratch[w * 33 + lane];
            a.gw[col] = t;
        }
        __syncthreads();
    }
}

}  // namespace rmsn
