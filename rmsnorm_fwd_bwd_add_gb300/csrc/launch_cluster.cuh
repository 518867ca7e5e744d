// launch_cluster.cuh -- picks the cluster_kernel instance for a plan.
#pragma once

#include "cluster.cuh"
#include "launch_util.h"

namespace rmsn {

// Instances: two vectors a thread up to CLUSTER_NT_V2 threads (slices of up
// to 2 * CLUSTER_NT_V2 vectors), four up to CLUSTER_NT_V4 (up to 2048).
template <typename T, int MODE, int NTMAX, int V, int CL, bool PIPE>
cudaError_t launch_cluster_inst(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    static std::atomic<uint64_t> smem_mask{0};
    auto kern = cluster_kernel<T, MODE, NTMAX, V, CL, PIPE>;
    cudaError_t e = allow_max_dynamic_smem((const void *)kern, smem_mask);
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(kern, dim3(p.grid), dim3(p.nt), p.smem, s, CL, a);
}

template <typename T, int MODE, int NTMAX, int V, bool PIPE>
cudaError_t launch_cluster_cl(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (p.cl) {
        case 2: return launch_cluster_inst<T, MODE, NTMAX, V, 2, PIPE>(p, a, s);
        case 4: return launch_cluster_inst<T, MODE, NTMAX, V, 4, PIPE>(p, a, s);
        case 8: return launch_cluster_inst<T, MODE, NTMAX, V, 8, PIPE>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int MODE>
cudaError_t launch_cluster_mode(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    if (p.nt < 32 || p.nt % 32 != 0) return cudaErrorInvalidValue;
    const bool pipe = p.stages >= 4;  // the plan's choice (see planner.h)
    if (p.v == 2 && p.nt <= CLUSTER_NT_V2)
        return pipe ? launch_cluster_cl<T, MODE, CLUSTER_NT_V2, 2, true>(p, a, s)
                    : launch_cluster_cl<T, MODE, CLUSTER_NT_V2, 2, false>(p, a, s);
    if (p.v == 4 && p.nt <= CLUSTER_NT_V4)
        return pipe ? launch_cluster_cl<T, MODE, CLUSTER_NT_V4, 4, true>(p, a, s)
                    : launch_cluster_cl<T, MODE, CLUSTER_NT_V4, 4, false>(p, a, s);
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_cluster_t(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (mode) {
        case MODE_FWD_RES: return launch_cluster_mode<T, MODE_FWD_RES>(p, a, s);
        case MODE_FWD_NORES: return launch_cluster_mode<T, MODE_FWD_NORES>(p, a, s);
        case MODE_VJP: return launch_cluster_mode<T, MODE_VJP>(p, a, s);
        case MODE_VJP_ADD: return launch_cluster_mode<T, MODE_VJP_ADD>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rmsn
