// launch_cluster.cuh -- picks the cluster_kernel instance for a plan.
#pragma once

#include "cluster.cuh"
#include "launch_util.h"

namespace rmsn {

template <typename T, int MODE, int NT, int V, int CL, bool PIPE>
cudaError_t launch_cluster_inst(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    static std::atomic<uint64_t> smem_mask{0};
    auto kern = cluster_kernel<T, MODE, NT, V, CL, PIPE>;
    cudaError_t e = allow_max_dynamic_smem((const void *)kern, smem_mask);
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(kern, dim3(p.grid), dim3(NT), p.smem, s, CL, a);
}

template <typename T, int MODE, int V, bool PIPE>
cudaError_t launch_cluster_cl(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (p.cl) {
        case 2: return launch_cluster_inst<T, MODE, CLUSTER_NT, V, 2, PIPE>(p, a, s);
        case 4: return launch_cluster_inst<T, MODE, CLUSTER_NT, V, 4, PIPE>(p, a, s);
        case 8: return launch_cluster_inst<T, MODE, CLUSTER_NT, V, 8, PIPE>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int MODE>
cudaError_t launch_cluster_mode(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    if (p.nt != CLUSTER_NT) return cudaErrorInvalidValue;
    const bool pipe = p.stages >= 4;  // the plan's choice (see planner.h)
    switch (p.v) {
        case 2: return pipe ? launch_cluster_cl<T, MODE, 2, true>(p, a, s)
                            : launch_cluster_cl<T, MODE, 2, false>(p, a, s);
        case 4: return pipe ? launch_cluster_cl<T, MODE, 4, true>(p, a, s)
                            : launch_cluster_cl<T, MODE, 4, false>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
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
