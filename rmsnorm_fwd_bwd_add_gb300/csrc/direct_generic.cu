// direct_generic.cu -- launchers for the direct and generic tiers, the gw
// stage-2 reduction, and the dtype switch of the staged tier.
#include "direct.cuh"
#include "generic.cuh"
#include "launch_util.h"

namespace rmsn {

cudaError_t launch_staged_f16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_staged_bf16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_staged_f32(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_staged_f16_sh(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_staged_bf16_sh(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_staged_f32_sh(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);

cudaError_t launch_staged(int dtype, int mode, const Plan &p, const KernelArgs &a,
                          cudaStream_t s) {
    if (p.shift) {
        switch (dtype) {
            case 0: return launch_staged_f16_sh(mode, p, a, s);
            case 1: return launch_staged_bf16_sh(mode, p, a, s);
            case 2: return launch_staged_f32_sh(mode, p, a, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (dtype) {
        case 0: return launch_staged_f16(mode, p, a, s);
        case 1: return launch_staged_bf16(mode, p, a, s);
        case 2: return launch_staged_f32(mode, p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

template <typename T, int MODE, int NT, int V>
cudaError_t direct_one(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    if constexpr (is_vjp(MODE)) {
        if (p.cl > 1) {  // a decode step's rows as one cluster that sums gw itself
            static std::atomic<uint64_t> smem_mask{0};
            auto kern = direct_kernel<T, MODE, NT, V, true>;
            cudaError_t e = allow_max_dynamic_smem((const void *)kern, smem_mask);
            if (e != cudaSuccess) return e;
            return launch_pdl_cluster(kern, dim3(p.grid), dim3(NT), p.smem, s, p.cl, a);
        }
    }
    return launch_pdl(direct_kernel<T, MODE, NT, V>, dim3(p.grid), dim3(NT), 0, s, a);
}

template <typename T, int MODE>
cudaError_t direct_mode(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    static_assert(N_DIRECT_CFG == 6, "keep this switch in step with DIRECT_CFGS");
    switch (p.cfg) {
        case 0: return direct_one<T, MODE, 128, 1>(p, a, s);
        case 1: return direct_one<T, MODE, 256, 1>(p, a, s);
        case 2: return direct_one<T, MODE, 512, 1>(p, a, s);
        case 3: return direct_one<T, MODE, 512, 2>(p, a, s);  // measured: 1024 x 1 is 0.35 us slower
        case 4: return direct_one<T, MODE, 1024, 2>(p, a, s);
        case 5:
            // Four vectors of x and g per thread plus gw accumulators do not
            // fit 1024 threads' registers; the VJP never plans this config.
            if constexpr (is_vjp(MODE)) return cudaErrorInvalidValue;
            else return direct_one<T, MODE, 1024, 4>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t direct_t(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (mode) {
        case MODE_FWD_RES: return direct_mode<T, MODE_FWD_RES>(p, a, s);
        case MODE_FWD_NORES: return direct_mode<T, MODE_FWD_NORES>(p, a, s);
        case MODE_VJP: return direct_mode<T, MODE_VJP>(p, a, s);
        case MODE_VJP_ADD: return direct_mode<T, MODE_VJP_ADD>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t generic_t(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    const dim3 grid(p.grid), block(GENERIC_NT);
    switch (mode) {
        case MODE_FWD_RES:
            return launch_pdl(generic_kernel<T, MODE_FWD_RES>, grid, block, 0, s, a);
        case MODE_FWD_NORES:
            return launch_pdl(generic_kernel<T, MODE_FWD_NORES>, grid, block, 0, s, a);
        case MODE_VJP: return launch_pdl(generic_kernel<T, MODE_VJP>, grid, block, 0, s, a);
        case MODE_VJP_ADD: return launch_pdl(generic_kernel<T, MODE_VJP_ADD>, grid, block, 0, s, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_direct(int dtype, int mode, const Plan &p, const KernelArgs &a,
                          cudaStream_t s) {
    switch (dtype) {
        case 0: return direct_t<__half>(mode, p, a, s);
        case 1: return direct_t<__nv_bfloat16>(mode, p, a, s);
        case 2: return direct_t<float>(mode, p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_generic(int dtype, int mode, const Plan &p, const KernelArgs &a,
                           cudaStream_t s) {
    switch (dtype) {
        case 0: return generic_t<__half>(mode, p, a, s);
        case 1: return generic_t<__nv_bfloat16>(mode, p, a, s);
        case 2: return generic_t<float>(mode, p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_cluster_f16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_cluster_bf16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);
cudaError_t launch_cluster_f32(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s);

cudaError_t launch_cluster(int dtype, int mode, const Plan &p, const KernelArgs &a,
                           cudaStream_t s) {
    switch (dtype) {
        case 0: return launch_cluster_f16(mode, p, a, s);
        case 1: return launch_cluster_bf16(mode, p, a, s);
        case 2: return launch_cluster_f32(mode, p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gw_reduce(const float *partials, float *gw, int P, int D, cudaStream_t s) {
    return launch_pdl(gw_reduce_kernel, dim3((unsigned int)((D + 31) / 32)), dim3(32 * GWR_CHUNKS),
                      0, s, partials, gw, P, D);
}

}  // namespace rmsn
