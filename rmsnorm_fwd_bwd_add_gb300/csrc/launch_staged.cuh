// launch_staged.cuh -- picks the staged_kernel instance for a plan.
#pragma once

#include "launch_util.h"
#include "staged.cuh"

namespace rmsn {

template <typename T, int MODE, int NT, int G, int V, bool GEN>
cudaError_t launch_staged_inst(const Plan &p, const KernelArgs &a, cudaStream_t stream) {
    constexpr int MINB = staged_max_ctas_per_sm(MODE, NT, G, V);
    static std::atomic<uint64_t> smem_mask{0};
    auto kern = staged_kernel<T, MODE, NT, G, V, MINB, GEN>;
    cudaError_t e = allow_max_dynamic_smem((const void *)kern, smem_mask);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(p.grid), dim3(NT), p.smem, stream, a);
}

// The dense instance unless a tensor the mode uses has rows a stride apart
// or rstd is given.
template <typename T, int MODE, int NT, int G, int V>
cudaError_t launch_staged_one(const Plan &p, const KernelArgs &a, cudaStream_t stream) {
    const int64_t D = a.D;
    bool gen = a.rstd != nullptr || a.ld_in0 != D || a.ld_out0 != D;
    if constexpr (input_tensors(MODE) >= 2) gen = gen || a.ld_in1 != D;
    if constexpr (input_tensors(MODE) == 3) gen = gen || a.ld_in2 != D;
    if constexpr (MODE == MODE_FWD_RES) gen = gen || a.ld_out1 != D;
    return gen ? launch_staged_inst<T, MODE, NT, G, V, true>(p, a, stream)
               : launch_staged_inst<T, MODE, NT, G, V, false>(p, a, stream);
}

template <typename T, int MODE>
cudaError_t launch_staged_mode(const Plan &p, const KernelArgs &a, cudaStream_t s) {
    static_assert(N_STAGED_CFG == 11, "keep this switch in step with STAGED_CFGS");
    switch (p.cfg) {
        case 0: return launch_staged_one<T, MODE, 256, 8, 1>(p, a, s);
        case 1: return launch_staged_one<T, MODE, 256, 16, 1>(p, a, s);
        case 2: return launch_staged_one<T, MODE, 256, 32, 1>(p, a, s);
        case 3: return launch_staged_one<T, MODE, 256, 32, 2>(p, a, s);
        case 4: return launch_staged_one<T, MODE, 256, 32, 3>(p, a, s);
        case 5: return launch_staged_one<T, MODE, 256, 32, 4>(p, a, s);
        case 6: return launch_staged_one<T, MODE, 128, 128, 2>(p, a, s);
        case 7: return launch_staged_one<T, MODE, 256, 256, 2>(p, a, s);
        case 8: return launch_staged_one<T, MODE, 512, 512, 2>(p, a, s);
        case 9: return launch_staged_one<T, MODE, 1024, 1024, 2>(p, a, s);
        case 10:
            if constexpr (is_vjp(MODE)) return cudaErrorInvalidValue;
            else return launch_staged_one<T, MODE, 256, 256, 4>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_staged_t(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    switch (mode) {
        case MODE_FWD_RES: return launch_staged_mode<T, MODE_FWD_RES>(p, a, s);
        case MODE_FWD_NORES: return launch_staged_mode<T, MODE_FWD_NORES>(p, a, s);
        case MODE_VJP: return launch_staged_mode<T, MODE_VJP>(p, a, s);
        case MODE_VJP_ADD: return launch_staged_mode<T, MODE_VJP_ADD>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rmsn
