// staged_bf16.cu -- bf16 instances of the staged kernels.
#include "launch_staged.cuh"

namespace rmsn {
cudaError_t launch_staged_bf16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_staged_t<__nv_bfloat16, false>(mode, p, a, s);
}
}  // namespace rmsn
