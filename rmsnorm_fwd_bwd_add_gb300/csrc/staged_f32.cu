// staged_f32.cu -- fp32 instances of the staged kernels.
#include "launch_staged.cuh"

namespace rmsn {
cudaError_t launch_staged_f32(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_staged_t<float, false>(mode, p, a, s);
}
}  // namespace rmsn
