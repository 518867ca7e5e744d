// staged_f16.cu -- fp16 instances of the staged kernels.
#include "launch_staged.cuh"

namespace rmsn {
cudaError_t launch_staged_f16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_staged_t<__half, false>(mode, p, a, s);
}
}  // namespace rmsn
