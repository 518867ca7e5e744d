// staged_f16_sh.cu -- fp16 instances of the staged kernels for shifted rows
// (dense rows whose tensors share one offset from a 16-byte boundary).
#include "launch_staged.cuh"

namespace rmsn {
cudaError_t launch_staged_f16_sh(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_staged_t<__half, true>(mode, p, a, s);
}
}  // namespace rmsn
