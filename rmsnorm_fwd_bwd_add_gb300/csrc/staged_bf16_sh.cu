// staged_bf16_sh.cu -- bf16 instances of the staged kernels for shifted rows
// (dense rows whose tensors share one offset from a 16-byte boundary).
#include "launch_staged.cuh"

namespace rmsn {
cudaError_t launch_staged_bf16_sh(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_staged_t<__nv_bfloat16, true>(mode, p, a, s);
}
}  // namespace rmsn
