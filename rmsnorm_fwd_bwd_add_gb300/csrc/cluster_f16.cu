// cluster_f16.cu -- fp16 instances of the cluster kernels.
#include "launch_cluster.cuh"

namespace rmsn {
cudaError_t launch_cluster_f16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_cluster_t<__half>(mode, p, a, s);
}
}  // namespace rmsn
