// cluster_f32.cu -- fp32 instances of the cluster kernels.
#include "launch_cluster.cuh"

namespace rmsn {
cudaError_t launch_cluster_f32(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_cluster_t<float>(mode, p, a, s);
}
}  // namespace rmsn
