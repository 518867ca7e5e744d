// cluster_bf16.cu -- bf16 instances of the cluster kernels.
#include "launch_cluster.cuh"

namespace rmsn {
cudaError_t launch_cluster_bf16(int mode, const Plan &p, const KernelArgs &a, cudaStream_t s) {
    return launch_cluster_t<__nv_bfloat16>(mode, p, a, s);
}
}  // namespace rmsn

namespace rmsn {

// Queried with the bf16 VJP instance of two vectors a thread, at 512 threads and 200 KB of
// shared memory, so that one CTA fills an SM as every cluster plan does.
int cluster_capacity(int cl) {
    constexpr int MAX_DEVICES = 64;
    static std::atomic<int> cache[MAX_DEVICES][9];  // 0: not queried; else capacity + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES || cl < 2 || cl > 8)
        return 0;
    const int got = cache[dev][cl].load();
    if (got) return got - 1;
    const void *kern = nullptr;
    static std::atomic<uint64_t> m2{0}, m4{0}, m8{0};
    std::atomic<uint64_t> *mask = nullptr;
    switch (cl) {
        case 2: kern = (const void *)cluster_kernel<__nv_bfloat16, MODE_VJP, CLUSTER_NT_V2, 2, 2, true>; mask = &m2; break;
        case 4: kern = (const void *)cluster_kernel<__nv_bfloat16, MODE_VJP, CLUSTER_NT_V2, 2, 4, true>; mask = &m4; break;
        case 8: kern = (const void *)cluster_kernel<__nv_bfloat16, MODE_VJP, CLUSTER_NT_V2, 2, 8, true>; mask = &m8; break;
        default: cache[dev][cl].store(1); return 0;
    }
    int n = 0;
    if (allow_max_dynamic_smem(kern, *mask) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned int)(cl * 64));
        cfg.blockDim = dim3(512);
        cfg.dynamicSmemBytes = 200 * 1024;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned int)cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
    } else {
        (void)cudaGetLastError();
    }
    cache[dev][cl].store(n + 1);
    return n;
}

}  // namespace rmsn
