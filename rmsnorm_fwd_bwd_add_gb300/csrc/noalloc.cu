// noalloc.cu -- rmsnorm_vjp_noalloc: the RMSNorm VJP for callers that must not
// allocate device memory.
//
// Some programs cannot call cudaMalloc (or any allocator) at the point where
// they run the backward pass: serving and training runtimes that reserve the
// device's memory once at start-up and treat any later allocation as an
// error, plugin interfaces that hand a kernel its tensors but neither an
// allocator nor a workspace, and code that must not take the implicit
// synchronisation or the failure modes of an allocation inside a
// latency-critical loop.  rmsnorm_vjp takes its gw scratch from a pool and
// rmsnorm_vjp_ws needs the caller to allocate it; this entry point instead uses
// a fixed array compiled into the library, so the caller passes only its inputs
// and outputs.
//
// The array lives in device memory of every GPU on which the library's module
// is loaded, from load until the process exits.  On the host its name is only a
// stand-in for that memory: the device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and handed to the
// kernels as their partials buffer.
#include <cuda_runtime.h>

#include <mutex>

#include "rmsnorm.h"

namespace rmsn {
size_t vjp_partials_bytes_for(const void *x, const void *w, const void *g, const void *gx,
                              int64_t rows, int64_t D, int dtype);
int record_cuda_error(cudaError_t e);
}  // namespace rmsn

// gw partial rows of rmsnorm_vjp_noalloc, shared by every call on a device.
static __device__ __align__(256) unsigned char g_vjp_noalloc_scratch[RMSNORM_VJP_NOALLOC_MAX_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void *g_scratch_addr[MAX_DEVICES];

// Device address of g_vjp_noalloc_scratch on the current device, looked up on
// the first call for that device.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return rmsn::record_cuda_error(e);
    if (dev < 0 || dev >= MAX_DEVICES) return RMSNORM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress((void **)&ptr, g_vjp_noalloc_scratch);
        if (e != cudaSuccess) return rmsn::record_cuda_error(e);
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return RMSNORM_OK;
}

}  // namespace

extern "C" int rmsnorm_vjp_noalloc(const void *x, const void *w, const void *g, float eps,
                                   float weight_bias, void *gx, float *gw, int64_t rows,
                                   int64_t D, int dtype, void *stream) {
    // Problems whose partial rows do not fit the fixed array are refused
    // before anything is enqueued.  (Invalid arguments size to 0 here and are
    // rejected by the validation of rmsnorm_vjp_ws below.)
    if (rmsn::vjp_partials_bytes_for(x, w, g, gx, rows, D, dtype) > RMSNORM_VJP_NOALLOC_MAX_BYTES)
        return RMSNORM_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != RMSNORM_OK) return st;
    // Every partial row the gw reduction reads is written in full by this
    // call's first kernel, so whatever the previous call left in the array
    // needs no clearing.
    return rmsnorm_vjp_ws(x, w, g, eps, weight_bias, gx, gw, rows, D, dtype, scratch,
                          RMSNORM_VJP_NOALLOC_MAX_BYTES, stream);
}
