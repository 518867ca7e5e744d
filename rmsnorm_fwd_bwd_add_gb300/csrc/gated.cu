// gated.cu -- the decode loop's gated activation, out = silu(a) * b with
// a = x[:, :d] and b = x[:, d:2d] of each row ("Fused residual-add RMSNorm and
// fused RoPE + KV-append decode kernels", Background, third bullet: a fused
// gate with 16-byte vectorised loads).
//
// Element-wise and HBM-bound: 2*d values read and d written per row, no
// reduction.  The vectorised kernel gives each thread one 16-byte column of
// the output (8 values) and walks the rows in steps of the grid's height with
// four rows in flight (eight 16-byte loads per thread).  silu(a) = a / (1 +
// e^-a) in fp32 (SFU exponential and reciprocal), the product rounded once.  Other shapes and alignments
// take an element-wise kernel.
#include "rmsnorm.h"

#include <algorithm>

#include "common.cuh"
#include "launch_util.h"

namespace rmsn {
int current_sm_count(int *sm);
int record_cuda_error(cudaError_t e);
}  // namespace rmsn

namespace {

using namespace rmsn;

constexpr int GATE_NT = 256;
constexpr int GATE_ROWS_IN_FLIGHT = 4;
constexpr int GATE_CTAS_PER_SM = 4;  // registers capped at 64 so four fit

// silu(a) = a / (1 + e^-a) with the SFU's exponential and reciprocal
// (__expf, __fdividef: a few ulp, far inside the fp16/bf16 rounding of the
// output); the full-precision expf and division left the vectorised kernel
// issue-bound at 85 % of the copy bandwidth.  For a < -87 the divisor
// overflows and the result is 0 (the true value is below 1e-36 in magnitude).
__device__ __forceinline__ float silu(float a) { return __fdividef(a, 1.f + __expf(-a)); }

template <typename T>
__global__ void __launch_bounds__(GATE_NT, GATE_CTAS_PER_SM) gated_silu_vec_kernel(const uint4 *x, uint4 *out,
                                                                 int64_t rows, int nv) {
    constexpr int U = GATE_ROWS_IN_FLIGHT;
    griddep_wait();
    const int c = blockIdx.x * GATE_NT + threadIdx.x;  // 16-byte column of the output
    if (c < nv) {
        const int64_t step = gridDim.y;
        for (int64_t r0 = blockIdx.y; r0 < rows; r0 += step * U) {
            uint4 va[U], vb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t r = r0 + u * step;
                if (r < rows) {
                    const uint4 *row = x + r * 2 * nv;
                    va[u] = ld_stream(row + c);
                    vb[u] = ld_stream(row + nv + c);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t r = r0 + u * step;
                if (r < rows) {
                    float2 a[4], b[4], o[4];
                    unpack8<T>(va[u], a);
                    unpack8<T>(vb[u], b);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        o[q] = make_float2(silu(a[q].x) * b[q].x, silu(a[q].y) * b[q].y);
                    st_global(out + r * nv + c, pack8<T>(o));
                }
            }
        }
    }
    griddep_launch_dependents();
}

template <typename T>
__global__ void __launch_bounds__(GATE_NT) gated_silu_any_kernel(const T *x, T *out, int64_t rows,
                                                                 int64_t d) {
    griddep_wait();
    const int64_t n = rows * d;
    for (int64_t i = (int64_t)blockIdx.x * GATE_NT + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * GATE_NT) {
        const int64_t r = i / d, j = i - r * d;
        const float a = Cvt<T>::load1(x + r * 2 * d + j);
        const float b = Cvt<T>::load1(x + r * 2 * d + d + j);
        Cvt<T>::store1(out + i, silu(a) * b);
    }
    griddep_launch_dependents();
}

template <typename T>
cudaError_t launch_gated(const void *x, void *out, int64_t rows, int64_t d, int sm_count,
                         cudaStream_t s) {
    const bool vec = d % 8 == 0 && ((uintptr_t)x & 15u) == 0 && ((uintptr_t)out & 15u) == 0 &&
                     d / 8 <= INT32_MAX;
    if (vec) {
        const int nv = (int)(d / 8);
        const unsigned gx = (unsigned)((nv + GATE_NT - 1) / GATE_NT);
        // one resident wave: GATE_CTAS_PER_SM CTAs per SM
        const int64_t want = std::max<int64_t>(1, (int64_t)sm_count * GATE_CTAS_PER_SM / gx);
        const unsigned gy = (unsigned)std::min<int64_t>({rows, want, 65535});
        return launch_pdl(gated_silu_vec_kernel<T>, dim3(gx, gy), dim3(GATE_NT), 0, s,
                          static_cast<const uint4 *>(x), static_cast<uint4 *>(out), rows, nv);
    }
    const int64_t blocks = std::min<int64_t>((rows * d + GATE_NT - 1) / GATE_NT, (int64_t)sm_count * 8);
    return launch_pdl(gated_silu_any_kernel<T>, dim3((unsigned)blocks), dim3(GATE_NT), 0, s,
                      static_cast<const T *>(x), static_cast<T *>(out), rows, d);
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" int rmsnorm_gated_silu(const void *x, void *out, int64_t rows, int64_t d, int dtype,
                                  void *stream) {
    if (dtype != RMSNORM_F16 && dtype != RMSNORM_BF16) return RMSNORM_ERR_INVALID_ARG;
    if (rows < 0 || d <= 0) return RMSNORM_ERR_INVALID_ARG;
    if (d > RMSNORM_MAX_D || rows > INT64_MAX / (4 * d)) return RMSNORM_ERR_UNSUPPORTED;
    if (rows == 0) return RMSNORM_OK;
    if (!x || !out) return RMSNORM_ERR_INVALID_ARG;
    if (ranges_overlap(x, (size_t)rows * (size_t)d * 4, out, (size_t)rows * (size_t)d * 2))
        return RMSNORM_ERR_INVALID_ARG;
    int sm = 0;
    const int st = current_sm_count(&sm);
    if (st != RMSNORM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == RMSNORM_F16 ? launch_gated<__half>(x, out, rows, d, sm, s)
                                               : launch_gated<__nv_bfloat16>(x, out, rows, d, sm, s);
    return e == cudaSuccess ? RMSNORM_OK : record_cuda_error(e);
}
