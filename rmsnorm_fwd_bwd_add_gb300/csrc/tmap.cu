// tmap.cu -- 2-D TMA tensor maps for the staged kernels' strided tiles.
//
// cuTensorMapEncodeTiled is a driver API entry point; it is fetched once
// through the runtime (cudaGetDriverEntryPointByVersion), so the library
// needs no link against the driver library.
#include <cudaTypedefs.h>

#include <mutex>

#include "plan.h"

namespace rmsn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

}  // namespace

bool encode_rows_tmap(CUtensorMap *map, const void *base, int64_t rows, int64_t D, int64_t ld,
                      int dtype, int box_cols, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || !base) return false;
    const int es = dtype == 2 ? 4 : 2;
    if ((D * es) % 8 || (box_cols * es) % 8) return false;
    // The copy only moves bytes, so the map counts 8-byte units: a box row
    // can then span 256 of them (2 KB) instead of 256 elements.
    const cuuint64_t dims[2] = {(cuuint64_t)(D * es / 8), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};  // bytes between rows
    const cuuint32_t box[2] = {(cuuint32_t)(box_cols * es / 8), (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rmsn
