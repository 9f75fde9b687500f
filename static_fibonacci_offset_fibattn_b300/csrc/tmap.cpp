// tmap.cpp -- TMA tensor-map encoding through the driver entry point exposed by the runtime.
#include "tmap.h"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace fibattn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

}  // namespace

namespace {

int make_map(CUtensorMap* m, const void* base, int64_t slices, int32_t T, uint32_t box_rows,
             int32_t d = 64) {
    auto fn = encode_fn();
    if (!fn) return -1;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)slices};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return (int)r;
}

}  // namespace

int make_bf16_rows_map(CUtensorMap* m, const void* base, int64_t slices, int32_t T) {
    return make_map(m, base, slices, T, kTmaBoxRows);
}

int make_bf16_rows_map_d(CUtensorMap* m, const void* base, int64_t slices, int32_t T, int32_t d) {
    return make_map(m, base, slices, T, kTmaBoxRows, d);
}

int make_bf16_rows8_map(CUtensorMap* m, const void* base, int64_t slices, int32_t T) {
    return make_map(m, base, slices, T, 8);
}

}  // namespace fibattn
