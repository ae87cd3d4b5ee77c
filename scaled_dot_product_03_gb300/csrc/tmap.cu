// tmap.cu -- TMA tensor-map encoding through the driver entry point (no
// link-time dependency on libcuda).
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "tmap.h"

namespace gbattn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

thread_local std::string t_refusal;

cudaError_t refused(CUresult r, int rank, const cuuint64_t *dims, const cuuint64_t *strides) {
    char buf[256];
    int n = snprintf(buf, sizeof buf, "driver error %d for dims (", (int)r);
    for (int i = 0; i < rank; ++i) n += snprintf(buf + n, sizeof buf - n, i ? ", %llu" : "%llu", (unsigned long long)dims[i]);
    n += snprintf(buf + n, sizeof buf - n, "), byte strides (");
    for (int i = 0; i + 1 < rank; ++i)
        n += snprintf(buf + n, sizeof buf - n, i ? ", %llu" : "%llu", (unsigned long long)strides[i]);
    snprintf(buf + n, sizeof buf - n, ")");
    t_refusal = buf;
    return kTmapRefused;
}

}  // namespace

const char *tmap_refusal() { return t_refusal.c_str(); }

cudaError_t make_tmap_16bit(CUtensorMap *map, const void *ptr, int dtype, const uint64_t dims[4],
                            const uint64_t strides_bytes[3], uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gstride[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t box[4] = {64, box_rows, 1, 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    4, const_cast<void *>(ptr), gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : refused(r, 4, gdim, gstride);
}

cudaError_t make_tmap_f32_acc(CUtensorMap *map, void *ptr, uint64_t cols, uint64_t rows, uint64_t heads,
                              uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (box_cols * 4 != 128) return cudaErrorInvalidValue;
    cuuint64_t gdim[3] = {cols, rows, heads};
    cuuint64_t gstride[2] = {cols * 4, rows * cols * 4};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, gdim, gstride, box, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : refused(r, 3, gdim, gstride);
}

}  // namespace gbattn
