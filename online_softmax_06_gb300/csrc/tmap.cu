// tmap.cu -- TMA tensor maps over the [rows, H, d] bf16 tensors of the
// attention kernels (built on the host, passed to kernels as __grid_constant__
// parameters).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "launch.h"

namespace fa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime (the
// library links no driver stub).
EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap *tm, const void *base, int64_t total, int H, int d, int box_rows,
                    int H_row)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    if (H_row <= 0)
        H_row = H;
    const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(H), cuuint64_t(total)};
    const cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(H_row) * d * 2};
    const cuuint32_t box[3] = {64, 1, cuuint32_t(box_rows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_e4m3_rows(CUtensorMap *tm, const void *base, int64_t total, int H, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(H), cuuint64_t(total)};
    const cuuint64_t strides[2] = {cuuint64_t(d), cuuint64_t(H) * d};
    const cuuint32_t box[3] = {cuuint32_t(d), 1, 128};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_seq_4d(CUtensorMap *tm, const void *base, bool e4m3, int B, int N, int H, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const cuuint64_t eb = e4m3 ? 1 : 2;
    const cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(H), cuuint64_t(N), cuuint64_t(B)};
    const cuuint64_t strides[3] = {cuuint64_t(d) * eb, cuuint64_t(H) * d * eb,
                                   cuuint64_t(N) * H * d * eb};
    const cuuint32_t box[4] = {cuuint32_t(128 / eb), 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(tm, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_e4m3_vt(CUtensorMap *tm, const void *base, int64_t rows, int64_t n_pad, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr)
        return false;
    const cuuint64_t dims[2] = {cuuint64_t(n_pad), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(n_pad)};
    const cuuint32_t box[2] = {128, cuuint32_t(d)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fa
