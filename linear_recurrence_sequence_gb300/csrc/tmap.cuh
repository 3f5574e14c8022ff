// Host-side TMA descriptor helper shared by the C entry points.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace lrs {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 3-D tensor map over a contiguous [B, L, D] BF16 tensor with a box of
// `rows` tokens x kGroup channels (rows past L read as zero).
inline bool make_bf16_map(CUtensorMap* map, const void* ptr, int B, int L, int D, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * (cuuint64_t)D * 2};
    cuuint32_t box[3] = {(cuuint32_t)kGroup, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same BF16 map with the 128-byte swizzle (the box rows are 128 bytes:
// kGroup channels), for boxes that feed the tensor cores; the destination
// must be 1024-byte aligned.
inline bool make_bf16_map_sw128(CUtensorMap* map, const void* ptr, int B, int L, int D, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * (cuuint64_t)D * 2};
    cuuint32_t box[3] = {(cuuint32_t)kGroup, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same over a contiguous [B, L, D] FP32 tensor (256-byte box rows).
inline bool make_f32_map(CUtensorMap* map, const void* ptr, int B, int L, int D, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)L * (cuuint64_t)D * 4};
    cuuint32_t box[3] = {(cuuint32_t)kGroup, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tensor map over the per-token control words [B, L] x 8 FP32 (each value
// duplicated, 32 bytes per token) with a box of `rows` tokens (rows past L
// read as zero).
inline bool make_ctrl_map(CUtensorMap* map, const void* ptr, int B, int L, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {8, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[2] = {32, (cuuint64_t)L * 32};
    cuuint32_t box[3] = {8, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace lrs
