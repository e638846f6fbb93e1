// Host-side construction of TMA tensor maps for [B, T, H, D] bf16 tensors.
// The driver entry point is looked up through the runtime, so the library
// does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

namespace nc {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// View a contiguous bf16 [B, T, H, D] tensor as the 4-D TMA tensor {D, H, T, B}
// (innermost first) with a {box_d, 1, box_t, 1} box and 128-byte swizzle.  Rows
// past T read as zero.  Returns false when the driver rejects the map.
inline bool make_tmap_bthd(CUtensorMap* map, const void* base, int B, int T, int H, int D, int box_d, int box_t) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_t, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// View a contiguous fp32 [B, T, H, D] tensor as {D, H, T, B} with a {box_d, 1, box_t, 1}
// box (used as the target of TMA reduce-adds): no swizzle, or the 128-byte swizzle for a 32-float box.
inline bool make_tmap_bthd_f32(CUtensorMap* map, const void* base, int B, int T, int H, int D, int box_d, int box_t,
                               bool swizzle128 = false) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4, (cuuint64_t)T * H * D * 4};
    const cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_t, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace nc
