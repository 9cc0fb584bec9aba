// Host-side construction of TMA tensor maps (bf16, 128-byte swizzle) through the
// driver's cuTensorMapEncodeTiled, looked up once via the runtime.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace mla {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A rank-`rank` bf16 tensor: dims[0] is the contiguous dimension; strides_bytes
// holds the byte strides of dims 1..rank-1 (multiples of 16).  The box's inner
// extent is at most 64 elements (128 bytes, one swizzle row).  Out-of-range
// elements of a box read as zero.
inline bool encode_bf16_sw128(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                              const uint64_t *strides_bytes, const uint32_t *box) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bd[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bd[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), gd, gs, bd, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A rank-`rank` tensor of 32-bit elements, no swizzle (rows land row-major in
// shared memory at the box's width): dims[0] is the contiguous dimension in
// 32-bit units, strides_bytes the byte strides of dims 1..rank-1 (multiples of
// 16), box[0] at most 256 elements.  Used to copy whole channel slices of cache
// rows (bf16 or FP8) with one copy per box.  Out-of-range elements read as zero.
inline bool encode_u32_plain(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                             const uint64_t *strides_bytes, const uint32_t *box) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bd[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bd[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, (cuuint32_t)rank, const_cast<void *>(base), gd, gs, bd, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mla
