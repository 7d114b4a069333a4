// tma_host.h -- host-side construction of TMA tensor maps (CUtensorMap) for
// bf16 tensors.  cuTensorMapEncodeTiled is a driver entry point; it is looked
// up once through the runtime so the library needs no link-time libcuda.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace carat {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tiled tensor map.  dims/box are innermost first; strides_bytes holds the
// byte strides of dims 1..rank-1 (multiples of 16).  swizzle128: 128-byte
// swizzle (box[0] * element size must then be <= 128).  Out-of-range
// elements read as 0.
inline bool make_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                            int rank, const uint64_t *dims, const uint64_t *strides_bytes,
                            const uint32_t *box, bool swizzle128) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gstride[i] = strides_bytes[i];
    CUresult r = enc(map, dtype, (cuuint32_t)rank,
                     const_cast<void *>(base), gdim, gstride, bdim, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

inline bool make_bf16_tensor_map(CUtensorMap *map, const void *base, int rank,
                                 const uint64_t *dims, const uint64_t *strides_bytes,
                                 const uint32_t *box, bool swizzle128) {
    return make_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes,
                           box, swizzle128);
}

// Tiled map of 1-byte elements (FP8 e4m3 caches): box[0] <= 128 with the
// 128-byte swizzle.
inline bool make_u8_tensor_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                               const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128) {
    return make_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides_bytes, box,
                           swizzle128);
}

}  // namespace carat
