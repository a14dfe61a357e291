// la_tma_host.h -- host-side creation of TMA tensor maps.  The CUDA driver API's
// cuTensorMapEncodeTiled is reached through the runtime's entry-point query,
// so the library needs no link-time dependency on libcuda.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace la {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A rank-3 bf16 tensor [d2][d1][d0] (d0 contiguous) read or written in boxes
// of box1 rows x box0 columns of one d2 slice, with the 128-byte swizzle
// (box0 * 2 bytes must be <= 128).  Out-of-range box rows load as zero and
// are skipped by stores.
inline bool make_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                              uint64_t d2, uint32_t box0, uint32_t box1) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A rank-3 fp32 tensor [d2][d1][d0] (d0 contiguous) read in boxes of box1 rows
// x box0 columns of one d2 slice, without swizzle (box0 * 4 bytes a multiple of
// 16, box0 and box1 <= 256): the box lands as dense rows of box0 floats.
inline bool make_tmap_f32_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1,
                             uint64_t d2, uint32_t box0, uint32_t box1) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace la
