// Host-side TMA tensor-map encoding (cuTensorMapEncodeTiled reached through the
// runtime's driver entry point, so the library links no libcuda stub).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace sage {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D tiled map over a contiguous [outer][rows][inner] tensor of `esize`-byte
// elements, box = [1][box_rows][box_inner].  With the default 128-byte swizzle
// box_inner * esize must be 128; without swizzle the box is a dense row-major
// [box_rows][box_inner] block in shared memory.  Out-of-range rows read as zero.
// Returns false on error.
inline bool make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int esize,
                         uint64_t inner, uint64_t rows, uint64_t outer, uint32_t box_inner,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * (uint64_t)esize, inner * rows * (uint64_t)esize};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sage
