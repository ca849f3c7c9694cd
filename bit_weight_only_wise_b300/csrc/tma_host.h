// Host side of the TMA copies: building 2-D tensor maps.
//
// cuTensorMapEncodeTiled is a driver entry point; it is looked up through the
// runtime (cudaGetDriverEntryPointByVersion) so that the library links only
// the static CUDA runtime and loads without a GPU or libcuda at hand.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include <atomic>
#include <cstdint>

namespace w4a16 {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once (an atomic, so threads making their first call together do
// not race; a failed lookup is retried on the next call).
inline PFN_encodeTiled tensor_map_encoder() {
  static std::atomic<PFN_encodeTiled> cached{nullptr};
  PFN_encodeTiled fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_encodeTiled>(ptr);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// A row-major [outer, inner] matrix with rows `row_bytes` apart, copied in
// boxes of [box_outer, box_inner] elements; out-of-range elements read as 0.
inline bool encode_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace w4a16
