// tmap.h — host-side driver calls reached through the runtime's entry-point
// lookup (no link against libcuda): TMA descriptor encoding and a 32-bit fill.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace osm {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {  // looked up once, thread-safe
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// cuMemsetD32Async (32-bit fill on a stream), fetched the same way
using MemsetD32Fn = CUresult (*)(CUdeviceptr, unsigned int, size_t, CUstream);
inline MemsetD32Fn memset_d32_fn() {
  static MemsetD32Fn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemsetD32Async", &p, 3020, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<MemsetD32Fn>(p);
    return static_cast<MemsetD32Fn>(nullptr);
  }();
  return fn;
}

// A [outer, rows, inner] bf16 tensor (inner contiguous) read in boxes of
// box_inner x box_rows x 1 with 128-byte swizzle (or none, for boxes stored
// from a plain row-major stage); out-of-range rows read 0 (and are not written
// by a store).
inline bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                              uint64_t outer, uint32_t box_inner, uint32_t box_rows,
                              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = tmap_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace osm
