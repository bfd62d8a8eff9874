// tmap.h -- host-side construction of TMA tensor maps for the token-major [rows, H, d]
// tensors the chunk kernels stream.  cuTensorMapEncodeTiled is fetched through the runtime's
// driver entry point so that the library has no link-time dependency on libcuda.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

#include <cstdint>

namespace gla {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A 16-bit tensor viewed as 3-D (innermost first): {d, H, rows} with rows = B*T, so a box
// {box_d, 1, box_rows} is a tile of `box_rows` consecutive tokens of one head.  The shared
// memory image of a box is box_rows rows of box_d*2 bytes, swizzled with `sw` (the row
// length must equal the swizzle span: 64 B for SW64, 128 B for SW128).
inline bool make_tmap_3d_16bit(CUtensorMap* map, const void* base, int d, int H, long long rows,
                               int box_d, int box_rows, CUtensorMapSwizzle sw, bool is_bf16) {
  auto fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)H};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace gla
