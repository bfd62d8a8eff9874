// tmap.h -- host-side construction of TMA tensor maps for the token-major [B, T, H, d]
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

// A 16-bit tensor [B, T, H, d] viewed as 4-D (innermost first): {d, H, T, B}.  A box
// {box_d, 1, box_rows, 1} is a tile of `box_rows` consecutive tokens of one head of one
// sequence; rows past the sequence's T tokens load as zeros.
inline bool make_tmap_seq_16bit(CUtensorMap* map, const void* base, int d, int H, int T, int B,
                                int box_d, int box_rows, CUtensorMapSwizzle sw, bool is_bf16) {
  auto fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * H, (cuuint64_t)d * 2 * H * T};
  cuuint32_t box[4] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 token-major output [B, T, H, d] as 4-D {d, H, T, B}, stored from shared memory in boxes
// of `box_d` (16 or 8) channels x 32 consecutive tokens of one head (64-byte rows with a 64-byte
// swizzle, or 32-byte rows with a 32-byte swizzle); rows past the sequence's T tokens are not
// written.
inline bool make_tmap_seq_out_f32(CUtensorMap* map, const void* base, int d, int H, int T, int B,
                                  int box_d = 16) {
  auto fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 4, (cuuint64_t)d * 4 * H, (cuuint64_t)d * 4 * H * T};
  cuuint32_t box[4] = {(cuuint32_t)box_d, 1u, 32u, 1u};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_d == 8 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A generic 3-D tensor map: dims / box innermost first, strides in bytes of dims 1 and 2.
inline bool make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         const unsigned long long (&dims)[3], const unsigned long long (&strides)[2],
                         const unsigned (&box)[3], CUtensorMapSwizzle sw) {
  auto fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// fp32 states [BH, 96, 192] stored in boxes of `box_c` (16 or 8) value channels x 32 key
// channels (64- or 32-byte swizzle, as the output maps).
inline bool make_tmap_state_f32(CUtensorMap* map, const void* base, long long bh, int box_c = 16) {
  const unsigned long long dims[3] = {192, 96, (unsigned long long)bh};
  const unsigned long long strides[2] = {192 * 4, 192 * 96 * 4};
  const unsigned box[3] = {(unsigned)box_c, 32, 1};
  return make_tmap_3d(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dims, strides, box,
                      box_c == 8 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace gla
