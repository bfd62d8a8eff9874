// scan_common.cuh -- pieces shared by the chunk-scan kernels (forward and the backward
// roles): the bounded wait with a CTA-wide abort flag, 16-bit conversions, the power-of-two
// scaled fp16 copy of a fp32 state row, and the coalesced store of fp32 output rows.
//
// Epilogue layout used by every scan kernel: 8 warps, warp w owns TMEM lane quadrant
// q = w & 3 (token rows 32q..32q+31, one row per thread) and column half hf = w >> 2.
#pragma once
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gla {
namespace scan {

constexpr int C = 128, DK = 96, DV = 192;
constexpr int EPI_WARPS = 8, EPI_THREADS = 256;
constexpr uint64_t DRAIN_NS = 4000000000ull;  // limit of the exit-time drain waits

struct Cta {
  uint8_t* base;      // 1024-aligned dynamic shared memory
  uint32_t sb;        // its shared-window address
  uint32_t bar_off;   // offset of the mbarrier array
  uint32_t abort_off; // offset of the abort flag (int)
  __device__ uint32_t bar(uint32_t i) const { return sb + bar_off + 8 * i; }
  __device__ volatile int* abort_flag() const { return (volatile int*)(base + abort_off); }
};

// Bounded wait that also returns false as soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait(const Cta& cta, uint32_t bar, uint32_t parity,
                                     const DevCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*cta.abort_flag()) return false;
      if (globaltimer() - t0 > ctl.wait_ns) {
        record_error(ctl, DEV_TIMEOUT);
        *cta.abort_flag() = 1;
        return false;
      }
    }
  }
}

template <bool BF16>
__device__ __forceinline__ float ld16(uint32_t bits16) {
  if constexpr (BF16) return __uint_as_float(bits16 << 16);
  else return __half2float(__ushort_as_half((unsigned short)bits16));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float h_lo(uint32_t u) {
  return __half2float(__ushort_as_half((unsigned short)(u & 0xFFFFu)));
}
__device__ __forceinline__ float h_hi(uint32_t u) {
  return __half2float(__ushort_as_half((unsigned short)(u >> 16)));
}
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }
__device__ __forceinline__ float sigmoid(float z) { return 1.f / (1.f + expf(-z)); }

// Scale 8 values and convert them to fp16 in place inside a 16-byte chunk of 16-bit data;
// `vmax` tracks the largest magnitude written (>= 65504 means the fp16 range was left).
template <bool SRC_BF16>
__device__ __forceinline__ void scale_chunk_to_half(uint4* p, float s, float& vmax) {
  uint4 x = *p;
  uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = ld16<SRC_BF16>(w[e] & 0xFFFFu) * s, b = ld16<SRC_BF16>(w[e] >> 16) * s;
    vmax = fmaxf(vmax, fmaxf(fabsf(a), fabsf(b)));
    w[e] = pack_h2(a, b);
  }
  *p = x;
}

// Power-of-two exponent e >= 0 such that m * 2^-e < 2^14 (fp16 copy with headroom).
// Returns -1 for a non-finite m.
__device__ __forceinline__ int state_exponent(float m) {
  if (!(m <= 3.0e38f)) return -1;
  if (m <= 0.f) return 0;
  int ex;
  frexpf(m, &ex);
  return ex > 14 ? ex - 14 : 0;
}

// Store 32 rows x NC (16 or 32) fp32 columns held one row per lane (`r`) to global memory
// with row-contiguous writes: the warp transposes through a staging area of 32 x NC x 4
// bytes (16-byte chunks XOR-swizzled by row), then each store instruction writes whole
// row segments (4 rows x 128 B, or 8 rows x 64 B).  `row_ptr(rr)` is the address of this
// block's first column in row rr (0..31).
template <int NC, typename RowPtr>
__device__ __forceinline__ void store_rows_coalesced(uint8_t* stage, const float* r, int lane,
                                                     RowPtr row_ptr) {
  static_assert(NC == 16 || NC == 32, "block width");
  constexpr int CH = NC / 4;            // 16-byte chunks per row
  constexpr int RB = NC * 4;            // row bytes
  constexpr int RPI = 32 / CH;          // rows per store instruction
#pragma unroll
  for (int c = 0; c < CH; ++c)
    *reinterpret_cast<float4*>(stage + lane * RB + ((c ^ (lane & (CH - 1))) << 4)) =
        make_float4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const int rr = RPI * k + lane / CH, c = lane % CH;
    const float4 x =
        *reinterpret_cast<const float4*>(stage + rr * RB + ((c ^ (rr & (CH - 1))) << 4));
    *reinterpret_cast<float4*>(row_ptr(rr) + 4 * c) = x;
  }
  __syncwarp();
}

// Write 32 rows x 16 fp32 columns (one row per lane, `r`) into a 2 KB staging buffer in
// the layout a 64-byte-swizzled TMA box {16, 1, 32} expects: row rr at rr * 64 bytes, its
// 16-byte chunk c at position c ^ ((rr >> 1) & 3).  `buf` must be 512-byte aligned.
__device__ __forceinline__ void stage_rows16_sw64(uint8_t* buf, const float* r, int lane) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<float4*>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
        make_float4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
}

// Emit a warp's 32 rows x (32 * NB) fp32 columns, produced block by block by `produce(k, r)`
// (k = 0..2*NB-1 fills the 16 columns of block k), through two 2 KB staging buffers
// (`buf0`, `buf0 + 2048`) and TMA stores.  `store(k, smem)` issues the TMA store of block k
// from the shared address `smem`.  Called by all 32 lanes; lane 0 issues the stores.
template <int NBLK16, typename Produce, typename Store>
__device__ __forceinline__ void emit_rows_tma(uint8_t* buf0, int lane, Produce produce,
                                              Store store) {
#pragma unroll
  for (int k = 0; k < NBLK16; ++k) {
    uint8_t* buf = buf0 + (k & 1) * 2048;
    float r[16];
    produce(k, r);
    if (k >= 2) {  // the store that last read this buffer must have finished reading it
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    stage_rows16_sw64(buf, r, lane);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      store(k, smem_u32(buf));
      bulk_commit();
    }
  }
}

}  // namespace scan
}  // namespace gla
