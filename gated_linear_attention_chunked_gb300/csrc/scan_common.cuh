// scan_common.cuh -- pieces shared by the chunk-scan kernels (forward, the backward roles and
// the segment passes): the bounded wait with a CTA-wide abort flag, 16-bit conversions, the
// power-of-two exponent of a state copy, and the TMA emission of fp32 output rows.
//
// In every scan kernel an epilogue warp w reads TMEM lane quadrant q = w & 3 (token rows
// 32q..32q+31, one row per thread); the kernels differ in how many warps share a quadrant.
#pragma once
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gla {
namespace scan {

constexpr int C = 128, DK = 96, DV = 192;
constexpr uint64_t DRAIN_NS = 4000000000ull;  // limit of the exit-time drain waits

struct Cta {
  uint8_t* base;      // 1024-aligned dynamic shared memory
  uint32_t sb;        // its shared-window address
  uint32_t bar_off;   // offset of the mbarrier array
  uint32_t abort_off; // offset of the abort flag (int)
  __device__ uint32_t bar(uint32_t i) const { return sb + bar_off + 8 * i; }
  __device__ volatile int* abort_flag() const { return (volatile int*)(base + abort_off); }
};

// The polling part of a bounded wait, kept out of line: every wait site then costs one
// try_wait and a call, which keeps the unrolled chunk loops small enough for the
// instruction cache.
static __device__ __noinline__ bool wait_slow(volatile int* abort, uint32_t bar, uint32_t parity,
                                              int* err, unsigned long long wait_ns) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > wait_ns) {
        DevCtl c;
        c.err = err;
        c.wait_ns = wait_ns;
        record_error(c, DEV_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}
// Bounded wait that also returns false as soon as another role of the CTA has given up.
__device__ __forceinline__ bool wait(const Cta& cta, uint32_t bar, uint32_t parity,
                                     const DevCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(cta.abort_flag(), bar, parity, ctl.err, ctl.wait_ns);
}

// The bounded wait as taken by all 32 lanes of a warp, with one outcome for the whole warp:
// false on every lane if any lane's wait gave up (or saw the abort flag).  A lane can see the
// barrier complete while another lane of its warp gives up at the same instant; the vote keeps
// the warp on one path, so the warp-collective instructions after it (shuffles, the
// .sync.aligned TMEM loads and stores, __syncwarp) are never reached by part of a warp.
__device__ __forceinline__ bool wait_warp(const Cta& cta, uint32_t bar, uint32_t parity,
                                          const DevCtl& ctl) {
  return __all_sync(0xffffffffu, wait(cta, bar, parity, ctl));
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

// Convert NCH 16-byte chunks of one tile row in place (scale s, to fp16), G chunks at a
// time with their loads issued together so that the shared-memory latency overlaps.
// `off(c)` is the byte offset of chunk c.
template <bool SRC_BF16, int NCH, int G = 4, typename Off>
__device__ __forceinline__ void convert_row(uint8_t* tile, Off off, float s, float& vmax) {
  static_assert(NCH % G == 0, "whole batches of chunks");
#pragma unroll 1  // batches of G chunks; a rolled loop keeps the code small
  for (int c0 = 0; c0 < NCH; c0 += G) {
    uint4 x[G];
#pragma unroll
    for (int u = 0; u < G; ++u) x[u] = *(const uint4*)(tile + off(c0 + u));
#pragma unroll
    for (int u = 0; u < G; ++u) {
      uint32_t* w = reinterpret_cast<uint32_t*>(&x[u]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = ld16<SRC_BF16>(w[e] & 0xFFFFu) * s, b = ld16<SRC_BF16>(w[e] >> 16) * s;
        vmax = fmaxf(vmax, fmaxf(fabsf(a), fabsf(b)));
        w[e] = pack_h2(a, b);
      }
    }
#pragma unroll
    for (int u = 0; u < G; ++u) *(uint4*)(tile + off(c0 + u)) = x[u];
  }
}

// Two rows' conversions interleaved (tile a scaled by sa, tile b by sb), G chunks of each per
// batch, so that 2G shared-memory loads are in flight together.
template <bool SRC_BF16, int NCH, int G, typename OffA, typename OffB>
__device__ __forceinline__ void convert_rows2(uint8_t* ta, OffA offa, float sa, float& ma,
                                              uint8_t* tb, OffB offb, float sb, float& mb) {
  static_assert(NCH % G == 0, "whole batches of chunks");
#pragma unroll 1
  for (int c0 = 0; c0 < NCH; c0 += G) {
    uint4 x[G], y[G];
#pragma unroll
    for (int u = 0; u < G; ++u) {
      x[u] = *(const uint4*)(ta + offa(c0 + u));
      y[u] = *(const uint4*)(tb + offb(c0 + u));
    }
#pragma unroll
    for (int u = 0; u < G; ++u) {
      uint32_t* w = reinterpret_cast<uint32_t*>(&x[u]);
      uint32_t* z = reinterpret_cast<uint32_t*>(&y[u]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a0 = ld16<SRC_BF16>(w[e] & 0xFFFFu) * sa, a1 = ld16<SRC_BF16>(w[e] >> 16) * sa;
        const float b0 = ld16<SRC_BF16>(z[e] & 0xFFFFu) * sb, b1 = ld16<SRC_BF16>(z[e] >> 16) * sb;
        ma = fmaxf(ma, fmaxf(fabsf(a0), fabsf(a1)));
        mb = fmaxf(mb, fmaxf(fabsf(b0), fabsf(b1)));
        w[e] = pack_h2(a0, a1);
        z[e] = pack_h2(b0, b1);
      }
    }
#pragma unroll
    for (int u = 0; u < G; ++u) {
      *(uint4*)(ta + offa(c0 + u)) = x[u];
      *(uint4*)(tb + offb(c0 + u)) = y[u];
    }
  }
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

// Emit a warp's 32 rows x (8 * NBLK8) fp32 columns, produced block by block by
// `produce(k, r)` (8 columns of block k), through two 1 KB staging buffers (`buf0`,
// `buf0 + 1024`) and TMA stores of 32-byte-swizzled boxes {8, 1, 32}: row rr at rr * 32
// bytes, its two 16-byte chunks exchanged when bit 2 of rr is set.  Blocks go two at a time:
// both staged, one proxy fence, both stores in one bulk group; the next pair reuses the
// buffers once those stores have read them.  `store(k, smem)` issues the TMA store of block
// k.  `buf0` must be 256-byte aligned.  Called by all 32 lanes; lane 0 issues the stores.
template <int NBLK8, typename Produce, typename Store>
__device__ __forceinline__ void emit_rows8_tma(uint8_t* buf0, int lane, Produce produce,
                                               Store store) {
  const int sw = (lane >> 2) & 1;
#pragma unroll
  for (int k0 = 0; k0 < NBLK8; k0 += 2) {
    const int nb = k0 + 1 < NBLK8 ? 2 : 1;
    float r[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (j < nb) produce(k0 + j, r[j]);
    if (k0 >= 2) {  // the previous pair's stores must have finished reading the buffers
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j < nb) {
        uint8_t* buf = buf0 + j * 1024;
        *reinterpret_cast<float4*>(buf + lane * 32 + (sw << 4)) =
            make_float4(r[j][0], r[j][1], r[j][2], r[j][3]);
        *reinterpret_cast<float4*>(buf + lane * 32 + ((sw ^ 1) << 4)) =
            make_float4(r[j][4], r[j][5], r[j][6], r[j][7]);
      }
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (j < nb) store(k0 + j, smem_u32(buf0 + j * 1024));
      bulk_commit();
    }
  }
}

}  // namespace scan
}  // namespace gla
