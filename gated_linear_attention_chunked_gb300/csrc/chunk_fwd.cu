// chunk_fwd.cu -- chunked forward of the Simple GLA mixer on tcgen05 tensor cores.
//
// Method ("Beyond the KV cache ... Laplace 3B ...", section "Challenge 1", the chunked form
// of the "GLA mixer" recurrence).  Per (b, h) and chunk c of C = 128 tokens, with
// D_ij = lambda^(i-j) (i >= j, else 0), Lq = diag(lambda^(i+1)), Lk = diag(lambda^(C-1-j)):
//   O_c     = (Q K^T o D) V + Lq Q S_c  + sigmoid(z) v      (intra + inter + self-augmentation)
//   S_{c+1} = lambda^C S_c + K^T Lk V                         (the only serial step)
//
// One CTA owns one (b, h) and walks its chunks in order; the fp32 state never leaves the chip.
//   warp 4      TMA producer: q, k tiles (3 boxes of 32 channels, 64-byte swizzle) and v tiles
//               (3 boxes of 64 channels, 128-byte swizzle) into a 2-stage ring.
//   warp 5      tcgen05 issuer (one thread) and TMEM owner (512 columns):
//                 D_P [cols 384,512)  P = Q K^T                  (bf16/fp16 inputs as given)
//                 D_O [cols   0,192)  O = Q'' S_c + P'' V          (fp16 operands)
//                 D_S [cols 192,384)  S = lambda^C S + K'^T V      (fp16 operands, fp32 state;
//                                    rows 96..127 are padding and never read)
//   warps 0..3  epilogue, thread = token row (= TMEM lane):
//                 (a) z = q.(a*k); Q'' = fp16(lambda^(i+1) q), K' = fp16(lambda^(127-i) k),
//                     V -> fp16 in place; P'' = fp16(mask(P) * 2^-e) into shared memory;
//                 (b) o = 2^e D_O + sigmoid(z) v, stored as fp32;
//                 (c) S -> fp16(S * 2^-e') into the drained q/k slot (B operand of the next
//                     Q'' S), and D_S <- lambda^C D_S ready for the next accumulation.
// fp16 operands (11-bit significand) keep the long-memory heads accurate; the state copy is
// scaled by a power of two e' chosen from max|S| so it never overflows fp16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "tmap.h"

namespace gla {
namespace {

constexpr int C = kChunk, DK = kDK, DV = kDV;
constexpr uint32_t Q_BOX = 8192;    // 128 rows x 64 B (32 channels), SW64
constexpr uint32_t V_BOX = 16384;   // 128 rows x 128 B (64 channels), SW128
constexpr uint32_t OFF_Q = 0, OFF_K = 3 * Q_BOX, OFF_V = 6 * Q_BOX;
constexpr uint32_t STAGE = OFF_V + 3 * V_BOX;  // 98304
constexpr uint32_t OFF_P = 2 * STAGE;          // 196608: P'' 2 atoms x 16 KB (K-major SW128)
constexpr uint32_t P_ATOM = 16384;
constexpr uint32_t S_ATOM = 12288;             // S copy: 3 atoms of 96 rows x 128 B (MN-major)
constexpr uint32_t OFF_BAR = OFF_P + 2 * P_ATOM;  // 229376
constexpr uint32_t OFF_TMEM = OFF_BAR + 16 * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_RED = OFF_TMEM + 16;     // float red[2][4]
constexpr uint32_t OFF_PW = OFF_BAR + 256;      // float pw[128]
constexpr uint32_t OFF_A = OFF_PW + 512;        // float a[96]
constexpr uint32_t SMEM_USED = OFF_A + 384;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(3 * S_ATOM <= 2 * 3 * Q_BOX, "state copy fits in a drained q/k slot");

constexpr uint32_t QK_BYTES = 6 * Q_BOX, V_BYTES = 3 * V_BOX;
constexpr uint32_t TM_O = 0, TM_S = 192, TM_P = 384;

enum Bar : uint32_t {
  QK_FULL = 0,   // +stage
  V_FULL = 2,    // +stage
  QK_EMPTY = 4,  // +stage: the state copy held in that slot has been consumed
  V_EMPTY = 6,   // +stage
  P_DONE = 8,
  O_DONE = 9,
  S_DONE = 10,
  EP_CONV = 11,
  EP_O = 12,
  EP_S = 13,
  DRAIN = 14,
  RED = 15,      // exchange of the per-warp max|S| (bounded wait, unlike bar.sync)
};

constexpr int THREADS = 192;
constexpr uint64_t DRAIN_NS = 4000000000ull;

struct Smem {
  uint8_t* base;
  uint32_t sb;
  __device__ uint32_t bar(uint32_t i) const { return sb + OFF_BAR + 8 * i; }
  __device__ volatile int* abort_flag() const { return (volatile int*)(base + OFF_ABORT); }
};

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(const Smem& sm, uint32_t bar, uint32_t parity,
                                              const DevCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*sm.abort_flag()) return false;
      if (globaltimer() - t0 > ctl.wait_ns) {
        record_error(ctl, DEV_TIMEOUT);
        *sm.abort_flag() = 1;
        return false;
      }
    }
  }
}

template <bool BF16>
__device__ __forceinline__ float ld16(uint16_t bits) {
  if constexpr (BF16) return __uint_as_float((uint32_t)bits << 16);
  else return __half2float(__ushort_as_half(bits));
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float h2lo(uint32_t u) { return __half2float(__ushort_as_half((uint16_t)(u & 0xFFFF))); }
__device__ __forceinline__ float h2hi(uint32_t u) { return __half2float(__ushort_as_half((uint16_t)(u >> 16))); }
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }  // |e| < 127

template <bool BF16>
__global__ void __launch_bounds__(THREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const float* __restrict__ log_decay,
           const float* __restrict__ aug, const float* __restrict__ init, float* __restrict__ out,
           float* __restrict__ fin, int T, int H, DevCtl ctl) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  sm.base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  sm.sb = smem_u32(sm.base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, b = bh / H, h = bh % H;
  const int nc = T / C;
  const float gamma = __ldg(log_decay + h);
  float* pw = (float*)(sm.base + OFF_PW);
  float* sa = (float*)(sm.base + OFF_A);
  float* red = (float*)(sm.base + OFF_RED);
  uint32_t* tmem_slot = (uint32_t*)(sm.base + OFF_TMEM);

  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == 128) {
    for (uint32_t s = 0; s < 2; ++s) {
      mbar_init(sm.bar(QK_FULL + s), 1);
      mbar_init(sm.bar(V_FULL + s), 1);
      mbar_init(sm.bar(QK_EMPTY + s), 1);
      mbar_init(sm.bar(V_EMPTY + s), 1 + 128);
    }
    mbar_init(sm.bar(P_DONE), 1);
    mbar_init(sm.bar(O_DONE), 1);
    mbar_init(sm.bar(S_DONE), 1);
    mbar_init(sm.bar(DRAIN), 1);
    mbar_init(sm.bar(EP_CONV), 128);
    mbar_init(sm.bar(EP_O), 128);
    mbar_init(sm.bar(EP_S), 128);
    mbar_init(sm.bar(RED), 128);
    *sm.abort_flag() = 0;
    fence_barrier_init();
  }
  if (tid < C) pw[tid] = expf((float)tid * gamma);  // lambda^d, d = 0..127
  if (tid < DK) sa[tid] = __ldg(aug + h * DK + tid);
  if ((sm.sb & 1023u) != 0) record_error(ctl, DEV_LAYOUT);  // cannot happen: base aligned above
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const int row0 = b * T;
      int armed_qk[2] = {0, 0}, armed_v[2] = {0, 0};
      for (int c = 0; c < nc; ++c) {
        const uint32_t s = c & 1, st = sm.sb + s * STAGE;
        const int row = row0 + c * C;
        if (c >= 2 && !wait_or_abort(sm, sm.bar(V_EMPTY + s), ((c >> 1) - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(sm.bar(V_FULL + s), V_BYTES);
        for (int j = 0; j < 3; ++j)
          tma_load_3d(st + OFF_V + j * V_BOX, &map_v, sm.bar(V_FULL + s), 64 * j, h, row);
        ++armed_v[s];
        if (c >= 1 && !wait_or_abort(sm, sm.bar(QK_EMPTY + s), ((c - 1) >> 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(sm.bar(QK_FULL + s), QK_BYTES);
        for (int j = 0; j < 3; ++j) {
          tma_load_3d(st + OFF_Q + j * Q_BOX, &map_q, sm.bar(QK_FULL + s), 32 * j, h, row);
          tma_load_3d(st + OFF_K + j * Q_BOX, &map_k, sm.bar(QK_FULL + s), 32 * j, h, row);
        }
        ++armed_qk[s];
      }
      // drain: every armed load has landed before the CTA may exit
      for (int s = 0; s < 2; ++s) {
        if (armed_v[s]) mbar_wait(sm.bar(V_FULL + s), (armed_v[s] - 1) & 1, ctl, DRAIN_NS);
        if (armed_qk[s]) mbar_wait(sm.bar(QK_FULL + s), (armed_qk[s] - 1) & 1, ctl, DRAIN_NS);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_f16(128, 128, BF16, BF16, false, false);
      constexpr uint32_t ID_QS = idesc_f16(128, 192, false, false, false, true);
      constexpr uint32_t ID_PV = idesc_f16(128, 192, false, false, false, true);
      constexpr uint32_t ID_KV = idesc_f16(128, 192, false, false, true, true);
      for (int c = 0; c < nc; ++c) {
        const uint32_t s = c & 1, st = sm.sb + s * STAGE;
        const uint32_t slot = sm.sb + (s ^ 1) * STAGE;  // state copy for this chunk
        if (!wait_or_abort(sm, sm.bar(QK_FULL + s), (c >> 1) & 1, ctl)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 6; ++ks) {
          const uint32_t off = (ks >> 1) * Q_BOX + (ks & 1) * 32;
          mma_f16_ss(tmem + TM_P, smem_desc(st + OFF_Q + off, 16, 512, SW_64),
                     smem_desc(st + OFF_K + off, 16, 512, SW_64), ID_QK, ks > 0);
        }
        mma_commit(sm.bar(P_DONE));
        if (!wait_or_abort(sm, sm.bar(EP_CONV), c & 1, ctl)) break;
        if (!wait_or_abort(sm, sm.bar(EP_S), c & 1, ctl)) break;
        if (c >= 1 && !wait_or_abort(sm, sm.bar(EP_O), (c - 1) & 1, ctl)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 6; ++ks) {  // O = Q'' S
          const uint32_t off = (ks >> 1) * Q_BOX + (ks & 1) * 32;
          mma_f16_ss(tmem + TM_O, smem_desc(st + OFF_Q + off, 16, 512, SW_64),
                     smem_desc(slot + ks * 2048, S_ATOM, 1024, SW_128), ID_QS, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // O += P'' V
          mma_f16_ss(tmem + TM_O,
                     smem_desc(sm.sb + OFF_P + (ks >> 2) * P_ATOM + (ks & 3) * 32, 16, 1024, SW_128),
                     smem_desc(st + OFF_V + ks * 2048, V_BOX, 1024, SW_128), ID_PV, 1);
        }
        mma_commit(sm.bar(O_DONE));
        mma_commit(sm.bar(QK_EMPTY + (s ^ 1)));
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // S += K'^T V
          mma_f16_ss(tmem + TM_S, smem_desc(st + OFF_K + ks * 1024, Q_BOX, 512, SW_64),
                     smem_desc(st + OFF_V + ks * 2048, V_BOX, 1024, SW_128), ID_KV, 1);
        }
        mma_commit(sm.bar(S_DONE));
        mma_commit(sm.bar(V_EMPTY + s));
      }
      mma_commit(sm.bar(DRAIN));
      mbar_wait(sm.bar(DRAIN), 0, ctl, DRAIN_NS);
    }
  } else {
    // ------------------------------------------------------------------ epilogue, row i
    const int i = tid;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const float lamC = expf((float)C * gamma);
    const float lq = (i + 1 < C) ? pw[i + 1] : lamC;  // lambda^(i+1)
    const float lk = pw[C - 1 - i];                   // lambda^(C-1-i)
    bool range_bad = false;
    int e_cur = 0;

    // Make a scaled fp16 copy of the state rows in the q/k slot at `slot_off`, and set
    // D_S <- lambda^C S.  Row i of S (fp32) comes from TMEM or from init_state (`g_row`,
    // null = zeros).  `use` counts the calls (parity of the RED exchange).  Returns the
    // power-of-two exponent e of the copy (copy = S * 2^-e), or -1 if it gave up waiting.
    auto publish_state = [&](uint32_t slot_off, int use, const float* g_row, bool from_tmem) {
      const int par = use & 1;
      float m = 0.f;
      uint32_t r[32];
      if (warp < 3) {
        for (int nb = 0; nb < 6; ++nb) {
          if (from_tmem) {
            tmem_ld32(trow + TM_S + nb * 32, r);
            tmem_wait_ld();
          } else {
            for (int j = 0; j < 32; ++j)
              r[j] = __float_as_uint(g_row ? __ldg(g_row + nb * 32 + j) : 0.f);
          }
          for (int j = 0; j < 32; ++j) m = fmaxf(m, fabsf(__uint_as_float(r[j])));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[par * 4 + warp] = m;
      mbar_arrive(sm.bar(RED));
      if (!wait_or_abort(sm, sm.bar(RED), par, ctl)) return -1;
      m = fmaxf(fmaxf(red[par * 4 + 0], red[par * 4 + 1]), fmaxf(red[par * 4 + 2], red[par * 4 + 3]));
      int e = 0;
      if (!(m <= 3.0e38f)) {  // inf or nan in the state
        range_bad = true;
      } else if (m > 0.f) {
        int ex;
        frexpf(m, &ex);
        e = ex > 14 ? ex - 14 : 0;
      }
      if (warp < 3) {
        const float sc = pow2i(-e);
        for (int nb = 0; nb < 6; ++nb) {
          if (from_tmem) {
            tmem_ld32(trow + TM_S + nb * 32, r);
            tmem_wait_ld();
          } else {
            for (int j = 0; j < 32; ++j)
              r[j] = __float_as_uint(g_row ? __ldg(g_row + nb * 32 + j) : 0.f);
          }
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {  // 4 chunks of 8 value channels
            const int n = nb * 32 + q8 * 8;
            uint4 pk;
            pk.x = pack_h2(__uint_as_float(r[q8 * 8 + 0]) * sc, __uint_as_float(r[q8 * 8 + 1]) * sc);
            pk.y = pack_h2(__uint_as_float(r[q8 * 8 + 2]) * sc, __uint_as_float(r[q8 * 8 + 3]) * sc);
            pk.z = pack_h2(__uint_as_float(r[q8 * 8 + 4]) * sc, __uint_as_float(r[q8 * 8 + 5]) * sc);
            pk.w = pack_h2(__uint_as_float(r[q8 * 8 + 6]) * sc, __uint_as_float(r[q8 * 8 + 7]) * sc);
            *(uint4*)(sm.base + slot_off + (n >> 6) * S_ATOM + swz_off(i, (n & 63) >> 3, 128)) = pk;
          }
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * lamC);
          tmem_st32(trow + TM_S + nb * 32, r);
        }
        tmem_wait_st();
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(sm.bar(EP_S));
      return e;
    };

    // initial state -> copy in stage 1's q/k slot, D_S = lambda^C S_0
    {
      const float* g_row = (init && i < DK) ? init + ((size_t)bh * DK + i) * DV : nullptr;
      e_cur = publish_state(1 * STAGE + OFF_Q, 0, g_row, false);
    }

    bool ok = e_cur >= 0;
    for (int c = 0; c < nc && ok; ++c) {
      const uint32_t s = c & 1;
      uint8_t* stg = sm.base + s * STAGE;
      // ---- (a) gate, in-place operand conversion, masked scores
      if (!(ok = wait_or_abort(sm, sm.bar(P_DONE), c & 1, ctl))) break;
      if (!(ok = wait_or_abort(sm, sm.bar(QK_FULL + s), (c >> 1) & 1, ctl))) break;
      if (!(ok = wait_or_abort(sm, sm.bar(V_FULL + s), (c >> 1) & 1, ctl))) break;
      tc_fence_after();
      float z = 0.f;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t off = j * Q_BOX + swz_off(i, ch, 64);
          uint4 qv = *(uint4*)(stg + OFF_Q + off);
          uint4 kv = *(uint4*)(stg + OFF_K + off);
          const uint32_t* qw = (const uint32_t*)&qv;
          const uint32_t* kw = (const uint32_t*)&kv;
          uint4 qo, ko;
          uint32_t* qow = (uint32_t*)&qo;
          uint32_t* kow = (uint32_t*)&ko;
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int d = j * 32 + ch * 8 + e2 * 2;
            const float q0 = ld16<BF16>((uint16_t)(qw[e2] & 0xFFFF)), q1 = ld16<BF16>((uint16_t)(qw[e2] >> 16));
            const float k0 = ld16<BF16>((uint16_t)(kw[e2] & 0xFFFF)), k1 = ld16<BF16>((uint16_t)(kw[e2] >> 16));
            z = fmaf(sa[d] * q0, k0, z);
            z = fmaf(sa[d + 1] * q1, k1, z);
            const float a0 = q0 * lq, a1 = q1 * lq, b0 = k0 * lk, b1 = k1 * lk;
            range_bad |= fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))) >= 65504.f;
            qow[e2] = pack_h2(a0, a1);
            kow[e2] = pack_h2(b0, b1);
          }
          *(uint4*)(stg + OFF_Q + off) = qo;
          *(uint4*)(stg + OFF_K + off) = ko;
        }
      }
      if constexpr (BF16) {  // v -> fp16 in place (exact for |v| < 65504 normal range)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint32_t off = OFF_V + j * V_BOX + swz_off(i, ch, 128);
            uint4 vv = *(uint4*)(stg + off);
            uint32_t* vw = (uint32_t*)&vv;
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float v0 = ld16<true>((uint16_t)(vw[e2] & 0xFFFF)), v1 = ld16<true>((uint16_t)(vw[e2] >> 16));
              range_bad |= fmaxf(fabsf(v0), fabsf(v1)) >= 65504.f;
              vw[e2] = pack_h2(v0, v1);
            }
            *(uint4*)(stg + off) = vv;
          }
        }
      }
      {
        const float psc = pow2i(-e_cur);
        uint32_t r[32];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
          tmem_ld32(trow + TM_P + jb * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            float p[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int jj = jb * 32 + q8 * 8 + u;
              const float x = __uint_as_float(r[q8 * 8 + u]);
              p[u] = (jj <= i) ? x * pw[i - jj] * psc : 0.f;
              range_bad |= fabsf(p[u]) >= 65504.f;
            }
            uint4 pk;
            pk.x = pack_h2(p[0], p[1]);
            pk.y = pack_h2(p[2], p[3]);
            pk.z = pack_h2(p[4], p[5]);
            pk.w = pack_h2(p[6], p[7]);
            const int j0 = jb * 32 + q8 * 8;
            *(uint4*)(sm.base + OFF_P + (j0 >> 6) * P_ATOM + swz_off(i, (j0 & 63) >> 3, 128)) = pk;
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(sm.bar(EP_CONV));

      // ---- (b) output row: o = 2^e D_O + sigmoid(z) v
      if (!(ok = wait_or_abort(sm, sm.bar(O_DONE), c & 1, ctl))) break;
      tc_fence_after();
      {
        const float sg = 1.f / (1.f + expf(-z));
        const float osc = pow2i(e_cur);
        float* orow = out + (((size_t)b * T + (size_t)c * C + i) * H + h) * DV;
        uint32_t r[32];
#pragma unroll 1
        for (int nb = 0; nb < 6; ++nb) {
          tmem_ld32(trow + TM_O + nb * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            const int n = nb * 32 + q8 * 8;
            const uint4 vv = *(const uint4*)(stg + OFF_V + (n >> 6) * V_BOX + swz_off(i, (n & 63) >> 3, 128));
            const uint32_t* vw = (const uint32_t*)&vv;
            float4 o0, o1;
            o0.x = fmaf(__uint_as_float(r[q8 * 8 + 0]), osc, sg * h2lo(vw[0]));
            o0.y = fmaf(__uint_as_float(r[q8 * 8 + 1]), osc, sg * h2hi(vw[0]));
            o0.z = fmaf(__uint_as_float(r[q8 * 8 + 2]), osc, sg * h2lo(vw[1]));
            o0.w = fmaf(__uint_as_float(r[q8 * 8 + 3]), osc, sg * h2hi(vw[1]));
            o1.x = fmaf(__uint_as_float(r[q8 * 8 + 4]), osc, sg * h2lo(vw[2]));
            o1.y = fmaf(__uint_as_float(r[q8 * 8 + 5]), osc, sg * h2hi(vw[2]));
            o1.z = fmaf(__uint_as_float(r[q8 * 8 + 6]), osc, sg * h2lo(vw[3]));
            o1.w = fmaf(__uint_as_float(r[q8 * 8 + 7]), osc, sg * h2hi(vw[3]));
            __stcs(reinterpret_cast<float4*>(orow + n), o0);
            __stcs(reinterpret_cast<float4*>(orow + n + 4), o1);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(sm.bar(EP_O));
      mbar_arrive(sm.bar(V_EMPTY + s));

      // ---- (c) state: publish the next chunk's state copy, or write the final state
      if (!(ok = wait_or_abort(sm, sm.bar(S_DONE), c & 1, ctl))) break;
      tc_fence_after();
      if (c == nc - 1) {
        if (fin && warp < 3) {
          float* frow = fin + ((size_t)bh * DK + i) * DV;
          uint32_t r[32];
          for (int nb = 0; nb < 6; ++nb) {
            tmem_ld32(trow + TM_S + nb * 32, r);
            tmem_wait_ld();
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(frow + nb * 32 + j) =
                  make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                              __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
          }
        }
      } else {
        e_cur = publish_state(s * STAGE + OFF_Q, c + 1, nullptr, true);
        if (!(ok = e_cur >= 0)) break;
      }
    }
    if (range_bad) record_error(ctl, DEV_RANGE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_chunk_fwd(const FwdArgs& a, DevCtl ctl, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const long long rows = (long long)a.B * a.T;
  if (!make_tmap_3d_16bit(&mq, a.q, DK, a.H, rows, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_3d_16bit(&mk, a.k, DK, a.H, rows, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_3d_16bit(&mv, a.v, DV, a.H, rows, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, a.bf16))
    return cudaErrorInvalidValue;
  auto kern = a.bf16 ? fwd_kernel<true> : fwd_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.H, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, a.log_decay, a.aug, a.init, a.o,
                                                   a.fin, a.T, a.H, ctl);
  return cudaGetLastError();
}

}  // namespace gla
