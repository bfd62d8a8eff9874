// chunk_bwd.cu -- chunked backward of the Simple GLA mixer on tcgen05 tensor cores.
//
// Method: the gradient through every sequential state update ("Beyond the KV cache ...
// Laplace 3B ...", section "Challenge 3"), in the chunked form of section "Challenge 1".
// Per (b, h) and chunk c, with S_c the state entering the chunk, dS_{c+1} the adjoint of the
// state leaving it, D_ij = lambda^(i-j) (i >= j), Lq = diag(lambda^(i+1)),
// Lk = diag(lambda^(C-1-j)), z = q.(a*k), r = sigmoid'(z) (dO.v):
//   dQ  = (dO V^T o D) K + Lq dO S_c^T + r (a*k)           (needs the forward state scan)
//   dK  = (dO V^T o D)^T Q + Lk V dS_{c+1}^T + r (a*q)      (needs the reverse adjoint scan)
//   dV  = (Q K^T o D)^T dO + Lk K dS_{c+1} + sigmoid(z) dO   (needs the reverse adjoint scan)
//   dS_c = lambda^C dS_{c+1} + Q^T Lq dO,  d_init = dS_0,  d_a = sum r (q*k)
//
// One launch runs three independent CTA roles per (b, h), each a chunk scan with its state
// (or adjoint) kept on chip, so no role waits for another:
//   role DQ  forward order : score dP = dO V^T, out dq = dP'' K + dO'' S^T, state S += K^T V'
//   role DV  reverse order : score P^T = K Q^T, out dv = P''^T dO + K' dS,  adjoint dS += Q''^T dO
//                            (sigmoid(z) dO enters through the diagonal of P''^T)
//   role DK  reverse order : score dP^T = V dO^T, out dk = dP''^T Q + V' dS^T, adjoint dS += Q^T dO''
// (X'' denotes an fp16 copy of X scaled by its decay factors; scores are masked with D and
// scaled by 2^-e in fp32 before their fp16 copy.)  Warp layout:
//   warp 16 TMA producer (one buffer of the q, k, v, dO tiles of a chunk, in two groups with
//           barriers of their own, so the tiles the state update reads last are refilled
//           first; L2 prefetch of the next chunk),
//   warp 17 tcgen05 issuer + TMEM owner (D_X [0,192) output, D_S [192,384) state,
//           D_P [384,512) score),
//   warps 0..15 epilogue, four warps per row quadrant (row = token = TMEM lane), each with a
//           quarter of the row: gate dot products, in-place fp16 operands, two blocks of the
//           masked score copy written back into TMEM as an MMA operand; then the next state
//           copy (the serial step) while the output MMA's TMEM-operand part runs, and the
//           output rows, TMA-stored from per-warp staging.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "scan_common.cuh"
#include "tmap.h"

namespace gla {
namespace {

using namespace scan;

enum Role : int { R_DQ = 0, R_DV = 1, R_DK = 2 };

constexpr uint32_t Q_BOX = 8192, V_BOX = 16384;
constexpr uint32_t OFF_Q = 0, OFF_K = 3 * Q_BOX, OFF_V = 6 * Q_BOX, OFF_G = OFF_V + 3 * V_BOX;
constexpr uint32_t OFF_CP = OFF_G + 3 * V_BOX;  // state copy, 3 atoms x 12 KB
constexpr uint32_t S_ATOM = 12288;
constexpr uint32_t OFF_STG = OFF_CP + 3 * S_ATOM;  // output staging, 2 KB per epilogue warp
constexpr uint32_t OFF_BAR = OFF_STG + 16 * 2048;
constexpr uint32_t NBAR = 21;
constexpr uint32_t OFF_TMEM = (OFF_BAR + NBAR * 8 + 15) & ~15u;  // 16-byte aligned from here
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_RED = OFF_TMEM + 16;  // float red[3][16]: per-warp max|S|
constexpr uint32_t OFF_ES = OFF_RED + 192;   // int es[2]
constexpr uint32_t OFF_AB = OFF_ES + 16;     // float abmax[2][32]: state-MMA operand maxima
constexpr uint32_t OFF_GP = OFF_AB + 256;    // float gate_part[4][128]: gate partial sums
constexpr uint32_t OFF_DP = OFF_GP + 2048;   // float dpv[128]: dO.v per row (DQ, DK)
constexpr uint32_t OFF_A = OFF_DP + 512;     // float a[96] (read as float4)
constexpr uint32_t OFF_PW = OFF_A + 384;     // float pw[128]
constexpr uint32_t SMEM_USED = OFF_PW + 512;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_A % 16 == 0, "a[] is read as float4");

constexpr uint32_t TM_X = 0, TM_A = 96, TM_S = 192, TM_P = 384;  // TM_A: d_a (DQ role)

// A chunk's tiles come in two groups with barriers of their own: the early group holds the
// tiles whose last reader is the state (adjoint) update, so the next chunk's copies of them
// start while this chunk's masked scores are made; the late group holds the rest.
enum Bar : uint32_t {
  FULL_E = 0,   // early tiles landed
  FULL_L = 1,   // late tiles landed
  EMPTY_E = 2,  // early tiles free: the state (adjoint) update has read them
  EMPTY_L = 3,  // late tiles free: the output MMAs are done and the epilogue has its operands
  P_DONE = 4,
  X_DONE = 5,
  S_DONE = 6,  // the state (adjoint) update is done
  EP_CONV = 7,
  EP_X = 8,
  EP_S = 9,
  RED = 10,
  DRAIN = 11,
  QG0 = 12,  // 12..15: quadrant q's four gate partial sums are in shared memory
  QS0 = 16,  // 16..19: quadrant q's four parts have read their score blocks
  EP_C1 = 20,  // the fp16 operands are in place (the MMAs that need no masked score may run)
};

constexpr int NEPI = 16;  // epilogue warps: four per TMEM lane quadrant
constexpr int THREADS = (NEPI + 2) * 32;
constexpr int PRODUCER_WARP = NEPI, MMA_WARP = NEPI + 1;
constexpr int EPI_THREADS = NEPI * 32;

struct BwdParams {
  const float* log_decay;
  const float* aug;
  const float* init;
  const float* dfin;
  float* da_part;  // [B*H, 96]: d_aug partial sums of the whole pairs
  int T, H;
  bool want_dinit;
  SplitPlan plan;
  const float* seg_state;  // cut pairs: state entering each part (DQ's start)
  const float* seg_adj;    // cut pairs: adjoint leaving each part (DV's and DK's start)
  float* da_split;         // cut pairs: d_aug partial sums per part, [96] each
  const float* gate;       // [B,H,T] sigmoid(z) saved by the forward, or null (recomputed)
  SavedStates saved;       // the forward's state copies (DQ reads them instead of scanning)
};

enum Tile : int { T_Q = 0, T_K = 1, T_V = 2, T_G = 3 };

// Group of a tile for a role: 0 early, 1 late, -1 not loaded.  DQ: v, dO are last read by the
// state update (K^T V') and the output MMA's state part (dO'' S^T); DK: k (gate only: not
// loaded when the gate is given), v, dO; DV: q, k.  The late tiles are read by the output
// MMA's TMEM-operand part or by the rows.
template <int ROLE, bool SAVED>
__device__ __forceinline__ constexpr int tile_group(int tile) {
  if (ROLE == R_DQ) return tile == T_V || tile == T_G ? 0 : 1;
  if (ROLE == R_DK) return tile == T_Q ? 1 : (SAVED && tile == T_K ? -1 : 0);
  return tile == T_V ? -1 : (tile == T_G ? 1 : 0);
}
template <int ROLE, bool SAVED, bool SC>
__device__ __forceinline__ constexpr uint32_t group_bytes(int g) {
  return (tile_group<ROLE, SAVED>(T_Q) == g ? 3 * Q_BOX : 0) +
         (tile_group<ROLE, SAVED>(T_K) == g ? 3 * Q_BOX : 0) +
         (tile_group<ROLE, SAVED>(T_V) == g ? 3 * V_BOX : 0) +
         (tile_group<ROLE, SAVED>(T_G) == g ? 3 * V_BOX : 0) +
         (SC && ROLE == R_DQ && g == 0 ? (uint32_t)kCopyBytes : 0u);  // the saved state copy
}

// Chunk handled at step t of the role's scan over chunks [c0, c0 + n): DQ scans forward when
// it carries the state itself; with the forward's saved state copies it has no chain and runs
// in reverse with DV and DK, so the three roles of a pair read each chunk at about the same
// time and share its tiles through L2.
template <int ROLE, bool SC>
__device__ __forceinline__ int chunk_at(int t, int c0, int n) {
  return ROLE == R_DQ && !SC ? c0 + t : c0 + n - 1 - t;
}

// 16-byte chunk `cc` of row `i` of a 16-bit tile: q/k tiles have 3 boxes of 32 channels
// (64-byte rows), v/dO tiles 3 boxes of 64 channels (128-byte rows).
__device__ __forceinline__ uint32_t qk_chunk(uint32_t i, int cc) {
  return (cc >> 2) * Q_BOX + swz_off(i, cc & 3, 64);
}
__device__ __forceinline__ uint32_t vg_chunk(uint32_t i, int cc) {
  return (cc >> 3) * V_BOX + swz_off(i, cc & 7, 128);
}

template <bool SRC_BF16>
__device__ __forceinline__ void unpack8(const uint4& x, float (&f)[8]) {
  const uint32_t* w = (const uint32_t*)&x;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = ld16<SRC_BF16>(w[e] & 0xFFFFu);
    f[2 * e + 1] = ld16<SRC_BF16>(w[e] >> 16);
  }
}

__device__ __forceinline__ float max16(const float* v) {
  float m = v[0];
#pragma unroll
  for (int w = 1; w < 16; ++w) m = fmaxf(m, v[w]);
  return m;
}

// SAVED: the gate sigmoid(z) comes from p.gate (saved by the forward) instead of being
// recomputed; a template parameter so that each variant gets its own register allocation.
template <int ROLE, bool BF16, bool SAVED, bool SC>
__device__ __forceinline__ void run_role(
    uint8_t* base, const Cta& cta, int bh, int c0, int n, int cut_idx, const BwdParams& p,
    const CUtensorMap& map_q,
    const CUtensorMap& map_k, const CUtensorMap& map_v, const CUtensorMap& map_g,
    const CUtensorMap& map_out, const CUtensorMap& map_dinit, const DevCtl& ctl) {
  constexpr int NX = ROLE == R_DV ? 192 : 96;  // output columns
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, T = p.T, b = bh / H, h = bh % H;
  // chunks of this sequence; the last one holds L_last = 1..C tokens (rows past T are zeros)
  const int nc = (T + C - 1) / C, L_last = T - (nc - 1) * C;
  const float gamma = __ldg(p.log_decay + h);
  float* pw = (float*)(base + OFF_PW);
  float* red = (float*)(base + OFF_RED);
  int* es = (int*)(base + OFF_ES);
  float* abmax = (float*)(base + OFF_AB);
  float* gate_part = (float*)(base + OFF_GP);
  float* dpv = (float*)(base + OFF_DP);
  float* sa = (float*)(base + OFF_A);
  uint32_t* tmem_slot = (uint32_t*)(base + OFF_TMEM);

  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == PRODUCER_WARP * 32) {
    mbar_init(cta.bar(FULL_E), 1);
    mbar_init(cta.bar(FULL_L), 1);
    mbar_init(cta.bar(EMPTY_E), 1);
    mbar_init(cta.bar(EMPTY_L), 1 + EPI_THREADS);
    mbar_init(cta.bar(P_DONE), 1);
    mbar_init(cta.bar(X_DONE), 1);
    mbar_init(cta.bar(S_DONE), 1);
    mbar_init(cta.bar(DRAIN), 1);
    mbar_init(cta.bar(EP_CONV), EPI_THREADS);
    mbar_init(cta.bar(EP_C1), EPI_THREADS);
    mbar_init(cta.bar(EP_X), EPI_THREADS);
    mbar_init(cta.bar(EP_S), EPI_THREADS);
    mbar_init(cta.bar(RED), EPI_THREADS);
    for (int q = 0; q < 4; ++q) {
      mbar_init(cta.bar(QG0 + q), 128);
      mbar_init(cta.bar(QS0 + q), 128);
    }
    *cta.abort_flag() = 0;
    fence_barrier_init();
  }
  if (tid < C) pw[tid] = expf((float)tid * gamma);
  if (tid < DK) sa[tid] = __ldg(p.aug + h * DK + tid);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = cta.sb;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // the tiles of group g of chunk c (or an L2 prefetch of them)
      auto load = [&](int c, int g, bool prefetch_only) {
        const int t0 = c * C;
        const uint32_t bar = cta.bar(g == 0 ? FULL_E : FULL_L);
        for (int j = 0; j < 3; ++j) {
          if (prefetch_only) {
            if (tile_group<ROLE, SAVED>(T_Q) == g) tma_prefetch_4d(&map_q, 32 * j, h, t0, b);
            if (tile_group<ROLE, SAVED>(T_K) == g) tma_prefetch_4d(&map_k, 32 * j, h, t0, b);
            if (tile_group<ROLE, SAVED>(T_V) == g) tma_prefetch_4d(&map_v, 64 * j, h, t0, b);
            if (tile_group<ROLE, SAVED>(T_G) == g) tma_prefetch_4d(&map_g, 64 * j, h, t0, b);
          } else {
            if (tile_group<ROLE, SAVED>(T_Q) == g)
              tma_load_4d(sb + OFF_Q + j * Q_BOX, &map_q, bar, 32 * j, h, t0, b);
            if (tile_group<ROLE, SAVED>(T_K) == g)
              tma_load_4d(sb + OFF_K + j * Q_BOX, &map_k, bar, 32 * j, h, t0, b);
            if (tile_group<ROLE, SAVED>(T_V) == g)
              tma_load_4d(sb + OFF_V + j * V_BOX, &map_v, bar, 64 * j, h, t0, b);
            if (tile_group<ROLE, SAVED>(T_G) == g)
              tma_load_4d(sb + OFF_G + j * V_BOX, &map_g, bar, 64 * j, h, t0, b);
          }
        }
        if (SC && ROLE == R_DQ && g == 0 && !prefetch_only)  // the state copy S_c 2^-e_c
          bulk_load(sb + OFF_CP, p.saved.copy + ((size_t)bh * nc + c) * kCopyBytes, kCopyBytes, bar);
      };
      int armed_e = 0, armed_l = 0;
      for (int t = 0; t < n; ++t) {
        const int c = chunk_at<ROLE, SC>(t, c0, n);
        if (t >= 1 && !wait(cta, cta.bar(EMPTY_E), (t - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(cta.bar(FULL_E), group_bytes<ROLE, SAVED, SC>(0));
        load(c, 0, false);
        ++armed_e;
        if (t >= 1 && !wait(cta, cta.bar(EMPTY_L), (t - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(cta.bar(FULL_L), group_bytes<ROLE, SAVED, SC>(1));
        load(c, 1, false);
        ++armed_l;
        if (t + 1 < n) {
          load(chunk_at<ROLE, SC>(t + 1, c0, n), 0, true);
          load(chunk_at<ROLE, SC>(t + 1, c0, n), 1, true);
        }
      }
      if (armed_e) mbar_wait(cta.bar(FULL_E), (armed_e - 1) & 1, ctl, DRAIN_NS);
      if (armed_l) mbar_wait(cta.bar(FULL_L), (armed_l - 1) & 1, ctl, DRAIN_NS);
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int t = 0; t < n; ++t) {
        const uint32_t par = t & 1;
        // the give-up path's diagnostic: the drain barrier's first phase completes only after
        // this loop, so this bounded wait runs out and the CTA gives up
        if (t == ctl.stall_step) {
          wait(cta, cta.bar(DRAIN), 0, ctl);
          break;
        }
        if (!wait(cta, cta.bar(FULL_E), par, ctl)) break;
        // the previous chunk's TMEM-operand MMAs have read D_P
        if (t >= 1 && !wait(cta, cta.bar(X_DONE), (t - 1) & 1, ctl)) break;
        tc_fence_after();
        // score (inputs as given, bf16 or fp16; early tiles)
        if constexpr (ROLE == R_DQ || ROLE == R_DK) {
          // DQ: dP = dO V^T (A = dO, B = V);  DK: dP^T = V dO^T (A = V, B = dO); K = 192
          constexpr uint32_t ID = idesc_f16(128, 128, BF16, BF16, false, false);
          const uint32_t A = sb + (ROLE == R_DQ ? OFF_G : OFF_V), B = sb + (ROLE == R_DQ ? OFF_V : OFF_G);
#pragma unroll 1
          for (int ks = 0; ks < 12; ++ks) {
            const uint32_t off = (ks >> 2) * V_BOX + (ks & 3) * 32;
            mma_f16_ss(tmem + TM_P, smem_desc(A + off, 16, 1024, SW_128),
                       smem_desc(B + off, 16, 1024, SW_128), ID, ks > 0);
          }
        } else {  // DV: P^T = K Q^T, K = 96
          constexpr uint32_t ID = idesc_f16(128, 128, BF16, BF16, false, false);
#pragma unroll 1
          for (int ks = 0; ks < 6; ++ks) {
            const uint32_t off = (ks >> 1) * Q_BOX + (ks & 1) * 32;
            mma_f16_ss(tmem + TM_P, smem_desc(sb + OFF_K + off, 16, 512, SW_64),
                       smem_desc(sb + OFF_Q + off, 16, 512, SW_64), ID, ks > 0);
          }
        }
        mma_commit(cta.bar(P_DONE));
        // ---- the MMAs that need no masked score, once the fp16 operands are in place
        if (!wait(cta, cta.bar(EP_C1), par, ctl)) break;
        if (!(SC && ROLE == R_DQ) && !wait(cta, cta.bar(EP_S), par, ctl)) break;
        if (t >= 1 && !wait(cta, cta.bar(EP_X), (t - 1) & 1, ctl)) break;
        if (!wait(cta, cta.bar(FULL_L), par, ctl)) break;
        tc_fence_after();
        const uint32_t CP = sb + OFF_CP;
        if constexpr (ROLE == R_DQ) {
          // dq = dO'' S^T  (A = dO'' K-major, K = dv; B = state copy as [dk rows][dv], K-major)
          constexpr uint32_t ID1 = idesc_f16(128, 96, false, false, false, false);
#pragma unroll 1
          for (int ks = 0; ks < 12; ++ks)
            mma_f16_ss(tmem + TM_X,
                       smem_desc(sb + OFF_G + (ks >> 2) * V_BOX + (ks & 3) * 32, 16, 1024, SW_128),
                       smem_desc(CP + (ks >> 2) * S_ATOM + (ks & 3) * 32, 16, 1024, SW_128), ID1,
                       ks > 0);
        } else if constexpr (ROLE == R_DV) {
          // dv = K' dS  (A = K' K-major, K = dk; B = adjoint copy [dk][dv], MN-major)
          constexpr uint32_t ID1 = idesc_f16(128, 192, false, false, false, true);
#pragma unroll 1
          for (int ks = 0; ks < 6; ++ks)
            mma_f16_ss(tmem + TM_X,
                       smem_desc(sb + OFF_K + (ks >> 1) * Q_BOX + (ks & 1) * 32, 16, 512, SW_64),
                       smem_desc(CP + ks * 2048, S_ATOM, 1024, SW_128), ID1, ks > 0);
        } else {
          // dk = V' dS^T  (A = V' K-major, K = dv; B = adjoint copy [dk][dv], K-major)
          constexpr uint32_t ID2 = idesc_f16(128, 96, false, false, false, false);
#pragma unroll 1
          for (int ks = 0; ks < 12; ++ks)
            mma_f16_ss(tmem + TM_X,
                       smem_desc(sb + OFF_V + (ks >> 2) * V_BOX + (ks & 3) * 32, 16, 1024, SW_128),
                       smem_desc(CP + (ks >> 2) * S_ATOM + (ks & 3) * 32, 16, 1024, SW_128), ID2,
                       ks > 0);
        }
        // state / adjoint update, M = 128 (96 key channels + padding rows never read); DQ
        // with the forward's saved copies has no state to carry
        if constexpr (!(SC && ROLE == R_DQ)) {
          constexpr uint32_t ID = idesc_f16(128, 192, false, false, true, true);
          const uint32_t A = sb + (ROLE == R_DQ ? OFF_K : OFF_Q);  // K^T (DQ) or Q''^T / Q^T
          const uint32_t B = sb + (ROLE == R_DQ ? OFF_V : OFF_G);  // V' (DQ) or dO / dO''
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ss(tmem + TM_S, smem_desc(A + ks * 1024, Q_BOX, 512, SW_64),
                       smem_desc(B + ks * 2048, V_BOX, 1024, SW_128), ID, 1);
        }
        mma_commit(cta.bar(EMPTY_E));  // the early tiles' last readers are the MMAs above
        mma_commit(cta.bar(S_DONE));
        // ---- the masked scores are in TMEM (and DQ's r q in place)
        if (!wait(cta, cta.bar(EP_CONV), par, ctl)) break;
        tc_fence_after();
        if constexpr (ROLE == R_DQ) {
          //    + dP'' K  (A = dP'' from TMEM, K = j; B = K as [j][dk], MN-major)
          constexpr uint32_t ID2 = idesc_f16(128, 96, false, false, false, true);
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ts(tmem + TM_X, tmem + TM_P + 8 * ks,
                       smem_desc(sb + OFF_K + ks * 1024, Q_BOX, 512, SW_64), ID2, 1);
        } else if constexpr (ROLE == R_DV) {
          //    + P''^T dO  (A = P''^T from TMEM, K = i; B = dO as [i][dv], MN-major)
          constexpr uint32_t ID1 = idesc_f16(128, 192, false, false, false, true);
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ts(tmem + TM_X, tmem + TM_P + 8 * ks,
                       smem_desc(sb + OFF_G + ks * 2048, V_BOX, 1024, SW_128), ID1, 1);
        } else {
          //    + dP''^T Q  (A = dP''^T from TMEM, K = i; B = Q as [i][dk], MN-major)
          constexpr uint32_t ID1 = idesc_f16(128, 96, false, false, false, true);
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ts(tmem + TM_X, tmem + TM_P + 8 * ks,
                       smem_desc(sb + OFF_Q + ks * 1024, Q_BOX, 512, SW_64), ID1, 1);
        }
        mma_commit(cta.bar(X_DONE));
        if constexpr (ROLE == R_DQ) {
          // d_a: diag((r q)^T k) accumulated over every chunk (A = r q as [i][dk] MN-major,
          // B = K as [i][dk] MN-major); rows 96..127 are padding
          constexpr uint32_t ID = idesc_f16(128, 96, false, false, true, true);
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ss(tmem + TM_A, smem_desc(sb + OFF_Q + ks * 1024, Q_BOX, 512, SW_64),
                       smem_desc(sb + OFF_K + ks * 1024, Q_BOX, 512, SW_64), ID, (t > 0 || ks > 0));
        }
        mma_commit(cta.bar(EMPTY_L));
      }
      mma_commit(cta.bar(DRAIN));
      mbar_wait(cta.bar(DRAIN), 0, ctl, DRAIN_NS);
    }
  } else {
    // ------------------------------------------------------------------ epilogue warps 0..15
    // Warp w serves rows 32q..32q+31 (q = w & 3, one row per thread = TMEM lane) and part
    // sub = w >> 2 (0..3) of the work on each row: a quarter of the channels for the gate dot
    // products and the in-place conversions, two of the eight 16-column score blocks, a quarter
    // of the columns of the state copy and of the output rows.
    const int q4 = warp & 3, sub = warp >> 2;
    const int i = 32 * q4 + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const float lam = pw[1], lamC = expf((float)C * gamma);
    const float lamL = L_last == C ? lamC : pw[L_last];  // lambda^(tokens of the last chunk)
    const float lq = (i + 1 < C) ? pw[i + 1] : lamC;  // lambda^(row+1)
    const float lk_full = pw[C - 1 - i];              // lambda^(C-1-row)
    // in the last chunk: lambda^(L_last-1-row), and 0 on the zero rows past T
    const float lk_last = i < L_last ? pw[L_last - 1 - i] : 0.f;
    // the decay applied to the state (adjoint) before step t's update is lambda^(tokens of
    // chunk_at(t)): lamL only for the last chunk, which is the first step of the reverse scans
    // and the last of the forward one
    const float dec_first =
        (ROLE == R_DQ ? c0 == nc - 1 : c0 + n == nc) ? lamL : lamC;  // step 0
    uint8_t* const stage = base + OFF_STG + warp * 2048;  // two 1 KB output staging buffers
    auto qk = [&](int cc) { return qk_chunk(i, 3 * sub + cc); };  // this part's q/k chunks
    auto vg = [&](int cc) { return vg_chunk(i, 6 * sub + cc); };  // this part's v/dO chunks
    float range_max = 0.f;
    bool bad = false;

    // state copy S * 2^-e (rows < 96, this part's 48 columns) into the copy buffer,
    // D_S <- dec S (dec = lambda^(tokens of the chunk whose update follows)), and this warp's
    // max|S| into red[use & 1]
    auto publish_state = [&](int use, int e, float dec, const float* g_row, bool from_tmem) {
      float m = 0.f;
      if (q4 < 3) {
        const float sc = pow2i(-e);
        const int col = 48 * sub;
        uint32_t r[48];
        if (from_tmem) {
          tmem_ld32(trow + TM_S + col, *reinterpret_cast<uint32_t(*)[32]>(r));
          tmem_ld16(trow + TM_S + col + 32, *reinterpret_cast<uint32_t(*)[16]>(r + 32));
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j4 = 0; j4 < 12; ++j4) {  // 12 loads in flight (rows are 16-byte aligned)
            const float4 x = g_row ? __ldg(reinterpret_cast<const float4*>(g_row + col) + j4)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            r[4 * j4] = __float_as_uint(x.x);
            r[4 * j4 + 1] = __float_as_uint(x.y);
            r[4 * j4 + 2] = __float_as_uint(x.z);
            r[4 * j4 + 3] = __float_as_uint(x.w);
          }
        }
        const float2 sc2 = make_float2(sc, sc), dec2 = make_float2(dec, dec);
#pragma unroll
        for (int q8 = 0; q8 < 6; ++q8) {
          const int nn = col + 8 * q8;
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 x = make_float2(__uint_as_float(r[8 * q8 + 2 * u]),
                                         __uint_as_float(r[8 * q8 + 2 * u + 1]));
            const float2 y = __fmul2_rn(x, sc2);
            w[u] = pack_h2(y.x, y.y);
          }
          *(uint4*)(base + OFF_CP + (nn >> 6) * S_ATOM + swz_off(i, (nn & 63) >> 3, 128)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
#pragma unroll
        for (int j = 0; j < 48; j += 2) {
          const float2 x = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
          m = fmaxf(m, fmaxf(fabsf(x.x), fabsf(x.y)));
          const float2 y = __fmul2_rn(x, dec2);
          r[j] = __float_as_uint(y.x);
          r[j + 1] = __float_as_uint(y.y);
        }
        tmem_st32(trow + TM_S + col, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_st16(trow + TM_S + col + 32, *reinterpret_cast<uint32_t(*)[16]>(r + 32));
        tmem_wait_st();
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[(use & 1) * 16 + warp] = m;
      if (tid == 0) es[use & 1] = e;
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(cta.bar(EP_S));
    };

    // starting state (DQ) or adjoint (DV, DK): the caller's initial state / d_final_state for
    // a whole pair, the segment passes' for a part of a cut one; its exact max first
    const float* src0 = cut_idx >= 0 ? (ROLE == R_DQ ? p.seg_state : p.seg_adj)
                                     : (ROLE == R_DQ ? p.init : p.dfin);
    const long long slot0 = cut_idx >= 0 ? cut_idx : bh;
    const float* g_row0 = (src0 && i < DK) ? src0 + ((size_t)slot0 * DK + i) * DV : nullptr;
    int e_cur = 0;
    {
      float m = 0.f;
      if (g_row0) {
        const float4* g4 = reinterpret_cast<const float4*>(g_row0 + 48 * sub);
#pragma unroll
        for (int j4 = 0; j4 < 12; ++j4) {
          const float4 x = __ldg(g4 + j4);
          m = fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[32 + warp] = m;
      mbar_arrive(cta.bar(RED));
    }
    bool ok = SC && ROLE == R_DQ ? true : wait_warp(cta, cta.bar(RED), 0, ctl);
    if (ok && !(SC && ROLE == R_DQ)) {
      e_cur = state_exponent(max16(red + 32));
      if (e_cur < 0) {
        bad = true;
        e_cur = 0;
      }
      publish_state(0, e_cur, dec_first, g_row0, false);
    }

    // in-register fp16 copy of three q/k chunks of this part (x: 16-bit input words), scaled
    // by s and stored back in place
    auto cvt3 = [&](uint4 (&x)[3], uint32_t tile_off, float s, float& vmax) {
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) {
        uint32_t* w = reinterpret_cast<uint32_t*>(&x[cc]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = ld16<BF16>(w[e] & 0xFFFFu) * s, a1 = ld16<BF16>(w[e] >> 16) * s;
          vmax = fmaxf(vmax, fmaxf(fabsf(a0), fabsf(a1)));
          w[e] = pack_h2(a0, a1);
        }
        *(uint4*)(base + tile_off + qk(cc)) = x[cc];
      }
    };

    for (int t = 0; t < n && ok; ++t) {
      const uint32_t par = t & 1;
      const int c = chunk_at<ROLE, SC>(t, c0, n);
      const float lk = c == nc - 1 ? lk_last : lk_full;
      // the saved gate of this row (issued before the waits; rows past T, all zeros, have
      // sigmoid(0))
      float sg_saved = 0.5f;
      if (SAVED && c * C + i < T) sg_saved = __ldg(p.gate + (size_t)bh * T + c * C + i);
      // DQ with the forward's saved copies: the exponent of this chunk's copy
      if (SC && ROLE == R_DQ) e_cur = __ldg(p.saved.exp + (size_t)bh * nc + c);
      if (!(ok = wait_warp(cta, cta.bar(FULL_E), par, ctl))) break;
      if (!(ok = wait_warp(cta, cta.bar(FULL_L), par, ctl))) break;
      // ---- gate partial sum z = q.(a*k) over this part's 24 channels (unless the gate is
      // given), fused with the fp16 copy of whichever of q, k the score MMA does not read
      // (DQ: k, DK: q, both scale 1); DV's score reads both, so DV converts them once the
      // score MMA is done
      float amax = 0.f, bmax = 0.f;  // A and B operands of the state MMA
      uint4 xq[3], xk[3];
      if (!SAVED || ROLE == R_DK) {
#pragma unroll
        for (int cc = 0; cc < 3; ++cc) xq[cc] = *(const uint4*)(base + OFF_Q + qk(cc));
      }
      if (!SAVED || ROLE == R_DQ) {
#pragma unroll
        for (int cc = 0; cc < 3; ++cc) xk[cc] = *(const uint4*)(base + OFF_K + qk(cc));
      }
      if (!SAVED) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int cc = 0; cc < 3; ++cc) {
          const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xq[cc]);
          const uint32_t* yw = reinterpret_cast<const uint32_t*>(&xk[cc]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = 24 * sub + 8 * cc + 2 * e;
            acc0 = fmaf(ld16<BF16>(xw[e] & 0xFFFFu) * sa[d], ld16<BF16>(yw[e] & 0xFFFFu), acc0);
            acc1 = fmaf(ld16<BF16>(xw[e] >> 16) * sa[d + 1], ld16<BF16>(yw[e] >> 16), acc1);
          }
        }
        gate_part[sub * 128 + i] = acc0 + acc1;
        mbar_arrive(cta.bar(QG0 + q4));
      }
      if constexpr (ROLE == R_DQ) cvt3(xk, OFF_K, 1.f, amax);  // K (state A, dP''K B)
      if constexpr (ROLE == R_DK) cvt3(xq, OFF_Q, 1.f, amax);  // Q (adjoint A, dP''^T Q B)
      if constexpr (ROLE == R_DV) convert_row<BF16, 6, 3>(base + OFF_G, vg, 1.f, bmax);  // dO
      // ---- once the score MMA has read its 16-bit tiles: their fp16 copies
      if (!(ok = wait_warp(cta, cta.bar(P_DONE), par, ctl))) break;
      tc_fence_after();
      if constexpr (ROLE == R_DQ) {
        if constexpr (!SC)  // V' (state B), dO'' (A of dO'' S^T)
          convert_rows2<BF16, 6, 3>(base + OFF_V, vg, lk, bmax, base + OFF_G, vg, lq, range_max);
        else
          convert_row<BF16, 6, 3>(base + OFF_G, vg, lq, range_max);
      } else if constexpr (ROLE == R_DV) {
        // Q'' (adjoint A), K' (A of K' dS)
        convert_rows2<BF16, 3, 3>(base + OFF_Q, qk, lq, amax, base + OFF_K, qk, lk, range_max);
      } else {
        // V' (A of V' dS^T), dO'' (adjoint B)
        convert_rows2<BF16, 6, 3>(base + OFF_V, vg, lk, range_max, base + OFF_G, vg, lq, bmax);
      }
      // every fp16 operand but DQ's r q is in place: the state MMA and the output MMA's
      // state-copy part may run while the masked scores are made
      fence_proxy_async();
      mbar_arrive(cta.bar(EP_C1));
      range_max = fmaxf(range_max, fmaxf(amax, bmax));
      {
        float am = amax, bm = bmax;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        }
        if (lane == 0) {
          abmax[par * 32 + warp] = am;
          abmax[par * 32 + 16 + warp] = bm;
        }
      }
      // ---- the row's gate: the saved one, or the four partial sums
      float sg = sg_saved;
      if (!SAVED) {
        if (!(ok = wait_warp(cta, cta.bar(QG0 + q4), par, ctl))) break;
        sg = sigmoid((gate_part[i] + gate_part[128 + i]) + (gate_part[256 + i] + gate_part[384 + i]));
      }
      // ---- masked score copy, scaled by 2^-e of this step's state copy: this part's 16-column
      // blocks hb = sub, sub+4 of the quadrant's rows, packed to fp16 pairs in registers.
      // Block hb's pairs go to 32-bit columns 8hb..8hb+7, inside block hb/2's fp32 columns, so
      // the four parts of a quadrant finish reading before any of them writes.
      if (!(SC && ROLE == R_DQ) && !(ok = wait_warp(cta, cta.bar(EP_S), par, ctl))) break;
      {
        const float psc = pow2i(-(SC && ROLE == R_DQ ? e_cur : es[par]));
        float pmax = 0.f;
        uint32_t pk[2][8];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int hb = sub + 4 * m;
          const int cb = 16 * hb;
          // DQ keeps columns j <= i (rows = queries i), DV and DK columns i >= j (rows = keys j)
          const bool live = ROLE == R_DQ ? hb <= 2 * q4 + 1 : hb >= 2 * q4;
          // every element of the block is kept for all 32 rows of the quadrant (all but the two
          // blocks on the diagonal): no per-element mask, no diagonal (warp-uniform)
          const bool full = ROLE == R_DQ ? hb <= 2 * q4 - 1 : hb >= 2 * q4 + 2;
          float sc[16];
          if (full) {
            uint32_t r[16];
            tmem_ld16(trow + TM_P + cb, r);
            tmem_wait_ld();
            if constexpr (ROLE == R_DQ) {
              float f = pw[i - (cb + 15)] * psc;  // going left from cb+15
#pragma unroll
              for (int u = 15; u >= 0; --u) {
                sc[u] = __uint_as_float(r[u]) * f;
                f = f * lam;
              }
            } else {
              float f = pw[cb - i] * psc;  // going right from cb
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                sc[u] = __uint_as_float(r[u]) * f;
                f = f * lam;
              }
            }
          } else if (live) {
            uint32_t r[16];
            tmem_ld16(trow + TM_P + cb, r);
            tmem_wait_ld();
            float dg = 0.f;
            if constexpr (ROLE == R_DQ) {
              float f = pw[max(i - (cb + 15), 0)] * psc;  // going left from min(i, cb+15)
#pragma unroll
              for (int u = 15; u >= 0; --u) {
                const bool in = cb + u <= i;
                sc[u] = in ? __uint_as_float(r[u]) * f : 0.f;
                f = in ? f * lam : f;
                dg = (cb + u == i) ? __uint_as_float(r[u]) : dg;
              }
            } else {
              float f = pw[max(cb - i, 0)] * psc;  // going right from max(j, cb)
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const bool in = cb + u >= i;
                sc[u] = in ? __uint_as_float(r[u]) * f : 0.f;
                f = in ? f * lam : f;
                dg = (cb + u == i) ? __uint_as_float(r[u]) : dg;
                // DV: the self-augmentation sigmoid(z_j) dO_j rides on the diagonal, so that
                // P''^T dO includes it: (P^T + diag(sigmoid(z))) 2^-e
                if (ROLE == R_DV && cb + u == i) sc[u] += sg * psc;
              }
            }
            // DQ, DK: the score's diagonal is dO_i . v_i, the gate's other factor
            if (ROLE != R_DV && (i >> 4) == hb) dpv[i] = dg;
          } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) sc[u] = 0.f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            pmax = fmaxf(pmax, fmaxf(fabsf(sc[2 * u]), fabsf(sc[2 * u + 1])));
            pk[m][u] = pack_h2(sc[2 * u], sc[2 * u + 1]);
          }
        }
        range_max = fmaxf(range_max, pmax);
        tc_fence_before();
        mbar_arrive(cta.bar(QS0 + q4));
        if (!(ok = wait_warp(cta, cta.bar(QS0 + q4), par, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < 2; ++m) tmem_st8(trow + TM_P + 8 * (sub + 4 * m), pk[m]);
        tmem_wait_st();
      }
      float rr = 0.f;  // r = sigmoid'(z) (dO.v) (DQ, DK)
      if constexpr (ROLE != R_DV) rr = sg * (1.f - sg) * dpv[i];
      if constexpr (ROLE == R_DQ) convert_row<BF16, 3, 3>(base + OFF_Q, qk, rr, range_max);  // r q
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(cta.bar(EP_CONV));
      // ---- the self-augmentation operand of the rows (DQ: k, DK: q, this part's 24 channels,
      // fp16) into registers; then this warp is done with the late tiles.  DV's term is inside
      // D_X already.
      uint4 vv[3];
      if constexpr (ROLE != R_DV) {
#pragma unroll
        for (int ch = 0; ch < 3; ++ch)
          vv[ch] = *(const uint4*)(base + (ROLE == R_DQ ? OFF_K : OFF_Q) + qk(ch));
      }
      mbar_arrive(cta.bar(EMPTY_L));
      // ---- the state update ran: next state copy (the serial step), while the output MMA's
      // TMEM-operand part runs
      int e_next = e_cur;
      if (!(SC && ROLE == R_DQ) && !(ok = wait_warp(cta, cta.bar(S_DONE), par, ctl))) break;
      tc_fence_after();
      if (!(SC && ROLE == R_DQ) && t < n - 1) {
        // bound on the next state: all parts' operand maxima and max|S| of this step's copy
        // (decayed by this step's factor)
        if (!(ok = wait_warp(cta, cta.bar(EP_CONV), par, ctl))) break;
        e_next = state_exponent((t == 0 ? dec_first : lamC) * max16(red + par * 16) +
                                (float)C * max16(abmax + par * 32) * max16(abmax + par * 32 + 16));
        if (e_next < 0) {
          bad = true;
          e_next = 0;
        }
        publish_state(t + 1, e_next, (ROLE == R_DQ && c0 + t + 2 == nc) ? lamL : lamC, nullptr,
                      true);
      }
      // ---- output rows, this part's columns: x = 2^e D_X (+ r (a * k|q) for DQ, DK)
      if (!(ok = wait_warp(cta, cta.bar(X_DONE), par, ctl))) break;
      tc_fence_after();
      if (lane == 0) bulk_wait_read<0>();  // the staging buffers are free again
      __syncwarp();
      {
        const float osc = pow2i(e_cur);
        const int t0 = c * C + 32 * q4;  // first token of this warp's rows (boxes past T: none)
        constexpr int NCOL = NX / 4;  // 24 (DQ, DK) or 48 (DV)
        uint32_t rbuf[16];  // blocks read in pairs: one TMEM round trip per two blocks
        emit_rows8_tma<NCOL / 8>(
            stage, lane,
            [&](int k, float (&x)[8]) {
              const int col = NCOL * sub + 8 * k;
              if ((k & 1) == 0) {
                if (k + 1 < NCOL / 8)
                  tmem_ld16(trow + TM_X + col, rbuf);
                else
                  tmem_ld8(trow + TM_X + col, *reinterpret_cast<uint32_t(*)[8]>(rbuf));
                tmem_wait_ld();
              }
              const uint32_t* r = rbuf + 8 * (k & 1);
              if constexpr (ROLE == R_DV) {
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(r[j]) * osc;
              } else {
                float f8[8];
                unpack8<false>(vv[k], f8);
                const float4 a0 = *reinterpret_cast<const float4*>(sa + col);
                const float4 a1 = *reinterpret_cast<const float4*>(sa + col + 4);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  x[j] = fmaf(__uint_as_float(r[j]), osc, rr * av[j] * f8[j]);
              }
            },
            [&](int k, uint32_t src) {
              if (t0 < T) tma_store_4d(&map_out, src, NCOL * sub + 8 * k, h, t0, b);
            });
      }
      tc_fence_before();
      mbar_arrive(cta.bar(EP_X));
      // ---- adjoint of the initial state (DV, after the last step = chunk 0)
      if (ROLE == R_DV && t == n - 1 && c0 == 0 && p.want_dinit && q4 < 3) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint32_t rb[16];
        emit_rows8_tma<6>(
            stage, lane,
            [&](int k, float (&f)[8]) {
              if ((k & 1) == 0) {
                tmem_ld16(trow + TM_S + 48 * sub + 8 * k, rb);
                tmem_wait_ld();
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(rb[8 * (k & 1) + j]);
            },
            [&](int k, uint32_t src) { tma_store_3d(&map_dinit, src, 48 * sub + 8 * k, 32 * q4, bh); });
      }
      e_cur = e_next;
    }
    // DQ: d_a of this (b, h) is the diagonal of the accumulated (r q)^T k; row d (lane of
    // quadrant d / 32) takes column d, once the last step's d_a MMAs are done
    if (ROLE == R_DQ && ok && sub == 0 && q4 < 3 && wait_warp(cta, cta.bar(EMPTY_L), (n - 1) & 1, ctl)) {
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(trow + TM_A + 32 * q4, r);
      tmem_wait_ld();
      float dd = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) dd = (j == lane) ? __uint_as_float(r[j]) : dd;
      float* da = cut_idx >= 0 ? p.da_split + (size_t)cut_idx * DK : p.da_part + (size_t)bh * DK;
      da[32 * q4 + lane] = dd;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (bad || range_max >= 65504.f) record_error(ctl, DEV_RANGE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16, bool SAVED, bool SC>
__global__ void __launch_bounds__(THREADS, 1)
bwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_g,
           const __grid_constant__ CUtensorMap map_dq, const __grid_constant__ CUtensorMap map_dk,
           const __grid_constant__ CUtensorMap map_dv, const __grid_constant__ CUtensorMap map_dinit,
           BwdParams p, DevCtl ctl) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Cta cta;
  cta.base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  cta.sb = smem_u32(cta.base);
  cta.bar_off = OFF_BAR;
  cta.abort_off = OFF_ABORT;
  // three roles per pair, adjacent so that they read each chunk's tiles at about the same time
  // (through L2), the longest first -- DV, DK, then DQ -- so that the launch's last CTAs tend to
  // be the short ones; the whole pairs first, then the parts of the cut ones
  const int nc = (p.T + C - 1) / C;
  const int role = ((int)blockIdx.x + 1) % 3, w = blockIdx.x / 3;
  const bool cut = w >= p.plan.whole;
  const int cut_idx = cut ? w - p.plan.whole : -1;
  const int part = cut ? cut_idx % p.plan.parts : 0;
  const int bh = cut ? p.plan.whole + cut_idx / p.plan.parts : w;
  const int c0 = cut ? part_begin(part, nc, p.plan.parts) : 0;
  const int n = cut ? part_begin(part + 1, nc, p.plan.parts) - c0 : nc;
  // the d_aug reduction, launched next as this grid's programmatic dependent, may start once
  // every CTA has (it waits for this grid to finish)
  griddep_launch_dependents();
  // a part starts from the states the segment passes leave: when this grid is launched as
  // their programmatic dependent it may be running before they finish (whole pairs need none)
  if (cut) griddep_wait();
  if (role == R_DQ)
    run_role<R_DQ, BF16, SAVED, SC>(cta.base, cta, bh, c0, n, cut_idx, p, map_q, map_k, map_v, map_g, map_dq,
                         map_dinit, ctl);
  else if (role == R_DV)
    run_role<R_DV, BF16, SAVED, false>(cta.base, cta, bh, c0, n, cut_idx, p, map_q, map_k, map_v, map_g, map_dv,
                         map_dinit, ctl);
  else
    run_role<R_DK, BF16, SAVED, false>(cta.base, cta, bh, c0, n, cut_idx, p, map_q, map_k, map_v, map_g, map_dk,
                         map_dinit, ctl);
}

// d_aug[h, d] = sum over b of the per-(b, h) partial sums (a cut pair's: its parts' in order).
// One warp per output: lane l adds b = l, l + 32, ... in order, then a fixed shuffle tree, whose
// lane 0 writes (deterministic).  Launched as the chunked kernel's programmatic dependent, so its
// launch overlaps that kernel's last wave; it waits for the kernel's partial sums.
constexpr int RED_WARPS = 8;
__global__ void __launch_bounds__(RED_WARPS * 32)
reduce_daug_kernel(const float* __restrict__ part, const float* __restrict__ split,
                   float* __restrict__ d_aug, int B, int H, SplitPlan plan) {
  griddep_wait();
  const int idx = blockIdx.x * RED_WARPS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (idx >= H * DK) return;  // (a whole warp)
  const int h = idx / DK, d = idx % DK;
  // whole pairs are b*H + h < whole: b < b_whole
  const int b_whole = min(B, (plan.whole - h + H - 1) / H);
  float s = 0.f;
  for (int b = lane; b < B; b += 32) {
    float t = 0.f;
    if (b < b_whole) {
      t = part[((size_t)b * H + h) * DK + d];
    } else {
      const size_t x = (size_t)b * H + h - plan.whole;
      for (int j = 0; j < plan.parts; ++j) t += split[(x * plan.parts + j) * DK + d];
    }
    s += t;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) d_aug[idx] = s;
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int B, int T, int H) {
  (void)T;
  return (((size_t)B * H * DK * sizeof(float)) + 255) & ~(size_t)255;
}

cudaError_t launch_chunk_bwd(const BwdArgs& a, DevCtl ctl, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mg, mdq, mdk, mdv, mdi;
  if (!make_tmap_seq_16bit(&mq, a.q, DK, a.H, a.T, a.B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_seq_16bit(&mk, a.k, DK, a.H, a.T, a.B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_seq_16bit(&mv, a.v, DV, a.H, a.T, a.B, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, a.bf16) ||
      !make_tmap_seq_16bit(&mg, a.dO, DV, a.H, a.T, a.B, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, a.bf16) ||
      !make_tmap_seq_out_f32(&mdq, a.dq, DK, a.H, a.T, a.B, 8) ||
      !make_tmap_seq_out_f32(&mdk, a.dk, DK, a.H, a.T, a.B, 8) ||
      !make_tmap_seq_out_f32(&mdv, a.dv, DV, a.H, a.T, a.B, 8) ||
      !make_tmap_state_f32(&mdi, a.dinit ? (const void*)a.dinit : (const void*)a.dv,
                           (long long)a.B * a.H, 8))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.log_decay = a.log_decay;
  p.aug = a.aug;
  p.init = a.init;
  p.dfin = a.dfin;
  p.da_part = static_cast<float*>(a.workspace);
  p.T = a.T;
  p.H = a.H;
  p.want_dinit = a.dinit != nullptr;
  p.plan = a.plan;
  const bool sc = a.saved.copy != nullptr;  // DQ reads the forward's state copies
  if (p.plan.parts <= 1 || (!a.seg_state && !sc) || !a.seg_adj || !a.da_split) {
    p.plan.whole = a.B * a.H;
    p.plan.parts = 1;
    p.plan.overlap = false;
  }
  p.seg_state = a.seg_state;
  p.seg_adj = a.seg_adj;
  p.da_split = a.da_split;
  p.gate = a.gate;
  p.saved = a.saved;
  using Kern = decltype(&bwd_kernel<true, true, true>);
  const Kern kerns[2][2][2] = {
      {{bwd_kernel<false, false, false>, bwd_kernel<false, false, true>},
       {bwd_kernel<false, true, false>, bwd_kernel<false, true, true>}},
      {{bwd_kernel<true, false, false>, bwd_kernel<true, false, true>},
       {bwd_kernel<true, true, false>, bwd_kernel<true, true, true>}}};
  const Kern kern = kerns[a.bf16 ? 1 : 0][a.gate ? 1 : 0][sc ? 1 : 0];
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid =
      3 * (p.plan.whole + ((long long)a.B * a.H - p.plan.whole) * p.plan.parts);
  {
    // with plan.overlap: the segment passes' programmatic dependent (see the forward)
    PdlLaunch L(dim3((unsigned)grid), dim3(THREADS), SMEM_BYTES, stream, p.plan.overlap);
    if ((e = cudaLaunchKernelEx(&L.cfg, kern, mq, mk, mv, mg, mdq, mdk, mdv, mdi, p, ctl)) !=
        cudaSuccess)
      return e;
  }
  const int n = a.H * DK;
  PdlLaunch R(dim3((n + RED_WARPS - 1) / RED_WARPS), dim3(RED_WARPS * 32), 0, stream, true);
  return cudaLaunchKernelEx(&R.cfg, reduce_daug_kernel, (const float*)p.da_part,
                            (const float*)p.da_split, a.d_aug, a.B, a.H, p.plan);
}

}  // namespace gla
