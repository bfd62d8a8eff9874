// chunk_fwd.cu -- chunked forward of the Simple GLA mixer on tcgen05 tensor cores.
//
// Method ("Beyond the KV cache ... Laplace 3B ...", section "Challenge 1", the chunked form
// of the "GLA mixer" recurrence).  Per (b, h) and chunk c of C = 128 tokens, with
// D_ij = lambda^(i-j) (i >= j, else 0), Lq = diag(lambda^(i+1)), Lk = diag(lambda^(C-1-j)):
//   O_c     = (Q K^T o D + diag(sigmoid(z))) V + Lq Q S_c   (intra + self-augmentation + inter)
//   S_{c+1} = lambda^C S_c + K^T Lk V                        (the only serial step)
//
// One CTA owns one (b, h) and walks its chunks in order; the fp32 state never leaves the chip.
//   producer  TMA producer: q, k tiles (3 boxes of 32 channels, 64-byte swizzle) and v tiles
//               (3 boxes of 64 channels, 128-byte swizzle) into a 2-stage ring (no L2
//               prefetch: measured, it slowed the loads it was meant to hide); the first
//               tiles are issued by the thread that initialises the barriers, during setup.
//   MMA warp  tcgen05 issuer (one thread) and TMEM owner (512 columns):
//                 D_P [384,512)  P = Q K^T (bf16/fp16 inputs as given); the masked fp16
//                                copy P'' is written back in place (64 columns) and read
//                                from TMEM as the A operand of P'' V
//                 D_O [  0,192)  O = Q'' S_c + P'' V           (fp16 operands)
//                 D_S [192,384)  S = lambda^C S + K'^T V       (fp16 operands, fp32 state;
//                                rows 96..127 are padding and never read)
//   convert     warps 0..7 (the plain forward: two per row quadrant splitting the channels
//               and score blocks) or 0..3 (with the fused output epilogue: one per quadrant),
//               thread = token row i (= TMEM lane), one chunk ahead of the
//               emit group: V -> fp16 in place; z = q.(a*k); Q'' = fp16(lambda^(i+1) q) and
//               K' = fp16(lambda^(127-i) k) in place; P'' = fp16((mask(P) + diag(sigmoid(z)))
//               * 2^-e) into TMEM -- the self-augmentation rides on the diagonal of P''.
//   emit        the next 8 warps, same rows, two warps per row quadrant splitting the value
//               columns: (1) the serial step -- S -> fp16(S * 2^-e') into the drained q/k
//               slot (B operand of the next Q'' S) and D_S <- lambda^C D_S; (2) the output rows
//               o = 2^e D_O as fp32, TMA-stored from per-warp staging.
// The output MMA is issued in two parts: Q''S as soon as Q'' is in place (it releases the
// slot of the state copy, so the next chunk's q, k load starts early), P''V once the masked
// scores are in TMEM.
// fp16 operands (11-bit significand) keep the long-memory heads accurate; the state copy is
// scaled by a power of two e' chosen from a bound on max|S| so it never overflows fp16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "scan_common.cuh"
#include "tmap.h"

namespace gla {
namespace {

using namespace scan;

constexpr uint32_t Q_BOX = 8192;    // 128 rows x 64 B (32 channels), SW64
constexpr uint32_t V_BOX = 16384;   // 128 rows x 128 B (64 channels), SW128
constexpr uint32_t OFF_Q = 0, OFF_K = 3 * Q_BOX, OFF_V = 6 * Q_BOX;
constexpr uint32_t STAGE = OFF_V + 3 * V_BOX;  // 98304
constexpr uint32_t OFF_STG = 2 * STAGE;        // output staging, 8 emit warps x 4 KB
constexpr uint32_t S_ATOM = 12288;             // state copy: 3 atoms of 96 rows x 128 B
constexpr uint32_t OFF_BAR = OFF_STG + 8 * 4096;
constexpr uint32_t NBAR = 32;
constexpr uint32_t OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_RED = OFF_TMEM + 16;     // float red[3][8]: per-warp max|S|
constexpr uint32_t OFF_ES = OFF_RED + 96;       // int es[2]: state-copy exponent per chunk parity
constexpr uint32_t OFF_KV = OFF_ES + 16;        // float kvmax[2][16]: per-warp max|K'|, max|V|
constexpr uint32_t OFF_A = OFF_KV + 128;        // float a[96]: aug_balance of the head
constexpr uint32_t OFF_PW = OFF_A + 384;        // float pw[128] = lambda^d
constexpr uint32_t OFF_XCH = OFF_PW + 512;      // float xch[2][128]: row sums of o^2 (gated)
constexpr uint32_t OFF_ZX = OFF_XCH + 1024;     // float zx[128]: second-half gate partial sums
constexpr uint32_t SMEM_USED = OFF_ZX + 512;
// The whole opt-in maximum is requested; the kernel aligns its base to 1024 bytes and
// refuses to run (GLA_ERR_LAYOUT, before touching shared memory) if the padding that
// takes would not fit.  The dynamic shared window normally starts 1024-aligned.
constexpr uint32_t SMEM_BYTES = 232448;
static_assert(SMEM_USED <= SMEM_BYTES, "shared memory budget");
static_assert(3 * S_ATOM <= 6 * Q_BOX, "state copy fits in a drained q/k slot");

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
  RED = 15,  // exchange of the per-warp max|S| inside the emit group
  QX = 16,   // 16..19 (gated output): the two warps of row quadrant q have their row sums
  EP_Q = 20,  // convert group: Q'' of the chunk is in place (the Q''S MMA may start)
  ZX0 = 24,   // 24..27: quadrant q's second convert warp has written its gate partial sums
  QS0 = 28,   // 28..31: both convert warps of quadrant q have read their score blocks
};

// Warp layout by variant: CW convert warps per row quadrant (warps 0..4CW-1), then 8 emit
// warps, the TMA producer and the MMA issuer.  The plain forward splits the convert work over
// two warps per quadrant (18 warps, 96 registers); the forward with the fused output epilogue,
// whose emit warps need more registers, keeps one (14 warps, 128 registers).
template <bool GATED>
struct Layout {
  static constexpr int CW = GATED ? 1 : 2;
  static constexpr int CONVERT_WARPS = 4 * CW;
  static constexpr int PRODUCER_WARP = CONVERT_WARPS + 8, MMA_WARP = PRODUCER_WARP + 1;
  static constexpr int THREADS = (MMA_WARP + 1) * 32;
  static constexpr int CONVERT_THREADS = 32 * CONVERT_WARPS;
};
constexpr int EMIT_THREADS = 256;  // 8 emit warps

template <bool BF16, bool GATED>
__global__ void __launch_bounds__(Layout<GATED>::THREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
           const __grid_constant__ CUtensorMap map_fin, const float* __restrict__ log_decay,
           const float* __restrict__ aug, const float* __restrict__ init, float* __restrict__ out,
           float* __restrict__ fin, int T, int H, SplitPlan plan,
           const float* __restrict__ seg_init, const float* __restrict__ seg_max, StatePages sp,
           const __grid_constant__ CUtensorMap map_y, OutGate og, float* __restrict__ gate_out,
           SavedStates saved, DevCtl ctl) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Cta cta;
  cta.base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  if ((uint32_t)(cta.base - smem_raw) + SMEM_USED > SMEM_BYTES) {
    if (threadIdx.x == 0) record_error(ctl, DEV_LAYOUT);
    return;
  }
  cta.sb = smem_u32(cta.base);
  cta.bar_off = OFF_BAR;
  cta.abort_off = OFF_ABORT;
  uint8_t* const base = cta.base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  using L = Layout<GATED>;
  constexpr int CW = L::CW, CONVERT_WARPS = L::CONVERT_WARPS;
  constexpr int PRODUCER_WARP = L::PRODUCER_WARP, MMA_WARP = L::MMA_WARP;
  // chunks of a sequence; the last one holds L_last = 1..C tokens (rows past T are zeros)
  const int nc = (T + C - 1) / C, L_last = T - (nc - 1) * C;
  // this CTA's pair and chunk range [c0, c0 + n): a whole pair, or part `part` of a cut one
  const bool cut = (int)blockIdx.x >= plan.whole;
  const int cut_idx = cut ? (int)blockIdx.x - plan.whole : 0;
  const int part = cut_idx % plan.parts;
  const int bh = cut ? plan.whole + cut_idx / plan.parts : (int)blockIdx.x, b = bh / H, h = bh % H;
  const int c0 = cut ? part_begin(part, nc, plan.parts) : 0;
  const int n = cut ? part_begin(part + 1, nc, plan.parts) - c0 : nc;
  // a part starts from the state the segment passes leave: when this grid is launched as their
  // programmatic dependent it may be running before they finish (whole pairs need nothing)
  if (cut) griddep_wait();
  const float gamma = __ldg(log_decay + h);
  float* pw = (float*)(base + OFF_PW);
  float* red = (float*)(base + OFF_RED);
  int* es = (int*)(base + OFF_ES);
  float* kvmax = (float*)(base + OFF_KV);
  float* sa = (float*)(base + OFF_A);
  uint32_t* tmem_slot = (uint32_t*)(base + OFF_TMEM);

  // the TMA copies of step c (chunk c0 + c) into ring stage c & 1 (the producer thread)
  auto load_v = [&](int c) {
    const uint32_t s = c & 1, st = cta.sb + s * STAGE;
    mbar_arrive_expect_tx(cta.bar(V_FULL + s), V_BYTES);
    for (int j = 0; j < 3; ++j)
      tma_load_4d(st + OFF_V + j * V_BOX, &map_v, cta.bar(V_FULL + s), 64 * j, h, (c0 + c) * C, b);
  };
  auto load_qk = [&](int c) {
    const uint32_t s = c & 1, st = cta.sb + s * STAGE;
    mbar_arrive_expect_tx(cta.bar(QK_FULL + s), QK_BYTES);
    for (int j = 0; j < 3; ++j) {
      tma_load_4d(st + OFF_Q + j * Q_BOX, &map_q, cta.bar(QK_FULL + s), 32 * j, h, (c0 + c) * C, b);
      tma_load_4d(st + OFF_K + j * Q_BOX, &map_k, cta.bar(QK_FULL + s), 32 * j, h, (c0 + c) * C, b);
    }
  };

  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (tid == PRODUCER_WARP * 32) {
    for (uint32_t s = 0; s < 2; ++s) {
      mbar_init(cta.bar(QK_FULL + s), 1);
      mbar_init(cta.bar(V_FULL + s), 1);
      mbar_init(cta.bar(QK_EMPTY + s), 1);
      mbar_init(cta.bar(V_EMPTY + s), 1);  // the MMAs are the only readers of v
    }
    mbar_init(cta.bar(P_DONE), 1);
    mbar_init(cta.bar(O_DONE), 1);
    mbar_init(cta.bar(S_DONE), 1);
    mbar_init(cta.bar(DRAIN), 1);
    mbar_init(cta.bar(EP_CONV), L::CONVERT_THREADS);
    mbar_init(cta.bar(EP_Q), L::CONVERT_THREADS);
    mbar_init(cta.bar(EP_O), EMIT_THREADS);     // emit group
    mbar_init(cta.bar(EP_S), EMIT_THREADS);     // emit group
    mbar_init(cta.bar(RED), EMIT_THREADS);      // emit group
    for (int q = 0; q < 4; ++q) {
      mbar_init(cta.bar(QX + q), 64);
      mbar_init(cta.bar(ZX0 + q), 32);
      mbar_init(cta.bar(QS0 + q), 32 * CW);
    }
    *cta.abort_flag() = 0;
    fence_barrier_init();
    // the first tiles load while the CTA finishes setting up (the initialised barriers made
    // visible to the async proxy first): v, q, k of step 0 and v of step 1 -- q, k of step 1
    // go into the slot of step 0's state copy and wait for its Q''S (QK_EMPTY)
    fence_proxy_async();
    // a part's starting state (72 KB, read twice by the emit warps) starts on its way to L2
    if (cut) bulk_prefetch_l2(seg_init + (size_t)cut_idx * DK * DV, DK * DV * sizeof(float));
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    load_v(0);
    load_qk(0);
    if (n > 1) load_v(1);
  }
  if (tid < C) pw[tid] = expf((float)tid * gamma);  // lambda^d, d = 0..127
  if (tid < DK) sa[tid] = __ldg(aug + h * DK + tid);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_o);
      // steps 0 (v, q, k) and 1 (v) were issued before the CTA's barrier
      int armed_qk[2] = {1, 0}, armed_v[2] = {1, n > 1 ? 1 : 0};
      for (int c = 1; c < n; ++c) {  // c: step of this CTA, chunk c0 + c
        const uint32_t s = c & 1;
        if (c >= 2) {
          if (!wait(cta, cta.bar(V_EMPTY + s), ((c >> 1) - 1) & 1, ctl)) break;
          load_v(c);
          ++armed_v[s];
        }
        if (!wait(cta, cta.bar(QK_EMPTY + s), ((c - 1) >> 1) & 1, ctl)) break;
        load_qk(c);
        ++armed_qk[s];
      }
      // drain: every armed load has landed before the CTA may exit
      for (int s = 0; s < 2; ++s) {
        if (armed_v[s]) mbar_wait(cta.bar(V_FULL + s), (armed_v[s] - 1) & 1, ctl, DRAIN_NS);
        if (armed_qk[s]) mbar_wait(cta.bar(QK_FULL + s), (armed_qk[s] - 1) & 1, ctl, DRAIN_NS);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_f16(128, 128, BF16, BF16, false, false);
      constexpr uint32_t ID_QS = idesc_f16(128, 192, false, false, false, true);
      constexpr uint32_t ID_PV = idesc_f16(128, 192, false, false, false, true);
      constexpr uint32_t ID_KV = idesc_f16(128, 192, false, false, true, true);
      for (int c = 0; c < n; ++c) {
        const uint32_t s = c & 1, st = cta.sb + s * STAGE;
        const uint32_t slot = cta.sb + (s ^ 1) * STAGE;  // state copy for this chunk
        // the give-up path's diagnostic: the drain barrier's first phase completes only after
        // this loop, so this bounded wait runs out and the CTA gives up
        if (c == ctl.stall_step) {
          wait(cta, cta.bar(DRAIN), 0, ctl);
          break;
        }
        if (!wait(cta, cta.bar(QK_FULL + s), (c >> 1) & 1, ctl)) break;
        // P'' of the previous chunk lives in D_P's columns: P'' V must be done before Q K^T
        // overwrites them
        if (c >= 1 && !wait(cta, cta.bar(O_DONE), (c - 1) & 1, ctl)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 6; ++ks) {  // P = Q K^T
          const uint32_t off = (ks >> 1) * Q_BOX + (ks & 1) * 32;
          mma_f16_ss(tmem + TM_P, smem_desc(st + OFF_Q + off, 16, 512, SW_64),
                     smem_desc(st + OFF_K + off, 16, 512, SW_64), ID_QK, ks > 0);
        }
        mma_commit(cta.bar(P_DONE));
        if (!wait(cta, cta.bar(EP_Q), c & 1, ctl)) break;
        if (!wait(cta, cta.bar(EP_S), c & 1, ctl)) break;
        if (c >= 1 && !wait(cta, cta.bar(EP_O), (c - 1) & 1, ctl)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 6; ++ks) {  // O = Q'' S
          const uint32_t off = (ks >> 1) * Q_BOX + (ks & 1) * 32;
          mma_f16_ss(tmem + TM_O, smem_desc(st + OFF_Q + off, 16, 512, SW_64),
                     smem_desc(slot + ks * 2048, S_ATOM, 1024, SW_128), ID_QS, ks > 0);
        }
        // the state copy this Q''S reads, saved for the backward: one bulk store from the
        // slot, read out before the slot is released for the next chunk's q, k
        if (saved.copy) {
          bulk_store(saved.copy + ((size_t)bh * nc + c0 + c) * kCopyBytes, slot, kCopyBytes);
          bulk_commit();
          bulk_wait_read<0>();
        }
        // the state copy has been read: the next chunk's q, k may load into that slot
        mma_commit(cta.bar(QK_EMPTY + (s ^ 1)));
        if (!wait(cta, cta.bar(EP_CONV), c & 1, ctl)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // O += P'' V  (P'' from TMEM)
          mma_f16_ts(tmem + TM_O, tmem + TM_P + 8 * ks,
                     smem_desc(st + OFF_V + ks * 2048, V_BOX, 1024, SW_128), ID_PV, 1);
        }
        mma_commit(cta.bar(O_DONE));
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {  // S += K'^T V
          mma_f16_ss(tmem + TM_S, smem_desc(st + OFF_K + ks * 1024, Q_BOX, 512, SW_64),
                     smem_desc(st + OFF_V + ks * 2048, V_BOX, 1024, SW_128), ID_KV, 1);
        }
        mma_commit(cta.bar(S_DONE));
        mma_commit(cta.bar(V_EMPTY + s));
      }
      mma_commit(cta.bar(DRAIN));
      mbar_wait(cta.bar(DRAIN), 0, ctl, DRAIN_NS);
      if (saved.copy) bulk_wait_all();  // the saved copies have reached global memory
    }
  } else if (warp < CONVERT_WARPS) {
    // ------------------------------------------------------------------ convert group
    // Warp w serves rows 32q..32q+31 (q = w & 3, thread = token row i = TMEM lane) and part
    // hv = w >> 2 of CW of the work on them: v chunks, q/k chunks (with their part of the gate
    // dot product) and some of the eight 16-column score blocks.  With two parts, part 0 owns
    // the quadrant's two diagonal blocks (and so adds the self-augmentation, for which it
    // takes part 1's gate partial sums); the blocks below the diagonal are shared out so that
    // the busiest quadrant gives each part four; each part zero-fills the blocks above the
    // diagonal of its parity.
    const int q4 = warp & 3, hv = warp >> 2;
    const int i = 32 * q4 + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const float lam = pw[1], lamC = expf((float)C * gamma);
    const float lq = (i + 1 < C) ? pw[i + 1] : lamC;  // lambda^(i+1)
    const float lk_full = pw[C - 1 - i];              // lambda^(C-1-i)
    // in the last chunk (L_last tokens): lambda^(L_last-1-i), and 0 on the zero rows past T
    const float lk_last = i < L_last ? pw[L_last - 1 - i] : 0.f;
    float* zx = (float*)(base + OFF_ZX);
    // this warp's blocks at or below the diagonal: hb_first + m for half 1, the diagonal pair
    // then 0, 1, ... for half 0
    constexpr int NV = 24 / CW, MAXB = 8 / CW;  // v chunks and live score blocks per part
    const int below = max(0, q4 - 1);  // with two parts, part 0 takes the blocks hb < below
    const int nlive = CW == 1 ? 2 * q4 + 2 : hv == 0 ? 2 + below : 2 * q4 - below;
    auto live_block = [&](int m) {
      return CW == 1 ? m : hv == 0 ? (m < 2 ? 2 * q4 + m : m - 2) : below + m;
    };
    float range_max = 0.f;
    for (int c = 0; c < n; ++c) {
      const uint32_t s = c & 1, par = c & 1;
      const float lk = c0 + c == nc - 1 ? lk_last : lk_full;
      uint8_t* stg = base + s * STAGE;
      float vmax = 0.f, kmax = 0.f, qmax = 0.f;
      if (!wait_warp(cta, cta.bar(V_FULL + s), (c >> 1) & 1, ctl)) break;
      if constexpr (BF16) {  // v -> fp16 in place (exact for |v| in the fp16 normal range)
#pragma unroll 4
        for (int cc = NV * hv; cc < NV * hv + NV; ++cc)
          scale_chunk_to_half<true>(
              (uint4*)(stg + OFF_V + (cc >> 3) * V_BOX + swz_off(i, cc & 7, 128)), 1.f, vmax);
      } else {
#pragma unroll 4
        for (int cc = NV * hv; cc < NV * hv + NV; ++cc) {
          const uint4 x = *(const uint4*)(stg + OFF_V + (cc >> 3) * V_BOX + swz_off(i, cc & 7, 128));
          const uint32_t* w = (const uint32_t*)&x;
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) vmax = fmaxf(vmax, fmaxf(fabsf(h_lo(w[e2])), fabsf(h_hi(w[e2]))));
        }
      }
      if (!wait_warp(cta, cta.bar(P_DONE), par, ctl)) break;
      if (!wait_warp(cta, cta.bar(QK_FULL + s), (c >> 1) & 1, ctl)) break;
      tc_fence_after();
      // channels 8cc..8cc+7 of q, k: their part of the gate sum into `zacc`, Q'' and K' in place
      auto qk_chunk = [&](int cc, float& zacc) {
        const uint32_t off = (cc >> 2) * Q_BOX + swz_off(i, cc & 3, 64);
        uint4 qv = *(uint4*)(stg + OFF_Q + off);
        uint4 kv = *(uint4*)(stg + OFF_K + off);
        uint32_t* qw = (uint32_t*)&qv;
        uint32_t* kw = (uint32_t*)&kv;
        const float4 a0 = *reinterpret_cast<const float4*>(sa + 8 * cc);
        const float4 a1 = *reinterpret_cast<const float4*>(sa + 8 * cc + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const float q0 = ld16<BF16>(qw[e2] & 0xFFFFu), q1 = ld16<BF16>(qw[e2] >> 16);
          const float k0 = ld16<BF16>(kw[e2] & 0xFFFFu), k1 = ld16<BF16>(kw[e2] >> 16);
          zacc = fmaf(av[2 * e2] * q0, k0, zacc);
          zacc = fmaf(av[2 * e2 + 1] * q1, k1, zacc);
          const float x0 = q0 * lq, x1 = q1 * lq, y0 = k0 * lk, y1 = k1 * lk;
          qmax = fmaxf(qmax, fmaxf(fabsf(x0), fabsf(x1)));
          kmax = fmaxf(kmax, fmaxf(fabsf(y0), fabsf(y1)));
          qw[e2] = pack_h2(x0, x1);
          kw[e2] = pack_h2(y0, y1);
        }
        *(uint4*)(stg + OFF_Q + off) = qv;
        *(uint4*)(stg + OFF_K + off) = kv;
      };
      // the gate sum is always formed as (channels 0..47) + (channels 48..95), whichever
      // layout, so both give bit-identical outputs
      float z = 0.f, z_hi = 0.f;
#pragma unroll 2
      for (int cc = 6 * hv; cc < 6 * hv + 6; ++cc) qk_chunk(cc, z);
      if constexpr (CW == 1) {
#pragma unroll 2
        for (int cc = 6; cc < 12; ++cc) qk_chunk(cc, z_hi);
      }
      if (CW == 2 && hv == 1) {  // part 0 adds the diagonal term: it needs the whole gate sum
        zx[i] = z;
        mbar_arrive(cta.bar(ZX0 + q4));
      }
      // Q'' is in place: the Q''S MMA can run (and release the state copy's slot) while the
      // masked scores are still being made
      fence_proxy_async();
      mbar_arrive(cta.bar(EP_Q));
      // chunk maxima of |K'| and |V| (for the emit group's bound on the next state)
      {
        float km = kmax, vm = vmax;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, off));
          vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
        }
        if (lane == 0) {
          kvmax[par * 16 + warp] = km;
          kvmax[par * 16 + 8 + warp] = vm;
        }
      }
      // the state exponent of this chunk (and P'' of the previous chunk consumed)
      if (!wait_warp(cta, cta.bar(EP_S), par, ctl)) break;
      float sg = 0.f;
      if (CW == 1) {
        sg = sigmoid(z + z_hi);
      } else if (hv == 0) {
        if (!wait_warp(cta, cta.bar(ZX0 + q4), par, ctl)) break;
        sg = sigmoid(z + zx[i]);
      }
      // the gate, saved for the backward if asked (the warp that holds the whole sum); head
      // major [B,H,T], so a warp's 32 rows are one contiguous 128-byte store
      if (gate_out && (CW == 1 || hv == 0)) {
        const int t = (c0 + c) * C + i;
        if (t < T) gate_out[((size_t)b * H + h) * T + t] = sg;
      }
      const float psc = pow2i(-es[par]);
      float pmax = 0.f;
      {
        // fp16 pairs, in place over the fp32 scores: block hb's 8 packed columns land on fp32
        // columns 8hb..8hb+7, inside block hb/2.  One warp per quadrant takes its blocks in
        // increasing order, so it writes each as soon as it is made; with two, both read first.
        uint32_t pk[CW == 1 ? 1 : MAXB][8];
#pragma unroll
        for (int m = 0; m < MAXB; ++m) {
          if (m < nlive) {
            const int cb = 16 * live_block(m);
            uint32_t r[16];
            tmem_ld16(trow + TM_P + cb, r);
            tmem_wait_ld();
            // lambda^(i-j) by repeated multiplication going left from j = min(i, cb+15)
            float f = pw[max(i - (cb + 15), 0)] * psc;
            float p[16];
#pragma unroll
            for (int u = 15; u >= 0; --u) {
              const bool in = cb + u <= i;
              p[u] = in ? __uint_as_float(r[u]) * f : 0.f;
              f = in ? f * lam : f;
              // the self-augmentation sigmoid(z_i) v_i rides on the diagonal, so P'' V
              // includes it: (P o D + diag(sigmoid(z))) 2^-e
              if (cb + u == i) p[u] += sg * psc;
              pmax = fmaxf(pmax, fabsf(p[u]));
            }
            uint32_t(&dst)[8] = pk[CW == 1 ? 0 : m];
#pragma unroll
            for (int u = 0; u < 8; ++u) dst[u] = pack_h2(p[2 * u], p[2 * u + 1]);
            if constexpr (CW == 1) tmem_st8(trow + TM_P + cb / 2, dst);
          }
        }
        if constexpr (CW == 2) {
          tc_fence_before();
          mbar_arrive(cta.bar(QS0 + q4));
          if (!wait_warp(cta, cta.bar(QS0 + q4), par, ctl)) break;
          tc_fence_after();
#pragma unroll
          for (int m = 0; m < MAXB; ++m)
            if (m < nlive) tmem_st8(trow + TM_P + 8 * live_block(m), pk[m]);
        }
        const uint32_t zero8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        for (int hb = 2 * q4 + 2 + hv; hb < 8; hb += CW) tmem_st8(trow + TM_P + 8 * hb, zero8);
      }
      range_max = fmaxf(range_max, fmaxf(fmaxf(vmax, kmax), fmaxf(qmax, pmax)));
      tmem_wait_st();
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(cta.bar(EP_CONV));
    }
    if (range_max >= 65504.f) record_error(ctl, DEV_RANGE);
  } else if (warp < PRODUCER_WARP) {
    // ------------------------------------------------------------------ emit group
    // Warp w serves rows 32(w&3)..+31 and value columns [96hf, 96hf+96), hf = (w-8)>>2.
    // State copy for the next chunk (the serial chain, first), then the output rows.
    const int q4 = warp & 3, hf = (warp - CONVERT_WARPS) >> 2, ew = warp - CONVERT_WARPS;
    const int i = 32 * q4 + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
    const float lamC = expf((float)C * gamma);
    const float lamL = L_last == C ? lamC : pw[L_last];  // lambda^(tokens of the last chunk)
    bool bad = false;

    // fp16 copy S * 2^-e of this warp's state rows / column half into the q/k slot at
    // `slot_off`, D_S <- dec S (dec = lambda^(tokens of chunk `use`, whose update follows)),
    // and the warp's max|S| into red[use & 1].  Row i comes from TMEM (the state after the
    // chunk's update) or from init_state (`g_row`).
    auto publish_state = [&](uint32_t slot_off, int use, int e, float dec, const float* g_row,
                             bool from_tmem) {
      float m = 0.f;
      if (q4 < 3) {
        const float sc = pow2i(-e);
        float r[32];
#pragma unroll 1
        for (int nb = 0; nb < 3; ++nb) {
          const int col = 96 * hf + 32 * nb;
          if (from_tmem) {
            tmem_ld32(trow + TM_S + col, *reinterpret_cast<uint32_t(*)[32]>(r));
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {  // 8 loads in flight (rows are 16-byte aligned)
              const float4 x = g_row ? __ldg(reinterpret_cast<const float4*>(g_row + col) + j4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
              r[4 * j4] = x.x;
              r[4 * j4 + 1] = x.y;
              r[4 * j4 + 2] = x.z;
              r[4 * j4 + 3] = x.w;
            }
          }
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            const int n = col + 8 * q8;
            uint4 pk;
            pk.x = pack_h2(r[8 * q8 + 0] * sc, r[8 * q8 + 1] * sc);
            pk.y = pack_h2(r[8 * q8 + 2] * sc, r[8 * q8 + 3] * sc);
            pk.z = pack_h2(r[8 * q8 + 4] * sc, r[8 * q8 + 5] * sc);
            pk.w = pack_h2(r[8 * q8 + 6] * sc, r[8 * q8 + 7] * sc);
            *(uint4*)(base + slot_off + (n >> 6) * S_ATOM + swz_off(i, (n & 63) >> 3, 128)) = pk;
          }
          uint32_t u[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            m = fmaxf(m, fabsf(r[j]));
            u[j] = __float_as_uint(r[j] * dec);
          }
          tmem_st32(trow + TM_S + col, u);
        }
        tmem_wait_st();
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[(use & 1) * 8 + ew] = m;
      if (ew == 0 && lane == 0) {
        es[use & 1] = e;
        if (saved.exp) saved.exp[(size_t)bh * nc + c0 + use] = e;
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(cta.bar(EP_S));
    };
    auto red_max = [&](int slot) {
      float m = red[slot * 8];
#pragma unroll
      for (int w = 1; w < 8; ++w) m = fmaxf(m, red[slot * 8 + w]);
      return m;
    };

    // slot of this sequence's initial/final state: [b][h] of the caller's arrays, or its page
    // of a state pool
    long long zst = (long long)b * H + h;
    bool page_ok = true;
    if (sp.page) {
      const int pg = __ldg(sp.page + b);
      page_ok = pg >= 0 && pg < sp.n_pages;
      zst = ((long long)pg * sp.pool_layers + sp.layer) * H + h;
      if (!page_ok && ew == 0 && lane == 0 && (!cut || part == plan.parts - 1))
        record_error(ctl, DEV_RANGE);
    }
    const long long zinit = sp.init_paged ? zst : bh;
    // starting state: the caller's (whole pair) or the one the segment passes left for this
    // part; its exponent needs its exact max first (one exchange in the group)
    const float* g_row0 =
        i >= DK ? nullptr
        : cut   ? seg_init + ((size_t)cut_idx * DK + i) * DV
        : (init && page_ok) ? init + ((size_t)zinit * DK + i) * DV
                            : nullptr;
    // the final state is this CTA's to write if it ends the sequence
    const bool ends_seq = !cut || part == plan.parts - 1;
    int e_cur = 0;
    bool ok = true;
    if (cut && seg_max) {
      // the segment passes left this part's max |state| (as partial maxima): the same exponent
      // without a pass over the state or the exchange
      const float* pm = seg_max + (size_t)cut_idx * 4;
      e_cur = state_exponent(fmaxf(fmaxf(__ldg(pm), __ldg(pm + 1)), __ldg(pm + 2)));
    } else {
      float m = 0.f;
      if (g_row0) {
        const float4* g4 = reinterpret_cast<const float4*>(g_row0 + 96 * hf);
#pragma unroll
        for (int j4 = 0; j4 < 24; ++j4) {
          const float4 x = __ldg(g4 + j4);
          m = fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[16 + ew] = m;
      mbar_arrive(cta.bar(RED));
      ok = wait_warp(cta, cta.bar(RED), 0, ctl);
      if (ok) e_cur = state_exponent(red_max(2));
    }
    if (ok) {
      if (e_cur < 0) {
        bad = true;
        e_cur = 0;
      }
      publish_state(1 * STAGE + OFF_Q, 0, e_cur, c0 == nc - 1 ? lamL : lamC, g_row0, false);
    }

    for (int c = 0; c < n && ok; ++c) {
      const uint32_t s = c & 1, par = c & 1;
      if (!(ok = wait_warp(cta, cta.bar(O_DONE), par, ctl))) break;
      if (!(ok = wait_warp(cta, cta.bar(S_DONE), par, ctl))) break;
      if (!(ok = wait_warp(cta, cta.bar(EP_CONV), par, ctl))) break;
      tc_fence_after();
      // ---- next chunk's state copy first: it is on the serial chain.  Its exponent comes
      // from a bound, |S_{c+1}| <= lambda^C max|S_c| + 128 max|K'_c| max|V_c|, so the copy
      // needs a single pass over the state.
      int e_next = e_cur;
      if (c < n - 1) {
        // every emit thread has stored its part of max|S_c| (EP_S phase c is complete)
        if (!(ok = wait_warp(cta, cta.bar(EP_S), par, ctl))) break;
        const float ms = red_max(par);
        float km = kvmax[par * 16], vm = kvmax[par * 16 + 8];
#pragma unroll
        for (int w = 1; w < CONVERT_WARPS; ++w) {
          km = fmaxf(km, kvmax[par * 16 + w]);
          vm = fmaxf(vm, kvmax[par * 16 + 8 + w]);
        }
        e_next = state_exponent(lamC * ms + (float)C * km * vm);
        if (e_next < 0) {
          bad = true;
          e_next = 0;
        }
        publish_state(s * STAGE + OFF_Q, c + 1, e_next, c0 + c + 2 == nc ? lamL : lamC, nullptr,
                      true);
      }
      // ---- output rows: o = 2^e D_O for columns [96hf, 96hf+96) (the self-augmentation
      // sigmoid(z) v is already in D_O through the diagonal of P''), TMA-stored
      uint8_t* const stage_o = base + OFF_STG + ew * 4096;
      if constexpr (!GATED) {
        const float osc = pow2i(e_cur);
        const int t0 = (c0 + c) * C + 32 * q4;  // first token of this warp's rows (none past T)
        emit_rows_tma<6>(
            stage_o, lane,
            [&](int k, float (&o)[16]) {
              uint32_t r[16];
              tmem_ld16(trow + TM_O + 96 * hf + 16 * k, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __uint_as_float(r[j]) * osc;
            },
            [&](int k, uint32_t src) {
              if (t0 < T) tma_store_4d(&map_o, src, 96 * hf + 16 * k, h, t0, b);
            });
      } else {
        // y = o r w[tier] SiLU(g), r = (mean over the row's 192 channels of o^2 + eps)^-1/2:
        // pass 1 sums o^2 over this warp's 96 columns (writing o too if asked), the two warps
        // of the row quadrant exchange their sums, pass 2 writes y
        const float osc = pow2i(e_cur);
        const int t0 = (c0 + c) * C + 32 * q4;  // first token of this warp's rows (none past T)
        const bool live = (c0 + c) * C + i < T;  // this thread's row is a token of the sequence
        const long long tok = (long long)b * T + (c0 + c) * C + i;  // token row of this thread
        float* xch = (float*)(base + OFF_XCH);
        float ss = 0.f;
        if (og.want_o) {
          emit_rows_tma<6>(
              stage_o, lane,
              [&](int k, float (&o)[16]) {
                uint32_t r[16];
                tmem_ld16(trow + TM_O + 96 * hf + 16 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  o[j] = __uint_as_float(r[j]) * osc;
                  ss = fmaf(o[j], o[j], ss);
                }
              },
              [&](int k, uint32_t src) {
                if (t0 < T) tma_store_4d(&map_o, src, 96 * hf + 16 * k, h, t0, b);
              });
        } else {
#pragma unroll 1
          for (int k = 0; k < 6; ++k) {
            uint32_t r[16];
            tmem_ld16(trow + TM_O + 96 * hf + 16 * k, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float o = __uint_as_float(r[j]) * osc;
              ss = fmaf(o, o, ss);
            }
          }
        }
        // the row's gate values, all 12 loads in flight together
        const uint4* gp = reinterpret_cast<const uint4*>(og.g + (tok * H + h) * DV + 96 * hf);
        uint4 gq[12];
#pragma unroll
        for (int u = 0; u < 12; ++u) gq[u] = live ? __ldg(gp + u) : make_uint4(0u, 0u, 0u, 0u);
        xch[hf * 128 + i] = ss;
        mbar_arrive(cta.bar(QX + q4));
        if (!(ok = wait_warp(cta, cta.bar(QX + q4), par, ctl))) break;
        const float rr = 1.f / sqrtf((xch[i] + xch[128 + i]) * (1.f / DV) + og.eps);
        if (og.rstd && hf == 0 && live) og.rstd[tok * H + h] = rr;
        const float* wrow = og.w + (h / og.heads_per_tier) * DV + 96 * hf;
        if (lane == 0) bulk_wait_read<0>();  // pass 1's stores have read the staging
        __syncwarp();
        emit_rows_tma<6>(
            stage_o, lane,
            [&](int k, float (&y)[16]) {
              uint32_t r[16];
              tmem_ld16(trow + TM_O + 96 * hf + 16 * k, r);
              tmem_wait_ld();
              const float f = osc * rr;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const uint4 gv = j < 8 ? gq[2 * k] : gq[2 * k + 1];
                const uint32_t w2 = (j & 7) < 2 ? gv.x : (j & 7) < 4 ? gv.y : (j & 7) < 6 ? gv.z : gv.w;
                const float gj = ld16<true>((j & 1) ? (w2 >> 16) : (w2 & 0xFFFFu));
                const float sl = __fdividef(gj, 1.f + __expf(-gj));
                y[j] = __uint_as_float(r[j]) * f * __ldg(wrow + 16 * k + j) * sl;
              }
            },
            [&](int k, uint32_t src) {
              if (t0 < T) tma_store_4d(&map_y, src, 96 * hf + 16 * k, h, t0, b);
            });
      }
      tc_fence_before();
      mbar_arrive(cta.bar(EP_O));
      // ---- final state (after the last chunk), staged through the same rows
      // (only the CTA that ends the sequence: a whole pair or the last part of a cut one)
      if (c == n - 1 && fin && q4 < 3 && ends_seq && page_ok) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        emit_rows_tma<6>(
            stage_o, lane,
            [&](int k, float (&f)[16]) {
              uint32_t r[16];
              tmem_ld16(trow + TM_S + 96 * hf + 16 * k, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(r[j]);
            },
            [&](int k, uint32_t src) {
              tma_store_3d(&map_fin, src, 96 * hf + 16 * k, 32 * q4, (int)zst);
            });
      }
      if (lane == 0) bulk_wait_read<0>();  // the staging buffers are free for the next chunk
      __syncwarp();
      e_cur = e_next;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    if (bad) record_error(ctl, DEV_RANGE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_chunk_fwd(const FwdArgs& a, DevCtl ctl, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo, mfin, my;
  float* const o_any = a.o ? a.o : a.og.y;  // stand-in for a map that is never used
  if (!make_tmap_seq_16bit(&mq, a.q, DK, a.H, a.T, a.B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_seq_16bit(&mk, a.k, DK, a.H, a.T, a.B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_seq_16bit(&mv, a.v, DV, a.H, a.T, a.B, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, a.bf16) ||
      !make_tmap_seq_out_f32(&mo, o_any, DV, a.H, a.T, a.B) ||
      !make_tmap_seq_out_f32(&my, a.og.y ? a.og.y : o_any, DV, a.H, a.T, a.B) ||
      !make_tmap_state_f32(&mfin, a.fin ? (const void*)a.fin : (const void*)o_any,
                           a.sp.page ? (long long)a.sp.n_pages * a.sp.pool_layers * a.H
                                     : (long long)a.B * a.H))
    return cudaErrorInvalidValue;
  const bool gated = a.og.g != nullptr;
  auto kern = gated ? (a.bf16 ? fwd_kernel<true, true> : fwd_kernel<false, true>)
                    : (a.bf16 ? fwd_kernel<true, false> : fwd_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  SplitPlan plan = a.plan;
  if (plan.parts <= 1 || !a.seg_init) {
    plan.whole = a.B * a.H;
    plan.parts = 1;
    plan.overlap = false;
  }
  const long long grid = plan.whole + ((long long)a.B * a.H - plan.whole) * plan.parts;
  const unsigned threads = gated ? Layout<true>::THREADS : Layout<false>::THREADS;
  // with plan.overlap the kernel is the segment passes' programmatic dependent: its whole pairs
  // start beside the passes, its parts wait for them (griddep_wait)
  PdlLaunch L(dim3((unsigned)grid), dim3(threads), SMEM_BYTES, stream, plan.overlap);
  return cudaLaunchKernelEx(&L.cfg, kern, mq, mk, mv, mo, mfin, a.log_decay, a.aug, a.init, a.o,
                            a.fin, a.T, a.H, plan, a.seg_init, a.seg_max, a.sp, my, a.og, a.gate,
                            a.saved, ctl);
}

}  // namespace gla
