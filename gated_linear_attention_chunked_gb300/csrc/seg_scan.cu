// seg_scan.cu -- cutting (b, h) pairs into chunk ranges that run as separate CTAs.
//
// Method: the chunked forward and backward ("Beyond the KV cache ... Laplace 3B ...", sections
// "Challenge 1" and "Challenge 3") carry a state (forward) or its adjoint (backward) from chunk
// to chunk, so each (b, h) is a serial chain of ceil(T/128) steps.  When the pairs do not fill
// the last wave of SMs -- or there are fewer pairs than SMs, as in long-context prefill -- the
// chains of the pairs in that wave are cut into parts.  The recurrence S_t = lambda S_{t-1} +
// k_t v_t^T (section "i14 and the Laplace 3B architecture", "GLA mixer") is linear, and so is
// its adjoint dS_{t-1} = lambda dS_t + q_t dO_t^T, so for a part j of L_j tokens, s_j its first
// token and e_j its last,
//
//     S entering part j+1  = lambda^(L_j) S entering part j + U_j,
//                            U_j  = sum_{t in j} lambda^(e_j - t) k_t v_t^T
//     dS leaving part j-1  = lambda^(L_j) dS leaving part j + U'_j,
//                            U'_j = sum_{t in j} lambda^(t - s_j + 1) q_t dO_t^T.
//
//   pass A  (seg_sum_kernel, one item per cut pair and part, a CTA taking one or several in
//           turn): U_j (parts 0..p-2) or U'_j (parts 1..p-1) on the tensor cores, the pair's
//           K''^T V or Q''^T dO over the part's chunks into one fp32 TMEM accumulator, the decay
//           folded into the fp16 copy of k (q);
//   pass B  (seg_link_kernel): the recurrences above per cut pair, giving every part its
//           starting state (the caller's initial state, a pool page or zero for part 0) and
//           its starting adjoint (d_final_state or zero for the last part) -- with two parts
//           one step per direction, which pass A's items take themselves (no pass B);
//   then    the chunked kernel runs the whole pairs and every part as its own CTA.
//
// Extra traffic: pass A reads k, v (q, dO) of all parts but the last (first).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <map>

#include "kernels.h"
#include "scan_common.cuh"
#include "tmap.h"

namespace gla {
namespace {

using namespace scan;

constexpr int STAGES = 3;
constexpr uint32_t K_BOX = 8192;                   // 128 rows x 32 channels x 2 B, 64-B swizzle
constexpr uint32_t V_BOX = 16384;                  // 128 rows x 64 channels x 2 B, 128-B swizzle
constexpr uint32_t STAGE = 3 * K_BOX + 3 * V_BOX;  // k then v of one chunk: 72 KB
constexpr uint32_t OFF_BAR = STAGES * STAGE;
constexpr uint32_t NBAR = 11;
constexpr uint32_t OFF_TMEM = (OFF_BAR + NBAR * 8 + 15) & ~15u;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t SMEM_USED = OFF_TMEM + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment of the dynamic base
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

enum Bar : uint32_t {
  FULL = 0,   // 0..2: stage s landed
  CONV = 3,   // 3..5: stage s converted to fp16 operands
  EMPTY = 6,  // 6..8: the MMAs of stage s are done
  DONE = 9,   // every MMA of the current item is done (one phase per item)
  DRAIN = 10,  // every MMA the CTA issued is done (the MMA thread's own wait before exit)
};

constexpr int THREADS = 192;  // warps 0..3 convert + epilogue (row = token = TMEM lane)
constexpr int PRODUCER_WARP = 4, MMA_WARP = 5;

// 16-byte chunk `cc` of row `i`: k has 3 boxes of 32 channels (64-byte rows), v 3 boxes of 64
// channels (128-byte rows), v after k within a stage.
__device__ __forceinline__ uint32_t k_chunk(uint32_t i, int cc) {
  return (cc >> 2) * K_BOX + swz_off(i, cc & 3, 64);
}
__device__ __forceinline__ uint32_t v_chunk(uint32_t i, int cc) {
  return 3 * K_BOX + (cc >> 3) * V_BOX + swz_off(i, cc & 7, 128);
}

// Item `it` of pass A: it < n_fwd is the forward sum U_j of part j = it % (p-1) of cut pair
// x = it / (p-1), into states[x*p + j + 1]; it >= n_fwd the reverse sum U'_j of part
// j = 1 + it' % (p-1) (it' = it - n_fwd), into adj[x*p + j - 1].  Those slots are then
// completed by pass B in place -- or, with two parts (`fold`), by the item itself.
// full != 0 (a sequence-sharded call's slice sums): ncol items per pair bh, its one part being
// the whole sequence and item `nb` of the pair summing value columns [nb*192/ncol, ...) only
// (ncol = 1 or 3: a third is one 64-column v box); items it < n_fwd write U of pair it / ncol
// into states, it >= n_fwd U' of pair (it - n_fwd) / ncol into adj.
struct SumItem {
  bool rev;
  int x, j, nb, bh, b, h, c_lo, c_hi;
};
__device__ __forceinline__ SumItem sum_item(int it, int n_fwd, int full, int ncol, int whole,
                                            int parts, int H, int nc) {
  SumItem I;
  I.rev = it >= n_fwd;
  const int idx = I.rev ? it - n_fwd : it;
  I.x = full ? idx / ncol : idx / (parts - 1);
  I.nb = full ? idx % ncol : 0;
  I.j = full ? 0 : idx % (parts - 1) + (I.rev ? 1 : 0);
  I.bh = whole + I.x;
  I.b = I.bh / H;
  I.h = I.bh % H;
  I.c_lo = full ? 0 : part_begin(I.j, nc, parts);
  I.c_hi = full ? nc : part_begin(I.j + 1, nc, parts);
  return I;
}

// Pass A.  The CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ... in order; its TMA ring
// runs on across them (the next item's first chunks load while this one's sum is written out).
// fold (two parts, not full): the item also applies its pair's one recurrence step, as pass B
// would: forward, states[x*2] = S_0 (the caller's initial state, its pool page or zeros) and
// states[x*2 + 1] = lambda^(L_0) S_0 + U_0; reverse, adj[x*2 + 1] = A_1 (d_final_state or
// zeros) and adj[x*2] = lambda^(L_1) A_1 + U'_1; and, given state_max, each forward slot's
// three 32-row groups' max |state| into state_max[slot][0..2] (one per epilogue warp, so no
// warp waits on another).
template <bool BF16>
__global__ void __launch_bounds__(THREADS, 1)
seg_sum_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
               const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_g,
               const float* __restrict__ log_decay, float* __restrict__ states,
               float* __restrict__ adj, const float* __restrict__ init,
               const float* __restrict__ dfin, StatePages sp, float* __restrict__ state_max,
               int T, int H, int whole, int parts, int n_fwd, int n_items, int full, int ncol,
               int fold, DevCtl ctl) {
  // the next launch may start: pass B (which waits for these sums) or, with two parts, the
  // chunked kernel, whose whole pairs need nothing from this pass
  griddep_launch_dependents();
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
  const int nc = (T + C - 1) / C;
  const int it0 = (int)blockIdx.x, it_step = (int)gridDim.x;
  uint32_t* tmem_slot = (uint32_t*)(base + OFF_TMEM);

  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  if (tid == PRODUCER_WARP * 32) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(cta.bar(FULL + s), 1);
      mbar_init(cta.bar(CONV + s), 128);
      mbar_init(cta.bar(EMPTY + s), 1);
    }
    mbar_init(cta.bar(DONE), 1);
    mbar_init(cta.bar(DRAIN), 1);
    *cta.abort_flag() = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = cta.sb;

  // g: this CTA's chunk step over all its items (ring stage g % STAGES, phase g / STAGES)
  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      int armed0 = 0, armed1 = 0, armed2 = 0;  // loads issued per stage
      bool ok = true;
      int g = 0;
      for (int it = it0; it < n_items && ok; it += it_step) {
        const SumItem I = sum_item(it, n_fwd, full, ncol, whole, parts, H, nc);
        const CUtensorMap* map_a = I.rev ? &map_q : &map_k;
        const CUtensorMap* map_b = I.rev ? &map_g : &map_v;
        for (int m = 0; m < I.c_hi - I.c_lo; ++m, ++g) {
          const int s = g % STAGES;
          if (g >= STAGES && !(ok = wait(cta, cta.bar(EMPTY + s), (g / STAGES - 1) & 1, ctl)))
            break;
          // k (q) whole; v (dO) whole, or the one 64-column box of this item's column third
          mbar_arrive_expect_tx(cta.bar(FULL + s), 3 * K_BOX + (ncol == 3 ? 1 : 3) * V_BOX);
          const int t0 = (I.c_lo + m) * C;
          const uint32_t st = sb + s * STAGE;
          for (int jb = 0; jb < 3; ++jb) {
            tma_load_4d(st + jb * K_BOX, map_a, cta.bar(FULL + s), 32 * jb, I.h, t0, I.b);
            if (ncol == 1 || jb == 0)
              tma_load_4d(st + 3 * K_BOX + jb * V_BOX, map_b, cta.bar(FULL + s),
                          64 * (ncol == 3 ? I.nb : jb), I.h, t0, I.b);
          }
          armed0 += s == 0;
          armed1 += s == 1;
          armed2 += s == 2;
        }
      }
      // no copy may still be landing when the CTA exits
      if (armed0) mbar_wait(cta.bar(FULL + 0), (armed0 - 1) & 1, ctl, DRAIN_NS);
      if (armed1) mbar_wait(cta.bar(FULL + 1), (armed1 - 1) & 1, ctl, DRAIN_NS);
      if (armed2) mbar_wait(cta.bar(FULL + 2), (armed2 - 1) & 1, ctl, DRAIN_NS);
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      // U (rows = 96 key channels + 32 padding rows never read) += A''^T B, K = 16 tokens per
      // instruction: A = k (q) tile as [token][channel] (MN-major), B = v (dO) tile likewise.
      // One DONE phase per item; the next item's first MMA overwrites the accumulator, which
      // the convert warps have read out before they release that item's first stage (CONV).
      constexpr uint32_t ID192 = idesc_f16(128, 192, false, false, true, true);
      constexpr uint32_t ID64 = idesc_f16(128, 64, false, false, true, true);
      const uint32_t ID = ncol == 3 ? ID64 : ID192;
      bool ok = true;
      int g = 0, k = 0;
      for (int it = it0; it < n_items && ok; it += it_step, ++k) {
        const SumItem I = sum_item(it, n_fwd, full, ncol, whole, parts, H, nc);
        for (int m = 0; m < I.c_hi - I.c_lo; ++m, ++g) {
          const int s = g % STAGES;
          if (g == ctl.stall_step) {  // the give-up path's diagnostic (see the chunk kernels):
            // DONE's phase k completes only after this item's MMAs, so the wait runs out
            wait(cta, cta.bar(DONE), k & 1, ctl);
            ok = false;
            break;
          }
          if (!(ok = wait(cta, cta.bar(CONV + s), (g / STAGES) & 1, ctl))) break;
          tc_fence_after();
          const uint32_t st = sb + s * STAGE;
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ss(tmem, smem_desc(st + ks * 1024, K_BOX, 512, SW_64),
                       smem_desc(st + 3 * K_BOX + ks * 2048, V_BOX, 1024, SW_128), ID,
                       (m > 0 || ks > 0) ? 1u : 0u);
          mma_commit(cta.bar(EMPTY + s));
        }
        if (ok) mma_commit(cta.bar(DONE));
      }
      // every MMA issued (the items' and any an abort left behind) has completed before the
      // accumulator is freed.  Its own barrier: one more phase of DONE could complete before a
      // convert warp has seen the last item's, which would then look incomplete to it.
      mma_commit(cta.bar(DRAIN));
      mbar_wait(cta.bar(DRAIN), 0, ctl, DRAIN_NS);
    }
  } else {
    // ---- warps 0..3: in-place fp16 operands of chunk m, row i = token i of the chunk: k
    // scaled by lambda^(e_j - t) (forward) or q by lambda^(t - s_j + 1) (reverse), v / dO as
    // they are.  Rows past T are zeros (the tensor map's fill); in the forward direction e_j
    // is the part's last token, so a ragged last chunk weighs its rows by
    // lambda^(last_len - 1 - i) and its rows past T by 0.  Every wait is voted per warp, so
    // a warp stays on one path through the items and its collective TMEM loads.
    const int i = tid;
    float vmax = 0.f;
    bool ok = true;
    int g = 0, k = 0;
    for (int it = it0; it < n_items && ok; it += it_step, ++k) {
      const SumItem I = sum_item(it, n_fwd, full, ncol, whole, parts, H, nc);
      const int M = I.c_hi - I.c_lo;  // chunks of the part (>= 1)
      // tokens of the part, and of its last chunk (C unless it is the sequence's ragged one)
      const int len = min(I.c_hi * C, T) - I.c_lo * C;
      const int last_len = min(I.c_hi * C, T) - (I.c_hi - 1) * C;
      const float gamma = __ldg(log_decay + I.h);
      // lambda^d as exp(d gamma), d = i + 1 (reverse) or C - 1 - i (forward)
      const float row_w = expf((float)(I.rev ? i + 1 : C - 1 - i) * gamma);
      const float row_w_last =
          I.rev ? row_w : (i < last_len ? expf((float)(last_len - 1 - i) * gamma) : 0.f);
      for (int m = 0; m < M; ++m, ++g) {
        const int s = g % STAGES;
        if (!(ok = wait_warp(cta, cta.bar(FULL + s), (g / STAGES) & 1, ctl))) break;
        uint8_t* st = base + s * STAGE;
        // reverse: the chunks between this one and s_j; forward: the tokens after this chunk
        // up to e_j (whole chunks, then the last chunk's last_len)
        const float sk = I.rev ? expf(gamma * (float)(C * m)) * row_w
                               : (m == M - 1 ? row_w_last
                                             : expf(gamma * (float)(C * (M - 2 - m) + last_len)) *
                                                   row_w);
        convert_row<BF16, 12>(st, [&](int cc) { return k_chunk(i, cc); }, sk, vmax);
        if (ncol == 3)
          convert_row<BF16, 8>(st, [&](int cc) { return v_chunk(i, cc); }, 1.f, vmax);
        else
          convert_row<BF16, 24>(st, [&](int cc) { return v_chunk(i, cc); }, 1.f, vmax);
        fence_proxy_async();
        tc_fence_before();  // (the previous item's TMEM loads come before this stage's MMAs)
        mbar_arrive(cta.bar(CONV + s));
      }
      // ---- the sum out: rows 0..95 (warps 0..2), 192 fp32 each
      if (ok) ok = wait_warp(cta, cta.bar(DONE), k & 1, ctl);
      ok = __all_sync(0xffffffffu, ok && *cta.abort_flag() == 0);
      if (ok && warp < 3) {
        tc_fence_after();
        float* const out = I.rev ? adj : states;
        const long long slot =
            full ? (long long)I.x : (long long)I.x * parts + (I.rev ? I.j - 1 : I.j + 1);
        const int ncols = DV / ncol;  // this item's value columns, from column ncols * nb
        float* dst = out + (size_t)slot * DK * DV + (size_t)i * DV + (size_t)ncols * I.nb;
        // fold: the boundary row (the pair's initial state or d_final_state; null = zeros),
        // its slot, and lambda^(tokens of this part)
        const float* bnd = nullptr;
        float* dst0 = nullptr;
        float lam = 0.f;
        if (fold) {
          dst0 = out + ((size_t)I.x * parts + (I.rev ? parts - 1 : 0)) * DK * DV + (size_t)i * DV;
          lam = expf(gamma * (float)len);
          if (I.rev) {
            if (dfin) bnd = dfin + ((size_t)I.bh * DK + i) * DV;
          } else {
            long long zi = I.bh;  // [b][h] of the caller's initial states, or a pool page
            if (sp.init_paged) {
              const int pg = __ldg(sp.page + I.b);
              zi = (pg >= 0 && pg < sp.n_pages)
                       ? ((long long)pg * sp.pool_layers + sp.layer) * H + I.h
                       : -1;
            }
            if (init && zi >= 0) bnd = init + ((size_t)zi * DK + i) * DV;
          }
        }
        float m0 = 0.f, m1 = 0.f;  // max |S_0|, |S_1| over this thread's row (forward fold)
#pragma unroll 1
        for (int cb = 0; cb < ncols / 32; ++cb) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * cb, r);
          tmem_wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            float4 u = make_float4(__uint_as_float(r[jj]), __uint_as_float(r[jj + 1]),
                                   __uint_as_float(r[jj + 2]), __uint_as_float(r[jj + 3]));
            if (fold) {
              const float4 b4 =
                  bnd ? __ldg(reinterpret_cast<const float4*>(bnd + 32 * cb + jj))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
              *reinterpret_cast<float4*>(dst0 + 32 * cb + jj) = b4;
              u = make_float4(fmaf(lam, b4.x, u.x), fmaf(lam, b4.y, u.y), fmaf(lam, b4.z, u.z),
                              fmaf(lam, b4.w, u.w));
              m0 = fmaxf(m0, fmaxf(fmaxf(fabsf(b4.x), fabsf(b4.y)), fmaxf(fabsf(b4.z), fabsf(b4.w))));
              m1 = fmaxf(m1, fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w))));
            }
            *reinterpret_cast<float4*>(dst + 32 * cb + jj) = u;
          }
        }
        if (!fold && !I.rev && state_max && warp == 0 && lane < 4) {
          // pass B fills this item's slot's max (and slot 0's, with part 0) by atomicMax
          state_max[((size_t)I.x * parts + I.j + 1) * 4 + lane] = 0.f;
          if (I.j == 0) state_max[((size_t)I.x * parts) * 4 + lane] = 0.f;
        }
        if (fold && !I.rev && state_max) {  // the row group's maxima of both starting states
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
          }
          if (lane == 0) {
            state_max[((size_t)I.x * parts + 0) * 4 + warp] = m0;
            state_max[((size_t)I.x * parts + 1) * 4 + warp] = m1;
          }
        }
      }
    }
    if (vmax >= 65504.f) record_error(ctl, DEV_RANGE);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Pass B.  blockIdx.z = 0: states[x*p + j] (j >= 1) holds U_{j-1} on entry and the state
// entering part j on exit; slot x*p receives the pair's initial state (or zeros).
// blockIdx.z = 1: adj[x*p + j] (j <= p-2) holds U'_{j+1} on entry and the adjoint leaving
// part j on exit; slot x*p + p-1 receives d_final_state (or zeros).  One thread per 4
// consecutive state elements, walking the parts in order.
constexpr int LINK_THREADS = 1024;
// Pass B's CTAs when it overlaps the chunked kernel: few enough to wait beside pass A's
constexpr int LINK_CTAS_OVERLAP = 16;

// One item of pass B: elements 4e .. 4e+3 of cut pair x's starting states (rev = 0) or
// adjoints (rev = 1), walking the pair's parts in order.  MAX: also note each forward
// state's max |state| in state_max (a separate instantiation, so the plain link is unchanged).
template <bool MAX>
__device__ __forceinline__ void link_one(const float* __restrict__ init,
                                         const float* __restrict__ dfin,
                                         const float* __restrict__ log_decay,
                                         float* __restrict__ states, float* __restrict__ adj,
                                         int T, int H, int whole, int parts, const StatePages& sp,
                                         unsigned* state_max, int rev, int x, int e) {
  constexpr int N4 = DK * DV / 4;
  float* const slots = rev ? adj : states;
  if (!slots) return;
  const int bh = whole + x, b = bh / H, h = bh % H;
  const float gamma = __ldg(log_decay + h);
  const int nc = (T + C - 1) / C;
  auto tokens = [&](int j) {  // tokens of part j
    return min(part_begin(j + 1, nc, parts) * C, T) - part_begin(j, nc, parts) * C;
  };
  float4* out = reinterpret_cast<float4*>(slots) + (size_t)x * parts * N4 + e;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  // forward direction, given state_max: slot j's max |state| -- the warp's 128 elements (one
  // pair: items come in whole warps) reduced, then one atomicMax of the bits (non-negative
  // floats order as their bit patterns, so the result does not depend on the order)
  auto note_max = [&](int j) {
    if (!MAX || rev) return;
    float m = fmaxf(fmaxf(fabsf(s.x), fabsf(s.y)), fmaxf(fabsf(s.z), fabsf(s.w)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) atomicMax(state_max + ((size_t)x * parts + j) * 4, __float_as_uint(m));
  };
  // the steps in order, their sums loaded LB at a time ahead of the chain (each slot is read
  // before the step that overwrites it)
  constexpr int LB = 4;
  auto walk = [&](int first, int n_steps, int dir, int tok_off) {
    for (int q0 = 0; q0 < n_steps; q0 += LB) {
      float4 u[LB];
#pragma unroll
      for (int q = 0; q < LB; ++q)
        if (q0 + q < n_steps) u[q] = out[(size_t)(first + dir * (q0 + q)) * N4];
#pragma unroll
      for (int q = 0; q < LB; ++q) {
        if (q0 + q < n_steps) {
          const int j = first + dir * (q0 + q);
          const float lam = expf(gamma * (float)tokens(j + tok_off));
          s = make_float4(fmaf(lam, s.x, u[q].x), fmaf(lam, s.y, u[q].y), fmaf(lam, s.z, u[q].z),
                          fmaf(lam, s.w, u[q].w));
          out[(size_t)j * N4] = s;
          note_max(j);
        }
      }
    }
  };
  if (!rev) {
    long long zi = bh;  // slot of the caller's initial state: [b][h] or a pool page
    if (sp.init_paged) {
      const int pg = __ldg(sp.page + b);
      zi = (pg >= 0 && pg < sp.n_pages) ? ((long long)pg * sp.pool_layers + sp.layer) * H + h : -1;
    }
    if (init && zi >= 0) s = __ldg(reinterpret_cast<const float4*>(init) + (size_t)zi * N4 + e);
    out[0] = s;
    note_max(0);
    walk(1, parts - 1, 1, -1);  // j = 1 .. p-1: S_j = lambda^(L_{j-1}) S_{j-1} + U_{j-1}
  } else {
    if (dfin) s = __ldg(reinterpret_cast<const float4*>(dfin) + (size_t)bh * N4 + e);
    out[(size_t)(parts - 1) * N4] = s;
    walk(parts - 2, parts - 1, -1, 1);  // j = p-2 .. 0: A_j = lambda^(L_{j+1}) A_{j+1} + U'_{j+1}
  }
}

// Pass B: every (direction, cut pair, 4 state elements) item, grid-stride.
template <bool MAX>
__global__ void __launch_bounds__(LINK_THREADS)
seg_link_kernel(const float* __restrict__ init, const float* __restrict__ dfin,
                const float* __restrict__ log_decay, float* __restrict__ states,
                float* __restrict__ adj, int T, int H, int whole, int parts, StatePages sp,
                unsigned* __restrict__ state_max, int X) {
  // a chunked kernel launched as this grid's dependent may start its whole pairs; the sums are
  // read once pass A is complete
  griddep_launch_dependents();
  griddep_wait();
  constexpr int N4 = DK * DV / 4;
  const long long per_dir = (long long)X * N4;
  for (long long it = (long long)blockIdx.x * LINK_THREADS + threadIdx.x; it < 2 * per_dir;
       it += (long long)gridDim.x * LINK_THREADS)
    link_one<MAX>(init, dfin, log_decay, states, adj, T, H, whole, parts, sp, state_max,
                  (int)(it / per_dir), (int)(it % per_dir / N4), (int)(it % N4));
}

// The state entering slice `rank` of a sequence cut into consecutive slices across ranks
// (forward), or the adjoint of the state leaving it (reverse), from every slice's sum:
//   forward  S_0 = boundary;      S_{j+1} = lambda^(len_j) S_j + U_j;      out = S_rank
//   reverse  A_{R-1} = boundary;  A_{j-1} = lambda^(len_j) A_j + U'_j;     out = A_rank
// U [R][B*H][96*192].  One thread per 4 consecutive state elements, walking the slices in
// order (the same recurrences as pass B, over slices instead of parts).
__global__ void shard_link_kernel(const float* __restrict__ U, const float* __restrict__ boundary,
                                  const float* __restrict__ log_decay, float* __restrict__ out,
                                  ShardLens lens, int rank, int reverse, int BH, int H) {
  constexpr int N4 = DK * DV / 4;
  const int bh = blockIdx.y, e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= N4) return;
  const float gamma = __ldg(log_decay + bh % H);
  const float4* u4 = reinterpret_cast<const float4*>(U) + e;
  float4 s = boundary ? __ldg(reinterpret_cast<const float4*>(boundary) + (size_t)bh * N4 + e)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  const int j0 = reverse ? lens.n - 1 : 0, j1 = reverse ? rank : rank, step = reverse ? -1 : 1;
  for (int j = j0; j != j1; j += step) {
    const float lam = expf(gamma * (float)lens.len[j]);
    const float4 u = __ldg(u4 + ((size_t)j * BH + bh) * N4);
    s = make_float4(fmaf(lam, s.x, u.x), fmaf(lam, s.y, u.y), fmaf(lam, s.z, u.z),
                    fmaf(lam, s.w, u.w));
  }
  reinterpret_cast<float4*>(out)[(size_t)bh * N4 + e] = s;
}

// Finish time of `jobs` equal jobs of length d, list-scheduled in order on n_sm SMs of which
// n_hi become free at t_hi and the others at t_lo (t_lo <= t_hi); also the SMs' last finish.
double list_finish(long long jobs, double d, int n_sm, int n_hi, double t_lo, double t_hi) {
  std::map<double, long long> free_at;  // time -> SMs free from then on
  if (n_sm - n_hi > 0) free_at[t_lo] += n_sm - n_hi;
  if (n_hi > 0) free_at[t_hi] += n_hi;
  while (jobs > 0) {
    auto it = free_at.begin();
    const double t = it->first;
    const long long n = it->second;
    free_at.erase(it);
    const long long k = n < jobs ? n : jobs;
    free_at[t + d] += k;
    if (n > k) free_at[t] += n - k;
    jobs -= k;
  }
  return free_at.rbegin()->first;
}

}  // namespace

// Estimated costs in chunk steps of the main kernel (forward / backward), from GB300 launch
// lists: a CTA's start and drain (its pipeline fill and the read of its starting state), one
// chunk of a segment pass and a pass CTA's start, and the passes' two extra launches.  A cut
// must promise kMinGain of the uncut time, the estimate being rough.
namespace {
constexpr double kCtaStart = 3.0;
constexpr double kPassChunk[2] = {0.25, 0.2};
constexpr double kPassStart = 2.0;
constexpr double kPassLaunch = 2.0;
constexpr double kMinGain = 0.97;
constexpr int kMaxParts = 32;
// Automatic cuts keep at least this many chunks per part.  (At T = 2048 a sweep of 1, 2 and 4
// parts over B = 8..40 matched the estimate's ratios to about 3 %: cutting pays when the last
// wave is nearly empty -- backward B = 16, 32; forward B = 12, 40 -- and costs otherwise.)
constexpr int kMinPartChunks = 4;

// CTAs of a sum pass of `items` parts beside the whole CTAs: the SMs the last wave's `tail`
// part CTAs leave over (the others start with a whole CTA, so all the parts find an SM free at
// about the same time), but enough to end within half the whole CTAs' waves (t_lo steps).
long long pass_width(long long items, long long tail, double pre_len, double t_lo, int n_sm) {
  long long w = n_sm - tail;
  const long long w_min =
      t_lo > 0.0 ? (long long)std::ceil((double)items * pre_len * 2.0 / t_lo) : items;
  if (w < w_min) w = w_min;
  if (w > items) w = items;
  return w < 1 ? 1 : w;
}
}  // namespace

SplitPlan plan_split(long long BH, int nc, int roles, int n_sm, int force_parts, int pass_dirs,
                     bool overlap) {
  SplitPlan none;
  none.whole = (int)BH;
  none.parts = 1;
  if (nc < 2 || n_sm <= 0 || BH <= 0 || force_parts == 1) return none;
  const long long ctas = (long long)roles * BH;
  long long X;  // pairs to cut: those of the partial last wave, or all when one wave holds them
  if (ctas <= n_sm) {
    X = BH;
  } else {
    const long long rem = ctas % n_sm;
    if (rem == 0) return none;
    X = (rem + roles - 1) / roles;
  }
  const int bwd = roles > 1 ? 1 : 0;
  const long long W = (long long)roles * (BH - X);  // whole CTAs, launched first
  const double whole_len = nc + kCtaStart;
  const double t_lo = (double)(W / n_sm) * whole_len;
  const int n_hi = (int)(W % n_sm);
  // p = 1: the X pairs run whole too
  int best_p = 1;
  const double uncut =
      list_finish((long long)roles * X, whole_len, n_sm, n_hi, t_lo, t_lo + whole_len);
  double best = uncut * kMinGain;
  const int p_auto = nc / kMinPartChunks < kMaxParts ? nc / kMinPartChunks : kMaxParts;
  const int p_max = force_parts >= 2 ? (force_parts < nc ? force_parts : nc) : p_auto;
  for (int p = force_parts >= 2 ? p_max : 2; p <= p_max; ++p) {
    const double part_len = (double)((nc + p - 1) / p) + kCtaStart;
    const double main_t =
        list_finish((long long)roles * X * p, part_len, n_sm, n_hi, t_lo, t_lo + whole_len);
    const long long pre_ctas = X * (p - 1) * pass_dirs;
    const double pre_len = (double)((nc + p - 1) / p) * kPassChunk[bwd] + kPassStart;
    const double launches = p == 2 ? kPassLaunch / 2 : kPassLaunch;  // two parts: no pass B
    double pre_t = (double)((pre_ctas + n_sm - 1) / n_sm) * pre_len + launches;
    if (overlap && W >= n_sm) {
      // beside at least a wave of whole CTAs the passes take only their share of the SMs'
      // time (their CTAs start first, the whole CTAs on the other SMs); the parts wait for
      // them only if they end after the whole CTAs
      const long long width = pass_width(pre_ctas, roles * X * p, pre_len, t_lo, n_sm);
      const double pre_serial = (double)((pre_ctas + width - 1) / width) * pre_len + launches;
      pre_t = (double)pre_ctas * pre_len / n_sm + (pre_serial > t_lo ? pre_serial - t_lo : 0.0);
    }
    const double total = main_t + pre_t;
    if (force_parts >= 2 || total < best) {
      best = total;
      best_p = p;
    }
  }
  if (best_p == 1) return none;
  SplitPlan plan;
  plan.whole = (int)(BH - X);
  plan.parts = best_p;
  plan.overlap = overlap && W >= n_sm;
  if (plan.overlap) {
    const long long items = X * (best_p - 1) * pass_dirs;
    const double pre_len = (double)((nc + best_p - 1) / best_p) * kPassChunk[bwd] + kPassStart;
    plan.pass_ctas = (int)pass_width(items, roles * X * best_p, pre_len, t_lo, n_sm);
  }
  return plan;
}

long long split_slots(long long BH, const SplitPlan& p) {
  return p.parts > 1 ? (BH - p.whole) * (long long)p.parts : 0;
}

cudaError_t launch_segment_states(const void* q, const void* k, const void* v, const void* dO,
                                  bool bf16, const float* log_decay, const float* init,
                                  const float* dfin, const StatePages& sp, float* states,
                                  float* adj, int B, int T, int H, const SplitPlan& plan,
                                  DevCtl ctl, cudaStream_t stream, float* state_max) {
  const long long X = (long long)B * H - plan.whole;
  if (plan.parts <= 1 || X <= 0) return cudaSuccess;
  CUtensorMap mk, mv, mq, mg;
  if (!make_tmap_seq_16bit(&mk, k, DK, H, T, B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, bf16) ||
      !make_tmap_seq_16bit(&mv, v, DV, H, T, B, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, bf16))
    return cudaErrorInvalidValue;
  if (adj) {
    if (!make_tmap_seq_16bit(&mq, q, DK, H, T, B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, bf16) ||
        !make_tmap_seq_16bit(&mg, dO, DV, H, T, B, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, bf16))
      return cudaErrorInvalidValue;
  } else {
    mq = mk;  // stand-ins, never read
    mg = mv;
  }
  const long long n_fwd = states ? X * (plan.parts - 1) : 0;
  const long long n_rev = adj ? X * (plan.parts - 1) : 0;
  const long long n_items = n_fwd + n_rev;
  // two parts: one recurrence step per direction, which the sum pass takes itself
  const bool fold = plan.parts == 2;
  if (n_items > 0) {
    auto kern = bf16 ? seg_sum_kernel<true> : seg_sum_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long grid =
        plan.pass_ctas > 0 && plan.pass_ctas < n_items ? plan.pass_ctas : n_items;
    kern<<<(unsigned)grid, THREADS, SMEM_BYTES, stream>>>(
        mk, mv, mq, mg, log_decay, states, adj, init, dfin, sp, state_max, T, H, plan.whole,
        plan.parts, (int)n_fwd, (int)n_items, 0, 1, fold ? 1 : 0, ctl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (fold) return cudaSuccess;
  const long long items = 2LL * X * (DK * DV / 4);
  long long ctas = (items + LINK_THREADS - 1) / LINK_THREADS;
  if (plan.overlap) {
    // beside the whole pairs: about four items of the directions computed per thread, on at
    // most LINK_CTAS_OVERLAP CTAs (they hold their SMs while they wait for pass A)
    const long long work = (long long)((states ? 1 : 0) + (adj ? 1 : 0)) * X * (DK * DV / 4);
    ctas = (work + 4LL * LINK_THREADS - 1) / (4LL * LINK_THREADS);
    if (ctas > LINK_CTAS_OVERLAP) ctas = LINK_CTAS_OVERLAP;
    if (ctas < 1) ctas = 1;
  }
  PdlLaunch L(dim3((unsigned)ctas), dim3(LINK_THREADS), 0, stream, plan.overlap);
  auto kern = state_max ? seg_link_kernel<true> : seg_link_kernel<false>;
  return cudaLaunchKernelEx(&L.cfg, kern, init, dfin, log_decay, states, adj, T, H, plan.whole,
                            plan.parts, sp, reinterpret_cast<unsigned*>(state_max), (int)X);
}

cudaError_t launch_slice_sums(const void* a, const void* b, bool bf16, bool reverse,
                              const float* log_decay, float* out, int B, int T, int H, int n_sm,
                              DevCtl ctl, cudaStream_t stream) {
  // a, b = k, v (forward: U of the slice) or q, dO (reverse: U' of the slice)
  CUtensorMap ma, mb;
  if (!make_tmap_seq_16bit(&ma, a, DK, H, T, B, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, bf16) ||
      !make_tmap_seq_16bit(&mb, b, DV, H, T, B, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, bf16))
    return cudaErrorInvalidValue;
  const long long n = (long long)B * H;
  // fewer pairs than SMs: each pair's sum in three CTAs, one 64-column third of the value
  // channels each (k is read three times; every CTA writes its own columns, so no workspace)
  const int ncol = n < n_sm ? 3 : 1;
  const long long items = n * ncol;
  auto kern = bf16 ? seg_sum_kernel<true> : seg_sum_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)items, THREADS, SMEM_BYTES, stream>>>(
      ma, mb, ma, mb, log_decay, reverse ? nullptr : out, reverse ? out : nullptr, nullptr,
      nullptr, StatePages{}, nullptr, T, H, 0, 2, reverse ? 0 : (int)items, (int)items, 1, ncol, 0,
      ctl);
  return cudaGetLastError();
}

cudaError_t launch_shard_link(const float* U, const ShardLens& lens, int rank, bool reverse,
                              const float* log_decay, const float* boundary, float* out, int B,
                              int H, cudaStream_t stream) {
  const int BH = B * H;
  shard_link_kernel<<<dim3((DK * DV / 4 + 255) / 256, (unsigned)BH), 256, 0, stream>>>(
      U, boundary, log_decay, out, lens, rank, reverse ? 1 : 0, BH, H);
  return cudaGetLastError();
}

}  // namespace gla
