// seg_scan.cu -- segment-parallel chunked forward for few, long sequences.
//
// Method: the chunked forward ("Beyond the KV cache ... Laplace 3B ...", section "Challenge 1")
// carries the state from chunk to chunk, so each (b, h) is a serial chain of T/128 steps and a
// call with few (b, h) pairs -- long-context prefill -- leaves most SMs idle.  The state
// recurrence S_t = lambda S_{t-1} + k_t v_t^T (section "i14 and the Laplace 3B architecture",
// "GLA mixer") is linear, so for a sequence cut into G segments of L tokens, segment g ending
// at token e_g,
//
//     S_{e_g} = lambda^L S_{e_{g-1}} + U_g,     U_g = sum_{t in g} lambda^(e_g - t) k_t v_t^T.
//
//   pass A  (seg_state_kernel, one CTA per (b, h, g) for every segment but the last): U_g on
//           the tensor cores, K''^T V over the segment's chunks into one fp32 TMEM accumulator,
//           the decay folded into the fp16 copy of k (row t scaled by lambda^(e_g - t));
//   pass B  (seg_combine_kernel): the G-step recurrence above per (b, h), giving every
//           segment's initial state (segment 0: the caller's, or zero);
//   pass C  the ordinary chunked forward over the B*G segments as independent sequences --
//           [B][T][H][d] is the same memory as [B*G][T/G][H][d] -- with only the last segment
//           of each sequence writing the final state.
//
// Extra traffic: pass A reads k and v of all but the last segment (576 B per token-head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

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
constexpr uint32_t NBAR = 10;
constexpr uint32_t OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4;
constexpr uint32_t OFF_PW = OFF_TMEM + 16;  // float pw[128] = lambda^i
constexpr uint32_t SMEM_USED = OFF_PW + 512;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + alignment of the dynamic base
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

enum Bar : uint32_t {
  FULL = 0,   // 0..2: stage s landed
  CONV = 3,   // 3..5: stage s converted to fp16 operands
  EMPTY = 6,  // 6..8: the MMAs of stage s are done
  DONE = 9,   // every MMA is done
};

constexpr int THREADS = 192;  // warps 0..3 convert + epilogue (row = token = TMEM lane)
constexpr int PRODUCER_WARP = 4, MMA_WARP = 5;
constexpr int MIN_SEGMENT_CHUNKS = 16;  // shorter segments do not repay the extra pass

// 16-byte chunk `cc` of row `i`: k has 3 boxes of 32 channels (64-byte rows), v 3 boxes of 64
// channels (128-byte rows), v after k within a stage.
__device__ __forceinline__ uint32_t k_chunk(uint32_t i, int cc) {
  return (cc >> 2) * K_BOX + swz_off(i, cc & 3, 64);
}
__device__ __forceinline__ uint32_t v_chunk(uint32_t i, int cc) {
  return 3 * K_BOX + (cc >> 3) * V_BOX + swz_off(i, cc & 7, 128);
}

// Pass A.  CTA (b, h, g) writes U_g to u_out[b*G + g + 1][h] (the slot of the initial state of
// segment g + 1, which pass B then turns into that state in place).
template <bool BF16>
__global__ void __launch_bounds__(THREADS, 1)
seg_state_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                 const float* __restrict__ log_decay, float* __restrict__ u_out, int T, int H, int G,
                 DevCtl ctl) {
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
  const int g = blockIdx.x % (G - 1), bh = blockIdx.x / (G - 1), b = bh / H, h = bh % H;
  const int M = T / C / G;                     // chunks per segment
  const int row0 = b * T + g * M * C;          // first token row of the segment
  const float gamma = __ldg(log_decay + h);
  float* pw = (float*)(base + OFF_PW);
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
    *cta.abort_flag() = 0;
    fence_barrier_init();
  }
  if (tid < C) pw[tid] = expf((float)tid * gamma);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sb = cta.sb;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      int armed0 = 0, armed1 = 0, armed2 = 0;  // loads issued per stage
      for (int m = 0; m < M; ++m) {
        const int s = m % STAGES;
        if (m >= STAGES && !wait(cta, cta.bar(EMPTY + s), (m / STAGES - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(cta.bar(FULL + s), STAGE);
        const int row = row0 + m * C;
        const uint32_t st = sb + s * STAGE;
        for (int j = 0; j < 3; ++j) {
          tma_load_3d(st + j * K_BOX, &map_k, cta.bar(FULL + s), 32 * j, h, row);
          tma_load_3d(st + 3 * K_BOX + j * V_BOX, &map_v, cta.bar(FULL + s), 64 * j, h, row);
        }
        armed0 += s == 0;
        armed1 += s == 1;
        armed2 += s == 2;
      }
      // no copy may still be landing when the CTA exits
      if (armed0) mbar_wait(cta.bar(FULL + 0), (armed0 - 1) & 1, ctl, DRAIN_NS);
      if (armed1) mbar_wait(cta.bar(FULL + 1), (armed1 - 1) & 1, ctl, DRAIN_NS);
      if (armed2) mbar_wait(cta.bar(FULL + 2), (armed2 - 1) & 1, ctl, DRAIN_NS);
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      // U (rows = 96 key channels + 32 padding rows never read) += K''^T V, K = 16 tokens per
      // instruction: A = k tile as [token][channel] (MN-major), B = v tile as [token][channel]
      constexpr uint32_t ID = idesc_f16(128, 192, false, false, true, true);
      for (int m = 0; m < M; ++m) {
        const int s = m % STAGES;
        if (!wait(cta, cta.bar(CONV + s), (m / STAGES) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t st = sb + s * STAGE;
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks)
          mma_f16_ss(tmem, smem_desc(st + ks * 1024, K_BOX, 512, SW_64),
                     smem_desc(st + 3 * K_BOX + ks * 2048, V_BOX, 1024, SW_128), ID,
                     (m > 0 || ks > 0) ? 1u : 0u);
        mma_commit(cta.bar(EMPTY + s));
      }
      mma_commit(cta.bar(DONE));
      mbar_wait(cta.bar(DONE), 0, ctl, DRAIN_NS);
    }
  } else {
    // ---- warps 0..3: in-place fp16 operands of chunk m, row i = token i of the chunk:
    // k scaled by lambda^(e_g - t) for its token t, v as it is
    const int i = tid;
    float vmax = 0.f;
    bool ok = true;
    for (int m = 0; m < M && ok; ++m) {
      const int s = m % STAGES;
      if (!(ok = wait(cta, cta.bar(FULL + s), (m / STAGES) & 1, ctl))) break;
      uint8_t* st = base + s * STAGE;
      const float sk = expf(gamma * (float)(C * (M - 1 - m))) * pw[C - 1 - i];
      convert_row<BF16, 12>(st, [&](int cc) { return k_chunk(i, cc); }, sk, vmax);
      convert_row<BF16, 24>(st, [&](int cc) { return v_chunk(i, cc); }, 1.f, vmax);
      fence_proxy_async();
      mbar_arrive(cta.bar(CONV + s));
    }
    // ---- U_g out: rows 0..95 (warps 0..2), 192 fp32 each
    if (ok) ok = wait(cta, cta.bar(DONE), 0, ctl);
    ok = __all_sync(0xffffffffu, ok && *cta.abort_flag() == 0);
    if (ok && warp < 3) {
      tc_fence_after();
      float* dst = u_out + ((size_t)(b * G + g + 1) * H + h) * DK * DV + (size_t)i * DV;
      const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
      for (int cb = 0; cb < DV / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(trow + 32 * cb, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(dst + 32 * cb + j) =
              make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                          __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
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

// Pass B.  vinit[b*G + g][h] (g >= 1) holds U_{g-1} on entry and the initial state of segment
// g on exit; vinit[b*G][h] receives the caller's initial state (or zeros).  One thread per
// 4 consecutive state elements, walking the segments in order.
__global__ void seg_combine_kernel(const float* __restrict__ init, const float* __restrict__ log_decay,
                                   float* __restrict__ vinit, int H, int G, int L, StatePages sp) {
  constexpr int N4 = DK * DV / 4;
  const int bh = blockIdx.y, b = bh / H, h = bh % H;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= N4) return;
  const float lamL = expf(__ldg(log_decay + h) * (float)L);  // lambda^L
  long long zi = bh;  // slot of the caller's initial state: [b][h] or a pool page
  if (sp.init_paged) {
    const int pg = __ldg(sp.page + b);
    zi = (pg >= 0 && pg < sp.n_pages) ? ((long long)pg * sp.pool_layers + sp.layer) * H + h : -1;
  }
  float4 s = (init && zi >= 0) ? __ldg(reinterpret_cast<const float4*>(init) + (size_t)zi * N4 + e)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  float4* out = reinterpret_cast<float4*>(vinit);
  out[((size_t)b * G * H + h) * N4 + e] = s;
  for (int g = 1; g < G; ++g) {
    float4* p = out + ((size_t)(b * G + g) * H + h) * N4 + e;
    const float4 u = *p;
    s = make_float4(fmaf(lamL, s.x, u.x), fmaf(lamL, s.y, u.y), fmaf(lamL, s.z, u.z),
                    fmaf(lamL, s.w, u.w));
    *p = s;
  }
}

}  // namespace

int fwd_segments(int B, int T, int H, int n_sm) {
  const long long bh = (long long)B * H;
  const int nc = T / C;
  if (T % C != 0) return 1;                  // a ragged last chunk: one serial scan
  if (n_sm <= 0 || 2 * bh > n_sm) return 1;  // enough (b, h) pairs to fill the GPU already
  int best = 1;
  for (int G = 2; G <= nc / MIN_SEGMENT_CHUNKS && bh * G <= n_sm; ++G)
    if (nc % G == 0) best = G;
  return best;
}

size_t fwd_segment_workspace_bytes(int B, int H, int G) {
  return G > 1 ? (size_t)B * G * H * DK * DV * sizeof(float) : 0;
}

cudaError_t launch_chunk_fwd_segmented(const FwdArgs& a, int G, void* workspace, DevCtl ctl,
                                       cudaStream_t stream) {
  float* vinit = static_cast<float*>(workspace);
  CUtensorMap mk, mv;
  const long long rows = (long long)a.B * a.T;
  if (!make_tmap_3d_16bit(&mk, a.k, DK, a.H, rows, 32, C, CU_TENSOR_MAP_SWIZZLE_64B, a.bf16) ||
      !make_tmap_3d_16bit(&mv, a.v, DV, a.H, rows, 64, C, CU_TENSOR_MAP_SWIZZLE_128B, a.bf16))
    return cudaErrorInvalidValue;
  auto kern = a.bf16 ? seg_state_kernel<true> : seg_state_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.H * (G - 1), THREADS, SMEM_BYTES, stream>>>(mk, mv, a.log_decay, vinit, a.T, a.H,
                                                             G, ctl);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  seg_combine_kernel<<<dim3((DK * DV / 4 + 255) / 256, a.B * a.H), 256, 0, stream>>>(
      a.init, a.log_decay, vinit, a.H, G, a.T / G, a.sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  FwdArgs c = a;
  c.B = a.B * G;
  c.T = a.T / G;
  c.init = vinit;
  c.seg = G;
  c.sp.init_paged = false;  // the segments' initial states are in the workspace
  return launch_chunk_fwd(c, ctl, stream);
}

}  // namespace gla
