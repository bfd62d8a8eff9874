// head_norm.cu -- the mixer's output epilogue: Head RMSNorm per decay tier, then SiLU(g) gate.
//
// Method ("Beyond the KV cache ... Laplace 3B ...", section "i14 and the Laplace 3B
// architecture", "GLA mixer" and "Decay schedule's reach"): the per-head outputs pass through
// a Head RMSNorm shared within each decay tier, are concatenated and gated by SiLU(g_t).  Per
// token t and head h, with tier(h) = h / (H / n_tiers) (tiers of consecutive heads, i.e. of
// neighbouring half-lives) and C = 192 value channels:
//   r    = 1 / sqrt(mean_c o_c^2 + eps)
//   y_c  = o_c r w[tier(h), c] SiLU(g_c),          SiLU(x) = x sigmoid(x)
// and its gradient for the scalar loss sum(y . dy):
//   n_c = o_c r,  a_c = n_c w_c,  s_c = SiLU(g_c)
//   dg_c = dy_c a_c sigmoid(g_c) (1 + g_c (1 - sigmoid(g_c)))
//   dn_c = dy_c s_c w_c,   do_c = r (dn_c - n_c mean_c'(dn_c' n_c'))
//   dw[tier, c] = sum over tokens and the tier's heads of dy_c s_c n_c
// All fp32 (g may be bf16).  One half-warp per (t, h) row: 16 lanes x 3 float4 = 192 channels,
// coalesced 768-byte rows; the per-row sum is a 16-lane shuffle reduction.  dw: every
// half-warp slot sees one head only and keeps its partial sums in registers, each CTA sums its
// slots per tier, and a second kernel sums the CTAs in a fixed order (deterministic).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace gla {
namespace {

constexpr int C = 192, C4 = C / 4, LANES = 16, PER = C4 / LANES;  // 3 float4 per lane
static_assert(PER * LANES == C4, "row tiling");
constexpr int THREADS = 256, ROWS_PER_CTA = THREADS / LANES;   // 16 rows per pass

template <bool GBF16>
__device__ __forceinline__ float4 load_g(const void* g, long long row, int c4) {
  if constexpr (GBF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(g) +
                                                         row * C) + c4);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  } else {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(g) + row * C) + c4);
  }
}

// logistic function with the fast intrinsics (a few ulp, far inside the fp32 bar)
__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

__device__ __forceinline__ float sum16(float x) {
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// component j (a constant after unrolling) of a float4
__device__ __forceinline__ float& F4(float4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

template <bool GBF16>
__global__ void __launch_bounds__(THREADS)
head_norm_fwd_kernel(const float* __restrict__ o, const void* __restrict__ g,
                     const float* __restrict__ w, float* __restrict__ y, float* __restrict__ rstd,
                     long long rows, int H, int heads_per_tier, float eps) {
  const int lane = threadIdx.x % LANES, hw = threadIdx.x / LANES;
  // The loop runs on the warp's first row so that both half-warps take every shuffle; the
  // second half-warp's row may lie past the end (then it loads and stores nothing).
  for (long long row0 = (long long)blockIdx.x * ROWS_PER_CTA + (hw & ~1); row0 < rows;
       row0 += (long long)gridDim.x * ROWS_PER_CTA) {
    const long long row = row0 + (hw & 1);
    const bool live = row < rows;
    const int tier = (int)(row % H) / heads_per_tier;
    // every load of the row first, so that they overlap
    float4 x[PER], gv[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      x[p] = live ? __ldg(reinterpret_cast<const float4*>(o + row * C) + lane + LANES * p)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      gv[p] = live ? load_g<GBF16>(g, row, lane + LANES * p) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ss = 0.f;
#pragma unroll
    for (int p = 0; p < PER; ++p)
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(F4(x[p], j), F4(x[p], j), ss);
    const float r = 1.f / sqrtf(sum16(ss) / C + eps);
    if (!live) continue;
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int c4 = lane + LANES * p;
      float4 gg = gv[p];
      float4 ww = __ldg(reinterpret_cast<const float4*>(w + tier * C) + c4);
      float4 out;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        F4(out, j) = F4(x[p], j) * r * F4(ww, j) * (F4(gg, j) * sigm(F4(gg, j)));
      reinterpret_cast<float4*>(y + row * C)[c4] = out;
    }
    if (rstd && lane == 0) rstd[row] = r;
  }
}

// dw partial sums.  The grid stride (gridDim.x * 16 rows) is a multiple of H, so half-warp
// slot q = blockIdx.x * 16 + threadIdx.x / 16 always sees head (q % H): its lanes keep their
// 12 channels' partial sums of dy s n in registers.  At the end the CTA adds its 16 slots per
// tier, in slot order, into part[blockIdx.x][tier][c].
template <bool GBF16>
__global__ void __launch_bounds__(THREADS)
head_norm_bwd_kernel(const float* __restrict__ dy, const float* __restrict__ o,
                     const void* __restrict__ g, const float* __restrict__ w,
                     float* __restrict__ d_o, float* __restrict__ dg, float* __restrict__ part,
                     long long rows, int H, int heads_per_tier, int n_tiers, float eps) {
  griddep_launch_dependents();  // the dw reduction launched next waits for this whole grid
  __shared__ float4 sacc[ROWS_PER_CTA][C4];
  __shared__ int stier[ROWS_PER_CTA];
  const int lane = threadIdx.x % LANES, hw = threadIdx.x / LANES;
  const long long slot = (long long)blockIdx.x * ROWS_PER_CTA + hw;
  const int tier = (int)(slot % H) / heads_per_tier;
  float4 wt[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p)
    wt[p] = __ldg(reinterpret_cast<const float4*>(w + tier * C) + lane + LANES * p);
  float4 acc[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) acc[p] = make_float4(0.f, 0.f, 0.f, 0.f);
  // loop on the warp's first slot: both half-warps take every shuffle (see the forward)
  for (long long row0 = slot - (hw & 1); row0 < rows; row0 += (long long)gridDim.x * ROWS_PER_CTA) {
    const long long row = row0 + (hw & 1);
    const bool live = row < rows;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    // every load of the row first, so that they overlap
    float4 x[PER], gv[PER], dv[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int c4 = lane + LANES * p;
      x[p] = live ? __ldg(reinterpret_cast<const float4*>(o + row * C) + c4) : zero;
      gv[p] = live ? load_g<GBF16>(g, row, c4) : zero;
      dv[p] = live ? __ldg(reinterpret_cast<const float4*>(dy + row * C) + c4) : zero;
    }
    float ss = 0.f;
#pragma unroll
    for (int p = 0; p < PER; ++p)
#pragma unroll
      for (int j = 0; j < 4; ++j) ss = fmaf(F4(x[p], j), F4(x[p], j), ss);
    const float r = 1.f / sqrtf(sum16(ss) / C + eps);
    float4 dn[PER];
    float dot = 0.f;  // sum_c dn_c n_c
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int c4 = lane + LANES * p;
      float4 gg = gv[p];
      float4 ww = wt[p];
      float4 dd = dv[p];
      float4 dgo;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float n = F4(x[p], j) * r, gv = F4(gg, j), sg = sigm(gv), s = gv * sg;
        const float da = F4(dd, j) * s;  // d(loss)/d(n w)
        F4(dgo, j) = F4(dd, j) * n * F4(ww, j) * sg * (1.f + gv * (1.f - sg));
        F4(dn[p], j) = da * F4(ww, j);
        dot = fmaf(F4(dn[p], j), n, dot);
        F4(acc[p], j) = fmaf(da, n, F4(acc[p], j));
      }
      if (live) reinterpret_cast<float4*>(dg + row * C)[c4] = dgo;
    }
    const float m = sum16(dot) / C;
    if (!live) continue;
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      float4 out;
#pragma unroll
      for (int j = 0; j < 4; ++j) F4(out, j) = r * (F4(dn[p], j) - F4(x[p], j) * r * m);
      reinterpret_cast<float4*>(d_o + row * C)[lane + LANES * p] = out;
    }
  }
#pragma unroll
  for (int p = 0; p < PER; ++p) sacc[hw][lane + LANES * p] = acc[p];
  if (lane == 0) stier[hw] = tier;
  __syncthreads();
  const float* sa = reinterpret_cast<const float*>(sacc);
  for (int i = threadIdx.x; i < n_tiers * C; i += THREADS) {
    const int t = i / C, c = i % C;
    float sum = 0.f;
    for (int q = 0; q < ROWS_PER_CTA; ++q)
      if (stier[q] == t) sum += sa[q * C + c];
    part[(size_t)blockIdx.x * n_tiers * C + i] = sum;
  }
}

// dw[i] = sum over the CTAs' partial sums part[b][i].  One CTA of RED_WARPS warps per 32
// consecutive outputs: warp w adds b = w, w + RED_WARPS, ... in order (coalesced rows), then
// one thread per output adds the warps' sums in order (a fixed order: deterministic).
// Launched as the backward kernel's programmatic dependent: it waits for that grid first.
constexpr int RED_WARPS = 32;
__global__ void __launch_bounds__(RED_WARPS * 32)
head_norm_dw_reduce(const float* __restrict__ part, float* __restrict__ dw, int n_parts, int n) {
  __shared__ float acc[RED_WARPS][33];
  griddep_wait();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int i = blockIdx.x * 32 + lane;
  const bool live = i < n;
  float s = 0.f;
  if (live) {
#pragma unroll 8
    for (int b = wid; b < n_parts; b += RED_WARPS) s += part[(size_t)b * n + i];
  }
  acc[wid][lane] = s;
  __syncthreads();
  if (wid == 0 && live) {
    float t = 0.f;
#pragma unroll 8
    for (int w = 0; w < RED_WARPS; ++w) t += acc[w][lane];
    dw[i] = t;
  }
}

// CTAs for `rows` rows: at most 8 per SM, and a multiple of H / gcd(16, H) so that the grid
// stride (16 rows per CTA) is a multiple of H.
int grid_for(long long rows, int H, int n_sm) {
  int a = 16, b = H;
  while (b) { const int t = a % b; a = b; b = t; }
  const long long unit = H / a;
  const long long need = (rows + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  long long grid = (long long)(n_sm > 0 ? n_sm : 152) * 8;
  if (need < grid) grid = need;
  grid = (grid + unit - 1) / unit * unit;
  return (int)grid;
}

}  // namespace

size_t head_norm_bwd_workspace_bytes(long long rows, int H, int n_sm) {
  return (size_t)grid_for(rows, H, n_sm) * H * C * sizeof(float);  // n_tiers <= H
}

cudaError_t launch_head_norm_fwd(const float* o, const void* g, bool g_bf16, const float* w,
                                 float* y, float* rstd, long long rows, int H, int n_tiers,
                                 float eps, int n_sm, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int grid = grid_for(rows, H, n_sm);
  if (g_bf16)
    head_norm_fwd_kernel<true><<<grid, THREADS, 0, stream>>>(o, g, w, y, rstd, rows, H,
                                                               H / n_tiers, eps);
  else
    head_norm_fwd_kernel<false><<<grid, THREADS, 0, stream>>>(o, g, w, y, rstd, rows, H,
                                                                H / n_tiers, eps);
  return cudaGetLastError();
}

cudaError_t launch_head_norm_bwd(const float* dy, const float* o, const void* g, bool g_bf16,
                                 const float* w, float* d_o, float* dg, float* dw, float* part,
                                 long long rows, int H, int n_tiers, float eps, int n_sm,
                                 cudaStream_t stream) {
  if (rows <= 0) return cudaMemsetAsync(dw, 0, sizeof(float) * n_tiers * C, stream);
  const int grid = grid_for(rows, H, n_sm);
  if (g_bf16)
    head_norm_bwd_kernel<true><<<grid, THREADS, 0, stream>>>(dy, o, g, w, d_o, dg, part, rows, H,
                                                               H / n_tiers, n_tiers, eps);
  else
    head_norm_bwd_kernel<false><<<grid, THREADS, 0, stream>>>(dy, o, g, w, d_o, dg, part, rows, H,
                                                                H / n_tiers, n_tiers, eps);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = n_tiers * C;
  PdlLaunch R(dim3((n + 31) / 32), dim3(RED_WARPS * 32), 0, stream, true);
  return cudaLaunchKernelEx(&R.cfg, head_norm_dw_reduce, (const float*)part, dw, grid, n);
}

}  // namespace gla
