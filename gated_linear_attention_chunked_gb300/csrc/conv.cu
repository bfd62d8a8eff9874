// conv.cu -- the depth-wise causal Conv1d (width 4) with SiLU in front of the QKVG projection,
// and its 3-token recurrent state.
//
// Method ("Beyond the KV cache ... Laplace 3B ...", section "i14 and the Laplace 3B
// architecture", "Normalization and convolution"): every channel d of the residual stream
// (D = 3072) is filtered causally over the last 4 tokens, then SiLU:
//   z_t[d] = sum_{j=0..3} w[d][j] x_{t-3+j}[d] + b[d],     y_t[d] = SiLU(z_t[d])
// with x_{-3..-1} the conv state carried from earlier tokens (zeros for a new sequence); the
// state after the call is x_{T-3..T-1}.  Decode is the same with T = 1 on a state of 3 inputs.
// Gradient for the scalar loss sum(y . dy), with dz = dy SiLU'(z):
//   dx_s = sum_j w[j] dz_{s+3-j}   (s = -3..-1: the initial state),
//   dw[d][j] = sum_{b,t} dz_t x_{t-3+j},  db[d] = sum_{b,t} dz_t.
// Memory-bound streaming: one thread owns 4 consecutive channels of a 64-token tile (2 in the
// staged backward) and walks its tokens with the 4-token window in registers (3-token halo,
// ~5 % re-read).  dw, db: per
// tile partial sums, summed over tiles in a fixed order by a second kernel (deterministic).
// Each thread issues the loads of 8 tokens before using the first, so that several DRAM
// round trips overlap.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "kernels.h"

namespace gla {
namespace {

constexpr int K = 4;        // filter width
constexpr int TT = 32;      // tokens per tile (forward: more CTAs, a shorter tail; 64 measured
                            // 2.4 % slower, 16 the same as 32 with more halo re-reads)
constexpr int TTB = 128;    // tokens per tile (backward: half the weight-gradient partial sums
                            // and halo re-reads of 64; 256 measured slower)
constexpr int THREADS = 256;

template <bool BF16>
__device__ __forceinline__ float4 load_x(const void* x, long long idx4) {  // 4 channels
  if constexpr (BF16) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(x) + idx4);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  } else {
    return __ldg(reinterpret_cast<const float4*>(x) + idx4);
  }
}

// raw 4-channel load (bf16: 8 bytes, fp32: 16 bytes) and its conversion, so that a group of
// tokens' loads can all be issued before the first is used
template <bool BF16>
struct Raw {
  using T = typename std::conditional<BF16, uint2, float4>::type;
};
template <bool BF16>
__device__ __forceinline__ typename Raw<BF16>::T load_raw(const void* x, long long idx4) {
  if constexpr (BF16) return __ldg(reinterpret_cast<const uint2*>(x) + idx4);
  else return __ldg(reinterpret_cast<const float4*>(x) + idx4);
}
__device__ __forceinline__ float4 to_f4(uint2 u) {
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ float4 to_f4(float4 v) { return v; }

constexpr int GRP = 8;      // tokens whose loads are issued together (forward)
constexpr int GRP_BWD = 4;  // (backward: two loads per token, and two CTAs per SM)

__device__ __forceinline__ float& at(float4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
// logistic function with the fast intrinsics (a few ulp; the conv is issue bound, and the
// IEEE division and full-range expf were most of its instructions)
__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

// Four channels' arithmetic as two packed fp32 pairs: each lane is the same IEEE operation
// (round to nearest) as the scalar one, in half the instructions -- the conv is issue bound.
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 cat4(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {  // a * b + c
  return cat4(__ffma2_rn(lo2(a), lo2(b), lo2(c)), __ffma2_rn(hi2(a), hi2(b), hi2(c)));
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return cat4(__fmul2_rn(lo2(a), lo2(b)), __fmul2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return cat4(__fadd2_rn(lo2(a), lo2(b)), __fadd2_rn(hi2(a), hi2(b)));
}
// dz = dy SiLU'(z) = dy s (1 + z (1 - s)), s = sigmoid(z), for four channels
__device__ __forceinline__ float4 silu_grad4(float4 z, float4 dy) {
  const float4 s = make_float4(sigm(z.x), sigm(z.y), sigm(z.z), sigm(z.w));
  const float4 one = make_float4(1.f, 1.f, 1.f, 1.f), neg = make_float4(-1.f, -1.f, -1.f, -1.f);
  const float4 one_minus_s = fma4(s, neg, one);
  return mul4(mul4(dy, s), fma4(z, one_minus_s, one));
}

// x_t for token t of sequence b (t < 0: the initial state, row t + 3; zeros without one)
template <bool BF16>
__device__ __forceinline__ float4 x_at(const void* x, const float* init, int b, int t, int T,
                                       int D4, int d4) {
  if (t >= 0) return load_x<BF16>(x, ((long long)b * T + t) * D4 + d4);
  if (!init) return make_float4(0.f, 0.f, 0.f, 0.f);
  return __ldg(reinterpret_cast<const float4*>(init) + ((long long)b * 3 + (t + 3)) * D4 + d4);
}

struct Filt {
  float4 w[K];  // w[j] for the 4 channels
  float4 b;
};

__device__ __forceinline__ Filt load_filter(const float* w, const float* bias, int d4) {
  Filt f;
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 4 * d4 + 0);  // channel 4d4
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 4 * d4 + 1);
  const float4 w2 = __ldg(reinterpret_cast<const float4*>(w) + 4 * d4 + 2);
  const float4 w3 = __ldg(reinterpret_cast<const float4*>(w) + 4 * d4 + 3);
  // transpose: f.w[j] holds tap j of the 4 channels
  f.w[0] = make_float4(w0.x, w1.x, w2.x, w3.x);
  f.w[1] = make_float4(w0.y, w1.y, w2.y, w3.y);
  f.w[2] = make_float4(w0.z, w1.z, w2.z, w3.z);
  f.w[3] = make_float4(w0.w, w1.w, w2.w, w3.w);
  f.b = bias ? __ldg(reinterpret_cast<const float4*>(bias) + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
  return f;
}

// z for the window win[0..3] = x_{t-3..t}
__device__ __forceinline__ float4 conv4(Filt& f, float4 (&win)[K]) {
  float4 z = f.b;
#pragma unroll
  for (int j = 0; j < K; ++j) z = fma4(f.w[j], win[j], z);
  return z;
}

// grid: x = b * n_tiles + tile, y = channel groups of 4 * THREADS
template <bool BF16>
__global__ void __launch_bounds__(THREADS)
conv_fwd_kernel(const void* __restrict__ x, const float* __restrict__ w,
                const float* __restrict__ bias, const float* __restrict__ init,
                float* __restrict__ y, float* __restrict__ fin, int T, int D) {
  const int D4 = D / 4, d4 = blockIdx.y * THREADS + threadIdx.x;
  if (d4 >= D4) return;
  const int n_tiles = (T + TT - 1) / TT;
  const int b = blockIdx.x / n_tiles, t0 = (blockIdx.x % n_tiles) * TT;
  const int t1 = min(t0 + TT, T);
  Filt f = load_filter(w, bias, d4);
  float4 win[K];
#pragma unroll
  for (int j = 0; j < K - 1; ++j) win[j + 1] = x_at<BF16>(x, init, b, t0 - 3 + j, T, D4, d4);
  for (int tg = t0; tg < t1; tg += GRP) {
    typename Raw<BF16>::T raw[GRP];
#pragma unroll
    for (int u = 0; u < GRP; ++u)
      if (tg + u < t1) raw[u] = load_raw<BF16>(x, ((long long)b * T + tg + u) * D4 + d4);
#pragma unroll
    for (int u = 0; u < GRP; ++u) {
      if (tg + u >= t1) break;
      win[0] = win[1];
      win[1] = win[2];
      win[2] = win[3];
      win[3] = to_f4(raw[u]);
      float4 z = conv4(f, win);
      float4 o;
#pragma unroll
      for (int c = 0; c < 4; ++c) at(o, c) = at(z, c) * sigm(at(z, c));
      reinterpret_cast<float4*>(y)[((long long)b * T + tg + u) * D4 + d4] = o;
    }
  }
  if (fin && t1 == T) {  // the state after the call: x_{T-3..T-1}
#pragma unroll
    for (int j = 0; j < 3; ++j)
      reinterpret_cast<float4*>(fin)[((long long)b * 3 + j) * D4 + d4] = win[j + 1];
  }
}

// The forward with x staged through shared memory: each token's channel block of the CTA (4
// channels per thread, DC = 1024 channels) is one contiguous row that a single bulk copy moves
// into a ring of NST stages of SG tokens, so ~64 KB per CTA are in flight without holding
// registers (the register version above keeps 8 tokens of loads in flight per thread and was
// latency bound).  A ninth warp issues the copies and refills a stage as soon as every thread
// of the eight compute warps has read it (a compute thread that also issued them delayed each
// refill by its own share of the stage: the backward measured 0.422 -> 0.391 ms at B=32).
// Requires rows of 16-byte multiples: D % 8 == 0 for bf16 x, D % 4 == 0 for fp32 x.
constexpr int SG = 8;                  // tokens per stage
constexpr int NST = 4;                 // stages
constexpr int DC = 4 * THREADS;        // channels per CTA
constexpr uint64_t CONV_DRAIN_NS = 4000000000ull;
template <bool BF16>
constexpr uint32_t staged_fwd_smem() { return NST * SG * DC * (BF16 ? 2 : 4) + 2 * NST * 8; }

template <bool BF16>
__global__ void __launch_bounds__(THREADS + 32)
conv_fwd_staged_kernel(const void* __restrict__ x, const float* __restrict__ w,
                       const float* __restrict__ bias, const float* __restrict__ init,
                       float* __restrict__ y, float* __restrict__ fin, int T, int D, DevCtl ctl) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int ES = BF16 ? 2 : 4;
  constexpr uint32_t ROW = DC * ES, STAGE = SG * ROW;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * STAGE);  // full[NST], empty[NST]
  const int D4 = D / 4, c0 = blockIdx.y * DC, nch = min(DC, D - c0);
  const int d4 = c0 / 4 + threadIdx.x;
  const bool active = 4 * (int)threadIdx.x < nch;
  const int n_tiles = (T + TT - 1) / TT;
  const int b = blockIdx.x / n_tiles, t0 = (blockIdx.x % n_tiles) * TT;
  const int t1 = min(t0 + TT, T), ng = (t1 - t0 + SG - 1) / SG;
  const uint32_t row_bytes = (uint32_t)nch * ES, sb = smem_u32(smem);
  auto full = [&](int st) { return smem_u32(bars + st); };
  auto empty = [&](int st) { return smem_u32(bars + NST + st); };
  const uint8_t* xrow = static_cast<const uint8_t*>(x) + ((size_t)b * T * D + c0) * ES;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), THREADS);
    }
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;  // groups whose copies the producer has issued
  auto issue = [&](int g) {
    const int st = g % NST, ta = t0 + g * SG, tb = min(ta + SG, t1);
    mbar_arrive_expect_tx(full(st), (uint32_t)(tb - ta) * row_bytes);
    for (int t = ta; t < tb; ++t)
      bulk_load(sb + st * STAGE + (t - ta) * ROW, xrow + (size_t)t * D * ES, row_bytes, full(st));
    issued = g + 1;
  };
  if (threadIdx.x >= THREADS) {
    // the producer warp: refills a stage as soon as every compute thread has read it
    if (threadIdx.x == THREADS) {
      bool ok = true;
      for (int g = 0; g < ng && ok; ++g) {
        if (g >= NST) ok = mbar_wait(empty(g % NST), ((g - NST) / NST) & 1, ctl);
        if (ok) issue(g);
      }
      // every issued copy has landed before the CTA leaves (each stage's last phase)
      for (int g = issued - NST > 0 ? issued - NST : 0; g < issued; ++g)
        mbar_wait(full(g % NST), (g / NST) & 1, ctl, CONV_DRAIN_NS);
    }
    return;
  }
  Filt f;
  float4 win[K];
  if (active) {
    f = load_filter(w, bias, d4);
#pragma unroll
    for (int j = 0; j < K - 1; ++j) win[j + 1] = x_at<BF16>(x, init, b, t0 - 3 + j, T, D4, d4);
  }
  int consumed = 0;
  for (int g = 0; g < ng; ++g) {
    const int st = g % NST, ta = t0 + g * SG, tb = min(ta + SG, t1);
    if (!mbar_wait(full(st), (g / NST) & 1, ctl)) break;
    consumed = g + 1;
    if (active) {
      const uint8_t* rows = smem + st * STAGE + threadIdx.x * 4 * ES;
      auto tok = [&](int t) {
        win[0] = win[1];
        win[1] = win[2];
        win[2] = win[3];
        if constexpr (BF16) win[3] = to_f4(*reinterpret_cast<const uint2*>(rows + (t - ta) * ROW));
        else win[3] = *reinterpret_cast<const float4*>(rows + (t - ta) * ROW);
        float4 z = conv4(f, win);
        float4 o;
#pragma unroll
        for (int c = 0; c < 4; ++c) at(o, c) = at(z, c) * sigm(at(z, c));
        reinterpret_cast<float4*>(y)[((long long)b * T + t) * D4 + d4] = o;
      };
      if (tb - ta == SG) {  // a full stage: unrolled, so the window shifts become renames
#pragma unroll
        for (int u = 0; u < SG; ++u) tok(ta + u);
      } else {
        for (int t = ta; t < tb; ++t) tok(t);
      }
    }
    mbar_arrive(empty(st));
  }
  if (active && fin && t1 == T && consumed == ng) {  // the state after the call: x_{T-3..T-1}
#pragma unroll
    for (int j = 0; j < 3; ++j)
      reinterpret_cast<float4*>(fin)[((long long)b * 3 + j) * D4 + d4] = win[j + 1];
  }
}

// part[(b * n_tiles + tile)][d][5] = (dw[d][0..3], db[d]) over the tile's tokens
template <bool BF16>
__global__ void __launch_bounds__(THREADS, 2)
conv_bwd_kernel(const void* __restrict__ x, const float* __restrict__ w,
                const float* __restrict__ bias, const float* __restrict__ init,
                const float* __restrict__ dy, float* __restrict__ dx, float* __restrict__ dinit,
                float* __restrict__ part, int T, int D) {
  griddep_launch_dependents();  // the reduction launched next waits for this whole grid
  const int D4 = D / 4, d4 = blockIdx.y * THREADS + threadIdx.x;
  if (d4 >= D4) return;
  const int n_tiles = (T + TTB - 1) / TTB;
  const int b = blockIdx.x / n_tiles, t0 = (blockIdx.x % n_tiles) * TTB;
  const int t1 = min(t0 + TTB, T);
  Filt f = load_filter(w, bias, d4);
  float4 win[K], dz[K];  // dz[0..3] = dz_{t-3..t} after step t
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < K - 1; ++j) win[j + 1] = x_at<BF16>(x, init, b, t0 - 3 + j, T, D4, d4);
#pragma unroll
  for (int j = 0; j < K; ++j) dz[j] = zero;
  float4 gw[K], gb = zero;
#pragma unroll
  for (int j = 0; j < K; ++j) gw[j] = zero;
  // t runs to t1 + 2 so that dx_s for every s < t1 is complete (dz beyond T is 0)
  const int tend = t1 + 3;
  for (int tg = t0; tg < tend; tg += GRP_BWD) {
  typename Raw<BF16>::T rx[GRP_BWD];
  float4 rg[GRP_BWD];
#pragma unroll
  for (int u = 0; u < GRP_BWD; ++u)
    if (tg + u < tend && tg + u < T) {
      rx[u] = load_raw<BF16>(x, ((long long)b * T + tg + u) * D4 + d4);
      rg[u] = __ldg(reinterpret_cast<const float4*>(dy) + ((long long)b * T + tg + u) * D4 + d4);
    }
#pragma unroll
  for (int u = 0; u < GRP_BWD; ++u) {
    const int t = tg + u;
    if (t >= tend) break;
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      win[j] = win[j + 1];
      dz[j] = dz[j + 1];
    }
    if (t < T) {
      win[3] = to_f4(rx[u]);
      const float4 d = silu_grad4(conv4(f, win), rg[u]);
      dz[3] = d;
      if (t < t1) {  // this tile's tokens: weight and bias gradients
        gb = add4(gb, d);
#pragma unroll
        for (int j = 0; j < K; ++j) gw[j] = fma4(d, win[j], gw[j]);
      }
    } else {
      win[3] = zero;
      dz[3] = zero;
    }
    // dx_{t-3} = sum_j w_j dz_{t-j}
    const int s = t - 3;
    if (s >= t0 || (t0 == 0 && s >= -3)) {
      if (s >= t1) continue;
      float4 g = zero;
#pragma unroll
      for (int j = 0; j < K; ++j) g = fma4(f.w[j], dz[3 - j], g);
      if (s >= 0)
        reinterpret_cast<float4*>(dx)[((long long)b * T + s) * D4 + d4] = g;
      else if (dinit)
        reinterpret_cast<float4*>(dinit)[((long long)b * 3 + (s + 3)) * D4 + d4] = g;
    }
  }
  }
  float* p = part + ((long long)blockIdx.x * D + 4 * d4) * 5;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int j = 0; j < K; ++j) p[c * 5 + j] = at(gw[j], c);
    p[c * 5 + 4] = at(gb, c);
  }
}

// The backward's ring: NSTB stages of SGB tokens of x and dy rows.
constexpr int SGB = 4;   // tokens per stage (backward)
constexpr int NSTB = 4;  // stages (backward)

// The backward with x and dy staged through shared memory (their rows of the CTA's 512
// channels, NSTB stages of SGB tokens, refilled by a producer warp), two channels per thread:
// a thread's windows, dz and weight-gradient sums are fp32 pairs, small enough that three CTAs
// fit an SM (with four channels per thread, 1,024 per CTA, two did).  The same arithmetic as
// conv_bwd_kernel.
constexpr int DC2 = 2 * THREADS;  // channels per CTA
template <bool BF16>
constexpr uint32_t staged_bwd2_smem() {
  return NSTB * SGB * DC2 * ((BF16 ? 2 : 4) + 4) + 2 * NSTB * 8;
}
struct Filt2 {
  float2 w[K];  // tap j of the 2 channels
  float2 b;
};
__device__ __forceinline__ Filt2 load_filter2(const float* w, const float* bias, int d2) {
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * d2);  // channel 2 d2
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * d2 + 1);
  Filt2 f;
  f.w[0] = make_float2(w0.x, w1.x);
  f.w[1] = make_float2(w0.y, w1.y);
  f.w[2] = make_float2(w0.z, w1.z);
  f.w[3] = make_float2(w0.w, w1.w);
  f.b = bias ? __ldg(reinterpret_cast<const float2*>(bias) + d2) : make_float2(0.f, 0.f);
  return f;
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
// x_t for token t of sequence b, channels 2 d2 and 2 d2 + 1 (t < 0: the initial state)
template <bool BF16>
__device__ __forceinline__ float2 x_at2(const void* x, const float* init, int b, int t, int T,
                                        int D2, int d2) {
  const long long i = ((long long)b * T + t) * D2 + d2;
  if (t >= 0) {
    if constexpr (BF16) return bf2_to_f2(__ldg(reinterpret_cast<const uint32_t*>(x) + i));
    else return __ldg(reinterpret_cast<const float2*>(x) + i);
  }
  if (!init) return make_float2(0.f, 0.f);
  return __ldg(reinterpret_cast<const float2*>(init) + ((long long)b * 3 + (t + 3)) * D2 + d2);
}
__device__ __forceinline__ float2 silu_grad2(float2 z, float2 dy) {
  const float2 s = make_float2(sigm(z.x), sigm(z.y));
  const float2 one_minus_s = __ffma2_rn(s, make_float2(-1.f, -1.f), make_float2(1.f, 1.f));
  return __fmul2_rn(__fmul2_rn(dy, s), __ffma2_rn(z, one_minus_s, make_float2(1.f, 1.f)));
}

template <bool BF16>
__global__ void __launch_bounds__(THREADS + 32, 3)
conv_bwd_staged2_kernel(const void* __restrict__ x, const float* __restrict__ w,
                        const float* __restrict__ bias, const float* __restrict__ init,
                        const float* __restrict__ dy, float* __restrict__ dx,
                        float* __restrict__ dinit, float* __restrict__ part, int T, int D,
                        DevCtl ctl) {
  griddep_launch_dependents();  // the reduction launched next waits for this whole grid
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int ES = BF16 ? 2 : 4;
  constexpr uint32_t XROW = DC2 * ES, GROW = DC2 * 4, STAGE = SGB * (XROW + GROW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NSTB * STAGE);  // full[NSTB], empty[NSTB]
  const int D2 = D / 2, c0 = blockIdx.y * DC2, nch = min(DC2, D - c0);
  const int d2 = c0 / 2 + threadIdx.x;
  const bool active = 2 * (int)threadIdx.x < nch;
  const int n_tiles = (T + TTB - 1) / TTB;
  const int b = blockIdx.x / n_tiles, t0 = (blockIdx.x % n_tiles) * TTB;
  const int t1 = min(t0 + TTB, T);
  // t runs to t1 + 2 so that dx_s for every s < t1 is complete (dz beyond T is 0); the rows of
  // tokens t0 .. tload-1 come through the ring
  const int tend = t1 + 3, tload = min(tend, T), ng = (tload - t0 + SGB - 1) / SGB;
  const uint32_t xbytes = (uint32_t)nch * ES, gbytes = (uint32_t)nch * 4, sb = smem_u32(smem);
  auto full = [&](int st) { return smem_u32(bars + st); };
  auto empty = [&](int st) { return smem_u32(bars + NSTB + st); };
  const uint8_t* xrow = static_cast<const uint8_t*>(x) + ((size_t)b * T * D + c0) * ES;
  const uint8_t* grow = reinterpret_cast<const uint8_t*>(dy) + ((size_t)b * T * D + c0) * 4;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NSTB; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), THREADS);
    }
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;
  auto issue = [&](int g) {
    const int st = g % NSTB, ta = t0 + g * SGB, tb = min(ta + SGB, tload);
    mbar_arrive_expect_tx(full(st), (uint32_t)(tb - ta) * (xbytes + gbytes));
    for (int t = ta; t < tb; ++t) {
      bulk_load(sb + st * STAGE + (t - ta) * XROW, xrow + (size_t)t * D * ES, xbytes, full(st));
      bulk_load(sb + st * STAGE + SGB * XROW + (t - ta) * GROW, grow + (size_t)t * D * 4, gbytes,
                full(st));
    }
    issued = g + 1;
  };
  if (threadIdx.x >= THREADS) {
    // the producer warp: refills a stage as soon as every compute thread has read it
    if (threadIdx.x == THREADS) {
      bool ok = true;
      for (int g = 0; g < ng && ok; ++g) {
        if (g >= NSTB) ok = mbar_wait(empty(g % NSTB), ((g - NSTB) / NSTB) & 1, ctl);
        if (ok) issue(g);
      }
      // every issued copy has landed before the CTA leaves (each stage's last phase)
      for (int g = issued - NSTB > 0 ? issued - NSTB : 0; g < issued; ++g)
        mbar_wait(full(g % NSTB), (g / NSTB) & 1, ctl, CONV_DRAIN_NS);
    }
    return;
  }
  const float2 zero = make_float2(0.f, 0.f);
  Filt2 f;
  float2 win[K], dz[K];  // dz[0..3] = dz_{t-3..t} after step t
  float2 gw[K], gb = zero;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    dz[j] = zero;
    gw[j] = zero;
  }
  if (active) {
    f = load_filter2(w, bias, d2);
#pragma unroll
    for (int j = 0; j < K - 1; ++j) win[j + 1] = x_at2<BF16>(x, init, b, t0 - 3 + j, T, D2, d2);
  }
  // one token: shift the windows, dz_t (zero past T), the tile's weight and bias sums, dx_{t-3}
  auto step = [&](int t, float2 xv, float2 g, bool in_seq) {
#pragma unroll
    for (int j = 0; j < K - 1; ++j) {
      win[j] = win[j + 1];
      dz[j] = dz[j + 1];
    }
    if (in_seq) {
      win[3] = xv;
      float2 z = f.b;
#pragma unroll
      for (int j = 0; j < K; ++j) z = __ffma2_rn(f.w[j], win[j], z);
      const float2 d = silu_grad2(z, g);
      dz[3] = d;
      if (t < t1) {
        gb = __fadd2_rn(gb, d);
#pragma unroll
        for (int j = 0; j < K; ++j) gw[j] = __ffma2_rn(d, win[j], gw[j]);
      }
    } else {
      win[3] = zero;
      dz[3] = zero;
    }
    const int s = t - 3;
    if ((s >= t0 || (t0 == 0 && s >= -3)) && s < t1) {
      float2 o = zero;
#pragma unroll
      for (int j = 0; j < K; ++j) o = __ffma2_rn(f.w[j], dz[3 - j], o);
      if (s >= 0)
        reinterpret_cast<float2*>(dx)[((long long)b * T + s) * D2 + d2] = o;
      else if (dinit)
        reinterpret_cast<float2*>(dinit)[((long long)b * 3 + (s + 3)) * D2 + d2] = o;
    }
  };
  int consumed = 0;
  for (int g = 0; g < ng; ++g) {
    const int st = g % NSTB, ta = t0 + g * SGB, tb = min(ta + SGB, tload);
    if (!mbar_wait(full(st), (g / NSTB) & 1, ctl)) break;
    consumed = g + 1;
    if (active) {
      const uint8_t* xs = smem + st * STAGE + threadIdx.x * 2 * ES;
      const uint8_t* gs = smem + st * STAGE + SGB * XROW + threadIdx.x * 8;
      auto tok = [&](int t) {
        float2 xv;
        if constexpr (BF16) xv = bf2_to_f2(*reinterpret_cast<const uint32_t*>(xs + (t - ta) * XROW));
        else xv = *reinterpret_cast<const float2*>(xs + (t - ta) * XROW);
        step(t, xv, *reinterpret_cast<const float2*>(gs + (t - ta) * GROW), true);
      };
      if (tb - ta == SGB) {  // a full stage: unrolled, so the window shifts become renames
#pragma unroll
        for (int u = 0; u < SGB; ++u) tok(ta + u);
      } else {
        for (int t = ta; t < tb; ++t) tok(t);
      }
    }
    mbar_arrive(empty(st));
  }
  if (consumed < ng) return;
  if (active) {
    for (int t = tload; t < tend; ++t) step(t, zero, zero, false);  // past T: dz = 0
    float* p = part + ((long long)blockIdx.x * D + 2 * d2) * 5;
#pragma unroll
    for (int j = 0; j < K; ++j) {
      p[j] = gw[j].x;
      p[5 + j] = gw[j].y;
    }
    p[4] = gb.x;
    p[9] = gb.y;
  }
}

// dw[d][j], db[d] = sums over the n_parts tiles.  One CTA of RED_WARPS warps per 32
// consecutive outputs i = d * 5 + j: warp w adds tiles w, w + RED_WARPS, ... in order (each
// load a coalesced 128-byte row of the partial sums), then one thread per output adds the
// warps' sums in order (a fixed order: deterministic).  Launched as the backward kernel's
// programmatic dependent: it waits for that grid before reading the partial sums.
constexpr int RED_WARPS = 32;
__global__ void __launch_bounds__(RED_WARPS * 32)
conv_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw,
                   float* __restrict__ db, int n_parts, int D) {
  __shared__ float acc[RED_WARPS][33];
  griddep_wait();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int i = blockIdx.x * 32 + lane;  // d * 5 + j
  const bool live = i < D * 5;
  float s = 0.f;
  if (live) {
#pragma unroll 8
    for (int q = wid; q < n_parts; q += RED_WARPS) s += part[(size_t)q * D * 5 + i];
  }
  acc[wid][lane] = s;
  __syncthreads();
  if (wid == 0 && live) {
    float t = 0.f;
#pragma unroll 8
    for (int w = 0; w < RED_WARPS; ++w) t += acc[w][lane];
    const int d = i / 5, j = i % 5;
    if (j < K) dw[d * K + j] = t;
    else if (db) db[d] = t;
  }
}

cudaError_t launch_conv_reduce(const float* part, float* dw, float* db, int n_parts, int D,
                               cudaStream_t stream) {
  PdlLaunch R(dim3((D * 5 + 31) / 32), dim3(RED_WARPS * 32), 0, stream, true);
  return cudaLaunchKernelEx(&R.cfg, conv_reduce_kernel, part, dw, db, n_parts, D);
}

__global__ void __launch_bounds__(THREADS)
conv_decode_kernel(float* __restrict__ state, const float* __restrict__ x,
                   const float* __restrict__ w, const float* __restrict__ bias,
                   float* __restrict__ y, long long n, int D) {
  const int D4 = D / 4;
  const long long i = (long long)blockIdx.x * THREADS + threadIdx.x;  // n * D4 + d4
  if (i >= n * D4) return;
  const long long r = i / D4;
  const int d4 = (int)(i % D4);
  Filt f = load_filter(w, bias, d4);
  float4* st = reinterpret_cast<float4*>(state) + r * 3 * D4 + d4;
  float4 win[K] = {st[0], st[D4], st[2 * D4], __ldg(reinterpret_cast<const float4*>(x) + i)};
  float4 z = conv4(f, win);
  float4 o;
#pragma unroll
  for (int c = 0; c < 4; ++c) at(o, c) = at(z, c) * sigm(at(z, c));
  reinterpret_cast<float4*>(y)[i] = o;
  st[0] = win[1];
  st[D4] = win[2];
  st[2 * D4] = win[3];
}

}  // namespace

size_t conv_bwd_workspace_bytes(int B, int T, int D) {
  return (size_t)B * ((T + TTB - 1) / TTB) * D * 5 * sizeof(float);
}

cudaError_t launch_conv_fwd(const void* x, bool bf16, const float* w, const float* bias,
                            const float* init, float* y, float* fin, int B, int T, int D,
                            DevCtl ctl, cudaStream_t stream) {
  if (D % (bf16 ? 8 : 4) == 0) {  // rows of 16-byte multiples: the staged kernel
    const dim3 grid(B * ((T + TT - 1) / TT), (D + DC - 1) / DC);
    cudaError_t e;
    if (bf16) {
      e = cudaFuncSetAttribute(conv_fwd_staged_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, staged_fwd_smem<true>());
      if (e != cudaSuccess) return e;
      conv_fwd_staged_kernel<true><<<grid, THREADS + 32, staged_fwd_smem<true>(), stream>>>(
          x, w, bias, init, y, fin, T, D, ctl);
    } else {
      e = cudaFuncSetAttribute(conv_fwd_staged_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, staged_fwd_smem<false>());
      if (e != cudaSuccess) return e;
      conv_fwd_staged_kernel<false><<<grid, THREADS + 32, staged_fwd_smem<false>(), stream>>>(
          x, w, bias, init, y, fin, T, D, ctl);
    }
    return cudaGetLastError();
  }
  const dim3 grid(B * ((T + TT - 1) / TT), (D / 4 + THREADS - 1) / THREADS);
  if (bf16)
    conv_fwd_kernel<true><<<grid, THREADS, 0, stream>>>(x, w, bias, init, y, fin, T, D);
  else
    conv_fwd_kernel<false><<<grid, THREADS, 0, stream>>>(x, w, bias, init, y, fin, T, D);
  return cudaGetLastError();
}

cudaError_t launch_conv_bwd(const void* x, bool bf16, const float* w, const float* bias,
                            const float* init, const float* dy, float* dx, float* dinit,
                            float* dw, float* db, float* part, int B, int T, int D,
                            DevCtl ctl, cudaStream_t stream) {
  const int n_tiles = (T + TTB - 1) / TTB;
  if (D % (bf16 ? 8 : 4) == 0) {  // rows of 16-byte multiples: the staged kernel
    const dim3 grid(B * n_tiles, (D + DC2 - 1) / DC2);
    cudaError_t e;
    if (bf16) {
      e = cudaFuncSetAttribute(conv_bwd_staged2_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, staged_bwd2_smem<true>());
      if (e != cudaSuccess) return e;
      conv_bwd_staged2_kernel<true><<<grid, THREADS + 32, staged_bwd2_smem<true>(), stream>>>(
          x, w, bias, init, dy, dx, dinit, part, T, D, ctl);
    } else {
      e = cudaFuncSetAttribute(conv_bwd_staged2_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, staged_bwd2_smem<false>());
      if (e != cudaSuccess) return e;
      conv_bwd_staged2_kernel<false><<<grid, THREADS + 32, staged_bwd2_smem<false>(), stream>>>(
          x, w, bias, init, dy, dx, dinit, part, T, D, ctl);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_conv_reduce(part, dw, db, B * n_tiles, D, stream);
  }
  const dim3 grid(B * n_tiles, (D / 4 + THREADS - 1) / THREADS);
  if (bf16)
    conv_bwd_kernel<true><<<grid, THREADS, 0, stream>>>(x, w, bias, init, dy, dx, dinit, part, T, D);
  else
    conv_bwd_kernel<false><<<grid, THREADS, 0, stream>>>(x, w, bias, init, dy, dx, dinit, part, T,
                                                          D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_conv_reduce(part, dw, db, B * n_tiles, D, stream);
}

cudaError_t launch_conv_decode(float* state, const float* x, const float* w, const float* bias,
                               float* y, long long n, int D, cudaStream_t stream) {
  const long long work = n * (D / 4);
  if (work <= 0) return cudaSuccess;
  conv_decode_kernel<<<(unsigned)((work + THREADS - 1) / THREADS), THREADS, 0, stream>>>(
      state, x, w, bias, y, n, D);
  return cudaGetLastError();
}

}  // namespace gla
