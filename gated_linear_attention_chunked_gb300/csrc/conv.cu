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
// Memory-bound streaming: one thread owns 4 consecutive channels of a 64-token tile and walks
// its tokens with the 4-token window in registers (3-token halo, ~5 % re-read).  dw, db: per
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
constexpr int TT = 64;      // tokens per tile
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
__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

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
  for (int j = 0; j < K; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) at(z, c) = fmaf(at(f.w[j], c), at(win[j], c), at(z, c));
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

// part[(b * n_tiles + tile)][d][5] = (dw[d][0..3], db[d]) over the tile's tokens
template <bool BF16>
__global__ void __launch_bounds__(THREADS, 2)
conv_bwd_kernel(const void* __restrict__ x, const float* __restrict__ w,
                const float* __restrict__ bias, const float* __restrict__ init,
                const float* __restrict__ dy, float* __restrict__ dx, float* __restrict__ dinit,
                float* __restrict__ part, int T, int D) {
  const int D4 = D / 4, d4 = blockIdx.y * THREADS + threadIdx.x;
  if (d4 >= D4) return;
  const int n_tiles = (T + TT - 1) / TT;
  const int b = blockIdx.x / n_tiles, t0 = (blockIdx.x % n_tiles) * TT;
  const int t1 = min(t0 + TT, T);
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
      float4 z = conv4(f, win);
      float4 g = rg[u];
      float4 d;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float zc = at(z, c), sg = sigm(zc);
        at(d, c) = at(g, c) * sg * (1.f + zc * (1.f - sg));
      }
      dz[3] = d;
      if (t < t1) {  // this tile's tokens: weight and bias gradients
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          at(gb, c) += at(d, c);
#pragma unroll
          for (int j = 0; j < K; ++j) at(gw[j], c) = fmaf(at(d, c), at(win[j], c), at(gw[j], c));
        }
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
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) at(g, c) = fmaf(at(f.w[j], c), at(dz[3 - j], c), at(g, c));
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

// dw[d][j], db[d] = sums over the n_parts tiles, in order
__global__ void conv_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw,
                                   float* __restrict__ db, int n_parts, int D) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // d * 5 + j
  if (i >= D * 5) return;
  float s = 0.f;
  for (int q = 0; q < n_parts; ++q) s += part[(size_t)q * D * 5 + i];
  const int d = i / 5, j = i % 5;
  if (j < K) dw[d * K + j] = s;
  else if (db) db[d] = s;
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
  return (size_t)B * ((T + TT - 1) / TT) * D * 5 * sizeof(float);
}

cudaError_t launch_conv_fwd(const void* x, bool bf16, const float* w, const float* bias,
                            const float* init, float* y, float* fin, int B, int T, int D,
                            cudaStream_t stream) {
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
                            cudaStream_t stream) {
  const int n_tiles = (T + TT - 1) / TT;
  const dim3 grid(B * n_tiles, (D / 4 + THREADS - 1) / THREADS);
  if (bf16)
    conv_bwd_kernel<true><<<grid, THREADS, 0, stream>>>(x, w, bias, init, dy, dx, dinit, part, T, D);
  else
    conv_bwd_kernel<false><<<grid, THREADS, 0, stream>>>(x, w, bias, init, dy, dx, dinit, part, T,
                                                          D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  conv_reduce_kernel<<<(D * 5 + 255) / 256, 256, 0, stream>>>(part, dw, db, B * n_tiles, D);
  return cudaGetLastError();
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
