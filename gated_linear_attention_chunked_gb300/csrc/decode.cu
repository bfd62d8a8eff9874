// decode.cu -- one recurrent decode step over a pool of fp32 states.
//
// Per state (one sequence, one layer, one head; "Inference optimization on Trainium2":
// a fixed recurrent state per sequence, O(1) work per token):
//   S' = lambda_h S + k v^T          (in place)
//   o  = S'^T q + sigmoid(q . (a * k)) v
//
// The step is a single streaming pass over the 96x192 fp32 state (73,728 B read and
// written per state), so it is bound by HBM bandwidth.  One CTA of 384 threads owns one
// state: thread (g, c) with c = tid % 48 owns the float4 column block c (value channels
// 4c..4c+3) and rows 12g..12g+11 (key channels).  All 12 float4 loads of a thread are issued
// before any use (streaming, evict-first), the update and the partial readout are done in
// registers, and the 8 row-group partials of S'^T q are summed through shared memory.
//
// Paged variant (a state pool with one fixed page per sequence, as the vLLM wrapper of the
// same section keeps it): the CTA of active sequence n, layer l, head h updates the state of
// page[n] -- pool[(page[n] * pool_layers + layer0 + l) * H + h] -- so the active set is any
// list of pages, in any order, with no padding.  A page outside [0, n_pages) records
// DEV_RANGE and its CTA touches nothing.
#include <cuda_runtime.h>

#include "kernels.h"

namespace gla {

namespace {
constexpr int DK = 96, DV = 192, DV4 = DV / 4, RG = 8, ROWS = DK / RG, THREADS = DV4 * RG;
static_assert(ROWS * RG == DK && THREADS == 384, "decode tiling");

struct Pages {
  const int* page;  // null: state s is state[s]
  int n_pages, pool_layers, layer0;
  DevCtl ctl;
};

template <bool PAGED>
__global__ void __launch_bounds__(THREADS, 2)
decode_kernel(float* __restrict__ state, const float* __restrict__ q,
              const float* __restrict__ k, const float* __restrict__ v,
              const float* __restrict__ log_decay, const float* __restrict__ aug,
              float* __restrict__ o, int L, int H, Pages pg) {
  __shared__ float sq[DK], sk[DK];
  __shared__ float4 sv[DV4];
  __shared__ float4 part[RG][DV4];
  __shared__ float sgate;

  const long long s = blockIdx.x;  // index of q, k, v, o: ((seq * L + l) * H + h)
  const int t = threadIdx.x, c4 = t % DV4, g = t / DV4;
  long long ss = s;  // index of the state
  if constexpr (PAGED) {
    const long long n = s / ((long long)L * H);
    const int lh = (int)(s % ((long long)L * H));
    const int p = __ldg(pg.page + n);
    if (p < 0 || p >= pg.n_pages) {  // the same page for every thread of the CTA
      if (t == 0) record_error(pg.ctl, DEV_RANGE);
      return;
    }
    ss = ((long long)p * pg.pool_layers + pg.layer0 + lh / H) * H + lh % H;
  }
  float4* S = reinterpret_cast<float4*>(state + ss * (long long)(DK * DV)) + g * ROWS * DV4 + c4;

  float4 x[ROWS];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) x[r] = __ldcs(S + r * DV4);

  if (t < DK) {
    sq[t] = __ldg(q + s * DK + t);
    sk[t] = __ldg(k + s * DK + t);
  }
  if (t < DV4) sv[t] = __ldg(reinterpret_cast<const float4*>(v + s * DV) + t);
  __syncthreads();

  const int h = (int)(s % H);
  const float lam = expf(__ldg(log_decay + h));
  const float4 vv = sv[c4];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int row = g * ROWS + r;
    const float kr = sk[row], qr = sq[row];
    float4 y;
    y.x = fmaf(lam, x[r].x, kr * vv.x);
    y.y = fmaf(lam, x[r].y, kr * vv.y);
    y.z = fmaf(lam, x[r].z, kr * vv.z);
    y.w = fmaf(lam, x[r].w, kr * vv.w);
    __stcs(S + r * DV4, y);
    acc.x = fmaf(y.x, qr, acc.x);
    acc.y = fmaf(y.y, qr, acc.y);
    acc.z = fmaf(y.z, qr, acc.z);
    acc.w = fmaf(y.w, qr, acc.w);
  }
  part[g][c4] = acc;

  if (t < 32) {  // gate z = q . (a * k), a = aug_balance[l, h]
    const float* a = aug + (s % ((long long)L * H)) * DK;
    float z = 0.f;
    for (int i = t; i < DK; i += 32) z = fmaf(__ldg(a + i) * sq[i], sk[i], z);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (t == 0) sgate = 1.f / (1.f + expf(-z));
  }
  __syncthreads();

  if (t < DV4) {
    float4 r = part[0][t];
#pragma unroll
    for (int gg = 1; gg < RG; ++gg) {
      const float4 p = part[gg][t];
      r.x += p.x; r.y += p.y; r.z += p.z; r.w += p.w;
    }
    const float4 vt = sv[t];
    const float gt = sgate;
    r.x = fmaf(gt, vt.x, r.x);
    r.y = fmaf(gt, vt.y, r.y);
    r.z = fmaf(gt, vt.z, r.z);
    r.w = fmaf(gt, vt.w, r.w);
    reinterpret_cast<float4*>(o + s * DV)[t] = r;
  }
}
}  // namespace

cudaError_t launch_decode(float* state, const float* q, const float* k, const float* v,
                          const float* log_decay, const float* aug, float* o, long long n_states,
                          int L, int H, cudaStream_t stream) {
  if (n_states <= 0) return cudaSuccess;
  decode_kernel<false><<<(unsigned)n_states, THREADS, 0, stream>>>(state, q, k, v, log_decay, aug,
                                                                    o, L, H, Pages{});
  return cudaGetLastError();
}

cudaError_t launch_decode_paged(float* pool, const int* page, int n_pages, int pool_layers,
                                int layer0, const float* q, const float* k, const float* v,
                                const float* log_decay, const float* aug, float* o, int n_active,
                                int L, int H, DevCtl ctl, cudaStream_t stream) {
  const long long n_states = (long long)n_active * L * H;
  if (n_states <= 0) return cudaSuccess;
  Pages pg{page, n_pages, pool_layers, layer0, ctl};
  decode_kernel<true><<<(unsigned)n_states, THREADS, 0, stream>>>(pool, q, k, v, log_decay, aug, o,
                                                                   L, H, pg);
  return cudaGetLastError();
}

}  // namespace gla
