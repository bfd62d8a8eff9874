// noalloc.cu -- gla_chunk_bwd_noalloc: the chunked backward without a caller workspace.
//
// Some callers cannot hand the library a device buffer for scratch: code that runs inside
// an inference engine's or plugin's execution callback where device allocation is not
// allowed, processes whose device memory is fully reserved up front, and latency-critical
// loops where cudaMalloc / cudaFree (which may synchronise the whole device) are off limits.
// For them the backward's only scratch -- the per-(b, h) partial sums of d_aug, reduced
// over the batch after the main kernel -- lives in the fixed array below, which every GPU
// that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include "gla.h"
#include "kernels.h"

namespace {

// Scratch for B * H <= GLA_NOALLOC_MAX_BH partial-sum rows of 96 floats (768 KiB).
static __device__ __align__(256) float g_noalloc_scratch[GLA_NOALLOC_MAX_BH * 96];

// Device address of the scratch array in the current device's context, looked up on every
// call with that device current (the lookup is a cheap table read once the module is loaded,
// and a context that was reset and created again may place the module elsewhere, so no
// address is kept between calls).  The array's name in host code is only a stand-in for the
// symbol; a kernel must be given the address returned here.
gla_status scratch_address(void** scratch) {
  void* s = nullptr;
  if (cudaGetSymbolAddress(&s, g_noalloc_scratch) != cudaSuccess || !s) return GLA_ERR_CUDA;
  *scratch = s;
  return GLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

gla_status gla_chunk_bwd_noalloc(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                                 const float* log_decay, const float* aug_balance,
                                 const float* init_state, const void* dO,
                                 const float* d_final_state, const float* gate, float* dq,
                                 float* dk, float* dv, float* d_aug, float* d_init_state, int B,
                                 int T, int H, int dk_, int dv_, cudaStream_t stream) {
  if (B <= 0 || T <= 0 || H <= 0) return GLA_ERR_INVALID_ARG;
  if (dk_ != gla::kDK || dv_ != gla::kDV) return GLA_ERR_UNSUPPORTED;
  if (in_dtype != GLA_BF16 && in_dtype != GLA_FP16) return GLA_ERR_UNSUPPORTED;
  if ((long long)B * H > GLA_NOALLOC_MAX_BH) return GLA_ERR_WORKSPACE;
  if ((long long)B * T > (1ll << 31) - 1) return GLA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !log_decay || !aug_balance || !dO || !dq || !dk || !dv || !d_aug)
    return GLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_decay) ||
      !aligned16(aug_balance) || !aligned16(init_state) || !aligned16(dO) ||
      !aligned16(d_final_state) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(d_aug) || !aligned16(d_init_state) ||
      (reinterpret_cast<uintptr_t>(gate) & 3u) != 0)
    return GLA_ERR_ALIGNMENT;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != GLA_OK) return GLA_ERR_CUDA;
  gla::DevCtl ctl;  // the library's device error word and wait limit
  if (gla::current_device_ctl(&ctl) != cudaSuccess) return GLA_ERR_CUDA;

  gla::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.dO = dO; a.bf16 = in_dtype == GLA_BF16;
  a.log_decay = log_decay; a.aug = aug_balance; a.init = init_state; a.dfin = d_final_state;
  a.dq = dq; a.dk = dk; a.dv = dv; a.d_aug = d_aug; a.dinit = d_init_state; a.gate = gate;
  // Every partial sum the reduction reads is written by this call's kernel first, so the
  // contents left by an earlier call never need clearing.
  a.workspace = scratch;
  a.workspace_bytes = sizeof(float) * (size_t)GLA_NOALLOC_MAX_BH * 96;
  a.B = B; a.T = T; a.H = H;
  return gla::launch_chunk_bwd(a, ctl, stream) == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

}  // extern "C"
