// api.cu -- the C ABI declared in include/gla.h: argument checks, workspace layout, device
// error word, and the launches on the caller's stream.  No device memory is allocated here.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "gla.h"
#include "kernels.h"

namespace {

__device__ int g_device_error = 0;
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<int> g_split_parts{0};  // gla_set_split_parts: 0 automatic, 1 never, p >= 2 forced
std::atomic<int> g_stall_step{-1};  // gla_set_stall_step: the give-up path's diagnostic
std::atomic<int> g_pass_overlap{1};  // gla_set_pass_overlap: segment passes beside the whole pairs

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

gla_status ctl_for_current_device(gla::DevCtl* ctl) {
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ctl->err), g_device_error) != cudaSuccess)
    return GLA_ERR_CUDA;
  ctl->wait_ns = g_wait_ns.load();
  ctl->stall_step = g_stall_step.load();
  return GLA_OK;
}

bool valid_dtype(gla_dtype t) { return t == GLA_BF16 || t == GLA_FP16 || t == GLA_FP32; }

// Common checks of the chunked calls.
gla_status check_chunk_sizes(int B, int T, int H, int dk, int dv, gla_dtype t) {
  if (B <= 0 || T <= 0 || H <= 0) return GLA_ERR_INVALID_ARG;
  if (dk != gla::kDK || dv != gla::kDV || !valid_dtype(t))
    return GLA_ERR_UNSUPPORTED;
  if ((long long)B * T > (1ll << 31) - 1 || (long long)B * H > (1ll << 31) - 1)
    return GLA_ERR_UNSUPPORTED;
  return GLA_OK;
}

// fp32 inputs are narrowed to fp16 in the workspace: q, k [B,T,H,96], v (and dO) [B,T,H,192].
size_t half_copy_bytes(int B, int T, int H, bool with_dO) {
  const size_t tok = (size_t)B * T * H;
  size_t s = 2 * round256(tok * gla::kDK * 2) + round256(tok * gla::kDV * 2);
  if (with_dO) s += round256(tok * gla::kDV * 2);
  return s;
}

// SMs of the current device (0 if there is none).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Bytes the forward must have (fp16 copies of fp32 inputs); the cut pairs' states go on top,
// at the offset round256(must).
size_t fwd_min_workspace(int B, int T, int H, gla_dtype in_dtype) {
  return in_dtype == GLA_FP32 ? half_copy_bytes(B, T, H, false) : 0;
}

constexpr size_t kStateBytes = (size_t)gla::kDK * gla::kDV * sizeof(float);

// Bytes the backward must have: d_aug partial sums, then fp16 copies of fp32 inputs.
size_t bwd_min_workspace(int B, int T, int H, gla_dtype in_dtype) {
  size_t s = gla::chunk_bwd_workspace_bytes(B, T, H);
  if (in_dtype == GLA_FP32) s += half_copy_bytes(B, T, H, true);
  return s;
}

// How the last wave's pairs are cut on the current device (roles: 1 forward, 3 backward;
// pass_dirs: 1 for the forward and a backward reading the forward's state copies, 2 for a
// backward that scans the state itself).
gla::SplitPlan split_plan(int B, int T, int H, int roles, int n_sm, int pass_dirs) {
  const int nc = (T + gla::kChunk - 1) / gla::kChunk;
  return gla::plan_split((long long)B * H, nc, roles, n_sm, g_split_parts.load(), pass_dirs,
                         g_pass_overlap.load() != 0);
}

// Extra workspace of a plan: the forward's part states; the backward's part states, part
// adjoints and d_aug partial sums (three 256-byte aligned arrays).
size_t split_bytes(int B, int H, const gla::SplitPlan& plan, bool bwd) {
  const long long slots = gla::split_slots((long long)B * H, plan);
  if (!slots) return 0;
  // (the forward: the states, then each state's partial maxima)
  if (!bwd) return round256((size_t)slots * kStateBytes) + round256((size_t)slots * 4 * 4);
  return 2 * round256((size_t)slots * kStateBytes) + round256((size_t)slots * gla::kDK * 4);
}


gla_status chunk_fwd_impl(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                          const float* log_decay, const float* aug_balance,
                          const float* init_state, float* o, float* final_state, void* workspace,
                          size_t workspace_bytes, int B, int T, int H, int dk, int dv,
                          const gla::StatePages& sp, cudaStream_t stream,
                          const gla::OutGate& og = gla::OutGate{}, float* gate = nullptr,
                          void* saved = nullptr, size_t saved_bytes = 0) {
  gla_status st = check_chunk_sizes(B, T, H, dk, dv, in_dtype);
  if (st != GLA_OK) return st;
  if (saved && saved_bytes < gla::saved_states_bytes(B, T, H)) return GLA_ERR_WORKSPACE;
  if (!aligned256(saved)) return GLA_ERR_ALIGNMENT;
  if (!q || !k || !v || !log_decay || !aug_balance || (!o && !og.g)) return GLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_decay) ||
      !aligned16(aug_balance) || !aligned16(init_state) || !aligned16(o) ||
      !aligned16(final_state) || !aligned4(gate))
    return GLA_ERR_ALIGNMENT;
  const size_t must = fwd_min_workspace(B, T, H, in_dtype);
  if (must && (!workspace || workspace_bytes < must)) return GLA_ERR_WORKSPACE;
  if (must && !aligned256(workspace)) return GLA_ERR_ALIGNMENT;
  // the pairs of a partial last wave (or all of few, long sequences) are cut into parts when
  // the workspace has room for their starting states
  gla::SplitPlan plan = split_plan(B, T, H, 1, sm_count(), 1);
  const size_t extra = split_bytes(B, H, plan, false);
  if (extra && !(workspace && aligned256(workspace) && workspace_bytes >= round256(must) + extra)) {
    plan.whole = B * H;
    plan.parts = 1;
    plan.overlap = false;
  }
  gla::DevCtl ctl;
  if ((st = ctl_for_current_device(&ctl)) != GLA_OK) return st;

  gla::FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.bf16 = in_dtype == GLA_BF16;
  a.log_decay = log_decay; a.aug = aug_balance; a.init = init_state;
  a.o = o; a.fin = final_state; a.B = B; a.T = T; a.H = H; a.sp = sp; a.og = og; a.gate = gate;
  a.saved = gla::saved_states_at(saved, B, T, H);
  if (in_dtype == GLA_FP32) {
    const size_t tok = (size_t)B * T * H;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    void* hq = w;
    void* hk = w + round256(tok * dk * 2);
    void* hv = w + 2 * round256(tok * dk * 2);
    if (gla::launch_to_half((const float*)q, hq, (long long)(tok * dk), ctl, stream) != cudaSuccess ||
        gla::launch_to_half((const float*)k, hk, (long long)(tok * dk), ctl, stream) != cudaSuccess ||
        gla::launch_to_half((const float*)v, hv, (long long)(tok * dv), ctl, stream) != cudaSuccess)
      return GLA_ERR_CUDA;
    a.q = hq; a.k = hk; a.v = hv; a.bf16 = false;
  }
  a.plan = plan;
  if (plan.parts > 1) {
    // the segment passes; with plan.overlap the chunked kernel, launched as their programmatic
    // dependent, runs its whole pairs beside them
    float* states = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round256(must));
    // the starting states' maxima: from the two-part sum pass, or from pass B when the passes
    // run before the chunked kernel (beside the whole pairs pass B's extra work would delay the
    // SMs it holds, which measured slower than the parts' saving)
    float* maxes = plan.parts == 2 || !plan.overlap
                       ? reinterpret_cast<float*>(
                             reinterpret_cast<uint8_t*>(states) +
                             round256((size_t)gla::split_slots((long long)B * H, plan) *
                                      kStateBytes))
                       : nullptr;
    a.seg_init = states;
    a.seg_max = maxes;
    if (gla::launch_segment_states(nullptr, a.k, a.v, nullptr, a.bf16, log_decay, init_state,
                                   nullptr, sp, states, nullptr, B, T, H, plan, ctl, stream,
                                   maxes) != cudaSuccess)
      return GLA_ERR_CUDA;
  }
  return gla::launch_chunk_fwd(a, ctl, stream) == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}


// One thread waits on an mbarrier that nothing ever arrives on: the bounded wait gives up after
// the configured limit and records DEV_TIMEOUT -- the failure path of every kernel's waits,
// exercised without a fault.
__global__ void wait_probe_kernel(gla::DevCtl ctl) {
  __shared__ alignas(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    gla::mbar_init(gla::smem_u32(&bar), 1);
    gla::fence_barrier_init();
    gla::mbar_wait(gla::smem_u32(&bar), 0, ctl);
  }
}
}  // namespace

namespace gla {
cudaError_t current_device_ctl(DevCtl* ctl) {
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ctl->err), g_device_error);
  ctl->wait_ns = g_wait_ns.load();
  ctl->stall_step = g_stall_step.load();
  return e;
}
}  // namespace gla

extern "C" {

const char* gla_status_string(gla_status s) {
  switch (s) {
    case GLA_OK: return "ok";
    case GLA_ERR_INVALID_ARG: return "invalid argument";
    case GLA_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case GLA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case GLA_ERR_CUDA: return "CUDA error";
    case GLA_ERR_TIMEOUT: return "device wait timed out";
    case GLA_ERR_RANGE: return "operand outside the fp16 range";
    case GLA_ERR_WORKSPACE: return "workspace missing or too small";
    case GLA_ERR_LAYOUT: return "shared memory layout error";
  }
  return "unknown status";
}

gla_status gla_get_device_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return GLA_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return GLA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return GLA_ERR_CUDA;
  switch (v) {
    case gla::DEV_OK: return GLA_OK;
    case gla::DEV_TIMEOUT: return GLA_ERR_TIMEOUT;
    case gla::DEV_RANGE: return GLA_ERR_RANGE;
    case gla::DEV_LAYOUT: return GLA_ERR_LAYOUT;
  }
  return GLA_ERR_CUDA;
}

gla_status gla_set_wait_timeout_ns(unsigned long long ns) {
  g_wait_ns.store(ns ? ns : 2000000000ull);
  return GLA_OK;
}

gla_status gla_set_stall_step(int step) {
  g_stall_step.store(step < 0 ? -1 : step);
  return GLA_OK;
}

gla_status gla_wait_probe(cudaStream_t stream) {
  gla::DevCtl ctl;
  gla_status st = ctl_for_current_device(&ctl);
  if (st != GLA_OK) return st;
  wait_probe_kernel<<<1, 32, 0, stream>>>(ctl);
  return cudaGetLastError() == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

gla_status gla_decay_schedule(int H, double t_min, double t_max, float* log_decay) {
  if (H <= 0 || !(t_min > 0) || !(t_max > 0) || !log_decay) return GLA_ERR_INVALID_ARG;
  for (int h = 0; h < H; ++h) {
    const double frac = H > 1 ? (double)h / (double)(H - 1) : 0.0;
    const double half_life = t_min * std::pow(t_max / t_min, frac);
    log_decay[h] = (float)(-std::log(2.0) / half_life);
  }
  return GLA_OK;
}

size_t gla_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, gla_dtype in_dtype) {
  if (check_chunk_sizes(B, T, H, dk, dv, in_dtype) != GLA_OK) return 0;
  const size_t must = fwd_min_workspace(B, T, H, in_dtype);
  const size_t extra = split_bytes(B, H, split_plan(B, T, H, 1, sm_count(), 1), false);
  return extra ? round256(must) + extra : must;
}

size_t gla_chunk_saved_states_size(int B, int T, int H) {
  if (B <= 0 || T <= 0 || H <= 0 || (long long)B * T > (1ll << 31) - 1) return 0;
  return gla::saved_states_bytes(B, T, H);
}

gla_status gla_chunk_fwd(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                         const float* log_decay, const float* aug_balance,
                         const float* init_state, float* o, float* final_state, float* gate,
                         void* saved_states, size_t saved_states_bytes, void* workspace,
                         size_t workspace_bytes, int B, int T, int H, int dk, int dv,
                         cudaStream_t stream) {
  return chunk_fwd_impl(q, k, v, in_dtype, log_decay, aug_balance, init_state, o, final_state,
                        workspace, workspace_bytes, B, T, H, dk, dv, gla::StatePages{}, stream,
                        gla::OutGate{}, gate, saved_states, saved_states_bytes);
}

gla_status gla_chunk_fwd_gated(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                               const float* log_decay, const float* aug_balance,
                               const float* init_state, const void* g, const float* norm_weight,
                               int n_tiers, float eps, float* y, float* rstd, float* o,
                               float* final_state, void* workspace, size_t workspace_bytes, int B,
                               int T, int H, int dk, int dv, cudaStream_t stream) {
  if (!g || !norm_weight || !y) return GLA_ERR_INVALID_ARG;
  if (H <= 0 || n_tiers <= 0 || H % n_tiers != 0 || !(eps >= 0.f) || !(eps < 1e30f))
    return GLA_ERR_INVALID_ARG;
  if (!aligned16(g) || !aligned16(norm_weight) || !aligned16(y) || !aligned16(rstd))
    return GLA_ERR_ALIGNMENT;
  gla::OutGate og;
  og.g = static_cast<const uint16_t*>(g);
  og.w = norm_weight;
  og.y = y;
  og.rstd = rstd;
  og.eps = eps;
  og.heads_per_tier = H / n_tiers;
  og.want_o = o != nullptr;
  return chunk_fwd_impl(q, k, v, in_dtype, log_decay, aug_balance, init_state, o, final_state,
                        workspace, workspace_bytes, B, T, H, dk, dv, gla::StatePages{}, stream, og);
}

gla_status gla_chunk_fwd_paged(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                               const float* log_decay, const float* aug_balance, float* pool,
                               const int* page, int n_pages, int pool_layers, int layer,
                               int init_from_pool, float* o, void* workspace,
                               size_t workspace_bytes, int B, int T, int H, int dk, int dv,
                               cudaStream_t stream) {
  if (!pool || !page) return GLA_ERR_INVALID_ARG;
  if (n_pages <= 0 || pool_layers <= 0 || layer < 0 || layer >= pool_layers || H <= 0)
    return GLA_ERR_INVALID_ARG;
  if ((long long)n_pages * pool_layers * H > (1ll << 31) - 1) return GLA_ERR_UNSUPPORTED;
  if (!aligned16(page)) return GLA_ERR_ALIGNMENT;
  gla::StatePages sp;
  sp.page = page;
  sp.n_pages = n_pages;
  sp.pool_layers = pool_layers;
  sp.layer = layer;
  sp.init_paged = init_from_pool != 0;
  return chunk_fwd_impl(q, k, v, in_dtype, log_decay, aug_balance, sp.init_paged ? pool : nullptr,
                        o, pool, workspace, workspace_bytes, B, T, H, dk, dv, sp, stream);
}

size_t gla_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, gla_dtype in_dtype) {
  if (check_chunk_sizes(B, T, H, dk, dv, in_dtype) != GLA_OK) return 0;
  const size_t must = bwd_min_workspace(B, T, H, in_dtype);
  // enough for either backward: the one that scans the state itself and the one that reads
  // the forward's state copies (whose cheaper segment passes may favour more parts)
  const int n_sm = sm_count();
  const size_t extra = std::max(split_bytes(B, H, split_plan(B, T, H, 3, n_sm, 2), true),
                                split_bytes(B, H, split_plan(B, T, H, 3, n_sm, 1), true));
  return extra ? round256(must) + extra : must;
}

gla_status gla_set_split_parts(int parts) {
  if (parts < 0) return GLA_ERR_INVALID_ARG;
  g_split_parts.store(parts);
  return GLA_OK;
}

gla_status gla_set_pass_overlap(int on) {
  g_pass_overlap.store(on ? 1 : 0);
  return GLA_OK;
}

gla_status gla_chunk_split_plan(int B, int T, int H, int backward, int n_sm, int* whole_pairs,
                                int* parts) {
  if (B <= 0 || T <= 0 || H <= 0 || n_sm <= 0 || !whole_pairs || !parts)
    return GLA_ERR_INVALID_ARG;
  if ((long long)B * H > (1ll << 31) - 1) return GLA_ERR_UNSUPPORTED;
  const gla::SplitPlan plan =
      split_plan(B, T, H, backward ? 3 : 1, n_sm, backward == 1 ? 2 : 1);
  *whole_pairs = plan.whole;
  *parts = plan.parts;
  return GLA_OK;
}

gla_status gla_chunk_bwd(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                         const float* log_decay, const float* aug_balance,
                         const float* init_state, const void* dO, const float* d_final_state,
                         const float* gate, const void* saved_states, size_t saved_states_bytes,
                         float* dq, float* dk, float* dv, float* d_aug, float* d_init_state,
                         void* workspace, size_t workspace_bytes, int B, int T, int H, int dk_,
                         int dv_, cudaStream_t stream) {
  gla_status st = check_chunk_sizes(B, T, H, dk_, dv_, in_dtype);
  if (st != GLA_OK) return st;
  if (saved_states && saved_states_bytes < gla::saved_states_bytes(B, T, H))
    return GLA_ERR_WORKSPACE;
  if (!aligned256(saved_states)) return GLA_ERR_ALIGNMENT;
  if (!q || !k || !v || !log_decay || !aug_balance || !dO || !dq || !dk || !dv || !d_aug)
    return GLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_decay) ||
      !aligned16(aug_balance) || !aligned16(init_state) || !aligned16(dO) ||
      !aligned16(d_final_state) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(d_aug) || !aligned16(d_init_state) || !aligned4(gate))
    return GLA_ERR_ALIGNMENT;
  const size_t need = bwd_min_workspace(B, T, H, in_dtype);
  if (need && (!workspace || workspace_bytes < need)) return GLA_ERR_WORKSPACE;
  if (need && !aligned256(workspace)) return GLA_ERR_ALIGNMENT;
  // the pairs of a partial last wave (or all of few, long sequences) are cut into parts when
  // the workspace has room for their starting states and adjoints
  gla::SplitPlan plan = split_plan(B, T, H, 3, sm_count(), saved_states ? 1 : 2);
  const size_t extra = split_bytes(B, H, plan, true);
  if (extra && workspace_bytes < round256(need) + extra) {
    plan.whole = B * H;
    plan.parts = 1;
    plan.overlap = false;
  }
  gla::DevCtl ctl;
  if ((st = ctl_for_current_device(&ctl)) != GLA_OK) return st;

  gla::BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.dO = dO; a.bf16 = in_dtype == GLA_BF16;
  a.log_decay = log_decay; a.aug = aug_balance; a.init = init_state; a.dfin = d_final_state;
  a.dq = dq; a.dk = dk; a.dv = dv; a.d_aug = d_aug; a.dinit = d_init_state; a.gate = gate;
  a.saved = gla::saved_states_at(const_cast<void*>(saved_states), B, T, H);
  a.workspace = workspace; a.workspace_bytes = gla::chunk_bwd_workspace_bytes(B, T, H);
  a.B = B; a.T = T; a.H = H;
  if (in_dtype == GLA_FP32) {
    const size_t tok = (size_t)B * T * H;
    uint8_t* w = static_cast<uint8_t*>(workspace) + a.workspace_bytes;
    void* hq = w;
    void* hk = w + round256(tok * dk_ * 2);
    void* hv = w + 2 * round256(tok * dk_ * 2);
    void* hd = w + 2 * round256(tok * dk_ * 2) + round256(tok * dv_ * 2);
    if (gla::launch_to_half((const float*)q, hq, (long long)(tok * dk_), ctl, stream) != cudaSuccess ||
        gla::launch_to_half((const float*)k, hk, (long long)(tok * dk_), ctl, stream) != cudaSuccess ||
        gla::launch_to_half((const float*)v, hv, (long long)(tok * dv_), ctl, stream) != cudaSuccess ||
        gla::launch_to_half((const float*)dO, hd, (long long)(tok * dv_), ctl, stream) != cudaSuccess)
      return GLA_ERR_CUDA;
    a.q = hq; a.k = hk; a.v = hv; a.dO = hd; a.bf16 = false;
  }
  a.plan = plan;
  if (plan.parts > 1) {
    const size_t slots = (size_t)gla::split_slots((long long)B * H, plan);
    uint8_t* w = static_cast<uint8_t*>(workspace) + round256(need);
    a.seg_state = reinterpret_cast<float*>(w);
    a.seg_adj = reinterpret_cast<float*>(w + round256(slots * kStateBytes));
    a.da_split = reinterpret_cast<float*>(w + 2 * round256(slots * kStateBytes));
    // with the forward's saved state copies the DQ role needs no starting states: only the
    // adjoints (DV, DK) are summed and linked
    if (a.saved.copy) a.seg_state = nullptr;
    // the segment passes (with plan.overlap beside the whole pairs: see the forward)
    if (gla::launch_segment_states(a.q, a.k, a.v, a.dO, a.bf16, log_decay, init_state,
                                   d_final_state, gla::StatePages{}, a.seg_state, a.seg_adj, B, T,
                                   H, plan, ctl, stream) != cudaSuccess)
      return GLA_ERR_CUDA;
  }
  return gla::launch_chunk_bwd(a, ctl, stream) == cudaSuccess ? GLA_OK : GLA_ERR_CUDA;
}

gla_status gla_chunk_state_sum(const void* k, const void* v, gla_dtype in_dtype,
                               const float* log_decay, float* U, int B, int T, int H, int dk,
                               int dv, cudaStream_t stream) {
  gla_status st = check_chunk_sizes(B, T, H, dk, dv, in_dtype);
  if (st != GLA_OK) return st;
  if (in_dtype == GLA_FP32) return GLA_ERR_UNSUPPORTED;
  if (!k || !v || !log_decay || !U) return GLA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(log_decay) || !aligned16(U))
    return GLA_ERR_ALIGNMENT;
  gla::DevCtl ctl;
  if ((st = ctl_for_current_device(&ctl)) != GLA_OK) return st;
  return gla::launch_slice_sums(k, v, in_dtype == GLA_BF16, false, log_decay, U, B, T, H,
                                sm_count(), ctl, stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

gla_status gla_chunk_adjoint_sum(const void* q, const void* dO, gla_dtype in_dtype,
                                 const float* log_decay, float* U, int B, int T, int H, int dk,
                                 int dv, cudaStream_t stream) {
  gla_status st = check_chunk_sizes(B, T, H, dk, dv, in_dtype);
  if (st != GLA_OK) return st;
  if (in_dtype == GLA_FP32) return GLA_ERR_UNSUPPORTED;
  if (!q || !dO || !log_decay || !U) return GLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(dO) || !aligned16(log_decay) || !aligned16(U))
    return GLA_ERR_ALIGNMENT;
  gla::DevCtl ctl;
  if ((st = ctl_for_current_device(&ctl)) != GLA_OK) return st;
  return gla::launch_slice_sums(q, dO, in_dtype == GLA_BF16, true, log_decay, U, B, T, H,
                                sm_count(), ctl, stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

gla_status gla_state_link(const float* U_all, const int* lens, int n_slices, int slice,
                          int reverse, const float* log_decay, const float* boundary, float* out,
                          int B, int H, int dk, int dv, cudaStream_t stream) {
  if (B <= 0 || H <= 0 || n_slices <= 0 || slice < 0 || slice >= n_slices)
    return GLA_ERR_INVALID_ARG;
  if (dk != gla::kDK || dv != gla::kDV || n_slices > gla::kMaxShards) return GLA_ERR_UNSUPPORTED;
  if ((long long)B * H > 65535) return GLA_ERR_UNSUPPORTED;
  if (!U_all || !lens || !log_decay || !out) return GLA_ERR_INVALID_ARG;
  if (!aligned16(U_all) || !aligned16(log_decay) || !aligned16(boundary) || !aligned16(out))
    return GLA_ERR_ALIGNMENT;
  gla::ShardLens L;
  L.n = n_slices;
  for (int j = 0; j < n_slices; ++j) {
    if (lens[j] <= 0) return GLA_ERR_INVALID_ARG;
    L.len[j] = lens[j];
  }
  return gla::launch_shard_link(U_all, L, slice, reverse != 0, log_decay, boundary, out, B, H,
                                stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

gla_status gla_decode_step(float* state, const float* q, const float* k, const float* v,
                           const float* log_decay, const float* aug_balance, float* o, int N,
                           int L, int H, int dk, int dv, cudaStream_t stream) {
  if (N <= 0 || L <= 0 || H <= 0) return GLA_ERR_INVALID_ARG;
  if (dk != gla::kDK || dv != gla::kDV) return GLA_ERR_UNSUPPORTED;
  if (!state || !q || !k || !v || !log_decay || !aug_balance || !o) return GLA_ERR_INVALID_ARG;
  if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(log_decay) || !aligned16(aug_balance) || !aligned16(o))
    return GLA_ERR_ALIGNMENT;
  const long long n = (long long)N * L * H;
  if (n > (1ll << 31) - 1) return GLA_ERR_UNSUPPORTED;
  return gla::launch_decode(state, q, k, v, log_decay, aug_balance, o, n, L, H, stream) ==
                 cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

gla_status gla_decode_step_paged(float* pool, const int* page, int n_active, int n_pages,
                                 int pool_layers, int layer0, const float* q, const float* k,
                                 const float* v, const float* log_decay, const float* aug_balance,
                                 float* o, int L, int H, int dk, int dv, cudaStream_t stream) {
  if (n_active < 0 || n_pages <= 0 || pool_layers <= 0 || L <= 0 || H <= 0 || layer0 < 0 ||
      layer0 + L > pool_layers)
    return GLA_ERR_INVALID_ARG;
  if (dk != gla::kDK || dv != gla::kDV) return GLA_ERR_UNSUPPORTED;
  if (n_active == 0) return GLA_OK;
  if (!pool || !page || !q || !k || !v || !log_decay || !aug_balance || !o)
    return GLA_ERR_INVALID_ARG;
  if (!aligned16(pool) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(log_decay) || !aligned16(aug_balance) || !aligned16(o))
    return GLA_ERR_ALIGNMENT;
  if ((long long)n_active * L * H > (1ll << 31) - 1 ||
      (long long)n_pages * pool_layers * H > (1ll << 40))
    return GLA_ERR_UNSUPPORTED;
  gla::DevCtl ctl;
  gla_status st = ctl_for_current_device(&ctl);
  if (st != GLA_OK) return st;
  return gla::launch_decode_paged(pool, page, n_pages, pool_layers, layer0, q, k, v, log_decay,
                                  aug_balance, o, n_active, L, H, ctl, stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

static gla_status check_head_norm(const float* o, const void* g, gla_dtype g_dtype,
                                  const float* weight, int n_tiers, float eps, long long n_tokens,
                                  int H, int dv) {
  if (n_tokens < 0 || H <= 0 || n_tiers <= 0 || H % n_tiers != 0 || !(eps >= 0.f) ||
      !(eps < 1e30f))
    return GLA_ERR_INVALID_ARG;
  if (dv != gla::kDV || (g_dtype != GLA_BF16 && g_dtype != GLA_FP32)) return GLA_ERR_UNSUPPORTED;
  if (n_tokens > 0 && (!o || !g || !weight)) return GLA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(g) || !aligned16(weight)) return GLA_ERR_ALIGNMENT;
  return GLA_OK;
}

gla_status gla_head_norm_gate_fwd(const float* o, const void* g, gla_dtype g_dtype,
                                  const float* weight, int n_tiers, float eps, float* y,
                                  float* rstd, long long n_tokens, int H, int dv,
                                  cudaStream_t stream) {
  gla_status st = check_head_norm(o, g, g_dtype, weight, n_tiers, eps, n_tokens, H, dv);
  if (st != GLA_OK) return st;
  if (n_tokens > 0 && !y) return GLA_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(rstd)) return GLA_ERR_ALIGNMENT;
  return gla::launch_head_norm_fwd(o, g, g_dtype == GLA_BF16, weight, y, rstd, n_tokens * H, H,
                                   n_tiers, eps, sm_count(), stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

size_t gla_head_norm_gate_bwd_workspace_size(long long n_tokens, int H, int dv) {
  if (n_tokens <= 0 || H <= 0 || dv != gla::kDV) return 0;
  return gla::head_norm_bwd_workspace_bytes(n_tokens * H, H, sm_count());
}

gla_status gla_head_norm_gate_bwd(const float* dy, const float* o, const void* g,
                                  gla_dtype g_dtype, const float* weight, int n_tiers, float eps,
                                  float* d_o, float* dg, float* d_weight, void* workspace,
                                  size_t workspace_bytes, long long n_tokens, int H, int dv,
                                  cudaStream_t stream) {
  gla_status st = check_head_norm(o, g, g_dtype, weight, n_tiers, eps, n_tokens, H, dv);
  if (st != GLA_OK) return st;
  if (!d_weight || (n_tokens > 0 && (!dy || !d_o || !dg))) return GLA_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(d_o) || !aligned16(dg) || !aligned16(d_weight))
    return GLA_ERR_ALIGNMENT;
  const size_t need = gla_head_norm_gate_bwd_workspace_size(n_tokens, H, dv);
  if (need && (!workspace || workspace_bytes < need)) return GLA_ERR_WORKSPACE;
  if (need && !aligned256(workspace)) return GLA_ERR_ALIGNMENT;
  return gla::launch_head_norm_bwd(dy, o, g, g_dtype == GLA_BF16, weight, d_o, dg, d_weight,
                                   static_cast<float*>(workspace), n_tokens * H, H, n_tiers, eps,
                                   sm_count(), stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

static gla_status check_conv(const void* x, gla_dtype x_dtype, const float* weight,
                             const float* bias, const float* init, int B, int T, int D) {
  if (B <= 0 || T <= 0 || D <= 0) return GLA_ERR_INVALID_ARG;
  if (D % 4 != 0 || (x_dtype != GLA_BF16 && x_dtype != GLA_FP32)) return GLA_ERR_UNSUPPORTED;
  if ((long long)B * ((T + 63) / 64) > (1ll << 31) - 1 || (long long)B * T * D > (1ll << 40))
    return GLA_ERR_UNSUPPORTED;
  if (!x || !weight) return GLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(bias) || !aligned16(init))
    return GLA_ERR_ALIGNMENT;
  return GLA_OK;
}

gla_status gla_conv_fwd(const void* x, gla_dtype x_dtype, const float* weight, const float* bias,
                        const float* init_state, float* y, float* final_state, int B, int T,
                        int D, cudaStream_t stream) {
  gla_status st = check_conv(x, x_dtype, weight, bias, init_state, B, T, D);
  if (st != GLA_OK) return st;
  if (!y) return GLA_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(final_state)) return GLA_ERR_ALIGNMENT;
  gla::DevCtl ctl;
  if ((st = ctl_for_current_device(&ctl)) != GLA_OK) return st;
  return gla::launch_conv_fwd(x, x_dtype == GLA_BF16, weight, bias, init_state, y, final_state,
                              B, T, D, ctl, stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

size_t gla_conv_bwd_workspace_size(int B, int T, int D) {
  if (B <= 0 || T <= 0 || D <= 0 || D % 4 != 0) return 0;
  return gla::conv_bwd_workspace_bytes(B, T, D);
}

gla_status gla_conv_bwd(const void* x, gla_dtype x_dtype, const float* weight, const float* bias,
                        const float* init_state, const float* dy, float* dx,
                        float* d_init_state, float* d_weight, float* d_bias, void* workspace,
                        size_t workspace_bytes, int B, int T, int D, cudaStream_t stream) {
  gla_status st = check_conv(x, x_dtype, weight, bias, init_state, B, T, D);
  if (st != GLA_OK) return st;
  if (!dy || !dx || !d_weight) return GLA_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(dx) || !aligned16(d_init_state) || !aligned16(d_weight) ||
      !aligned16(d_bias))
    return GLA_ERR_ALIGNMENT;
  const size_t need = gla_conv_bwd_workspace_size(B, T, D);
  if (!workspace || workspace_bytes < need) return GLA_ERR_WORKSPACE;
  if (!aligned256(workspace)) return GLA_ERR_ALIGNMENT;
  gla::DevCtl ctl;
  if ((st = ctl_for_current_device(&ctl)) != GLA_OK) return st;
  return gla::launch_conv_bwd(x, x_dtype == GLA_BF16, weight, bias, init_state, dy, dx,
                              d_init_state, d_weight, d_bias, static_cast<float*>(workspace), B,
                              T, D, ctl, stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

gla_status gla_conv_decode_step(float* state, const float* x, const float* weight,
                                const float* bias, float* y, long long N, int D,
                                cudaStream_t stream) {
  if (N < 0 || D <= 0) return GLA_ERR_INVALID_ARG;
  if (D % 4 != 0) return GLA_ERR_UNSUPPORTED;
  if (N == 0) return GLA_OK;
  if (!state || !x || !weight || !y) return GLA_ERR_INVALID_ARG;
  if (!aligned16(state) || !aligned16(x) || !aligned16(weight) || !aligned16(bias) ||
      !aligned16(y))
    return GLA_ERR_ALIGNMENT;
  if (N * (D / 4) > (1ll << 40)) return GLA_ERR_UNSUPPORTED;
  return gla::launch_conv_decode(state, x, weight, bias, y, N, D, stream) == cudaSuccess
             ? GLA_OK
             : GLA_ERR_CUDA;
}

}  // extern "C"
