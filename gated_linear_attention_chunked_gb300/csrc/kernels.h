// kernels.h -- internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda_runtime_api.h>

#include <cstddef>
#include <cstdint>

#include "ptx.cuh"

namespace gla {

constexpr int kDK = 96, kDV = 192, kChunk = 128;

cudaError_t launch_decode(float* state, const float* q, const float* k, const float* v,
                          const float* log_decay, const float* aug, float* o, long long n_states,
                          int L, int H, cudaStream_t stream);

// The same step over a pool of pages: active sequence n uses the states of page[n], layers
// layer0 .. layer0+L-1 of the pool's pool_layers; pages outside [0, n_pages) record DEV_RANGE.
cudaError_t launch_decode_paged(float* pool, const int* page, int n_pages, int pool_layers,
                                int layer0, const float* q, const float* k, const float* v,
                                const float* log_decay, const float* aug, float* o, int n_active,
                                int L, int H, DevCtl ctl, cudaStream_t stream);

// fp32 -> fp16 copy (for GLA_FP32 inputs); values with |x| >= 65504 record DEV_RANGE.
cudaError_t launch_to_half(const float* src, void* dst, long long n, DevCtl ctl,
                           cudaStream_t stream);

// Initial/final states in a pool with one page per sequence: sequence b's slot is
// pool[(page[b] * pool_layers + layer) * H + h]; init_paged: the initial state is read from
// that slot too (else from init as [b][h]).  page == null: the caller's [B][H] arrays.
struct StatePages {
  const int* page = nullptr;
  int n_pages = 0, pool_layers = 1, layer = 0;
  bool init_paged = false;
};

// Output epilogue fused into the chunked forward: y = o r w[h / heads_per_tier] SiLU(g) with
// r = (mean_c o_c^2 + eps)^-1/2 per (token, head).  g == null: plain output o.
struct OutGate {
  const uint16_t* g = nullptr;  // [B*T, H, 192] bf16 gate stream (raw bits)
  const float* w = nullptr;     // [n_tiers, 192]
  float* y = nullptr;           // [B*T, H, 192] fp32
  float* rstd = nullptr;        // [B*T, H] fp32 or null
  float eps = 0.f;
  int heads_per_tier = 1;
  bool want_o = false;          // also write o
};

// How the (b, h) pairs of a chunked call are laid out over CTAs.  Pairs 0 .. whole-1 run whole
// (one CTA per pair, or per pair and role in the backward, over all nc chunks); the last
// BH - whole pairs -- the partial last wave -- are cut into `parts` consecutive chunk ranges,
// part j covering chunks [j*nc/parts, (j+1)*nc/parts), each its own CTA that starts from the
// state (forward) or adjoint (reverse) at its boundary, computed beforehand by the segment
// passes (seg_scan.cu).  parts == 1: no pair is cut.
// Launch configuration of a kernel that may be a programmatic dependent of the grid ahead of
// it on the stream (pdl): it may then start while that grid finishes, and reads what that grid
// writes only after griddep_wait.  Used in place (cfg points at attr).
struct PdlLaunch {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl) {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
  }
  PdlLaunch(const PdlLaunch&) = delete;
};

struct SplitPlan {
  int whole = 0;
  int parts = 1;
  // the segment passes overlap the whole pairs: each pass and then the chunked kernel is
  // launched as a programmatic dependent of the launch before it, so the chunked kernel's whole
  // pairs start beside the passes and only its parts wait for them (griddep_wait)
  bool overlap = false;
  // CTAs of the sum pass (0: one per summed part).  Beside the whole pairs the pass walks
  // several parts per CTA, so that the SMs it holds at the start stay few enough for every
  // part of the last wave to start on an SM that began with a whole pair.
  int pass_ctas = 0;
};
__host__ __device__ inline int part_begin(int j, int nc, int parts) {
  return (int)(((long long)j * nc) / parts);
}

// A chunked forward's state copies, saved for the backward (an activation of the training
// step, like the gate): per (b, h) pair and chunk c, the fp16 copy S_c 2^-e_c of the state
// entering the chunk -- the B operand the forward's Q''S product reads -- as the tensor cores'
// shared-memory image (three 64-column atoms of 96 key rows x 128 bytes, 128-byte swizzle), and
// its exponent e_c.  With them the backward's DQ role needs no state scan of its own.
constexpr int kCopyBytes = 36864;
struct SavedStates {
  uint8_t* copy = nullptr;  // [B*H][nc][kCopyBytes]
  int* exp = nullptr;       // [B*H][nc]
};
// Bytes of the saved states of B*H pairs of T tokens: the copies, 256-aligned, then the
// exponents.
inline size_t saved_states_bytes(int B, int T, int H) {
  const size_t n = (size_t)B * H * ((T + kChunk - 1) / kChunk);
  return ((n * kCopyBytes + 255) & ~(size_t)255) + n * sizeof(int);
}
inline SavedStates saved_states_at(void* base, int B, int T, int H) {
  SavedStates s;
  if (!base) return s;
  const size_t n = (size_t)B * H * ((T + kChunk - 1) / kChunk);
  s.copy = static_cast<uint8_t*>(base);
  s.exp = reinterpret_cast<int*>(s.copy + ((n * kCopyBytes + 255) & ~(size_t)255));
  return s;
}

struct FwdArgs {
  const void* q;  // [B,T,H,96] 16-bit
  const void* k;
  const void* v;  // [B,T,H,192] 16-bit
  bool bf16;      // element type of q,k,v: bf16 (true) or fp16 (false)
  const float* log_decay;  // [H]
  const float* aug;        // [H,96]
  const float* init;       // [B,H,96,192] or null
  float* o;                // [B,T,H,192]
  float* fin;              // [B,H,96,192] or null
  int B, T, H;
  SplitPlan plan;          // plan.whole = B*H unless some pairs are cut
  // cut pairs: [(BH - whole) * parts][96][192], slot x*parts + j = the state entering part j
  // of cut pair x (filled by the segment passes; slot x*parts is the pair's initial state)
  const float* seg_init = nullptr;
  // per part slot, max |state| of its starting state as up to four partial maxima [slot][4]
  // (written by the segment passes; null: the kernel finds the max itself)
  const float* seg_max = nullptr;
  StatePages sp;  // with sp.page: init and fin are the pool (see StatePages)
  OutGate og;     // with og.g: the fused output epilogue (o written only if og.want_o)
  float* gate = nullptr;  // [B,H,T] or null: sigmoid(z) per head and token, written
  SavedStates saved;      // copy == null: not saved
};
// Returns cudaErrorInvalidValue if a tensor map cannot be encoded.
cudaError_t launch_chunk_fwd(const FwdArgs& a, DevCtl ctl, cudaStream_t stream);

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dO;  // [B,T,H,192] 16-bit
  bool bf16;
  const float* log_decay;
  const float* aug;
  const float* init;
  const float* dfin;
  float* dq;
  float* dk;
  float* dv;
  float* d_aug;
  float* dinit;
  void* workspace;          // d_aug partial sums of the whole pairs: [B*H][96] fp32
  size_t workspace_bytes;
  int B, T, H;
  SplitPlan plan;           // plan.whole = B*H unless some pairs are cut
  // cut pairs (x = pair - whole, slot x*parts + j for part j):
  float* seg_state = nullptr;  // the state entering part j (the DQ role's start)
  float* seg_adj = nullptr;    // the adjoint of the state leaving part j (DV, DK roles' start)
  float* da_split = nullptr;   // d_aug partial sums of the parts, [96] each
  const float* gate = nullptr;  // [B,H,T] or null: sigmoid(z) per head and token, read
                                // instead of recomputing the gate
  SavedStates saved;            // copy != null: the forward's state copies; the DQ role reads
                                // them instead of scanning the state itself
};
size_t chunk_bwd_workspace_bytes(int B, int T, int H);

// ---- splitting the last wave (seg_scan.cu)
// The plan for B*H pairs of nc chunks with `roles` CTAs per pair (1 forward, 3 backward) on
// n_sm SMs: cut the pairs of the partial last wave (all pairs if they do not fill the SMs)
// into the number of parts that minimises the estimated time, passes included.  force_parts:
// 0 chooses, 1 never cuts, p >= 2 cuts the last wave's pairs into min(p, nc) parts.
// pass_dirs: the directions the segment passes sum (the forward and a backward reading the
// forward's state copies need one; a backward that scans the state itself, two).  overlap:
// the passes may run beside the whole pairs' CTAs (programmatic dependent launches, see
// SplitPlan::overlap) instead of before them; the plan then says whether they do.
SplitPlan plan_split(long long BH, int nc, int roles, int n_sm, int force_parts, int pass_dirs,
                     bool overlap);
// States the cut pairs need (each 96 x 192 fp32): (BH - whole) * parts.
long long split_slots(long long BH, const SplitPlan& p);
// The segment passes: U sums over the parts (forward direction for the states entering parts
// 1.., reverse direction for the adjoints leaving parts ..p-2), then their recurrences, which
// also place the initial state (init / pool page / zero) and the final-state adjoint (dfin /
// zero) in the first and last slots.  states (adj) null: that direction is not computed.
// q_or_null, dO_or_null are needed for the reverse direction only.  With two parts the sum
// pass applies the one step of each recurrence itself and pass B is not launched.  With
// plan.overlap pass B is pass A's programmatic dependent and runs on at most 16 CTAs (which
// wait beside pass A's), so that the chunked kernel launched next as its dependent can start
// its whole pairs at once; pass A runs on plan.pass_ctas CTAs.
// state_max (forward direction, may be null): [slot][4] receives partial maxima of each
// starting state: with two parts its three 32-row groups' max |state| (entries 0..2), with
// more the whole state's max |state| (entry 0, the others 0).
cudaError_t launch_segment_states(const void* q, const void* k, const void* v, const void* dO,
                                  bool bf16, const float* log_decay, const float* init,
                                  const float* dfin, const StatePages& sp, float* states,
                                  float* adj, int B, int T, int H, const SplitPlan& plan,
                                  DevCtl ctl, cudaStream_t stream, float* state_max = nullptr);

// ---- sequence-sharded calls (seg_scan.cu): a sequence cut into consecutive slices, one per
// rank.  launch_slice_sums: per (b, h) of this rank's slice of T tokens, U = sum_t
// lambda^(T-1-t) k_t v_t^T (reverse == false; a = k, b = v) or U' = sum_t lambda^(t+1) q_t dO_t^T
// (reverse; a = q, b = dO), into out [B*H][96][192].  launch_shard_link: the state entering
// slice `rank` (forward) or the adjoint of the state leaving it (reverse) from all slices' sums
// U [n][B*H][96][192] and the caller's boundary (initial state / d_final_state, or null).
constexpr int kMaxShards = 256;
struct ShardLens {
  int n = 0;
  int len[kMaxShards];
};
cudaError_t launch_slice_sums(const void* a, const void* b, bool bf16, bool reverse,
                              const float* log_decay, float* out, int B, int T, int H, int n_sm,
                              DevCtl ctl, cudaStream_t stream);
cudaError_t launch_shard_link(const float* U, const ShardLens& lens, int rank, bool reverse,
                              const float* log_decay, const float* boundary, float* out, int B,
                              int H, cudaStream_t stream);

// The device error word and wait limit of the current device (defined in api.cu).
cudaError_t current_device_ctl(DevCtl* ctl);
cudaError_t launch_chunk_bwd(const BwdArgs& a, DevCtl ctl, cudaStream_t stream);

// Head RMSNorm per decay tier + SiLU(g) gate (head_norm.cu).  rows = tokens * H rows of 192;
// n_tiers divides H; g bf16 or fp32.  rstd [rows] may be null.  The backward's partial sums
// of dw need head_norm_bwd_workspace_bytes(rows, H, n_sm) bytes at `part`.
size_t head_norm_bwd_workspace_bytes(long long rows, int H, int n_sm);
cudaError_t launch_head_norm_fwd(const float* o, const void* g, bool g_bf16, const float* w,
                                 float* y, float* rstd, long long rows, int H, int n_tiers,
                                 float eps, int n_sm, cudaStream_t stream);
cudaError_t launch_head_norm_bwd(const float* dy, const float* o, const void* g, bool g_bf16,
                                 const float* w, float* d_o, float* dg, float* dw, float* part,
                                 long long rows, int H, int n_tiers, float eps, int n_sm,
                                 cudaStream_t stream);

// Depth-wise causal Conv1d (width 4) + SiLU and its 3-token state (conv.cu).  x [B,T,D] bf16
// or fp32, w [D,4], bias [D] or null, init/fin [B,3,D] fp32 or null, D % 4 == 0.
size_t conv_bwd_workspace_bytes(int B, int T, int D);
cudaError_t launch_conv_fwd(const void* x, bool bf16, const float* w, const float* bias,
                            const float* init, float* y, float* fin, int B, int T, int D,
                            DevCtl ctl, cudaStream_t stream);
cudaError_t launch_conv_bwd(const void* x, bool bf16, const float* w, const float* bias,
                            const float* init, const float* dy, float* dx, float* dinit,
                            float* dw, float* db, float* part, int B, int T, int D,
                            DevCtl ctl, cudaStream_t stream);
cudaError_t launch_conv_decode(float* state, const float* x, const float* w, const float* bias,
                               float* y, long long n, int D, cudaStream_t stream);

}  // namespace gla
