/*
 * gla.h -- C ABI of libgla, the GB300 (sm_103a) Simple GLA mixer library.
 *
 * The method is the "Simple GLA" token mixer of the Laplace 3B linear-attention
 * model, as described in "Beyond the KV cache: Training and serving i14's
 * Laplace 3B linear attention model on AWS Trainium2 with native PyTorch":
 *   section "i14 and the Laplace 3B architecture", paragraph "GLA mixer":
 *     S_t = lambda_h S_{t-1} + k_t v_t^T     (per-head 96x192 matrix state)
 *     o_t = S_t^T q_t + sigmoid(sum_c a_{h,c} q_{t,c} k_{t,c}) v_t
 *   paragraph "Decay schedule": lambda_h fixed, half-lives geometric from
 *     T_min to T_max (lambda_0 = 0.5, lambda_15 ~ 0.9997 for 1..2048);
 *   section "Challenge 1": the chunked parallel form (intra-chunk masked
 *     attention, inter-chunk running state, state advanced by the decay
 *     compounded over the chunk), chunk C = 128;
 *   section "Challenge 3": the backward through the sequential updates;
 *   section "Inference optimization on Trainium2": one fixed recurrent state
 *     per sequence, updated one token at a time while serving.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Ownership: the caller owns every buffer.  Tensor arguments are DEVICE
 *    pointers unless a comment says "host".  The library allocates no device
 *    memory; scratch comes from the caller's `workspace`.
 *  - Streams: calls enqueue work on `stream` (NULL = legacy default stream)
 *    and return without synchronising.  gla_chunk_fwd, gla_chunk_bwd and
 *    gla_decode_step can be captured into a CUDA graph (stream capture) once
 *    the device has run them eagerly: a replay gives exactly the results of
 *    the same calls made then on the captured buffers' contents.
 *  - Errors: argument errors are returned before anything is launched, as
 *    GLA_ERR_INVALID_ARG / GLA_ERR_UNSUPPORTED / GLA_ERR_ALIGNMENT /
 *    GLA_ERR_WORKSPACE.  A failed launch returns GLA_ERR_CUDA.  Errors found
 *    on the device while a kernel runs (a bounded wait that gave up, an fp16
 *    operand out of range) are recorded in a device error word that
 *    gla_get_device_error() reads and clears.
 *  - Layout: token-major and contiguous.  q, k: [B, T, H, dk]; v, o, dO:
 *    [B, T, H, dv]; states: [B, H, dk, dv] (row i = key channel, column n =
 *    value channel); aug_balance: [H, dk]; log_decay: [H].
 *  - Supported sizes: dk = 96, dv = 192 (the model's head sizes); B, T, H > 0.
 *    The chunked calls take any T: a sequence is ceil(T / 128) chunks and the
 *    last one holds the remaining 1..128 tokens.
 *  - Alignment: every tensor pointer must be 16-byte aligned.
 *  - Decay: log_decay[h] = gamma_h = ln(lambda_h) (natural log, < 0 for a
 *    decaying head).  The decay is fixed, so there is no gradient for it.
 *  - No internal scaling: q is used as given (callers pre-scale it).
 */
#ifndef GLA_H
#define GLA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define GLA_API __attribute__((visibility("default")))
#else
#define GLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GLA_OK = 0,
  GLA_ERR_INVALID_ARG = 1, /* null pointer where one is required, size <= 0 */
  GLA_ERR_UNSUPPORTED = 2, /* dk != 96, dv != 192, unknown dtype, sizes past 2^31 tokens */
  GLA_ERR_ALIGNMENT = 3,   /* a tensor pointer is not 16-byte aligned */
  GLA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  GLA_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel gave up */
  GLA_ERR_RANGE = 6,       /* device: an operand or state left the fp16 range, or a pool page index was out of range */
  GLA_ERR_WORKSPACE = 7,   /* workspace missing or smaller than required */
  GLA_ERR_LAYOUT = 8       /* device: shared memory not aligned as required */
} gla_status;

/* Element type of the q, k, v, dO inputs.  Outputs and states are fp32. */
typedef enum {
  GLA_BF16 = 0, /* bfloat16.  The chunked calls' tensor cores take fp16 operands, so they
                   need |x| < 65504 for every input element, and the masked scores they form
                   (scaled with the state copy) within that range too; a violation is
                   reported as GLA_ERR_RANGE, not returned as a silent overflow */
  GLA_FP32 = 1, /* float32: converted to fp16 on the device (|x| < 65504) */
  GLA_FP16 = 2  /* IEEE half */
} gla_dtype;

/* Human-readable name of a status code (static string). */
GLA_API const char* gla_status_string(gla_status s);

/* Reads the device error word of the current device and clears it.  Blocks
 * until all work on the device has finished (it synchronises the device).
 * Returns GLA_OK, GLA_ERR_TIMEOUT, GLA_ERR_RANGE or GLA_ERR_LAYOUT, or
 * GLA_ERR_CUDA if the device cannot be queried. */
GLA_API gla_status gla_get_device_error(void);

/* Wall-clock limit, in nanoseconds, of every bounded wait inside the chunk
 * kernels (default 2e9).  A wait that runs out records GLA_ERR_TIMEOUT and
 * the kernel finishes early without touching memory outside its tensors.
 * Applies to calls made after it returns.  ns == 0 restores the default. */
GLA_API gla_status gla_set_wait_timeout_ns(unsigned long long ns);

/* Diagnostic of the failure path (no counterpart in the article): launches one
 * thread that waits on a barrier nothing ever completes.  Its bounded wait gives
 * up after the limit set by gla_set_wait_timeout_ns and sets the device error
 * word, so that gla_get_device_error() then returns GLA_ERR_TIMEOUT and the
 * context stays usable.  Takes about that limit to finish.  Asynchronous on
 * `stream`. */
GLA_API gla_status gla_wait_probe(cudaStream_t stream);

/* Diagnostic of the chunk kernels' give-up path (no counterpart in the article).  For calls
 * made after it returns (process-wide), the tensor-core issuer of every CTA of the chunked
 * forward, backward and segment-pass kernels, on reaching chunk step `step` of its loop,
 * waits on a barrier whose phase completes only after that loop.  The bounded wait gives up
 * after the limit of gla_set_wait_timeout_ns, records GLA_ERR_TIMEOUT and raises the CTA's
 * abort flag; every role then leaves its loop (one path per warp), drains its copies and
 * tensor-core work, frees its tensor memory and exits.  The call's outputs are then
 * undefined; the context stays usable.  step < 0 (the default) turns it off.  No fault,
 * trap or unbounded wait is involved.  The mbarrier wait instruction suspends the waiting
 * thread until the phase completes (up to a hardware limit), so ordinary waits end before
 * any limit of the timer can be checked: a stall like this is what makes a wait run out. */
GLA_API gla_status gla_set_stall_step(int step);

/* Decay schedule ("Decay schedule" paragraph): half-lives
 *   T_h = t_min * (t_max / t_min)^(h / (H - 1))   (T_0 = t_min if H == 1)
 * and log_decay[h] = ln(2^(-1/T_h)) = -ln(2) / T_h, computed in double and
 * stored as float.  log_decay is a HOST array of H floats.
 * Errors: GLA_ERR_INVALID_ARG if H <= 0, t_min <= 0, t_max <= 0 or
 * log_decay is NULL. */
GLA_API gla_status gla_decay_schedule(int H, double t_min, double t_max, float* log_decay);

/* ---------------------------------------------------------------------------
 * Chunked forward ("Challenge 1" chunked form of the "GLA mixer" recurrence).
 *
 *   o[b,t,h,:]          = S_t^T q_t + sigmoid(q_t . (a_h * k_t)) v_t
 *   final_state[b,h]    = S_T
 * with S_0 = init_state[b,h] (zeros if init_state is NULL).
 *
 *   q, k         [B,T,H,96]  in_dtype        v [B,T,H,192] in_dtype
 *   log_decay    [H] fp32 (device)           aug_balance [H,96] fp32 (device)
 *   init_state   [B,H,96,192] fp32 or NULL   (read only)
 *   o            [B,T,H,192] fp32 (written)
 *   final_state  [B,H,96,192] fp32 or NULL   (written)
 *   gate         [B,H,T] fp32 or NULL (written: sigmoid(z_t), z_t = q_t . (a_h * k_t), the
 *                self-augmentation gate, head-major so that a chunk's values are contiguous;
 *                4-byte aligned) -- an activation a training step saves for gla_chunk_bwd,
 *                which then need not recompute it
 *   saved_states device buffer or NULL, 256-byte aligned, of saved_states_bytes >=
 *                gla_chunk_saved_states_size(B, T, H) (GLA_ERR_WORKSPACE if smaller): written
 *                with every chunk's fp16 state copy S_c 2^-e_c -- the operand the chunked form
 *                multiplies the chunk's queries with ("Challenge 1") -- and e_c, 36,868 bytes per
 *                chunk of each (b, h), an activation a training step saves for gla_chunk_bwd,
 *                whose dq part then needs no state scan of its own
 *   workspace    device scratch, 256-byte aligned, of gla_chunk_fwd_workspace_size()
 *                bytes.  fp32 inputs need their fp16 copies there (GLA_ERR_WORKSPACE
 *                if it is smaller).  The size also covers cutting pairs into parts:
 *                one CTA per (b, h) runs its chunks in order, and the pairs that would
 *                leave the last wave of SMs partly empty (all pairs, when there are fewer
 *                than SMs -- few long sequences) are cut into consecutive chunk ranges
 *                that run as CTAs of their own, each starting from the state at its
 *                boundary, which two short passes compute first (the state recurrence
 *                is linear).  See gla_chunk_split_plan.  Given less (or NULL for 16-bit
 *                inputs), no pair is cut: same results up to rounding, more time.  The
 *                size depends on the device current at the call.
 * Arithmetic: the tensor cores take fp16 operands with fp32 accumulation; the
 * state is carried in fp32 across chunks.  Inputs must satisfy |x| < 65504.
 */
GLA_API size_t gla_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, gla_dtype in_dtype);
GLA_API size_t gla_chunk_saved_states_size(int B, int T, int H);
GLA_API gla_status gla_chunk_fwd(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                         const float* log_decay, const float* aug_balance,
                         const float* init_state, float* o, float* final_state, float* gate,
                         void* saved_states, size_t saved_states_bytes, void* workspace,
                         size_t workspace_bytes, int B, int T, int H, int dk, int dv,
                         cudaStream_t stream);

/* gla_chunk_fwd_gated: the same forward with the mixer's output epilogue fused
 * into it ("GLA mixer": a Head RMSNorm shared within each decay tier, then the
 * SiLU(g) gate; see gla_head_norm_gate_fwd for the formula):
 *   y[b,t,h,:] = o r w[h / (H / n_tiers), :] SiLU(g[b,t,h,:]),
 *   r = 1 / sqrt(mean_c o^2 + eps)
 * without o leaving the chip (o is also written if `o` is not NULL, as the
 * epilogue's backward, gla_head_norm_gate_bwd, needs it).
 *   g            [B,T,H,192] bf16       norm_weight [n_tiers,192] fp32
 *   y            [B,T,H,192] fp32 (written)
 *   rstd         [B,T,H] fp32 or NULL (written: r)
 *   o            [B,T,H,192] fp32 or NULL;  other arguments as gla_chunk_fwd.
 */
GLA_API gla_status gla_chunk_fwd_gated(const void* q, const void* k, const void* v,
                                       gla_dtype in_dtype, const float* log_decay,
                                       const float* aug_balance, const float* init_state,
                                       const void* g, const float* norm_weight, int n_tiers,
                                       float eps, float* y, float* rstd, float* o,
                                       float* final_state, void* workspace,
                                       size_t workspace_bytes, int B, int T, int H, int dk,
                                       int dv, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Chunked backward ("Challenge 3": the gradient through every sequential
 * state update), for the scalar loss  L = sum o.dO + <d_final_state, S_T>:
 *
 *   dq_t = S_t dO_t + r_t (a*k_t)        dk_t = G_t v_t + r_t (a*q_t)
 *   dv_t = G_t^T k_t + sigmoid(z_t) dO_t
 *   d_aug[h] = sum_{b,t} r_t (q_t * k_t)  d_init_state = lambda G_1
 * where G_t = q_t dO_t^T + lambda G_{t+1}, G_T = q_T dO_T^T + d_final_state,
 * z_t = q_t.(a*k_t), r_t = sigmoid'(z_t) (dO_t . v_t).
 *
 *   q, k, v, in_dtype, log_decay, aug_balance, init_state: as in the forward
 *   dO            [B,T,H,192] in_dtype
 *   d_final_state [B,H,96,192] fp32 or NULL (= zeros)
 *   gate          [B,H,T] fp32 or NULL: sigmoid(z_t) as gla_chunk_fwd writes it (4-byte
 *                 aligned); given, the backward reads it instead of recomputing z_t (the
 *                 results then follow the values given); NULL: recomputed
 *   saved_states  NULL, or what gla_chunk_fwd wrote there for the same q, k, v, log_decay and
 *                 init_state (size and alignment as there): the dq part reads the state copies
 *                 instead of recomputing the state scan, and its chunks run in the same order
 *                 as the other two parts'
 *   dq, dk        [B,T,H,96]  fp32 (written)    dv [B,T,H,192] fp32 (written)
 *   d_aug         [H,96] fp32 (written, summed over B and T)
 *   d_init_state  [B,H,96,192] fp32 or NULL (written)
 *   workspace     gla_chunk_bwd_workspace_size() bytes, 256-aligned: the d_aug partial
 *                 sums (and fp16 copies of fp32 inputs) are required (GLA_ERR_WORKSPACE
 *                 if the workspace cannot hold them); the rest lets pairs be cut into
 *                 parts as in gla_chunk_fwd (each part of the backward's three scans
 *                 starts from the state entering it, or the adjoint of the state leaving
 *                 it).  Given only the required part, no pair is cut.
 */
GLA_API size_t gla_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, gla_dtype in_dtype);
GLA_API gla_status gla_chunk_bwd(const void* q, const void* k, const void* v, gla_dtype in_dtype,
                         const float* log_decay, const float* aug_balance,
                         const float* init_state, const void* dO, const float* d_final_state,
                         const float* gate, const void* saved_states, size_t saved_states_bytes,
                         float* dq, float* dk, float* dv, float* d_aug, float* d_init_state,
                         void* workspace, size_t workspace_bytes, int B, int T, int H,
                         int dk_, int dv_, cudaStream_t stream);

/* How the chunked calls lay (b, h) pairs out over CTAs (no counterpart in the article: a
 * scheduling choice for the GPU).  Pairs 0 .. whole_pairs-1 run whole (one CTA per pair,
 * three per pair in the backward); pairs whole_pairs .. B*H-1 are each cut into `parts`
 * consecutive chunk ranges (part j: chunks [j*nc/parts, (j+1)*nc/parts), nc = ceil(T/128)).
 * The cut is chosen to shorten the estimated time on a device with n_sm SMs: the pairs of a
 * partial last wave, or all pairs when they do not fill one wave, into the number of parts
 * (at most 32 and nc) that minimises the estimate.  parts == 1: nothing is cut.  A host query
 * of the plan the calls use (with the current device's SM count); results do not depend on it
 * beyond rounding.  backward: 0 the forward, 1 the backward, 2 the backward reading the
 * forward's saved state copies (its segment passes sum one direction instead of two, so it
 * may cut into more parts; gla_chunk_bwd_workspace_size covers both backward plans).
 * Errors: GLA_ERR_INVALID_ARG for sizes or n_sm <= 0 or NULL outputs. */
GLA_API gla_status gla_chunk_split_plan(int B, int T, int H, int backward, int n_sm,
                                        int* whole_pairs, int* parts);
/* Overrides the choice of gla_chunk_split_plan for calls made after it returns (process-wide):
 * 0 = automatic (default), 1 = never cut, p >= 2 = cut the pairs it would consider into
 * min(p, nc) parts.  GLA_ERR_INVALID_ARG for p < 0. */
GLA_API gla_status gla_set_split_parts(int parts);
/* How a call that cuts pairs into parts orders its launches (process-wide; a scheduling choice
 * for the GPU, no counterpart in the article).  on != 0 (the default): when the whole pairs
 * fill at least one wave of SMs, the segment passes and the chunked kernel are chained as
 * programmatic dependent launches on the caller's stream -- the chunked kernel starts its
 * whole pairs' CTAs beside the passes, and each part's CTA waits (griddepcontrol.wait) for the
 * passes before it reads the state they leave; everything stays on the caller's stream, which
 * sees the call's results complete as before.  on == 0: the passes, then the chunked kernel,
 * each after the previous launch has finished.  The results are the same either way; the plan
 * (gla_chunk_split_plan) counts the passes as overlapped when on != 0.  Returns GLA_OK. */
GLA_API gla_status gla_set_pass_overlap(int on);

/* ---------------------------------------------------------------------------
 * A long sequence cut into consecutive slices, one per rank (GPU), for long-context
 * prefill and its backward.  Section "Challenge 1" carries one state from chunk to chunk,
 * and section "Inference optimization on Trainium2" keeps that state fixed in size whatever
 * the prompt's length; the recurrence S_t = lambda S_{t-1} + k_t v_t^T ("GLA mixer") is
 * linear, so a slice j of len_j tokens contributes
 *     S leaving slice j = lambda^(len_j) S entering slice j + U_j,
 *         U_j  = sum_{t in j} lambda^(e_j - t) k_t v_t^T           (e_j: its last token)
 * and, in the backward ("Challenge 3"), with A_j the adjoint of the state leaving slice j,
 *     A_{j-1} = lambda^(len_j) A_j + U'_j,
 *         U'_j = sum_{t in j} lambda^(t - s_j + 1) q_t dO_t^T      (s_j: its first token).
 * Each rank computes its slice's sums, the ranks exchange them (one all-gather of
 * B*H*96*192 floats each), and each rank then runs gla_chunk_fwd / gla_chunk_bwd on its own
 * slice from the state (adjoint) gla_state_link gives it.  The library makes no collective
 * call itself: the exchange is the caller's (for example NCCL through torch.distributed).
 *
 * gla_chunk_state_sum:   U[b,h]  = sum_t lambda_h^(T-1-t) k_t v_t^T   over this call's T tokens
 * gla_chunk_adjoint_sum: U'[b,h] = sum_t lambda_h^(t+1) q_t dO_t^T
 *   k, q [B,T,H,96] and v, dO [B,T,H,192] in_dtype (GLA_BF16 or GLA_FP16; GLA_FP32 ->
 *   GLA_ERR_UNSUPPORTED); log_decay [H]; U [B,H,96,192] fp32 (written).  Tensor cores with
 *   fp16 operands and fp32 accumulation, as the chunked calls (|x| < 65504, GLA_ERR_RANGE).
 *   U equals the final state of gla_chunk_fwd from a zero initial state; U' equals the
 *   d_init_state of gla_chunk_bwd with a zero d_final_state.
 *
 * gla_state_link: out[b,h] for slice `slice` of n_slices (1 <= n_slices <= 256) slices of
 *   lens[0..n_slices-1] tokens (a HOST int array, every entry >= 1):
 *     reverse == 0:  S_0 = boundary (initial state, NULL = zeros), S_{j+1} = lambda^(len_j) S_j
 *                    + U_j; out = S_slice, the state entering the slice
 *     reverse != 0:  A_{n-1} = boundary (d_final_state, NULL = zeros), A_{j-1} =
 *                    lambda^(len_j) A_j + U'_j; out = A_slice, the adjoint of the state
 *                    leaving the slice
 *   U_all [n_slices,B,H,96,192] fp32 (slice j's sums at index j, as an all-gather lays them
 *   out; only the entries the recurrence reaches are read); boundary, out [B,H,96,192] fp32.
 *   B*H <= 65535.
 */
GLA_API gla_status gla_chunk_state_sum(const void* k, const void* v, gla_dtype in_dtype,
                                       const float* log_decay, float* U, int B, int T, int H,
                                       int dk, int dv, cudaStream_t stream);
GLA_API gla_status gla_chunk_adjoint_sum(const void* q, const void* dO, gla_dtype in_dtype,
                                         const float* log_decay, float* U, int B, int T, int H,
                                         int dk, int dv, cudaStream_t stream);
GLA_API gla_status gla_state_link(const float* U_all, const int* lens, int n_slices, int slice,
                                  int reverse, const float* log_decay, const float* boundary,
                                  float* out, int B, int H, int dk, int dv, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Chunked backward that allocates nothing and takes no workspace.
 *
 * The article has no counterpart to this call; it exists for callers that cannot give the
 * library a device buffer: code running inside an engine's or plugin's execution callback
 * where device allocation is not allowed, processes whose device memory is reserved in full
 * up front, and latency-critical loops that must avoid cudaMalloc / cudaFree (which can
 * synchronise the whole device).  It computes exactly what gla_chunk_bwd computes, with the
 * same arguments minus the workspace, by running the same kernels; its only scratch -- the
 * per-(b, h) partial sums of d_aug -- is a fixed array of GLA_NOALLOC_MAX_BH x 96 floats
 * (768 KiB) inside the library, held by every GPU that loads the library until exit.
 *  - Sizes: B * H must be <= GLA_NOALLOC_MAX_BH, else GLA_ERR_WORKSPACE (nothing launched).
 *    Inputs must be GLA_BF16 or GLA_FP16 (fp32 inputs need a workspace for their fp16
 *    copies): GLA_ERR_UNSUPPORTED otherwise.  Other checks and errors as gla_chunk_bwd;
 *    device errors go to the same error word (gla_get_device_error()).
 *  - Every call looks up the array's device address in the current device's context
 *    (cudaGetSymbolAddress, with the return code checked), so a context that was reset and
 *    created again is handled.  The first call on a device may load the library's module
 *    there; make that first call before any stream capture.
 *  - Every call on a device shares the one array, and a call leaves its partial sums in it.
 *    Each call overwrites every entry it later reads, so nothing needs clearing, but calls
 *    that overlap on the GPU (in flight at once, e.g. on two streams) race on the array:
 *    order them on one stream or with events.
 */
#define GLA_NOALLOC_MAX_BH 2048
GLA_API gla_status gla_chunk_bwd_noalloc(const void* q, const void* k, const void* v,
                                         gla_dtype in_dtype, const float* log_decay,
                                         const float* aug_balance, const float* init_state,
                                         const void* dO, const float* d_final_state,
                                         const float* gate, float* dq, float* dk, float* dv,
                                         float* d_aug, float* d_init_state, int B, int T, int H,
                                         int dk_, int dv_, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * One recurrent decode step for a pool of N sequences x L layers x H heads
 * ("Inference optimization on Trainium2": a fixed state per sequence, read
 * and written in the serving pool, O(1) per token).  In place, fp32:
 *
 *   S'  = lambda_h S + k v^T
 *   o   = S'^T q + sigmoid(q . (a_{l,h} * k)) v
 *
 *   state        [N,L,H,96,192] fp32, read and overwritten with S'
 *   q, k         [N,L,H,96] fp32     v [N,L,H,192] fp32
 *   log_decay    [H] fp32            aug_balance [L,H,96] fp32
 *   o            [N,L,H,192] fp32 (written)
 * N*L*H may be any positive count; nothing is allocated.
 */
GLA_API gla_status gla_decode_step(float* state, const float* q, const float* k, const float* v,
                           const float* log_decay, const float* aug_balance, float* o, int N,
                           int L, int H, int dk, int dv, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * State pool with one fixed page per sequence ("Inference optimization on
 * Trainium2": the model declares itself attention-free, so the serving engine
 * gives every sequence one fixed page of recurrent state).  A page holds
 * pool_layers x H states of 96x192 fp32:
 *
 *   pool  [n_pages, pool_layers, H, 96, 192] fp32
 *   state of (page p, layer l, head h) = pool[(p * pool_layers + l) * H + h]
 *
 * gla_decode_step_paged: the decode step above for a variable active set, no
 * padding: active sequence n (0 <= n < n_active) uses page[n] and layers
 * layer0 .. layer0+L-1 of its page.
 *   page         [n_active] int32 (device); distinct pages -- two active
 *                sequences on one page race.  A page outside [0, n_pages)
 *                leaves that sequence untouched (o not written) and sets the
 *                device error word to GLA_ERR_RANGE (gla_get_device_error).
 *   q, k         [n_active,L,H,96] fp32   v, o [n_active,L,H,192] fp32
 *   log_decay    [H]     aug_balance [L,H,96] (the layers of this call)
 * n_active == 0 returns GLA_OK without launching.
 */
GLA_API gla_status gla_decode_step_paged(float* pool, const int* page, int n_active, int n_pages,
                                         int pool_layers, int layer0, const float* q,
                                         const float* k, const float* v, const float* log_decay,
                                         const float* aug_balance, float* o, int L, int H, int dk,
                                         int dv, cudaStream_t stream);

/* gla_chunk_fwd_paged: chunked prefill straight into the pool.  Sequence b of
 * the call (q, k, v, o as in gla_chunk_fwd) starts from the state in layer
 * `layer` of page[b] (init_from_pool != 0) or from zero (init_from_pool == 0:
 * the page need not be cleared), and its final state is written back to that
 * slot.  page [B] int32 (device), distinct pages; a page outside [0, n_pages)
 * leaves its slot untouched and sets the device error word to GLA_ERR_RANGE.
 * Workspace: gla_chunk_fwd_workspace_size(B, T, H, ...) as for gla_chunk_fwd
 * (pairs are cut into parts here too).
 */
GLA_API gla_status gla_chunk_fwd_paged(const void* q, const void* k, const void* v,
                                       gla_dtype in_dtype, const float* log_decay,
                                       const float* aug_balance, float* pool, const int* page,
                                       int n_pages, int pool_layers, int layer,
                                       int init_from_pool, float* o, void* workspace,
                                       size_t workspace_bytes, int B, int T, int H, int dk,
                                       int dv, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * The mixer's output epilogue ("i14 and the Laplace 3B architecture", "GLA
 * mixer" and "Decay schedule's reach": a Head RMSNorm shared within each decay
 * tier, then the SiLU(g_t) gate).  Per token t and head h, tier(h) =
 * h / (H / n_tiers) (consecutive heads, i.e. neighbouring half-lives):
 *
 *   r_th   = 1 / sqrt(mean_c o_thc^2 + eps)
 *   y_thc  = o_thc r_th weight[tier(h), c] SiLU(g_thc),   SiLU(x) = x sigmoid(x)
 *
 *   o, y         [n_tokens, H, 192] fp32 (tokens = B*T, any order)
 *   g            [n_tokens, H, 192] g_dtype (GLA_BF16 or GLA_FP32)
 *   weight       [n_tiers, 192] fp32, n_tiers divides H
 *   rstd         [n_tokens, H] fp32 or NULL (written: r_th)
 * All fp32 arithmetic, nothing allocated.
 */
GLA_API gla_status gla_head_norm_gate_fwd(const float* o, const void* g, gla_dtype g_dtype,
                                          const float* weight, int n_tiers, float eps, float* y,
                                          float* rstd, long long n_tokens, int H, int dv,
                                          cudaStream_t stream);

/* Its gradient for the scalar loss sum(y . dy): with n = o r, s = SiLU(g),
 *   dg        = dy n weight sigmoid(g) (1 + g (1 - sigmoid(g)))
 *   d_o       = r (dn - n mean_c(dn n)),   dn = dy s weight
 *   d_weight  [n_tiers, 192] = sum over tokens and each tier's heads of dy s n
 * (written, summed in a fixed order: deterministic).  dy, d_o, dg [n_tokens,
 * H, 192] fp32.  workspace: gla_head_norm_gate_bwd_workspace_size() bytes,
 * 256-byte aligned (per-row-slot partial sums of d_weight).
 */
GLA_API size_t gla_head_norm_gate_bwd_workspace_size(long long n_tokens, int H, int dv);
GLA_API gla_status gla_head_norm_gate_bwd(const float* dy, const float* o, const void* g,
                                          gla_dtype g_dtype, const float* weight, int n_tiers,
                                          float eps, float* d_o, float* dg, float* d_weight,
                                          void* workspace, size_t workspace_bytes,
                                          long long n_tokens, int H, int dv,
                                          cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Depth-wise causal Conv1d of width 4 with SiLU, in front of the QKVG
 * projection ("i14 and the Laplace 3B architecture", "Normalization and
 * convolution"), and its recurrent state of the last 3 inputs per sequence:
 *
 *   y_t[d] = SiLU(sum_{j=0..3} weight[d][j] x_{t-3+j}[d] + bias[d])
 *
 * with x_{-3..-1} = init_state (zeros if NULL) and final_state = x_{T-3..T-1}
 * (the state to continue from).
 *   x            [B,T,D] x_dtype (GLA_BF16 or GLA_FP32), D % 4 == 0
 *   weight       [D,4] fp32       bias [D] fp32 or NULL (= 0)
 *   init_state, final_state   [B,3,D] fp32 or NULL
 *   y            [B,T,D] fp32 (written)
 */
GLA_API gla_status gla_conv_fwd(const void* x, gla_dtype x_dtype, const float* weight,
                                const float* bias, const float* init_state, float* y,
                                float* final_state, int B, int T, int D, cudaStream_t stream);

/* Gradient for the scalar loss sum(y . dy): dz = dy SiLU'(z),
 *   dx_s = sum_j weight[j] dz_{s+3-j}    (d_init_state: s = -3..-1; may be NULL)
 *   d_weight[d][j] = sum_{b,t} dz_t x_{t-3+j},  d_bias[d] = sum_{b,t} dz_t (NULL: skipped)
 * (summed in a fixed order: deterministic).  The final state is a copy of
 * the last inputs: a caller that differentiates through it adds its gradient
 * to dx itself.  dy, dx [B,T,D] fp32; workspace gla_conv_bwd_workspace_size()
 * bytes, 256-byte aligned.
 */
GLA_API size_t gla_conv_bwd_workspace_size(int B, int T, int D);
GLA_API gla_status gla_conv_bwd(const void* x, gla_dtype x_dtype, const float* weight,
                                const float* bias, const float* init_state, const float* dy,
                                float* dx, float* d_init_state, float* d_weight, float* d_bias,
                                void* workspace, size_t workspace_bytes, int B, int T, int D,
                                cudaStream_t stream);

/* One decode token: state [N,3,D] fp32 holds x_{t-3..t-1} and becomes
 * x_{t-2..t} (in place); x, y [N,D] fp32.  N counts sequences (x layers, if
 * the caller lays a pool out as [N_seq, L, 3, D]). */
GLA_API gla_status gla_conv_decode_step(float* state, const float* x, const float* weight,
                                        const float* bias, float* y, long long N, int D,
                                        cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GLA_H */
