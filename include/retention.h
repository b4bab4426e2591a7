/*
 * retention.h — C ABI of libretention.so: RetNet multi-scale retention (MSR)
 * on one NVIDIA B300 (sm_103a).
 *
 * The operation (per batch row b and head h, decay γ_h, rotation
 * frequencies θ_i, absolute position n = pos0 + t of local index t):
 *
 *   q′_t = R(nθ) q_t,  k′_t = d_k^{-1/2} R(nθ) k_t          (Θ prologue)
 *   o_t  = Σ_{m≤t} γ^{t−m} (q′_t·k′_m) v_m + γ^{t+1} q′_t S_in
 *   S_out = γ^L S_in + Σ_m γ^{L−1−m} k′_mᵀ v_m
 *   optional per-head GroupNorm of o_t over its d_v channels.
 *
 * R(φ) rotates every interleaved pair (x_{2i}, x_{2i+1}) counter-clockwise by
 * φ_i = n·θ_i: theta_shift(x) = x·cos + rotate_every_two(x)·sin of
 * «从RoPE到Retention：一文拆解RetNet如何用'旋转'和'衰减'重塑序列建模» §2
 * (Q←Q⊙Θ, K←K⊙Θ̄; the real dot product of the two rotated vectors depends on
 * n − m only).  The decay mask D_nm = γ^{n−m} (n ≥ m, else exactly 0) is §3 of
 * that page; the parallel, recurrent and chunkwise-recurrent forms are its
 * §4.1–§4.3 and the sections 并行表征 / 循环表征 / 分块循环 of the RetNet
 * 保留网络 explainer (aiqz.cc); the 1/√d scale and GroupNorm are §5 of the
 * first page.  The three forms compute the same result up to rounding.
 *
 * Conventions for every entry point
 * ---------------------------------
 * Layout    q, k: [B, H, L, d_k]; v, out: [B, H, L, d_v]; states:
 *           [B, H, d_k, d_v] fp32; all row-major and contiguous.
 * Memory    q, k, v, out, state*, workspace, gn->weight, gn->bias are DEVICE
 *           pointers owned by the caller.  gamma[H] and theta[d_k/2] are HOST
 *           arrays, read during the call only.  The library allocates no
 *           device memory in any call.
 * Dtypes    RET_BF16 inputs run on the tensor cores (fp32 accumulate) when
 *           d_k ∈ {64, 128, 256}, d_v is a multiple of 128, chunk = 128 and
 *           every head has γ^127 ≥ 2^-60 (any L for the chunkwise entry
 *           points, L a multiple of 128 for ret_parallel); other bf16 calls
 *           and RET_F32 inputs run on fp32 FFMA kernels.  ret_*_plan reports
 *           the path.  out may be bf16 or fp32.
 * Sizes     1 ≤ H ≤ 128; d_k even, 2 ≤ d_k ≤ 512; 1 ≤ d_v ≤ 1024;
 *           0 ≤ pos0 and pos0 + L ≤ 2^24 (positions are exact in fp32);
 *           every pointer 16-byte aligned; 0 < γ_h ≤ 1; θ finite.
 * Errors    Arguments are validated synchronously: RET_EINVAL (bad argument)
 *           or RET_EUNSUPPORTED (valid but not implemented), no launch and no
 *           side effect.  A CUDA launch error returns RET_ECUDA.  Kernels
 *           never trap: a bounded wait that expires sets a device status word
 *           that ret_sync_status() reports as RET_ETIMEOUT.
 * Streams   Every call is asynchronous on `stream` (no host synchronisation).
 * Aliasing  state_in == state_out is allowed; out must not alias the inputs.
 */
#ifndef RETENTION_H
#define RETENTION_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RET_ABI_VERSION 1

typedef enum {
  RET_OK = 0,
  RET_EINVAL = 1,        /* an argument is out of range, NULL or misaligned   */
  RET_EUNSUPPORTED = 2,  /* valid arguments outside the implemented domain     */
  RET_ECUDA = 3,         /* a CUDA call or launch failed                       */
  RET_ETIMEOUT = 4,      /* a kernel's bounded wait expired (see sync_status)  */
  RET_EWORKSPACE = 5     /* workspace missing or smaller than required         */
} ret_status;

typedef enum { RET_F32 = 0, RET_BF16 = 1 } ret_dtype;

/* Per-head GroupNorm epilogue («从RoPE到Retention…» §5; one group = one head's d_v
 * channels of one token; biased variance).  weight/bias: DEVICE [H*d_v] fp32,
 * NULL means 1 / 0.  Pass a NULL ret_gn* (or enabled = 0) to skip it. */
typedef struct {
  int enabled;
  float eps;
  const float* weight;
  const float* bias;
} ret_gn;

/* Kernel path chosen for a call (reported by ret_*_plan). */
typedef enum {
  RET_PATH_TC = 1,     /* tcgen05 tensor-core kernels (bf16 inputs)       */
  RET_PATH_SIMT = 2,   /* fp32 FFMA kernels                               */
  RET_PATH_TC_SINGLE = 3, /* ret_force_path only: the tensor-core path with
                             one CTA per d_v tile instead of CTA pairs    */
  RET_PATH_TC_CARRY = 4   /* ret_force_path only: ret_chunkwise keeps the
                             carried layout where it would take the
                             chunk-parallel one for a small grid          */
} ret_path;

/* ------------------------------------------------------------------------
 * ret_chunkwise — chunkwise-recurrent form, carried-state layout.
 * Chunks of `chunk` tokens are processed in order: inside a chunk the
 * parallel form, across chunks the state S ← γ^b S + (ζ⊙K′)ᵀV with
 * ζ_j = γ^{b−1−j}, and the cross-chunk output term γ^{j+1} q′_j S
 * («从RoPE到Retention…» §4.3; RetNet 保留网络 explainer, 分块循环).
 * state_in: NULL means S_in = 0.  state_out: NULL skips the final state.
 * The per-chunk state is updated in fp32 as S_i = fmaf(γ^b, S_{i−1}, ΔS_i)
 * with ΔS_i accumulated from zero; ret_chunkwise_scan uses the same order,
 * so the two layouts return bit-identical state_out.
 * workspace: DEVICE scratch of at least ret_chunkwise_plan(...)->bytes
 * (NULL allowed when that is 0), or of at least ret_chunkwise_plan_compact's
 * bytes for the compact mode.  The required size depends on the path.
 * ------------------------------------------------------------------------ */
ret_status ret_chunkwise(const void* q, const void* k, const void* v, ret_dtype in_dt,
                         const float* gamma, const float* theta,
                         int B, int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                         const float* state_in, float* state_out,
                         void* out, ret_dtype out_dt, const ret_gn* gn,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ret_chunkwise with one start position per batch row: the tokens of row b
 * sit at positions row_pos0[b] … row_pos0[b] + L − 1 (row_pos0: HOST array
 * of B values, each ≥ 0 with row_pos0[b] + L ≤ 2^24).  B ≤ 256, else
 * RET_EUNSUPPORTED; row_pos0 == NULL is RET_EINVAL.  Same layouts, workspace
 * (ret_chunkwise_plan), paths and results as ret_chunkwise, which it equals
 * bit for bit when every row_pos0[b] equals its pos0. */
ret_status ret_chunkwise_rowpos(const void* q, const void* k, const void* v, ret_dtype in_dt,
                                const float* gamma, const float* theta,
                                int B, int H, int L, int d_k, int d_v, const int64_t* row_pos0,
                                int chunk, const float* state_in, float* state_out,
                                void* out, ret_dtype out_dt, const ret_gn* gn,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Path and workspace bytes ret_chunkwise would use for these arguments.
 * gamma may be NULL (then the tensor-core path is assumed allowed). */
ret_status ret_chunkwise_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                              int d_k, int d_v, int chunk, ret_dtype out_dt, int gn_enabled,
                              int* path, size_t* workspace_bytes);

/* The smallest workspace ret_chunkwise (and ret_chunkwise_rowpos) accepts
 * for these arguments.  On the tensor-core path with CTA pairs (d_k 128 or
 * 256, an even number of 128-wide d_v tiles) this is the compact mode: the
 * Θ prologue runs inside the chunk launch — producer CTAs on the SMs that
 * the consumer pairs leave free rotate q and k into a ring of 4 chunk slots
 * per head, which stays in L2 — instead of as a front pass that writes the
 * rotated Q′ and K̂′ of the whole sequence.  Workspace: the ring (4 chunks
 * of Q′ and K̂′ for at most 128/(d_v/128) heads), an angle table
 * [L][d_k/2] (cos, sin) and the same staging buffers as the plan's (25 MB at
 * the 7B shape against 268 MB).  ret_chunkwise takes this mode by itself
 * whenever its workspace is smaller than ret_chunkwise_plan's bytes but at
 * least these; the results are bit-identical to the front-pass mode's, and
 * it runs about 2.3× slower at the 7B shape (the producers' share of the SMs
 * cannot move and rotate q, k as fast as a front pass on all SMs).  Where
 * the ring is not smaller (sequences of a few chunks) and on every other
 * path it returns the same bytes as ret_chunkwise_plan. */
ret_status ret_chunkwise_plan_compact(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                                      int d_k, int d_v, int chunk, ret_dtype out_dt,
                                      int gn_enabled, int* path, size_t* workspace_bytes);

/* Chunk length for a chunkwise call of this shape: 128 (the tensor-core
 * tile) wherever the tensor-core path applies, otherwise b = round(√L), the
 * square-root balance of the RetNet 保留网络 explainer (分块循环: n/b chunks
 * of O(b²) work each, O(n·b) in total, with n/b sequential state steps),
 * at least 1.  √8192 ≈ 91, so at the 7B shape the tile is the nearest
 * power of two above the balance.  gamma: HOST [H] or NULL (then the
 * tensor-core path is assumed allowed).  Returns 0 for invalid arguments. */
int ret_chunk_size(ret_dtype in_dt, const float* gamma, int H, int L, int d_k, int d_v);

/* ------------------------------------------------------------------------
 * ret_chunkwise_noalloc — ret_chunkwise for callers that may not allocate
 * device memory themselves, e.g. plugins whose host application owns the
 * whole device memory budget, or latency-critical loops that cannot afford
 * a cudaMalloc (or a caching allocator's growth) inside them.  The RetNet
 * pages have no counterpart: this is a library convenience.
 * Scratch: instead of a caller workspace it uses one array of
 * RET_NOALLOC_SCRATCH_BYTES that lives in the library's own device image.
 * Every GPU that loads the library holds that array until the process
 * exits.  Arguments as ret_chunkwise (all data pointers still come from the
 * caller).  It runs the front-pass mode when ret_chunkwise_plan's bytes fit
 * in the array, else the compact mode when ret_chunkwise_plan_compact's
 * bytes do; a problem that fits neither returns RET_EWORKSPACE with no
 * launch.  Every call made outside stream capture looks the array's device
 * address up afresh (cudaGetSymbolAddress, with the caller's device
 * current), so a cudaDeviceReset or a re-created context is picked up; a
 * call made while its stream is capturing reuses the address found by the
 * last uncaptured call on that device, so make one call on each device
 * before any stream capture.  All calls share the one array and it keeps
 * whatever the previous call left; every kernel that reads it writes it
 * first, so nothing needs clearing, but calls that can overlap on the GPU
 * (different streams, or different host threads) race on it: serialise them.
 * The call itself allocates nothing.
 * ------------------------------------------------------------------------ */
#define RET_NOALLOC_SCRATCH_BYTES (32u << 20)

ret_status ret_chunkwise_noalloc(const void* q, const void* k, const void* v, ret_dtype in_dt,
                                 const float* gamma, const float* theta,
                                 int B, int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                                 const float* state_in, float* state_out,
                                 void* out, ret_dtype out_dt, const ret_gn* gn,
                                 cudaStream_t stream);

/* ------------------------------------------------------------------------
 * ret_chunkwise_scan — the same result as ret_chunkwise, computed in the
 * parallel-then-scan layout: every chunk's ΔS_i from zero (all chunks in
 * parallel), an fp32 scan S_i = fmaf(γ^b, S_{i−1}, ΔS_i) over chunks, then
 * every chunk's outputs from its entering state (all chunks in parallel).
 * Arguments as ret_chunkwise; the workspace holds one d_k×d_v fp32 state per
 * (b, h, chunk) (ret_chunkwise_scan_plan gives its size).  On both kernel
 * paths the two layouts run the same tile arithmetic in the same order, so
 * state_out and out are bit-identical to ret_chunkwise's.
 * ------------------------------------------------------------------------ */
ret_status ret_chunkwise_scan(const void* q, const void* k, const void* v, ret_dtype in_dt,
                              const float* gamma, const float* theta,
                              int B, int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                              const float* state_in, float* state_out,
                              void* out, ret_dtype out_dt, const ret_gn* gn,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);

ret_status ret_chunkwise_scan_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                                   int d_k, int d_v, int chunk, ret_dtype out_dt,
                                   int gn_enabled, int* path, size_t* workspace_bytes);

/* ------------------------------------------------------------------------
 * ret_chunkwise_backward — gradients of ret_chunkwise (without the GroupNorm
 * epilogue) with respect to q, k, v and state_in, given the gradient d_out
 * of out and d_state_out of state_out.  Per head, with the decay mask A,
 * ξ_t = γ^{t+1}, w_m = γ^{L−1−m} and G = (dO Vᵀ) ⊙ A (the chain rule applied
 * to the parallel form with state terms, «从RoPE到Retention…» §4.1):
 *   dQ′ = G K′ + ξ ⊙ (dO S_inᵀ)          dV = (Q′K′ᵀ ⊙ A)ᵀ dO + (w ⊙ K′) dS_out
 *   dK′ = Gᵀ Q′ + (w ⊙ V) dS_outᵀ         dS_in = (ξ ⊙ Q′)ᵀ dO + γ^L dS_out
 *   dq = R(−nθ) dQ′,  dk = d_k^{-1/2} R(−nθ) dK′    (the Θ prologue's adjoint)
 * Computed as three chunkwise evaluations: dQ′ in order, dK′ and dV as
 * anti-causal ones (sums over t ≥ m).  Paths: bf16 inputs with chunk = 128,
 * d_k ∈ {128, 256}, d_v a multiple of 128 and every γ^255 ≥ 2^-100 run
 * the evaluations on the tensor-core chunk kernels (bf16 operands, fp32
 * accumulation; the anti-causal ones walk the chunks from the last; the two
 * evaluations that contract over d_v run as sums of pieces of at most 256
 * columns, the pieces held in grad_dt and summed in fp32); everything else
 * runs on the fp32 kernels over the reversed
 * sequence, with `chunk` as the chunk length (any ≥ 1).
 * q, k, v, d_out: DEVICE, in_dt, layouts as above.  dq, dk [B, H, L, d_k]
 * and dv [B, H, L, d_v]: DEVICE, grad_dt; they must not alias any input.
 * state_in, d_state_out: DEVICE fp32 [B, H, d_k, d_v] or NULL (zero).
 * d_state_in: DEVICE fp32 or NULL (not computed); it may alias state_in or
 * d_state_out.  workspace: DEVICE, at least ret_chunkwise_backward_plan's
 * bytes (never 0).  B·H > 65535 or a γ_h below 2^-64 (the reversed
 * evaluations start from dS_out/γ) is RET_EUNSUPPORTED.  Validation and errors as for the other entry points.
 * ------------------------------------------------------------------------ */
ret_status ret_chunkwise_backward(const void* q, const void* k, const void* v, const void* d_out,
                                  ret_dtype in_dt, const float* gamma, const float* theta,
                                  int B, int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                                  const float* state_in, const float* d_state_out,
                                  void* dq, void* dk, void* dv, ret_dtype grad_dt,
                                  float* d_state_in, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/* Path and workspace bytes of ret_chunkwise_backward.  gamma may be NULL
 * (then the tensor-core path is assumed allowed). */
ret_status ret_chunkwise_backward_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                                       int d_k, int d_v, int chunk, int* path,
                                       size_t* workspace_bytes);

/* ------------------------------------------------------------------------
 * ret_chunkwise_param_grads — gradients of ret_chunkwise (without the
 * GroupNorm epilogue) with respect to the decay rates γ [H] and the rotation
 * frequencies θ [d_k/2] («从RoPE到Retention…» §2 makes θ learnable; §3 sets
 * γ per head), for the upstream gradients d_out and d_state_out.  Both are
 * sums over (query, key) pairs of the terms of <dO, out> + <dS_out, S_out>
 * weighted by the derivative of their decay γ^{n−m} (n − m)·γ^{n−m−1} or of
 * their rotation angle (m − n)·θ (§3, §4.1, §2), plus the state terms.  The
 * call evaluates them split at 128-token chunk boundaries, so that no weight
 * exceeds the chunk length except the genuine absolute-position weights of
 * the state terms (κ = 63.5, j the index inside a chunk, S_c / dS_c the state
 * after chunk c and its gradient, r the last chunk's length, J(a, b) =
 * (−b, a) on each rotation pair, Z_c = Σ_v S_c[2i+1]dS_c[2i] − S_c[2i]dS_c[2i+1]):
 *   γ·dγ = Σ_t (j−κ)(dO_t·o_t − v_t·dv_t) + (1+κ)<S_in, dS_in>
 *          + (r−1−κ)<S_out, dS_out> + 128·Σ_{interior c} <S_c, dS_c>
 *   dθ_i = Σ_t (j−κ)(dq_t·J q_t + dk_t·J k_t)_i + (pos0+κ)Z_{−1}
 *          − (pos0+L−r+κ)Z_{C−1} + 128·Σ_{interior c} Z_c
 * The row sums read the forward call's out and the backward call's dq, dk,
 * dv for the same inputs, upstream gradients and pos0; the states are
 * recomputed from q, k, v, d_out by two sequential walks over the chunks
 * with fp32 states: on the tensor cores for bf16 inputs with d_k and d_v
 * multiples of 128 (the rotated, decay-weighted q and k rows as bf16 hi +
 * lo parts, 16 significant bits), else in fp32 FMA (64 × 64 state tiles).
 * ret_force_path(RET_PATH_SIMT) selects the fp32 walks.
 * q, k, v, d_out: DEVICE, in_dt, [B, H, L, d_k|d_v].  out: DEVICE, out_dt,
 * [B, H, L, d_v] (the forward output before any GroupNorm; dγ only).  dq,
 * dk (dθ only), dv (dγ only): DEVICE, grad_dt.  state_in, d_state_out:
 * DEVICE fp32 [B, H, d_k, d_v] or NULL (zero).  gamma [H] in (0, 1], theta
 * [d_k/2]: HOST, read during the call.  d_gamma [H], d_theta [d_k/2]: DEVICE
 * fp32 outputs, overwritten; either may be NULL (not computed), not both.
 * workspace: DEVICE, at least ret_chunkwise_param_grads_plan's bytes
 * (B·H·⌈L/128⌉·d_k·d_v·4 bytes for the states, plus small terms).
 * Deterministic: fixed-order sums.  Validation and errors as for the other
 * entry points.
 * ------------------------------------------------------------------------ */
ret_status ret_chunkwise_param_grads(const void* q, const void* k, const void* v,
                                     const void* d_out, ret_dtype in_dt, const void* out,
                                     ret_dtype out_dt, const void* dq, const void* dk,
                                     const void* dv, ret_dtype grad_dt, const float* gamma,
                                     const float* theta, int B, int H, int L, int d_k, int d_v,
                                     int64_t pos0, const float* state_in,
                                     const float* d_state_out, float* d_gamma, float* d_theta,
                                     void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream);

/* Workspace bytes of ret_chunkwise_param_grads. */
ret_status ret_chunkwise_param_grads_plan(int B, int H, int L, int d_k, int d_v,
                                          size_t* workspace_bytes);

/* ------------------------------------------------------------------------
 * ret_groupnorm — the per-head GroupNorm epilogue as a call of its own
 * («从RoPE到Retention…» §5): each (b, h, t) row of x [B, H, L, d_v] is
 * normalised over its d_v channels (biased variance, gn->eps), then scaled
 * and shifted by gn->weight / gn->bias [H, d_v] (DEVICE fp32, 16-byte
 * aligned, each may be NULL).  gn->enabled is ignored.  x: DEVICE, x_dt; y: DEVICE, y_dt; both
 * 16-byte aligned; y may be x when the types agree.  With ret_groupnorm_backward it gives the
 * training path: forward ret_chunkwise without GroupNorm, then this call.
 * ------------------------------------------------------------------------ */
ret_status ret_groupnorm(const void* x, ret_dtype x_dt, void* y, ret_dtype y_dt, int B, int H,
                         int L, int d_v, const ret_gn* gn, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * ret_groupnorm_backward — gradients of ret_groupnorm for the upstream
 * gradient d_y: with x̂ = (x − μ)·rstd and g = d_y ⊙ weight per row,
 *   d_x = rstd·(g − mean(g) − x̂·mean(g ⊙ x̂)),
 *   d_weight = Σ_{b,t} d_y ⊙ x̂,   d_bias = Σ_{b,t} d_y   ([H, d_v]).
 * x (the GroupNorm input), d_y: DEVICE, x_dt, [B, H, L, d_v], 16-byte
 * aligned.  weight: DEVICE fp32 [H, d_v] or NULL (ones).  d_x: DEVICE,
 * grad_dt, must not alias x or d_y.  d_weight, d_bias: DEVICE fp32 [H, d_v]
 * or NULL (not computed); when either is wanted the workspace must hold
 * ret_groupnorm_backward_plan's bytes (else it may be NULL).  Sums are in a
 * fixed order (deterministic).
 * ------------------------------------------------------------------------ */
ret_status ret_groupnorm_backward(const void* x, const void* d_y, ret_dtype x_dt,
                                  const float* weight, float eps, int B, int H, int L, int d_v,
                                  void* d_x, ret_dtype grad_dt, float* d_weight, float* d_bias,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes of ret_groupnorm_backward (for d_weight / d_bias). */
ret_status ret_groupnorm_backward_plan(int B, int H, int L, int d_v, size_t* workspace_bytes);

/* ------------------------------------------------------------------------
 * ret_parallel — parallel form O = (Q′K′ᵀ ⊙ D) V + γ^{t+1} q′_t S_in
 * («从RoPE到Retention…» §4.1; RetNet 保留网络 explainer, 并行表征).
 * O(L²) work.  state_out (optional) is the closed-form final state.
 * ------------------------------------------------------------------------ */
ret_status ret_parallel(const void* q, const void* k, const void* v, ret_dtype in_dt,
                        const float* gamma, const float* theta,
                        int B, int H, int L, int d_k, int d_v, int64_t pos0,
                        const float* state_in, float* state_out,
                        void* out, ret_dtype out_dt, const ret_gn* gn,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

ret_status ret_parallel_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                             int d_k, int d_v, ret_dtype out_dt, int gn_enabled,
                             int state_out_wanted, int* path, size_t* workspace_bytes);

/* ------------------------------------------------------------------------
 * ret_step — one recurrent decode step at absolute position `pos`
 * («从RoPE到Retention…» §4.2: S_n = γS_{n−1} + K_nᵀV_n, output Q_nS_n with
 * the updated state).  q, k: [B, H, d_k]; v, out: [B, H, d_v];
 * state: [B, H, d_k, d_v] fp32, updated in place.  No workspace.
 * ------------------------------------------------------------------------ */
ret_status ret_step(const void* q, const void* k, const void* v, ret_dtype in_dt,
                    const float* gamma, const float* theta,
                    int B, int H, int d_k, int d_v, int64_t pos,
                    float* state, void* out, ret_dtype out_dt, const ret_gn* gn,
                    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * ret_rotate — the Θ prologue alone: y_t = scale·R((pos0+t)θ) x_t for
 * x, y: [B, H, L, d] («从RoPE到Retention…» §2 theta_shift).  Exposed for
 * testing the prologue that the other calls fuse or run in front.
 * ------------------------------------------------------------------------ */
ret_status ret_rotate(const void* x, ret_dtype in_dt, const float* theta,
                      int B, int H, int L, int d, int64_t pos0, float scale,
                      void* y, ret_dtype out_dt, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * ret_decay_row_norm — the row-normalised decay variant («从RoPE到Retention…»
 * §5: the decay weights normalised per row), applied in place to `out` of a
 * plain call (ret_chunkwise / ret_parallel without GroupNorm, or ret_step
 * with L = 1 and pos0 = its pos).  Row N of the decay mask covers positions
 * 0..N (the state term standing for the positions before pos0); divided by
 * its sum r_N = Σ_{i=0}^{N} γ^i it divides output row N by r_N, so
 *   out[b][h][t][:] /= r_{pos0+t},  r_N = (1 − γ_h^{N+1}) / (1 − γ_h).
 * The pages' "global scaling" has no stated value and is 1.  A GroupNorm
 * after the variant cancels it up to eps (GroupNorm is invariant to a
 * positive per-token scale), so the variant is meant for outputs without
 * GroupNorm.  out: DEVICE [B, H, L, d_v] in out_dt; gamma: HOST [H].
 * 0 < γ_h ≤ 1, else RET_EINVAL.  The state is not affected.
 * ------------------------------------------------------------------------ */
ret_status ret_decay_row_norm(void* out, ret_dtype out_dt, const float* gamma, int B, int H,
                              int L, int d_v, int64_t pos0, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * ret_matmul — C = A·W on the tensor cores (the projection GEMM of
 * ret_msr_block, exposed on its own).  A: DEVICE [M][K] bf16, W: DEVICE [K][N]
 * bf16, both row-major; C: DEVICE [M][N] in c_dt (bf16 rounded to nearest, or
 * fp32); fp32 accumulation.  N a multiple of 256 and K of 64, else
 * RET_EUNSUPPORTED; any M ≥ 1.  Tiles of 256 × 256 on CTA pairs
 * (tcgen05.mma.cta_group::2), operands staged by TMA.
 * ------------------------------------------------------------------------ */
ret_status ret_matmul(const void* a, const void* w, void* c, ret_dtype c_dt, int M, int N, int K,
                      cudaStream_t stream);

/* ------------------------------------------------------------------------
 * ret_msr_block — the multi-scale retention block around the core:
 *   q = x·W_Q, k = x·W_K, v = x·W_V per head (the SimpleRetention of
 *   «RetNet：Transformer的革命性继任者？»: one projection per head, the heads
 *   side by side), o = the chunkwise retention of q, k, v (with the Θ
 *   prologue, state_in / state_out as ret_chunkwise), per-head GroupNorm of
 *   o («从RoPE到Retention…» §5), then the gate and output projection of the
 *   published MSR definition, which the pages do not spell out:
 *   z = (swish(x·W_G) ⊙ concat_h GN(o_h))·W_O, swish(u) = u·σ(u).
 * x: DEVICE [B][L][D] bf16.  w_q, w_k: [D][H·d_k]; w_v, w_g: [D][H·d_v];
 * w_o: [H·d_v][D_out]; all DEVICE bf16 row-major (column h·d + c belongs to
 * head h).  z: DEVICE [B][L][D_out] in z_dt.  gamma, theta: HOST as for
 * ret_chunkwise.  GroupNorm: eps = gn_eps > 0, no affine terms.
 * The q and k projections' epilogues write the chunk kernels' rotated,
 * decay-folded operands directly (no separate Θ pass); v goes to the head
 * layout; the chunkwise core runs on the tensor cores (its shape rules:
 * bf16, d_k ∈ {64, 128, 256}, d_v = 64 or a multiple of 128, every
 * γ^127 ≥ 2^-60), and D a multiple of 64, H·d_k, H·d_v and D_out multiples
 * of 256; anything else is RET_EUNSUPPORTED.  workspace: DEVICE, at least
 * ret_msr_block_plan's bytes (the projected operands, the fp32 core output,
 * the gate and the gated, normalised rows: 1.6 GB at B2 L8192 D4096 H16
 * d_k256 d_v512).
 * ------------------------------------------------------------------------ */
ret_status ret_msr_block(const void* x, const void* w_q, const void* w_k, const void* w_v,
                         const void* w_g, const void* w_o, const float* gamma, const float* theta,
                         int B, int L, int D, int H, int d_k, int d_v, int D_out, int64_t pos0,
                         const float* state_in, float* state_out, void* z, ret_dtype z_dt,
                         float gn_eps, void* workspace, size_t workspace_bytes, cudaStream_t stream);

ret_status ret_msr_block_plan(const float* gamma, int B, int L, int D, int H, int d_k, int d_v,
                              int D_out, size_t* workspace_bytes);

/* Synchronise `stream`, then return and clear the device status word:
 * RET_ETIMEOUT if a kernel's bounded wait expired since the last call,
 * RET_ECUDA on a CUDA error, else RET_OK. */
ret_status ret_sync_status(cudaStream_t stream);

/* Launch a one-block kernel that waits on a barrier nothing will complete,
 * with a wait budget of `budget_us` microseconds (1 … 2,000,000); it must
 * give up, record RET_ETIMEOUT and exit.  Tests the failure path on a GPU
 * without faulting it. */
ret_status ret_selftest_timeout(int budget_us, cudaStream_t stream);

/* Profiling hook.  ret_profile_begin arms it with `n_events` caller-created
 * CUDA events; every later kernel launch of the library records events
 * [2i] and [2i+1] on the call's stream just before and after its i-th
 * launch (while 2i+1 < n_events).  ret_profile_end disarms it and returns the
 * number of kernels recorded; ret_profile_kernel(i) names the i-th one.
 * Process-wide and not thread-safe: for benchmarks. */
ret_status ret_profile_begin(cudaEvent_t* events, int n_events);
int ret_profile_end(void);
const char* ret_profile_kernel(int i);

/* Force every later call in this process onto one path (RET_PATH_SIMT),
 * onto the tensor-core path without CTA pairs (RET_PATH_TC_SINGLE), or back
 * to automatic selection (0).  For cross-checks between paths.  Plans still
 * report RET_PATH_TC for both tensor-core variants. */
ret_status ret_force_path(int path);

const char* ret_status_string(ret_status s);
int ret_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RETENTION_H */
