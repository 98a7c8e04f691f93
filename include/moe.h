/* C ABI of the single-GPU dropless top-k mixture-of-experts layer (sm_103a).
 *
 * The layer runs four stages, as laid out in "Scalable Training of
 * Mixture-of-Experts Models with Megatron Core" (summary page, section
 * "Method"): Route (a linear router kept in FP32 with softmax or sigmoid
 * scoring and top-k selection), Dispatch (permute tokens so that each
 * expert's tokens are contiguous), Compute (all experts run as one grouped
 * GEMM) and Combine (gate-weighted unpermute and sum).  The same section names
 * the compute recipes this library follows: grouped GEMM, kernel fusion and
 * sync-free dropless execution that CUDA Graphs can capture.
 *
 * Conventions for every entry point below:
 *  - Pointers marked (device) point to GPU memory; the caller allocates and
 *    owns every buffer, including the workspace.  The library never
 *    allocates, frees or synchronises on these calls.
 *  - bf16 tensors are passed as raw 16-bit patterns (moe_bf16).  All tensors
 *    are dense row-major with the shapes given, and 16-byte aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t, or NULL for the
 *    legacy default stream) and can be captured into a CUDA Graph: no call
 *    reads a device value back to the host.
 *  - Arguments are checked on the host before any launch; a bad argument
 *    returns MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED for a valid but
 *    unsupported shape) and launches nothing.  A launch failure returns
 *    MOE_ERR_CUDA.  Faults found inside kernels (a pipeline wait that ran out
 *    of time, inconsistent routing inputs) set an error word in the
 *    workspace, read by moe_read_device_error().
 *
 * Notation: T tokens, H hidden size, E experts, k experts per token, F expert
 * FFN size, Fs shared-expert FFN size, S = T*k assignments, and R =
 * moe_max_rows() rows in the permuted buffers (S plus per-expert padding).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_CUDA = 4,
  MOE_ERR_TIMEOUT = 5,
  MOE_ERR_DEVICE = 6
} moe_status;

/* Layer configuration (plain data, passed by pointer, read only during the call).
 *  T, H, E, k, F  sizes; H and F must be multiples of 128, 1 <= k <= E <= 256, k <= 32,
 *                 and E a multiple of 8 when E > 32.
 *  F_shared       size of the always-on shared expert (0: none); multiple of 128.
 *  score_fn       0: softmax over the E logits; 1: sigmoid of each logit.
 *  renorm         1: gates renormalised over the k selected experts.
 *  gate_scale     multiplies every gate after renormalisation (e.g. 2.5).
 *  n_group        >1: group-limited routing over n_group contiguous groups of E/n_group experts.
 *  topk_group     groups kept when n_group > 1 (topk_group * E/n_group >= k).
 *  group_score    0: group score = sum of the group's two largest keys; 1: its largest key.
 *  align          row alignment of every expert segment in the permuted buffers:
 *                 128 for the grouped GEMM; 1 is accepted by the routing/permute calls only.
 */
typedef struct {
  int32_t T, H, E, k, F, F_shared;
  int32_t score_fn;
  int32_t renorm;
  float gate_scale;
  int32_t n_group, topk_group, group_score;
  int32_t align;
  int32_t reserved;
} moe_config;

/* Short text for a status code (static storage). */
const char* moe_status_string(moe_status s);

/* R: rows of every permuted buffer (Xperm, GU, A, Yperm, dYperm, dGU, dXperm)
 * and entries of slot_src: T*k + E*(align-1).  Rows from offsets[E] to R are never written. */
moe_status moe_max_rows(const moe_config* cfg, int64_t* R);

/* Bytes of device workspace all calls of this configuration need.  The
 * workspace holds the device error word, per-chunk routing histograms, the router
 * forward's bf16 split of W_r and K-split partial logits, and the router-gradient
 * scratch.  Initialise it once with moe_workspace_init(). */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Zeroes the workspace (including the error word), asynchronously on stream. */
moe_status moe_workspace_init(const moe_config* cfg, void* ws, void* stream);

/* Synchronises `stream`, then returns the device error word (0 = none; else a
 * moe_status value) and clears it.  Not for use inside a graph capture. */
moe_status moe_read_device_error(void* ws, int32_t* err, void* stream);

/* Limit of every pipeline wait inside the tensor-core kernels (grouped GEMMs, router
 * projection) and of the one-launch small dispatch's wait for its token rows, in
 * nanoseconds; library-wide, read when each kernel is launched (a
 * captured graph keeps the value of its capture).  Default 4e9 (4 s).  The pages have
 * no counterpart: this is the library's failure detection.  A wait on another part of
 * the kernel's pipeline (a TMA copy landing, the MMAs of a tile, the epilogue freeing an
 * accumulator) that runs out of time sets MOE_ERR_TIMEOUT in the device error word
 * (moe_read_device_error) and the kernel unwinds: each CTA waits, with a fixed 4 s
 * bound, for the copies and MMAs it already issued (the two CTAs of a pair settle the
 * loads each of them issued), frees its tensor memory and exits, so the context stays
 * usable and the next call runs normally.  A limit of 0 makes every pipeline wait a
 * single non-blocking test, so that nearly every launch runs out: meant for testing the
 * unwind path, the outputs of such a launch are undefined.  Not thread-safe against
 * concurrent launches that expect another value. */
void moe_set_wait_limit_ns(uint64_t ns);
uint64_t moe_get_wait_limit_ns(void);

/* Route.  ("Method": the router is a learned linear projection, optionally kept
 * in FP32, followed by softmax or sigmoid scoring and top-k selection.)
 *  X        [T,H] bf16 (device)      tokens
 *  W_r      [E,H] fp32 (device)      router weight
 *  logit_bias [E] fp32 (device, nullable)  added to the logits (enters gates and gradients)
 *  sel_bias [E] fp32 (device, nullable)    added to the selection key only
 *  logits   [T,E] fp32 out           X W_r^T + logit_bias, FP32 accumulation
 *  scores   [T,E] fp32 out           softmax(logits) or sigmoid(logits)
 *  topk_idx [T,k] int32 out          selected experts in descending key order,
 *                                    key = logit + sel_bias (softmax) or score + sel_bias (sigmoid),
 *                                    exact ties to the lower expert index
 *  gates    [T,k] fp32 out           combine weights (renormalised, times gate_scale)
 *  counts   [E] int32 out            tokens per expert
 *  ws       workspace (moe_workspace_size) or NULL.  It holds the bf16 split of W_r that
 *           the tensor-core projection reads, the partial sums of its K splits, and the
 *           error word its bounded waits report to (MOE_ERR_TIMEOUT, read by
 *           moe_read_device_error).  With NULL the projection runs on the CUDA cores
 *           instead (FP32 FMA; one fused launch for E <= 32; same selection rule and
 *           bounds). */
moe_status moe_router_topk(const moe_config* cfg, const moe_bf16* X, const float* W_r,
                           const float* logit_bias, const float* sel_bias, float* logits, float* scores,
                           int32_t* topk_idx, float* gates, int32_t* counts, void* ws, void* stream);

/* Router replay.  (Summary page, "Key claims": router replay for reinforcement-learning
 * training, i.e. reusing routing decisions taken elsewhere.)  Same as moe_router_topk
 * except that the selection is an input: topk_in [T,k] int32 (device) lists, per token, k
 * distinct experts in [0,E) (not checked on the device; an id outside [0,E) is read as 0).
 * logits and scores are computed as usual; gates are those of the given selection (renorm
 * and gate_scale applied the same way); topk_idx receives a copy of topk_in; counts is the
 * histogram of topk_in.  No group limit or selection bias is applied. */
moe_status moe_router_replay(const moe_config* cfg, const moe_bf16* X, const float* W_r, const float* logit_bias,
                             const int32_t* topk_in, float* logits, float* scores, int32_t* topk_idx, float* gates,
                             int32_t* counts, void* ws, void* stream);

/* Dispatch.  ("Method": the dispatcher permutes tokens so that the tokens of
 * one expert are contiguous, as the grouped GEMM needs; dropless, no capacity.)
 *  X            [T,H] bf16 (device)
 *  topk_idx     [T,k] int32 (device), counts [E] int32 (device): from moe_router_topk
 *  offsets      [E+1] int32 out   segment starts; offsets[e+1]-offsets[e] = counts[e] rounded up to align
 *  tile_offsets [E+1] int32 out   prefix sums of ceil(counts[e]/128) (the grouped GEMM's M-tile schedule)
 *  row_id_map   [T,k] int32 out   permuted row of assignment (t,j); tokens keep their order within an expert
 *  slot_src     [R] int32 out     inverse map: row -> t*k+j, or -1 for a padding row
 *  Xperm        [R,H] bf16 out    permuted tokens; padding rows are zero.  NULL: the maps only
 *                                 (for moe_grouped_swiglu_mlp_gather); X may then be NULL too */
moe_status moe_permute(const moe_config* cfg, const moe_bf16* X, const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map, int32_t* slot_src,
                       moe_bf16* Xperm, void* ws, void* stream);

/* Dispatch with capacity-controlled token dropping.  (Summary page, "Results": listed
 * among the production features; the pages give no policy.)
 * Two policies; kept gates are never renormalised:
 *  - priority == NULL: each expert keeps its first `capacity` assignments in token order
 *    (t-major, then j) and drops the rest, as a fixed-capacity dispatch does;
 *  - priority [T,k] fp32 (device): an expert with more than `capacity` assignments keeps
 *    the `capacity` of largest priority (pass the gates to drop the least-weighted ones);
 *    equal priorities go to the earlier assignment in token order; -0 equals +0.
 * Either way the kept assignments take their rows in token order.
 * Arguments as moe_permute, plus:
 *  capacity     int32 >= 0        slots per expert (e.g. ceil(capacity_factor * T * k / E));
 *                                 a negative value is MOE_ERR_INVALID_ARG
 *  priority     [T,k] fp32 (device, nullable), see above
 *  kept_counts  [E] int32 out     min(counts[e], capacity)
 * offsets and tile_offsets are built from kept_counts; row_id_map is -1 for a dropped
 * assignment.  Pass kept_counts wherever a later call asks for counts (the grouped GEMMs'
 * backward and moe_unpermute_combine_bwd).  Combine, combine backward and permute backward
 * skip row -1, so a dropped assignment adds nothing to Y, gets dgates 0 and passes no
 * gradient to X.  capacity >= max(counts) gives exactly moe_permute's results. */
moe_status moe_permute_capacity(const moe_config* cfg, const moe_bf16* X, const int32_t* topk_idx,
                                const int32_t* counts, int32_t capacity, const float* priority,
                                int32_t* kept_counts, int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map,
                                int32_t* slot_src, moe_bf16* Xperm, void* ws, void* stream);

/* Compute: all experts' SwiGLU MLPs in two grouped GEMM launches.  ("Method":
 * all local experts run in one grouped GEMM call; SwiGLU is the GLU variant of
 * "GLU Variants Improve Transformer", cited on the index page.)
 *  Xperm   [R,H] bf16 (device)       offsets, tile_offsets: from moe_permute
 *  W13     [E,2F,H] bf16 (device)    rows 0..F-1 = W_gate, rows F..2F-1 = W_up
 *  W2      [E,H,F] bf16 (device)     W_down
 *  GU      [R,2F] bf16 out           pre-activations [g | u] (saved for backward)
 *  A       [R,F] bf16 out            silu(g) * u, formed from the FP32 accumulators
 *  Yperm   [R,H] bf16 out            expert outputs
 * Shared expert (only when F_shared > 0; all six pointers must then be non-null):
 *  X [T,H] bf16, W13_s [2Fs,H], W2_s [H,Fs] (device); GU_s [T,2Fs], A_s [T,Fs], Yshared [T,H] out. */
moe_status moe_grouped_swiglu_mlp(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                  const int32_t* tile_offsets, const moe_bf16* W13, const moe_bf16* W2,
                                  moe_bf16* GU, moe_bf16* A, moe_bf16* Yperm, const moe_bf16* X,
                                  const moe_bf16* W13_s, const moe_bf16* W2_s, moe_bf16* GU_s, moe_bf16* A_s,
                                  moe_bf16* Yshared, void* ws, void* stream);

/* Gathered-rows expert MLP: the dispatch without a permuted copy of the tokens.  (Summary
 * page, "Method": kernel fusion among the compute recipes; fusing the permutation into
 * the GEMM is a reading.)  FC1 reads row r of each expert segment as token
 * slot_src[r] / k of X [T,H] (zeros for padding rows, slot_src[r] < 0), through TMA
 * four-row gathers, so moe_permute can be called with Xperm = NULL (maps only).
 * Outputs and results are those of moe_grouped_swiglu_mlp on the Xperm that moe_permute
 * would have written.  Requires H % 256 == 0 (else MOE_ERR_UNSUPPORTED).
 *  X [T,H] bf16 (device): the token rows (also the shared expert's input)
 *  slot_src [R] int32 (device): from moe_permute / moe_permute_capacity
 *  other arguments as moe_grouped_swiglu_mlp. */
moe_status moe_grouped_swiglu_mlp_gather(const moe_config* cfg, const moe_bf16* X, const int32_t* slot_src,
                                         const int32_t* offsets, const int32_t* tile_offsets, const moe_bf16* W13,
                                         const moe_bf16* W2, moe_bf16* GU, moe_bf16* A, moe_bf16* Yperm,
                                         const moe_bf16* W13_s, const moe_bf16* W2_s, moe_bf16* GU_s,
                                         moe_bf16* A_s, moe_bf16* Yshared, void* ws, void* stream);

/* Backward of moe_grouped_swiglu_mlp_gather: as moe_grouped_swiglu_mlp_bwd, with FC1's
 * weight gradient gathering the token rows of X along K (dW13_e = dGU_e^T X[rows of e]);
 * dXperm is still the permuted input gradient (moe_permute_bwd reduces it into dX). */
moe_status moe_grouped_swiglu_mlp_bwd_gather(const moe_config* cfg, const moe_bf16* X, const int32_t* slot_src,
                                             const int32_t* offsets, const int32_t* tile_offsets,
                                             const int32_t* counts, const moe_bf16* W13, const moe_bf16* W2,
                                             const moe_bf16* GU, const moe_bf16* A, const moe_bf16* dYperm,
                                             moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* dW13, moe_bf16* dW2,
                                             const moe_bf16* dY, const moe_bf16* W13_s, const moe_bf16* W2_s,
                                             const moe_bf16* GU_s, const moe_bf16* A_s, moe_bf16* dGU_s,
                                             moe_bf16* dX_shared, moe_bf16* dW13_s, moe_bf16* dW2_s, void* ws,
                                             void* stream);

/* Memory-efficient expert MLP (gated rows).  (Summary page, "Method": memory-efficient
 * permutation and fine-grained activation recomputation are named among the memory
 * recipes; the pages give no mechanism, so this is a reading.)  The gate of permuted row r,
 * gates[slot_src[r]] (0 for padding rows), is applied to the activation before FC2:
 *  A  [R,F] bf16 out       gate * silu(g) * u
 *  Yperm [R,H] bf16 out    A W2^T, i.e. the gate-weighted expert outputs: combine them with
 *                          moe_unpermute_combine(gates = NULL).  Yperm is needed by nothing
 *                          in the backward, and A is recomputed there, so neither has to be
 *                          kept between the passes.
 * Other arguments as moe_grouped_swiglu_mlp; slot_src [R] int32 from moe_permute, gates
 * [T,k] fp32 from the router.  The shared expert (gate 1) is computed as there. */
moe_status moe_grouped_swiglu_mlp_gated(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                        const int32_t* tile_offsets, const int32_t* slot_src, const float* gates,
                                        const moe_bf16* W13, const moe_bf16* W2, moe_bf16* GU, moe_bf16* A,
                                        moe_bf16* Yperm, const moe_bf16* X, const moe_bf16* W13_s,
                                        const moe_bf16* W2_s, moe_bf16* GU_s, moe_bf16* A_s, moe_bf16* Yshared,
                                        void* ws, void* stream);

/* Combine.  ("Method": the fourth stage sums each token's gate-weighted expert outputs.)
 *  Y[t] = sum_j gates[t,j] * Yperm[row_id_map[t,j]] (+ Yshared[t]), FP32 sum, one bf16 rounding.
 *  gates NULL: unit weights (rows already gated by moe_grouped_swiglu_mlp_gated).
 *  Yshared [T,H] bf16 (device, nullable);  Y [T,H] bf16 out. */
moe_status moe_unpermute_combine(const moe_config* cfg, const moe_bf16* Yperm, const int32_t* row_id_map,
                                 const float* gates, const moe_bf16* Yshared, moe_bf16* Y, void* stream);

/* Backward of the combine for upstream gradient dY [T,H] bf16:
 *  dYperm[row_id_map[t,j]] = bf16(gates[t,j] * dY[t]); padding rows of dYperm are zeroed
 *    (offsets, counts locate them);
 *  dgates[t,j] = <dY[t], Yperm[row_id_map[t,j]]>, FP32 accumulation.
 *  dYperm [R,H] bf16 out; dgates [T,k] fp32 out.
 *  gates NULL: unit weights; dgates NULL: no gate gradient (Yperm is then not read and may
 *  be NULL).  The gated path passes both as NULL: dYperm rows are copies of dY. */
moe_status moe_unpermute_combine_bwd(const moe_config* cfg, const moe_bf16* dY, const moe_bf16* Yperm,
                                     const int32_t* row_id_map, const float* gates, const int32_t* offsets,
                                     const int32_t* counts, moe_bf16* dYperm, float* dgates, void* stream);

/* Backward of the experts (four grouped GEMM launches, plus four for the shared expert):
 *  dGU    [R,2F] bf16 out   dA = dYperm_e W2_e; dG = dA*u*silu'(g), dU = dA*silu(g) (fused epilogue)
 *  dXperm [R,H] bf16 out    dGU_e W13_e
 *  dW2    [E,H,F] bf16 out  dYperm_e^T A_e   (FP32 accumulation; an expert with no tokens gets 0)
 *  dW13   [E,2F,H] bf16 out dGU_e^T Xperm_e
 * Shared expert (F_shared > 0): X, dY [T,H], W13_s, W2_s, GU_s, A_s (device) in;
 *  dGU_s [T,2Fs], dX_shared [T,H], dW13_s [2Fs,H], dW2_s [H,Fs] bf16 out. */
moe_status moe_grouped_swiglu_mlp_bwd(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                      const int32_t* tile_offsets, const int32_t* counts, const moe_bf16* W13,
                                      const moe_bf16* W2, const moe_bf16* GU, const moe_bf16* A,
                                      const moe_bf16* dYperm, moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* dW13,
                                      moe_bf16* dW2, const moe_bf16* X, const moe_bf16* dY,
                                      const moe_bf16* W13_s, const moe_bf16* W2_s, const moe_bf16* GU_s,
                                      const moe_bf16* A_s, moe_bf16* dGU_s, moe_bf16* dX_shared,
                                      moe_bf16* dW13_s, moe_bf16* dW2_s, void* ws, void* stream);

/* Backward of moe_grouped_swiglu_mlp_gated.  dYperm is the gradient of the gated rows, i.e.
 * moe_unpermute_combine_bwd(gates = NULL, dgates = NULL).  With a = silu(g) * u recomputed from
 * the saved GU and gate = gates[slot_src[r]]:
 *  dA' = dYperm_e W2_e; dgates[t,j] = <dA'[r], a[r]> for r = row_id_map[t,j] (0 if dropped),
 *  summed over the FC2-dgrad tiles in a fixed order; dA = gate * dA', then dG, dU as above;
 *  A      [R,F] bf16 out   gate * a, rewritten here for dW2 (scratch: nothing reads it after)
 *  dW2    = dYperm_e^T A_e; dXperm, dW13 as in moe_grouped_swiglu_mlp_bwd.
 * counts are required; row_id_map [T,k], slot_src [R] from the dispatch; gates [T,k].
 * Shared expert: as in moe_grouped_swiglu_mlp_bwd (its A_s is the saved one). */
moe_status moe_grouped_swiglu_mlp_bwd_gated(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                            const int32_t* tile_offsets, const int32_t* counts,
                                            const int32_t* slot_src, const int32_t* row_id_map, const float* gates,
                                            const moe_bf16* W13, const moe_bf16* W2, const moe_bf16* GU,
                                            const moe_bf16* dYperm, moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* A,
                                            moe_bf16* dW13, moe_bf16* dW2, float* dgates, const moe_bf16* X,
                                            const moe_bf16* dY, const moe_bf16* W13_s, const moe_bf16* W2_s,
                                            const moe_bf16* GU_s, const moe_bf16* A_s, moe_bf16* dGU_s,
                                            moe_bf16* dX_shared, moe_bf16* dW13_s, moe_bf16* dW2_s, void* ws,
                                            void* stream);

/* Backward of the router.  dlogits = exact gradient of the gates w.r.t. the
 * logits for the fixed selection (zero for unselected experts when renorm=1);
 * no gradient flows through the selection or sel_bias.
 *  logits, scores [T,E] fp32, topk_idx [T,k], gates, dgates [T,k] fp32 (device) in
 *  dW_r [E,H] fp32 out = dlogits^T X;  dlogit_bias [E] fp32 out (nullable) = column sums of dlogits;
 *  dX_router [T,H] fp32 out = dlogits W_r.
 * For E > 32 the dW_r and dX_router products run on the tensor cores from exact three-term
 * bf16 splits of dlogits and W_r (FP32 accumulation), E must then be a multiple of 8. */
moe_status moe_router_topk_bwd(const moe_config* cfg, const moe_bf16* X, const float* W_r, const float* logits,
                               const float* scores, const int32_t* topk_idx, const float* gates,
                               const float* dgates, float* dW_r, float* dlogit_bias, float* dX_router, void* ws,
                               void* stream);

/* Backward of the dispatch: dX[t] = sum_j dXperm[row_id_map[t,j]] + dX_router[t] + dX_shared[t],
 * FP32 sum, one bf16 rounding.  dX_router [T,H] fp32 and dX_shared [T,H] bf16 are nullable. */
moe_status moe_permute_bwd(const moe_config* cfg, const moe_bf16* dXperm, const int32_t* row_id_map,
                           const float* dX_router, const moe_bf16* dX_shared, moe_bf16* dX, void* stream);

/* ---------------------------------------------------------------- FP8 E4M3 expert GEMMs
 * ("Abstract" of the index page and "Method" of the summary page: FP8 low-precision
 * training across the expert GEMMs, the router kept in higher precision.)  Every
 * operand of the six expert GEMMs is quantized to E4M3 in blocks of 128 values that
 * share one power-of-two scale (the smallest 2^e with 448*2^e >= the block's max |x|,
 * stored as the UE8M0 byte e+127): activations in 1x128 blocks along each GEMM's K,
 * weights in 128x128 blocks, weight-gradient operands in 128x1 blocks along the tokens.
 * The GEMMs run on the block-scaled FP8 tensor cores with FP32 accumulation; stored
 * tensors (GU, A, Yperm, dGU, dXperm, dW) stay bf16.  The router, gates, permute and
 * combine calls are the bf16 ones above. */

/* Bytes of the FP8 workspace (quantized activations and their scales). */
moe_status moe_fp8_workspace_size(const moe_config* cfg, size_t* bytes);

/* Quantizes the expert weights: W13 [E,2F,H] -> W13q [E,2F,H] e4m3 + W13sc [E,2F/128,H/128]
 * UE8M0; W2 [E,H,F] -> W2q + W2sc [E,H/128,F/128]; the shared expert's likewise
 * (with E = 1) when F_shared > 0.  All pointers device, outputs caller-owned. */
moe_status moe_quantize_weights_fp8(const moe_config* cfg, const moe_bf16* W13, const moe_bf16* W2,
                                    const moe_bf16* W13_s, const moe_bf16* W2_s, uint8_t* W13q, uint8_t* W13sc,
                                    uint8_t* W2q, uint8_t* W2sc, uint8_t* W13q_s, uint8_t* W13sc_s, uint8_t* W2q_s,
                                    uint8_t* W2sc_s, void* stream);

/* moe_grouped_swiglu_mlp with FP8 E4M3 GEMMs: quantized weights from
 * moe_quantize_weights_fp8; activations are quantized on the fly into fp8_ws. */
moe_status moe_grouped_swiglu_mlp_fp8(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                      const int32_t* tile_offsets, const uint8_t* W13q, const uint8_t* W13sc,
                                      const uint8_t* W2q, const uint8_t* W2sc, moe_bf16* GU, moe_bf16* A,
                                      moe_bf16* Yperm, const moe_bf16* X, const uint8_t* W13q_s,
                                      const uint8_t* W13sc_s, const uint8_t* W2q_s, const uint8_t* W2sc_s,
                                      moe_bf16* GU_s, moe_bf16* A_s, moe_bf16* Yshared, void* fp8_ws, void* ws,
                                      void* stream);

/* moe_grouped_swiglu_mlp_bwd with FP8 E4M3 GEMMs (same outputs, bf16). */
moe_status moe_grouped_swiglu_mlp_bwd_fp8(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                          const int32_t* tile_offsets, const int32_t* counts, const uint8_t* W13q,
                                          const uint8_t* W13sc, const uint8_t* W2q, const uint8_t* W2sc,
                                          const moe_bf16* GU, const moe_bf16* A, const moe_bf16* dYperm,
                                          moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* dW13, moe_bf16* dW2,
                                          const moe_bf16* X, const moe_bf16* dY, const uint8_t* W13q_s,
                                          const uint8_t* W13sc_s, const uint8_t* W2q_s, const uint8_t* W2sc_s,
                                          const moe_bf16* GU_s, const moe_bf16* A_s, moe_bf16* dGU_s,
                                          moe_bf16* dX_shared, moe_bf16* dW13_s, moe_bf16* dW2_s, void* fp8_ws,
                                          void* ws, void* stream);

/* Dispatch without a workspace, for callers that cannot allocate device memory.
 * The pages have no counterpart of this call; it exists because moe_permute
 * needs a caller-provided workspace, and some callers cannot provide one: code
 * running inside a memory arena sized once at start-up, a plugin that is handed
 * only its inputs and outputs, or a caller in the middle of recording a CUDA
 * graph (where cudaMalloc is not allowed).
 * Same arguments, outputs and results as moe_permute, minus `ws` (Xperm NULL
 * writes the maps only, as there).  The scratch it needs lives in a static
 * device array built into the library (512 KiB + 1.25 KiB, held by every GPU
 * that loads the library until the process exits), which limits it to
 * ceil(T/128) * E <= 65536 (for example T = 32768 with E = 256); larger
 * configurations return MOE_ERR_WORKSPACE and launch nothing.  Each call clears
 * the part of the array that must start at zero (the error word); the rest is
 * fully rewritten before it is read.
 * The first call on each device looks up the array's device address with
 * that device current, so make the first call on a device before any stream
 * capture.  Every call shares the one array: calls whose kernels can overlap
 * on the GPU (different streams with no ordering between them) race and must
 * not be issued.  Device-side consistency checks of this variant are not
 * reported (there is no workspace error word to read); host-side argument
 * checks are the same as moe_permute's.  Allocates, frees and syncs nothing. */
moe_status moe_permute_noalloc(const moe_config* cfg, const moe_bf16* X, const int32_t* topk_idx,
                               const int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                               int32_t* row_id_map, int32_t* slot_src, moe_bf16* Xperm, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
