// Internal launchers behind the C ABI (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Limit of each pipeline wait inside the tensor-core kernels, in nanoseconds (the
// library-wide setting of moe_set_wait_limit_ns; read at every launch).
uint64_t pipeline_wait_ns();

// Sizes of one grouped GEMM launch.
struct GemmShape {
  int E, H, F;                  // F: expert FFN size (Fs for the shared expert)
  int64_t rows;                 // rows of the row-indexed operands (R, or T for the dense segment)
  int dense_rows;               // > 0: one dense segment of this many rows (the shared expert)
  int max_mtiles;               // host-known upper bound on M tiles (grid sizing)
  const int32_t* offsets;       // [E+1] (device)
  const int32_t* tile_offsets;  // [E+1] (device)
  const int32_t* counts;        // [E] (device)
  int nsm;
};

// An FP8 E4M3 operand: values and their UE8M0 block scales.
struct Fp8Op {
  const uint8_t* q;
  const uint8_t* sc;
};

// Workspace pieces of the router forward on the tensor cores.
struct RouterFwdScratch {
  uint16_t* wsplit;  // [3*Ep, H] bf16 split of W_r (row blocks hi, mid, lo)
  float* part;       // [max_splits-1, T, E] K-split partial logits
  int max_splits;
  int* err;          // device error word
};

// Workspace pieces of the router backward.
struct RouterBwdScratch {
  float* dl;          // [T,E] fp32 dlogits
  float* part;        // [splits,E,H] partial dW_r (token splits)
  int splits;
  uint16_t* dl_rows;  // E > 32: [3*Tp, Ep] bf16 split of dl (row blocks hi, mid, lo)
  uint16_t* dl_cols;  // E > 32: [T, 3*Ep] bf16 split of dl (column blocks hi, hi, mid)
  uint16_t* wb;       // E > 32: [3*Ep, H] bf16 split of W_r (row blocks hi, mid, hi)
  int Tp, Ep;
};

cudaError_t launch_router_topk(const moe_config& c, const uint16_t* X, const float* Wr, const float* logit_bias,
                               const float* sel_bias, float* logits, float* scores, int32_t* topk_idx, float* gates,
                               int32_t* counts, cudaStream_t st, int nsm, const int32_t* given = nullptr,
                               const RouterFwdScratch* w = nullptr);
// P = X W_r^T on the tensor cores from wsplit = [3*Ep,H] bf16 (row blocks hi, mid, lo of
// W_r), split over K: split 0 into P0, split s > 0 into Pn + (s-1)*T*E; the routing pass
// adds them in that order.  router_tc_splits: how many splits (1..max_splits).
int router_tc_splits(int T, int H, int E, int nsm, int max_splits);
cudaError_t launch_router_logits_tc(int T, int H, int E, int Ep, const uint16_t* X, const uint16_t* wsplit, float* P0,
                                    float* Pn, int splits, int* err, cudaStream_t st);
cudaError_t launch_router_bwd(const moe_config& c, const uint16_t* X, const float* Wr, const float* logits,
                              const int32_t* topk_idx, const float* gates, const float* dgates, float* dW_r,
                              float* dlogit_bias, float* dX_router, const RouterBwdScratch& w, int* err, int nsm,
                              cudaStream_t st);
// cap: per-expert capacity (INT_MAX = dropless); kept [E] (required) receives the rows
// each expert keeps, min(histogram total, cap), and sizes the padding; priority [T,k]
// (nullable): drop the lowest-priority assignments instead of the last ones in token
// order, which needs drop_order [T*k] and drop_start [E+1].
cudaError_t launch_permute(const moe_config& c, const uint16_t* X, const int32_t* topk_idx, const int32_t* counts,
                           int cap, const float* priority, int32_t* kept, int32_t* offsets, int32_t* tile_offsets,
                           int32_t* row_id_map, int32_t* slot_src, uint16_t* Xperm, int32_t* chunk_counts,
                           int32_t* chunk_base, int32_t* drop_order, int32_t* drop_start, int* err, int nsm,
                           cudaStream_t st);
cudaError_t launch_combine(const moe_config& c, const uint16_t* Yperm, const int32_t* row_id_map, const float* gates,
                           const uint16_t* Ysh, uint16_t* Y, cudaStream_t st);
cudaError_t launch_combine_bwd(const moe_config& c, const uint16_t* dY, const uint16_t* Yperm,
                               const int32_t* row_id_map, const float* gates, const int32_t* offsets,
                               const int32_t* counts, uint16_t* dYperm, float* dgates, cudaStream_t st);
cudaError_t launch_dgates_reduce(const moe_config& c, const int32_t* row_id_map, const float* part, int ntile,
                                 float* dgates, int nsm, cudaStream_t st);
cudaError_t launch_permute_bwd(const moe_config& c, const uint16_t* dXperm, const int32_t* row_id_map,
                               const float* dXr, const uint16_t* dXs, uint16_t* dX, cudaStream_t st);

// The memory-efficient (gated) path: row r of the permuted buffers carries gate
// gates[slot_src[r]] (0 for padding rows).  FC1's epilogue then writes the gated
// activation gate * silu(g) * u; FC2-dgrad's epilogue takes the gradient of the gated
// activation, recomputes a = silu(g) * u from GU, writes gate * a to a_out [rows, F]
// (for FC2's wgrad) and per-tile partials of the gate gradient to dg_part
// [rows, F / tile width].
struct Gating {
  const int32_t* slot_src;
  const float* gates;
  float* dg_part;
  uint16_t* a_out;
};

// Gathered rows (no permuted copy of X): permuted row r of FC1's input is token
// slot_src[r] / k of X [src_rows, H], or zeros for a padding row (slot_src[r] < 0).
struct RowGather {
  const int32_t* slot_src;
  int k;
  int64_t src_rows;
};

cudaError_t launch_fc1_fwd(const GemmShape& s, const uint16_t* X1, const uint16_t* W13, uint16_t* GU, uint16_t* Aact,
                           int* err, cudaStream_t st, const Gating* gate = nullptr,
                           const RowGather* gather = nullptr);
cudaError_t launch_fc2_fwd(const GemmShape& s, const uint16_t* Aact, const uint16_t* W2, uint16_t* Y, int* err,
                           cudaStream_t st);
cudaError_t launch_fc2_dgrad(const GemmShape& s, const uint16_t* dYp, const uint16_t* W2, const uint16_t* GU,
                             uint16_t* dGU, int* err, cudaStream_t st, const Gating* gate = nullptr);
// columns of one FC2-dgrad tile (the dg_part row length is F / this)
int fc2_dgrad_tile_n(int F);
cudaError_t launch_fc1_dgrad(const GemmShape& s, const uint16_t* dGU, const uint16_t* W13, uint16_t* dX1, int* err,
                             cudaStream_t st);
cudaError_t launch_fc2_wgrad(const GemmShape& s, const uint16_t* dYp, const uint16_t* Aact, uint16_t* dW2, int* err,
                             cudaStream_t st);
cudaError_t launch_fc1_wgrad(const GemmShape& s, const uint16_t* dGU, const uint16_t* X1, uint16_t* dW13, int* err,
                             cudaStream_t st, const RowGather* gather = nullptr);

cudaError_t launch_fc1_fwd_fp8(const GemmShape& s, const Fp8Op& X1, const Fp8Op& W13, uint16_t* GU, uint16_t* Aact,
                               int* err, cudaStream_t st);
cudaError_t launch_fc2_fwd_fp8(const GemmShape& s, const Fp8Op& A1, const Fp8Op& W2, uint16_t* Y, int* err,
                               cudaStream_t st);
cudaError_t launch_fc2_dgrad_fp8(const GemmShape& s, const Fp8Op& dY1, const Fp8Op& W2, const uint16_t* GU,
                                 uint16_t* dGU, int* err, cudaStream_t st);
cudaError_t launch_fc1_dgrad_fp8(const GemmShape& s, const Fp8Op& dGU1, const Fp8Op& W13, uint16_t* dX1, int* err,
                                 cudaStream_t st);
cudaError_t launch_fc2_wgrad_fp8(const GemmShape& s, const Fp8Op& dYc, const Fp8Op& Ac, uint16_t* dW2, int* err,
                                 cudaStream_t st);
cudaError_t launch_fc1_wgrad_fp8(const GemmShape& s, const Fp8Op& dGUc, const Fp8Op& Xc, uint16_t* dW13, int* err,
                                 cudaStream_t st);
cudaError_t launch_quant_rows(const uint16_t* X, int64_t rows, int K, const int32_t* rows_valid, uint8_t* q,
                              uint8_t* sc, int nsm, cudaStream_t st);
cudaError_t launch_quant_cols(const uint16_t* X, int64_t rows, int N, const int32_t* rows_valid, uint8_t* q,
                              uint8_t* sc, cudaStream_t st);
cudaError_t launch_quant_weights(const uint16_t* W, int64_t nmat, int rows, int cols, uint8_t* q, uint8_t* sc,
                                 cudaStream_t st);

cudaError_t launch_router_dwr_tc(int T, int Tp, int H, int E, int Ep, const uint16_t* dlsplit, const uint16_t* X,
                                 float* dWr, int splits, int* err, int nsm, cudaStream_t st);
cudaError_t launch_router_dx_tc(int T, int H, int Ep, const uint16_t* dlA, const uint16_t* WB, float* dXr, int* err,
                                int nsm, cudaStream_t st);

}  // namespace moe
