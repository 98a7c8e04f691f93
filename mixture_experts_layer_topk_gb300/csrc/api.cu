// The exported C ABI (include/moe.h): host-side argument checks, workspace
// carving and the launches of each stage.  Nothing here allocates, frees or
// synchronises, except moe_read_device_error, which is documented to sync.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "moe_internal.h"

using namespace moe;

namespace {

int num_sms() {
  static std::atomic<int> cache[64];  // per device; 0 = not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// A buffer with a T dimension may be null when T == 0 (an empty batch).
inline bool tok_ok(const moe_config* c, const void* p) { return p != nullptr || c->T == 0; }

moe_status check_cfg(const moe_config* c, bool gemm) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H <= 0 || c->E <= 0 || c->k <= 0 || c->F <= 0 || c->F_shared < 0) return MOE_ERR_INVALID_ARG;
  if (c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->score_fn != 0 && c->score_fn != 1) return MOE_ERR_INVALID_ARG;
  if (c->renorm != 0 && c->renorm != 1) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->gate_scale)) return MOE_ERR_INVALID_ARG;
  if (c->group_score != 0 && c->group_score != 1) return MOE_ERR_INVALID_ARG;
  if (c->align < 1) return MOE_ERR_INVALID_ARG;
  if (c->n_group < 1 || c->E % c->n_group != 0) return MOE_ERR_INVALID_ARG;
  if (c->n_group > 1) {
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
    if ((int64_t)c->topk_group * (c->E / c->n_group) < c->k) return MOE_ERR_INVALID_ARG;
  }
  if (c->E > 256 || c->k > 32 || c->n_group > 32) return MOE_ERR_UNSUPPORTED;
  if (c->E > 32 && c->E % 8 != 0) return MOE_ERR_UNSUPPORTED;  // tensor-core router backward: 32-byte fp32 rows
  if (c->H % 128 != 0 || c->F % 128 != 0 || c->F_shared % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->k + (int64_t)c->E * (c->align - 1) >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->H >= (int64_t)1 << 40) return MOE_ERR_UNSUPPORTED;
  if (gemm && c->align != 128) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int64_t max_rows(const moe_config& c) { return (int64_t)c.T * c.k + (int64_t)c.E * (c.align - 1); }

int* err_word(void* ws, const moe_config& c) { return ws_ptr<int>(ws, ws_layout(c).err); }

GemmShape routed_shape(const moe_config& c, const int32_t* offsets, const int32_t* tile_offsets,
                       const int32_t* counts) {
  GemmShape s;
  s.E = c.E;
  s.H = c.H;
  s.F = c.F;
  s.rows = max_rows(c);
  s.dense_rows = 0;
  s.max_mtiles = (int)(((int64_t)c.T * c.k + 127) / 128 + c.E);
  s.offsets = offsets;
  s.tile_offsets = tile_offsets;
  s.counts = counts;
  s.nsm = num_sms();
  return s;
}

GemmShape shared_shape(const moe_config& c) {
  GemmShape s;
  s.E = 1;
  s.H = c.H;
  s.F = c.F_shared;
  s.rows = c.T;
  s.dense_rows = c.T;
  s.max_mtiles = (c.T + 127) / 128;
  s.offsets = s.tile_offsets = s.counts = nullptr;
  s.nsm = num_sms();
  return s;
}

// FP8 workspace: per operand the E4M3 values and their UE8M0 block scales.
// Routed operands have R rows, the shared expert's T rows.
struct Fp8Buf {
  uint8_t* q;
  uint8_t* sc;
};
struct Fp8Set {  // one expert family (routed or shared)
  Fp8Buf x, a, dy, dgu;      // row blocks (1x128 along K)
  Fp8Buf dyc, ac, dguc, xc;  // token blocks (128x1)
};
struct Fp8Layout {
  Fp8Set routed, shared;
  size_t total;
};

Fp8Layout fp8_layout(const moe_config& c, void* base) {
  Fp8Layout L{};
  char* b = static_cast<char*>(base);
  size_t o = 0;
  auto take = [&](size_t n) {
    char* p = b ? b + o : nullptr;
    o = align256(o + n);
    return reinterpret_cast<uint8_t*>(p);
  };
  auto rows_set = [&](Fp8Set& S, int64_t rows, int64_t H, int64_t F) {
    const int64_t rb = (rows + 127) / 128;
    S.x = {take(rows * H), take(rows * (H / 128))};
    S.a = {take(rows * F), take(rows * (F / 128))};
    S.dy = {take(rows * H), take(rows * (H / 128))};
    S.dgu = {take(rows * 2 * F), take(rows * (2 * F / 128))};
    S.dyc = {take(rows * H), take(rb * H)};
    S.ac = {take(rows * F), take(rb * F)};
    S.dguc = {take(rows * 2 * F), take(rb * 2 * F)};
    S.xc = {take(rows * H), take(rb * H)};
  };
  rows_set(L.routed, max_rows(c), c.H, c.F);
  if (c.F_shared > 0) rows_set(L.shared, c.T, c.H, c.F_shared);
  L.total = o;
  return L;
}

#define MOE_TRY(expr)                               \
  do {                                              \
    cudaError_t _e = (expr);                        \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;     \
  } while (0)

std::atomic<uint64_t> g_wait_ns{kWaitLimitNs};

}  // namespace

uint64_t moe::pipeline_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

extern "C" {

void moe_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

uint64_t moe_get_wait_limit_ns(void) { return g_wait_ns.load(std::memory_order_relaxed); }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA launch or runtime error";
    case MOE_ERR_TIMEOUT: return "a pipeline wait inside a kernel ran out of time";
    case MOE_ERR_DEVICE: return "inconsistent inputs detected on the device";
  }
  return "unknown status";
}

moe_status moe_max_rows(const moe_config* cfg, int64_t* R) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!R) return MOE_ERR_INVALID_ARG;
  *R = max_rows(*cfg);
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_workspace_init(const moe_config* cfg, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!ws) return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_layout(*cfg).total, (cudaStream_t)stream));
}

moe_status moe_read_device_error(void* ws, int32_t* err, void* stream) {
  if (!ws || !err) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  MOE_TRY(cudaStreamSynchronize(st));
  int32_t v[2] = {0, 0};
  MOE_TRY(cudaMemcpyAsync(v, ws, sizeof(v), cudaMemcpyDeviceToHost, st));
  MOE_TRY(cudaStreamSynchronize(st));
  *err = v[0];
  if (v[0]) MOE_TRY(cudaMemsetAsync(ws, 0, sizeof(v), st));
  MOE_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

moe_status moe_router_topk(const moe_config* cfg, const moe_bf16* X, const float* W_r, const float* logit_bias,
                           const float* sel_bias, float* logits, float* scores, int32_t* topk_idx, float* gates,
                           int32_t* counts, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!tok_ok(cfg, X) || !W_r || !tok_ok(cfg, logits) || !tok_ok(cfg, scores) || !tok_ok(cfg, topk_idx) ||
      !tok_ok(cfg, gates) || !counts)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W_r) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  const int nsm = num_sms();
  if (nsm <= 0) return MOE_ERR_CUDA;
  RouterFwdScratch w{};
  if (ws) {  // the tensor-core logits: W_r's bf16 split, K-split partials, the error word
    const WsLayout L = ws_layout(*cfg);
    w.wsplit = ws_ptr<uint16_t>(ws, L.wb);
    w.part = ws_ptr<float>(ws, L.rlog);
    w.max_splits = L.rlog_splits;
    w.err = ws_ptr<int>(ws, L.err);
  }
  return cuda_status(launch_router_topk(*cfg, X, W_r, logit_bias, sel_bias, logits, scores, topk_idx, gates, counts,
                                        (cudaStream_t)stream, nsm, nullptr, ws ? &w : nullptr));
}

moe_status moe_router_replay(const moe_config* cfg, const moe_bf16* X, const float* W_r, const float* logit_bias,
                             const int32_t* topk_in, float* logits, float* scores, int32_t* topk_idx, float* gates,
                             int32_t* counts, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!tok_ok(cfg, X) || !W_r || !tok_ok(cfg, topk_in) || !tok_ok(cfg, logits) || !tok_ok(cfg, scores) ||
      !tok_ok(cfg, topk_idx) || !tok_ok(cfg, gates) || !counts)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W_r) || !aligned16(logits)) return MOE_ERR_INVALID_ARG;
  const int nsm = num_sms();
  if (nsm <= 0) return MOE_ERR_CUDA;
  RouterFwdScratch w{};
  if (ws) {  // the tensor-core logits: W_r's bf16 split, K-split partials, the error word
    const WsLayout L = ws_layout(*cfg);
    w.wsplit = ws_ptr<uint16_t>(ws, L.wb);
    w.part = ws_ptr<float>(ws, L.rlog);
    w.max_splits = L.rlog_splits;
    w.err = ws_ptr<int>(ws, L.err);
  }
  return cuda_status(launch_router_topk(*cfg, X, W_r, logit_bias, nullptr, logits, scores, topk_idx, gates, counts,
                                        (cudaStream_t)stream, nsm, topk_in, ws ? &w : nullptr));
}

moe_status moe_permute(const moe_config* cfg, const moe_bf16* X, const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map, int32_t* slot_src,
                       moe_bf16* Xperm, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  // Xperm NULL: the dispatch maps only (X is then not read)
  if ((Xperm && !tok_ok(cfg, X)) || !tok_ok(cfg, topk_idx) || !counts || !offsets || !tile_offsets ||
      !tok_ok(cfg, row_id_map) || !slot_src)
    return MOE_ERR_INVALID_ARG;
  if (Xperm && (!aligned16(X) || !aligned16(Xperm))) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(*cfg);
  const int nsm = num_sms();
  if (nsm <= 0) return MOE_ERR_CUDA;
  return cuda_status(launch_permute(*cfg, X, topk_idx, counts, INT_MAX, nullptr, ws_ptr<int32_t>(ws, L.seg_rows),
                                    offsets, tile_offsets, row_id_map, slot_src, Xperm, ws_ptr<int32_t>(ws, L.chunk_counts),
                                    ws_ptr<int32_t>(ws, L.chunk_base), nullptr, nullptr, ws_ptr<int>(ws, L.err), nsm,
                                    (cudaStream_t)stream));
}

moe_status moe_permute_capacity(const moe_config* cfg, const moe_bf16* X, const int32_t* topk_idx,
                                const int32_t* counts, int32_t capacity, const float* priority,
                                int32_t* kept_counts, int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map,
                                int32_t* slot_src, moe_bf16* Xperm, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (capacity < 0) return MOE_ERR_INVALID_ARG;
  if (priority && !tok_ok(cfg, priority)) return MOE_ERR_INVALID_ARG;
  if ((Xperm && !tok_ok(cfg, X)) || !tok_ok(cfg, topk_idx) || !counts || !kept_counts || !offsets ||
      !tile_offsets || !tok_ok(cfg, row_id_map) || !slot_src)
    return MOE_ERR_INVALID_ARG;
  if (Xperm && (!aligned16(X) || !aligned16(Xperm))) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(*cfg);
  const int nsm = num_sms();
  if (nsm <= 0) return MOE_ERR_CUDA;
  return cuda_status(launch_permute(*cfg, X, topk_idx, counts, capacity, priority, kept_counts, offsets,
                                    tile_offsets, row_id_map, slot_src, Xperm, ws_ptr<int32_t>(ws, L.chunk_counts),
                                    ws_ptr<int32_t>(ws, L.chunk_base), ws_ptr<int32_t>(ws, L.drop_order),
                                    ws_ptr<int32_t>(ws, L.drop_start), ws_ptr<int>(ws, L.err), nsm,
                                    (cudaStream_t)stream));
}

moe_status moe_grouped_swiglu_mlp(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                  const int32_t* tile_offsets, const moe_bf16* W13, const moe_bf16* W2,
                                  moe_bf16* GU, moe_bf16* A, moe_bf16* Yperm, const moe_bf16* X,
                                  const moe_bf16* W13_s, const moe_bf16* W2_s, moe_bf16* GU_s, moe_bf16* A_s,
                                  moe_bf16* Yshared, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!Xperm || !offsets || !tile_offsets || !W13 || !W2 || !GU || !A || !Yperm) return MOE_ERR_INVALID_ARG;
  const void* al[] = {Xperm, W13, W2, GU, A, Yperm};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0) {
    if (!tok_ok(cfg, X) || !W13_s || !W2_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) || !tok_ok(cfg, Yshared))
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {X, W13_s, W2_s, GU_s, A_s, Yshared};
    for (const void* p : al2)
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int* err = err_word(ws, *cfg);
  const GemmShape rs = routed_shape(*cfg, offsets, tile_offsets, nullptr);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  MOE_TRY(launch_fc1_fwd(rs, Xperm, W13, GU, A, err, st));
  MOE_TRY(launch_fc2_fwd(rs, A, W2, Yperm, err, st));
  if (cfg->F_shared > 0 && cfg->T > 0) {
    const GemmShape ss = shared_shape(*cfg);
    MOE_TRY(launch_fc1_fwd(ss, X, W13_s, GU_s, A_s, err, st));
    MOE_TRY(launch_fc2_fwd(ss, A_s, W2_s, Yshared, err, st));
  }
  return MOE_OK;
}

// Gathered-rows variants: FC1 reads the token rows of X through slot_src instead of a
// permuted copy.  The CTA-pair kernels do the gathering, so H must be a multiple of 256.
moe_status moe_grouped_swiglu_mlp_gather(const moe_config* cfg, const moe_bf16* X, const int32_t* slot_src,
                                         const int32_t* offsets, const int32_t* tile_offsets, const moe_bf16* W13,
                                         const moe_bf16* W2, moe_bf16* GU, moe_bf16* A, moe_bf16* Yperm,
                                         const moe_bf16* W13_s, const moe_bf16* W2_s, moe_bf16* GU_s,
                                         moe_bf16* A_s, moe_bf16* Yshared, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (cfg->H % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (!tok_ok(cfg, X) || !slot_src || !offsets || !tile_offsets || !W13 || !W2 || !GU || !A || !Yperm)
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {X, W13, W2, GU, A, Yperm};
  for (const void* p : al)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0) {
    if (!W13_s || !W2_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) || !tok_ok(cfg, Yshared))
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {W13_s, W2_s, GU_s, A_s, Yshared};
    for (const void* p : al2)
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int* err = err_word(ws, *cfg);
  const GemmShape rs = routed_shape(*cfg, offsets, tile_offsets, nullptr);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  if (cfg->T > 0) {
    const RowGather rg{slot_src, cfg->k, cfg->T};
    MOE_TRY(launch_fc1_fwd(rs, X, W13, GU, A, err, st, nullptr, &rg));
  }
  MOE_TRY(launch_fc2_fwd(rs, A, W2, Yperm, err, st));
  if (cfg->F_shared > 0 && cfg->T > 0) {
    const GemmShape ss = shared_shape(*cfg);
    MOE_TRY(launch_fc1_fwd(ss, X, W13_s, GU_s, A_s, err, st));
    MOE_TRY(launch_fc2_fwd(ss, A_s, W2_s, Yshared, err, st));
  }
  return MOE_OK;
}

moe_status moe_grouped_swiglu_mlp_bwd_gather(const moe_config* cfg, const moe_bf16* X, const int32_t* slot_src,
                                             const int32_t* offsets, const int32_t* tile_offsets,
                                             const int32_t* counts, const moe_bf16* W13, const moe_bf16* W2,
                                             const moe_bf16* GU, const moe_bf16* A, const moe_bf16* dYperm,
                                             moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* dW13, moe_bf16* dW2,
                                             const moe_bf16* dY, const moe_bf16* W13_s, const moe_bf16* W2_s,
                                             const moe_bf16* GU_s, const moe_bf16* A_s, moe_bf16* dGU_s,
                                             moe_bf16* dX_shared, moe_bf16* dW13_s, moe_bf16* dW2_s, void* ws,
                                             void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (cfg->H % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (!tok_ok(cfg, X) || !slot_src || !offsets || !tile_offsets || !counts || !W13 || !W2 || !GU || !A ||
      !dYperm || !dGU || !dXperm || !dW13 || !dW2)
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {X, W13, W2, GU, A, dYperm, dGU, dXperm, dW13, dW2};
  for (const void* p : al)
    if (p && !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0) {
    if (!tok_ok(cfg, dY) || !W13_s || !W2_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) || !tok_ok(cfg, dGU_s) ||
        !tok_ok(cfg, dX_shared) || !dW13_s || !dW2_s)
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {dY, W13_s, W2_s, GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s};
    for (const void* p : al2)
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int* err = err_word(ws, *cfg);
  const GemmShape rs = routed_shape(*cfg, offsets, tile_offsets, counts);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  MOE_TRY(launch_fc2_dgrad(rs, dYperm, W2, GU, dGU, err, st));
  MOE_TRY(launch_fc2_wgrad(rs, dYperm, A, dW2, err, st));
  MOE_TRY(launch_fc1_dgrad(rs, dGU, W13, dXperm, err, st));
  if (cfg->T > 0) {
    const RowGather rg{slot_src, cfg->k, cfg->T};
    MOE_TRY(launch_fc1_wgrad(rs, dGU, X, dW13, err, st, &rg));
  } else {  // no tokens: every expert's gradient is zero
    MOE_TRY(cudaMemsetAsync(dW13, 0, sizeof(moe_bf16) * (size_t)cfg->E * 2 * cfg->F * cfg->H, st));
  }
  if (cfg->F_shared > 0) {
    if (cfg->T == 0) {
      MOE_TRY(cudaMemsetAsync(dW13_s, 0, sizeof(moe_bf16) * 2 * cfg->F_shared * cfg->H, st));
      MOE_TRY(cudaMemsetAsync(dW2_s, 0, sizeof(moe_bf16) * cfg->F_shared * cfg->H, st));
      return MOE_OK;
    }
    const GemmShape ss = shared_shape(*cfg);
    MOE_TRY(launch_fc2_dgrad(ss, dY, W2_s, GU_s, dGU_s, err, st));
    MOE_TRY(launch_fc2_wgrad(ss, dY, A_s, dW2_s, err, st));
    MOE_TRY(launch_fc1_dgrad(ss, dGU_s, W13_s, dX_shared, err, st));
    MOE_TRY(launch_fc1_wgrad(ss, dGU_s, X, dW13_s, err, st));
  }
  return MOE_OK;
}

moe_status moe_grouped_swiglu_mlp_gated(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                        const int32_t* tile_offsets, const int32_t* slot_src, const float* gates,
                                        const moe_bf16* W13, const moe_bf16* W2, moe_bf16* GU, moe_bf16* A,
                                        moe_bf16* Yperm, const moe_bf16* X, const moe_bf16* W13_s,
                                        const moe_bf16* W2_s, moe_bf16* GU_s, moe_bf16* A_s, moe_bf16* Yshared,
                                        void* ws, void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!slot_src || !tok_ok(cfg, gates)) return MOE_ERR_INVALID_ARG;
  // the argument checks and the shared expert are those of the plain call, which runs
  // after the gated routed pass below
  if (!Xperm || !offsets || !tile_offsets || !W13 || !W2 || !GU || !A || !Yperm) return MOE_ERR_INVALID_ARG;
  const void* al[] = {Xperm, W13, W2, GU, A, Yperm};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0) {
    if (!tok_ok(cfg, X) || !W13_s || !W2_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) || !tok_ok(cfg, Yshared))
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {X, W13_s, W2_s, GU_s, A_s, Yshared};
    for (const void* p : al2)
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int* err = err_word(ws, *cfg);
  const GemmShape rs = routed_shape(*cfg, offsets, tile_offsets, nullptr);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  const Gating gt{slot_src, gates, nullptr, nullptr};
  MOE_TRY(launch_fc1_fwd(rs, Xperm, W13, GU, A, err, st, &gt));
  MOE_TRY(launch_fc2_fwd(rs, A, W2, Yperm, err, st));
  if (cfg->F_shared > 0 && cfg->T > 0) {
    const GemmShape ss = shared_shape(*cfg);
    MOE_TRY(launch_fc1_fwd(ss, X, W13_s, GU_s, A_s, err, st));
    MOE_TRY(launch_fc2_fwd(ss, A_s, W2_s, Yshared, err, st));
  }
  return MOE_OK;
}

moe_status moe_unpermute_combine(const moe_config* cfg, const moe_bf16* Yperm, const int32_t* row_id_map,
                                 const float* gates, const moe_bf16* Yshared, moe_bf16* Y, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!Yperm || !tok_ok(cfg, row_id_map) || !tok_ok(cfg, Y)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(Yperm) || !aligned16(Y) || (Yshared && !aligned16(Yshared))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*cfg, Yperm, row_id_map, gates, Yshared, Y, (cudaStream_t)stream));
}

moe_status moe_unpermute_combine_bwd(const moe_config* cfg, const moe_bf16* dY, const moe_bf16* Yperm,
                                     const int32_t* row_id_map, const float* gates, const int32_t* offsets,
                                     const int32_t* counts, moe_bf16* dYperm, float* dgates, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!tok_ok(cfg, dY) || (dgates && !Yperm) || !tok_ok(cfg, row_id_map) || !offsets || !counts || !dYperm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(dY) || (Yperm && !aligned16(Yperm)) || !aligned16(dYperm)) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_combine_bwd(*cfg, dY, Yperm, row_id_map, gates, offsets, counts, dYperm, dgates, (cudaStream_t)stream));
}

moe_status moe_grouped_swiglu_mlp_bwd(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                      const int32_t* tile_offsets, const int32_t* counts, const moe_bf16* W13,
                                      const moe_bf16* W2, const moe_bf16* GU, const moe_bf16* A,
                                      const moe_bf16* dYperm, moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* dW13,
                                      moe_bf16* dW2, const moe_bf16* X, const moe_bf16* dY,
                                      const moe_bf16* W13_s, const moe_bf16* W2_s, const moe_bf16* GU_s,
                                      const moe_bf16* A_s, moe_bf16* dGU_s, moe_bf16* dX_shared,
                                      moe_bf16* dW13_s, moe_bf16* dW2_s, void* ws, void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!Xperm || !offsets || !tile_offsets || !counts || !W13 || !W2 || !GU || !A || !dYperm || !dGU || !dXperm ||
      !dW13 || !dW2)
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {Xperm, W13, W2, GU, A, dYperm, dGU, dXperm, dW13, dW2};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0) {
    if (!tok_ok(cfg, X) || !tok_ok(cfg, dY) || !W13_s || !W2_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) ||
        !tok_ok(cfg, dGU_s) || !tok_ok(cfg, dX_shared) || !dW13_s || !dW2_s)
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {X, dY, W13_s, W2_s, GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s};
    for (const void* p : al2)
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  int* err = err_word(ws, *cfg);
  const GemmShape rs = routed_shape(*cfg, offsets, tile_offsets, counts);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  MOE_TRY(launch_fc2_dgrad(rs, dYperm, W2, GU, dGU, err, st));
  MOE_TRY(launch_fc2_wgrad(rs, dYperm, A, dW2, err, st));
  MOE_TRY(launch_fc1_dgrad(rs, dGU, W13, dXperm, err, st));
  MOE_TRY(launch_fc1_wgrad(rs, dGU, Xperm, dW13, err, st));
  if (cfg->F_shared > 0) {
    if (cfg->T == 0) {
      MOE_TRY(cudaMemsetAsync(dW13_s, 0, sizeof(moe_bf16) * 2 * cfg->F_shared * cfg->H, st));
      MOE_TRY(cudaMemsetAsync(dW2_s, 0, sizeof(moe_bf16) * cfg->F_shared * cfg->H, st));
      return MOE_OK;
    }
    const GemmShape ss = shared_shape(*cfg);
    MOE_TRY(launch_fc2_dgrad(ss, dY, W2_s, GU_s, dGU_s, err, st));
    MOE_TRY(launch_fc2_wgrad(ss, dY, A_s, dW2_s, err, st));
    MOE_TRY(launch_fc1_dgrad(ss, dGU_s, W13_s, dX_shared, err, st));
    MOE_TRY(launch_fc1_wgrad(ss, dGU_s, X, dW13_s, err, st));
  }
  return MOE_OK;
}

moe_status moe_grouped_swiglu_mlp_bwd_gated(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                            const int32_t* tile_offsets, const int32_t* counts,
                                            const int32_t* slot_src, const int32_t* row_id_map, const float* gates,
                                            const moe_bf16* W13, const moe_bf16* W2, const moe_bf16* GU,
                                            const moe_bf16* dYperm, moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* A,
                                            moe_bf16* dW13, moe_bf16* dW2, float* dgates, const moe_bf16* X,
                                            const moe_bf16* dY, const moe_bf16* W13_s, const moe_bf16* W2_s,
                                            const moe_bf16* GU_s, const moe_bf16* A_s, moe_bf16* dGU_s,
                                            moe_bf16* dX_shared, moe_bf16* dW13_s, moe_bf16* dW2_s, void* ws,
                                            void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!slot_src || !tok_ok(cfg, row_id_map) || !tok_ok(cfg, gates) || !tok_ok(cfg, dgates))
    return MOE_ERR_INVALID_ARG;
  if (!Xperm || !offsets || !tile_offsets || !counts || !W13 || !W2 || !GU || !A || !dYperm || !dGU || !dXperm ||
      !dW13 || !dW2)
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {Xperm, W13, W2, GU, A, dYperm, dGU, dXperm, dW13, dW2};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0) {
    if (!tok_ok(cfg, X) || !tok_ok(cfg, dY) || !W13_s || !W2_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) ||
        !tok_ok(cfg, dGU_s) || !tok_ok(cfg, dX_shared) || !dW13_s || !dW2_s)
      return MOE_ERR_INVALID_ARG;
    const void* al2[] = {X, dY, W13_s, W2_s, GU_s, A_s, dGU_s, dX_shared, dW13_s, dW2_s};
    for (const void* p : al2)
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*cfg);
  int* err = ws_ptr<int>(ws, L.err);
  const GemmShape rs = routed_shape(*cfg, offsets, tile_offsets, counts);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  float* part = ws_ptr<float>(ws, L.dg_part);
  const Gating gt{slot_src, gates, part, A};
  MOE_TRY(launch_fc2_dgrad(rs, dYperm, W2, GU, dGU, err, st, &gt));
  MOE_TRY(launch_dgates_reduce(*cfg, row_id_map, part, cfg->F / fc2_dgrad_tile_n(cfg->F), dgates, rs.nsm, st));
  MOE_TRY(launch_fc2_wgrad(rs, dYperm, A, dW2, err, st));
  MOE_TRY(launch_fc1_dgrad(rs, dGU, W13, dXperm, err, st));
  MOE_TRY(launch_fc1_wgrad(rs, dGU, Xperm, dW13, err, st));
  if (cfg->F_shared > 0) {
    if (cfg->T == 0) {
      MOE_TRY(cudaMemsetAsync(dW13_s, 0, sizeof(moe_bf16) * 2 * cfg->F_shared * cfg->H, st));
      MOE_TRY(cudaMemsetAsync(dW2_s, 0, sizeof(moe_bf16) * cfg->F_shared * cfg->H, st));
      return MOE_OK;
    }
    const GemmShape ss = shared_shape(*cfg);
    MOE_TRY(launch_fc2_dgrad(ss, dY, W2_s, GU_s, dGU_s, err, st));
    MOE_TRY(launch_fc2_wgrad(ss, dY, A_s, dW2_s, err, st));
    MOE_TRY(launch_fc1_dgrad(ss, dGU_s, W13_s, dX_shared, err, st));
    MOE_TRY(launch_fc1_wgrad(ss, dGU_s, X, dW13_s, err, st));
  }
  return MOE_OK;
}

moe_status moe_fp8_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = fp8_layout(*cfg, nullptr).total;
  return MOE_OK;
}

moe_status moe_quantize_weights_fp8(const moe_config* cfg, const moe_bf16* W13, const moe_bf16* W2,
                                    const moe_bf16* W13_s, const moe_bf16* W2_s, uint8_t* W13q, uint8_t* W13sc,
                                    uint8_t* W2q, uint8_t* W2sc, uint8_t* W13q_s, uint8_t* W13sc_s, uint8_t* W2q_s,
                                    uint8_t* W2sc_s, void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!W13 || !W2 || !W13q || !W13sc || !W2q || !W2sc) return MOE_ERR_INVALID_ARG;
  const void* al[] = {W13, W2, W13q, W2q};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const moe_config& c = *cfg;
  MOE_TRY(launch_quant_weights(W13, c.E, 2 * c.F, c.H, W13q, W13sc, st));
  MOE_TRY(launch_quant_weights(W2, c.E, c.H, c.F, W2q, W2sc, st));
  if (c.F_shared > 0) {
    if (!W13_s || !W2_s || !W13q_s || !W13sc_s || !W2q_s || !W2sc_s) return MOE_ERR_INVALID_ARG;
    MOE_TRY(launch_quant_weights(W13_s, 1, 2 * c.F_shared, c.H, W13q_s, W13sc_s, st));
    MOE_TRY(launch_quant_weights(W2_s, 1, c.H, c.F_shared, W2q_s, W2sc_s, st));
  }
  return MOE_OK;
}

moe_status moe_grouped_swiglu_mlp_fp8(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                      const int32_t* tile_offsets, const uint8_t* W13q, const uint8_t* W13sc,
                                      const uint8_t* W2q, const uint8_t* W2sc, moe_bf16* GU, moe_bf16* A,
                                      moe_bf16* Yperm, const moe_bf16* X, const uint8_t* W13q_s,
                                      const uint8_t* W13sc_s, const uint8_t* W2q_s, const uint8_t* W2sc_s,
                                      moe_bf16* GU_s, moe_bf16* A_s, moe_bf16* Yshared, void* fp8_ws, void* ws,
                                      void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!Xperm || !offsets || !tile_offsets || !W13q || !W13sc || !W2q || !W2sc || !GU || !A || !Yperm)
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {Xperm, W13q, W2q, GU, A, Yperm};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0 &&
      (!tok_ok(cfg, X) || !W13q_s || !W13sc_s || !W2q_s || !W2sc_s || !tok_ok(cfg, GU_s) || !tok_ok(cfg, A_s) ||
       !tok_ok(cfg, Yshared)))
    return MOE_ERR_INVALID_ARG;
  if (!ws || !fp8_ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const moe_config& c = *cfg;
  int* err = err_word(ws, c);
  const Fp8Layout L = fp8_layout(c, fp8_ws);
  const GemmShape rs = routed_shape(c, offsets, tile_offsets, nullptr);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  const int32_t* rv = offsets + c.E;  // rows in use, read on the device
  const Fp8Set& R = L.routed;
  MOE_TRY(launch_quant_rows(Xperm, rs.rows, c.H, rv, R.x.q, R.x.sc, rs.nsm, st));
  MOE_TRY(launch_fc1_fwd_fp8(rs, {R.x.q, R.x.sc}, {W13q, W13sc}, GU, A, err, st));
  MOE_TRY(launch_quant_rows(A, rs.rows, c.F, rv, R.a.q, R.a.sc, rs.nsm, st));
  MOE_TRY(launch_fc2_fwd_fp8(rs, {R.a.q, R.a.sc}, {W2q, W2sc}, Yperm, err, st));
  if (c.F_shared > 0 && c.T > 0) {
    const GemmShape ss = shared_shape(c);
    const Fp8Set& Sh = L.shared;
    MOE_TRY(launch_quant_rows(X, c.T, c.H, nullptr, Sh.x.q, Sh.x.sc, rs.nsm, st));
    MOE_TRY(launch_fc1_fwd_fp8(ss, {Sh.x.q, Sh.x.sc}, {W13q_s, W13sc_s}, GU_s, A_s, err, st));
    MOE_TRY(launch_quant_rows(A_s, c.T, c.F_shared, nullptr, Sh.a.q, Sh.a.sc, rs.nsm, st));
    MOE_TRY(launch_fc2_fwd_fp8(ss, {Sh.a.q, Sh.a.sc}, {W2q_s, W2sc_s}, Yshared, err, st));
  }
  return MOE_OK;
}

moe_status moe_grouped_swiglu_mlp_bwd_fp8(const moe_config* cfg, const moe_bf16* Xperm, const int32_t* offsets,
                                          const int32_t* tile_offsets, const int32_t* counts, const uint8_t* W13q,
                                          const uint8_t* W13sc, const uint8_t* W2q, const uint8_t* W2sc,
                                          const moe_bf16* GU, const moe_bf16* A, const moe_bf16* dYperm,
                                          moe_bf16* dGU, moe_bf16* dXperm, moe_bf16* dW13, moe_bf16* dW2,
                                          const moe_bf16* X, const moe_bf16* dY, const uint8_t* W13q_s,
                                          const uint8_t* W13sc_s, const uint8_t* W2q_s, const uint8_t* W2sc_s,
                                          const moe_bf16* GU_s, const moe_bf16* A_s, moe_bf16* dGU_s,
                                          moe_bf16* dX_shared, moe_bf16* dW13_s, moe_bf16* dW2_s, void* fp8_ws,
                                          void* ws, void* stream) {
  moe_status s = check_cfg(cfg, true);
  if (s != MOE_OK) return s;
  if (!Xperm || !offsets || !tile_offsets || !counts || !W13q || !W13sc || !W2q || !W2sc || !GU || !A || !dYperm ||
      !dGU || !dXperm || !dW13 || !dW2)
    return MOE_ERR_INVALID_ARG;
  const void* al[] = {Xperm, W13q, W2q, GU, A, dYperm, dGU, dXperm, dW13, dW2};
  for (const void* p : al)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (cfg->F_shared > 0 &&
      (!tok_ok(cfg, X) || !tok_ok(cfg, dY) || !W13q_s || !W13sc_s || !W2q_s || !W2sc_s || !tok_ok(cfg, GU_s) ||
       !tok_ok(cfg, A_s) || !tok_ok(cfg, dGU_s) || !tok_ok(cfg, dX_shared) || !dW13_s || !dW2_s))
    return MOE_ERR_INVALID_ARG;
  if (!ws || !fp8_ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const moe_config& c = *cfg;
  int* err = err_word(ws, c);
  const Fp8Layout L = fp8_layout(c, fp8_ws);
  const GemmShape rs = routed_shape(c, offsets, tile_offsets, counts);
  if (rs.nsm <= 0) return MOE_ERR_CUDA;
  const int32_t* rv = offsets + c.E;
  const Fp8Set& R = L.routed;
  MOE_TRY(launch_quant_rows(dYperm, rs.rows, c.H, rv, R.dy.q, R.dy.sc, rs.nsm, st));
  MOE_TRY(launch_fc2_dgrad_fp8(rs, {R.dy.q, R.dy.sc}, {W2q, W2sc}, GU, dGU, err, st));
  MOE_TRY(launch_quant_cols(dYperm, rs.rows, c.H, rv, R.dyc.q, R.dyc.sc, st));
  MOE_TRY(launch_quant_cols(A, rs.rows, c.F, rv, R.ac.q, R.ac.sc, st));
  MOE_TRY(launch_fc2_wgrad_fp8(rs, {R.dyc.q, R.dyc.sc}, {R.ac.q, R.ac.sc}, dW2, err, st));
  MOE_TRY(launch_quant_rows(dGU, rs.rows, 2 * c.F, rv, R.dgu.q, R.dgu.sc, rs.nsm, st));
  MOE_TRY(launch_fc1_dgrad_fp8(rs, {R.dgu.q, R.dgu.sc}, {W13q, W13sc}, dXperm, err, st));
  MOE_TRY(launch_quant_cols(dGU, rs.rows, 2 * c.F, rv, R.dguc.q, R.dguc.sc, st));
  MOE_TRY(launch_quant_cols(Xperm, rs.rows, c.H, rv, R.xc.q, R.xc.sc, st));
  MOE_TRY(launch_fc1_wgrad_fp8(rs, {R.dguc.q, R.dguc.sc}, {R.xc.q, R.xc.sc}, dW13, err, st));
  if (c.F_shared > 0) {
    if (c.T == 0) {
      MOE_TRY(cudaMemsetAsync(dW13_s, 0, sizeof(moe_bf16) * 2 * c.F_shared * c.H, st));
      MOE_TRY(cudaMemsetAsync(dW2_s, 0, sizeof(moe_bf16) * c.F_shared * c.H, st));
      return MOE_OK;
    }
    const GemmShape ss = shared_shape(c);
    const Fp8Set& Sh = L.shared;
    const int Fs = c.F_shared;
    MOE_TRY(launch_quant_rows(dY, c.T, c.H, nullptr, Sh.dy.q, Sh.dy.sc, rs.nsm, st));
    MOE_TRY(launch_fc2_dgrad_fp8(ss, {Sh.dy.q, Sh.dy.sc}, {W2q_s, W2sc_s}, GU_s, dGU_s, err, st));
    MOE_TRY(launch_quant_cols(dY, c.T, c.H, nullptr, Sh.dyc.q, Sh.dyc.sc, st));
    MOE_TRY(launch_quant_cols(A_s, c.T, Fs, nullptr, Sh.ac.q, Sh.ac.sc, st));
    MOE_TRY(launch_fc2_wgrad_fp8(ss, {Sh.dyc.q, Sh.dyc.sc}, {Sh.ac.q, Sh.ac.sc}, dW2_s, err, st));
    MOE_TRY(launch_quant_rows(dGU_s, c.T, 2 * Fs, nullptr, Sh.dgu.q, Sh.dgu.sc, rs.nsm, st));
    MOE_TRY(launch_fc1_dgrad_fp8(ss, {Sh.dgu.q, Sh.dgu.sc}, {W13q_s, W13sc_s}, dX_shared, err, st));
    MOE_TRY(launch_quant_cols(dGU_s, c.T, 2 * Fs, nullptr, Sh.dguc.q, Sh.dguc.sc, st));
    MOE_TRY(launch_quant_cols(X, c.T, c.H, nullptr, Sh.xc.q, Sh.xc.sc, st));
    MOE_TRY(launch_fc1_wgrad_fp8(ss, {Sh.dguc.q, Sh.dguc.sc}, {Sh.xc.q, Sh.xc.sc}, dW13_s, err, st));
  }
  return MOE_OK;
}

moe_status moe_router_topk_bwd(const moe_config* cfg, const moe_bf16* X, const float* W_r, const float* logits,
                               const float* scores, const int32_t* topk_idx, const float* gates,
                               const float* dgates, float* dW_r, float* dlogit_bias, float* dX_router, void* ws,
                               void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  (void)scores;
  if (!tok_ok(cfg, X) || !W_r || !tok_ok(cfg, logits) || !tok_ok(cfg, topk_idx) || !tok_ok(cfg, gates) ||
      !tok_ok(cfg, dgates) || !dW_r || !tok_ok(cfg, dX_router))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W_r) || !aligned16(dX_router) || !aligned16(dW_r)) return MOE_ERR_INVALID_ARG;
  if (!ws) return MOE_ERR_WORKSPACE;
  const WsLayout L = ws_layout(*cfg);
  const int nsm = num_sms();
  if (nsm <= 0) return MOE_ERR_CUDA;
  RouterBwdScratch w;
  w.dl = ws_ptr<float>(ws, L.dlogits);
  w.part = ws_ptr<float>(ws, L.rbwd_part);
  w.splits = L.rbwd_splits;
  w.dl_rows = ws_ptr<uint16_t>(ws, L.dl_rows);
  w.dl_cols = ws_ptr<uint16_t>(ws, L.dl_cols);
  w.wb = ws_ptr<uint16_t>(ws, L.wb);
  w.Tp = L.Tp;
  w.Ep = L.Ep;
  return cuda_status(launch_router_bwd(*cfg, X, W_r, logits, topk_idx, gates, dgates, dW_r, dlogit_bias, dX_router, w,
                                       ws_ptr<int>(ws, L.err), nsm, (cudaStream_t)stream));
}

moe_status moe_permute_bwd(const moe_config* cfg, const moe_bf16* dXperm, const int32_t* row_id_map,
                           const float* dX_router, const moe_bf16* dX_shared, moe_bf16* dX, void* stream) {
  moe_status s = check_cfg(cfg, false);
  if (s != MOE_OK) return s;
  if (!dXperm || !tok_ok(cfg, row_id_map) || !tok_ok(cfg, dX)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dXperm) || !aligned16(dX) || (dX_router && !aligned16(dX_router)) ||
      (dX_shared && !aligned16(dX_shared)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_permute_bwd(*cfg, dXperm, row_id_map, dX_router, dX_shared, dX, (cudaStream_t)stream));
}

}  // extern "C"
