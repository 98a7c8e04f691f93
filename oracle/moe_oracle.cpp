// CPU oracle of the single-GPU dropless top-k MoE layer (forward and backward).
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
// load this file; only the tests, the smoke check and the benchmark's CPU
// baseline do.  It shares no code, header or table with the CUDA library.
//
// What it computes follows "Scalable Training of Mixture-of-Experts Models with
// Megatron Core" (summary page, section "Method"): a router (learned linear
// projection in FP32, softmax or sigmoid scoring, top-k selection), a
// dispatcher that groups each expert's tokens contiguously, SwiGLU experts
// ("GLU Variants Improve Transformer", cited on the index page under "Builds
// on"), and a combine stage that sums the gate-weighted expert outputs.  The
// layer is dropless (same page, "Method": sync-free dropless execution), so
// every one of the T*k assignments is kept.
//
// The pages give no formulas; the readings taken here are:
//  * top-k in descending key order, ties to the lower expert index;
//  * softmax key = logit (+ selection bias), sigmoid key = sigmoid(logit)
//    (+ selection bias); the bias never enters the gate values;
//  * group-limited routing: contiguous groups of E/n_group experts, group
//    score = sum of the two largest keys (or the max), keep topk_group groups
//    (ties to the lower group id), then top-k inside them;
//  * gates renormalised over the k winners (softmax over the selected logits,
//    or s_j / sum s), then multiplied by gate_scale;
//  * SwiGLU expert: y = W2 (silu(Wg x) * (Wu x)), no biases, silu(z)=z*sigmoid(z);
//  * shared expert: always on, gate 1, added in the combine;
//  * backward: the exact gradient of L = <dY, Y>, selection treated as
//    piecewise constant (no gradient through top-k, groups or the bias).
//
// Arithmetic: every dot product accumulates in double.  In "mirror" mode the
// values are rounded to bf16 (round-to-nearest-even) exactly where the GPU
// path stores bf16 tensors (GU, A, Yperm, Y, dYperm, dGU, dXperm, dX, dW) and
// nowhere else; in "pure" mode nothing is rounded (for finite differences).
//
// "Gated" mode (the memory-efficient path: summary page, "Method", memory recipes)
// computes the same function with each routed expert's gate applied to its
// activation before the down projection, so the expert output is already gate-
// weighted and the gate gradient is <dA', a> with dA' = W2^T dY and a = silu(g) u
// recomputed from the stored g, u.  In pure mode it equals the plain layer up to
// rounding; in mirror mode it rounds where that path stores bf16 (A' = g a, the
// gated expert output, the recomputed g a for dW2).
//
// The dispatch maps are built by a plain stable counting sort over tokens in
// increasing order, which the GPU path does not use.
//
// Parity pins live in tests/test_oracle_pins.py (brute-force selection, E=1
// dense SwiGLU, identical experts, bijection invariants, gate sums, finite
// differences, autograd).  Parity unpinned: values at the full workload sizes,
// for which the pages print nothing; there the oracle itself is the reference.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

extern "C" {
typedef struct {
  int32_t T, H, E, k, F, F_shared;
  int32_t score_fn;    // 0 softmax, 1 sigmoid
  int32_t renorm;      // 1: renormalise the k gates
  double gate_scale;   // multiplies the gates after renormalisation
  int32_t n_group;     // 1: no group limit
  int32_t topk_group;  // groups kept when n_group > 1
  int32_t group_score; // 0: sum of the two largest keys, 1: the largest key
  int32_t align;       // row alignment of each expert segment in the permuted buffer
  int32_t BM;          // rows per M tile, for tile_offsets
  int32_t mirror;      // 1: round to bf16 where the GPU stores bf16; 0: pure double
  int32_t nthreads;    // 0: all host cores
  int32_t fp8;         // 1: every expert GEMM operand passes through FP8 E4M3 block quantization
  int32_t gated;       // 1: routed experts take their gate before the down projection (see above)
} ora_cfg;
}

namespace {

inline double bf(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round a double to the nearest bf16 value (ties to even), returned as double.
inline double rbf(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e;
  double m = std::frexp(x, &e);               // x = m * 2^e, 0.5 <= |m| < 1
  double q = std::nearbyint(std::ldexp(m, 8)); // 8 significant bits, default mode = ties-to-even
  return std::ldexp(q, e - 8);
}

inline double maybe_r(const ora_cfg& c, double x) { return c.mirror ? rbf(x) : x; }

inline double sigm(double z) { return 1.0 / (1.0 + std::exp(-z)); }
inline double silu(double z) { return z * sigm(z); }
inline double dsilu(double z) {
  const double s = sigm(z);
  return s * (1.0 + z * (1.0 - s));
}

// ---------------------------------------------------------------- FP8 E4M3
// E4M3 ("fn" flavour): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
// infinities, largest finite 448, smallest normal 2^-6, subnormal spacing 2^-9.
// Round to nearest, ties to even.  Inputs here never exceed 448 in magnitude.
double e4m3_rne(double v) {
  if (v == 0.0) return 0.0;
  const double a = std::fabs(v);
  int ex;
  std::frexp(a, &ex);                  // a = m * 2^ex, 0.5 <= m < 1, so floor(log2 a) = ex - 1
  const int e = std::max(ex - 1, -6);  // below 2^-6 the spacing stays 2^-9
  const double ulp = std::ldexp(1.0, e - 3);
  const double q = std::nearbyint(a / ulp) * ulp;
  return v < 0 ? -q : q;
}

// Block scale: the smallest power of two s = 2^e with 448*s >= amax (s = 1 for an
// all-zero block).  Power-of-two scales are exact to apply and to undo.
double block_scale(double amax) {
  if (!(amax > 0.0)) return 1.0;
  int ex;
  std::frexp(amax / 448.0, &ex);
  int e = ex;                                          // 2^(ex-1) <= amax/448 < 2^ex
  while (e > -127 && 448.0 * std::ldexp(1.0, e - 1) >= amax) --e;  // exact comparisons
  while (448.0 * std::ldexp(1.0, e) < amax) ++e;
  return std::ldexp(1.0, e);
}

// Quantize-dequantize n consecutive values as blocks of `blk` elements.
void qdq_blocks(const double* in, double* out, int n, int blk) {
  for (int b0 = 0; b0 < n; b0 += blk) {
    const int b1 = std::min(n, b0 + blk);
    double amax = 0;
    for (int i = b0; i < b1; ++i) amax = std::max(amax, std::fabs(in[i]));
    const double s = block_scale(amax);
    for (int i = b0; i < b1; ++i) out[i] = e4m3_rne(in[i] / s) * s;
  }
}

// Column-wise blocks: rows [r0, r0+128) of each column of a [m x n] row-major array.
void qdq_columns(double* a, int64_t m, int n) {
  std::vector<double> col;
  for (int64_t r0 = 0; r0 < m; r0 += 128) {
    const int64_t r1 = std::min<int64_t>(m, r0 + 128);
    for (int j = 0; j < n; ++j) {
      double amax = 0;
      for (int64_t r = r0; r < r1; ++r) amax = std::max(amax, std::fabs(a[r * n + j]));
      const double s = block_scale(amax);
      for (int64_t r = r0; r < r1; ++r) a[r * n + j] = e4m3_rne(a[r * n + j] / s) * s;
    }
  }
}

int nthreads_of(const ora_cfg& c) {
  if (c.nthreads > 0) return c.nthreads;
  unsigned hc = std::thread::hardware_concurrency();
  return hc ? (int)hc : 1;
}

template <typename Fn>
void parallel_for(int64_t n, int nth, Fn fn) {
  if (nth <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> th;
  for (int w = 0; w < std::min<int64_t>(nth, n); ++w)
    th.emplace_back([&] {
      for (int64_t i; (i = next.fetch_add(1)) < n;) fn(i);
    });
  for (auto& t : th) t.join();
}

// Top-k selection with the optional group limit, on keys of type K.
// Keys are formed by the caller; returns experts in descending key order,
// ties to the lower index.
template <typename K>
void select_topk(const ora_cfg& c, const K* key, int32_t* out) {
  const int E = c.E;
  std::vector<char> allowed(E, 1);
  if (c.n_group > 1) {
    const int G = c.n_group, per = E / G;
    std::vector<K> gs(G);
    for (int g = 0; g < G; ++g) {
      // largest key in the group, then the largest of the others
      int i1 = g * per;
      for (int e = g * per; e < (g + 1) * per; ++e)
        if (key[e] > key[i1]) i1 = e;
      if (c.group_score == 1 || per == 1) {
        gs[g] = key[i1];
      } else {
        int i2 = -1;
        for (int e = g * per; e < (g + 1) * per; ++e)
          if (e != i1 && (i2 < 0 || key[e] > key[i2])) i2 = e;
        gs[g] = key[i1] + key[i2];
      }
    }
    std::vector<char> keep(G, 0);
    for (int r = 0; r < c.topk_group; ++r) {
      int best = -1;
      for (int g = 0; g < G; ++g)
        if (!keep[g] && (best < 0 || gs[g] > gs[best])) best = g;
      keep[best] = 1;
    }
    for (int e = 0; e < E; ++e) allowed[e] = keep[e / per];
  }
  std::vector<char> taken(E, 0);
  for (int j = 0; j < c.k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (allowed[e] && !taken[e] && (best < 0 || key[e] > key[best])) best = e;
    taken[best] = 1;
    out[j] = best;
  }
}

// Gates of one token from its double logits and its selection.
void token_gates(const ora_cfg& c, const double* l, const int32_t* sel, double* g) {
  const int k = c.k, E = c.E;
  if (c.score_fn == 0) {
    if (c.renorm) {
      double m = l[sel[0]];
      for (int j = 1; j < k; ++j) m = std::max(m, l[sel[j]]);
      double z = 0;
      for (int j = 0; j < k; ++j) z += std::exp(l[sel[j]] - m);
      for (int j = 0; j < k; ++j) g[j] = c.gate_scale * std::exp(l[sel[j]] - m) / z;
    } else {
      double m = l[0];
      for (int e = 1; e < E; ++e) m = std::max(m, l[e]);
      double z = 0;
      for (int e = 0; e < E; ++e) z += std::exp(l[e] - m);
      for (int j = 0; j < k; ++j) g[j] = c.gate_scale * std::exp(l[sel[j]] - m) / z;
    }
  } else {
    double S = 0;
    for (int j = 0; j < k; ++j) S += sigm(l[sel[j]]);
    for (int j = 0; j < k; ++j) g[j] = c.gate_scale * sigm(l[sel[j]]) / (c.renorm ? S : 1.0);
  }
}

// d(gates)/d(logits) applied to dg: exact gradient of token_gates for a fixed selection.
void token_dlogits(const ora_cfg& c, const double* l, const int32_t* sel, const double* g,
                   const double* dg, double* dl) {
  const int k = c.k, E = c.E;
  const double a = c.gate_scale;
  for (int e = 0; e < E; ++e) dl[e] = 0.0;
  if (c.score_fn == 0) {
    if (c.renorm) {
      // g_j = a * q_j, q = softmax over the selected logits
      double s = 0;
      for (int j = 0; j < k; ++j) s += (g[j] / a) * dg[j];
      for (int j = 0; j < k; ++j) dl[sel[j]] = a * (g[j] / a) * (dg[j] - s);
    } else {
      // g_j = a * p[sel_j], p = softmax over all E logits
      double m = l[0];
      for (int e = 1; e < E; ++e) m = std::max(m, l[e]);
      std::vector<double> p(E);
      double z = 0;
      for (int e = 0; e < E; ++e) z += (p[e] = std::exp(l[e] - m));
      for (int e = 0; e < E; ++e) p[e] /= z;
      double s = 0;
      for (int j = 0; j < k; ++j) s += dg[j] * p[sel[j]];
      for (int e = 0; e < E; ++e) dl[e] = -a * p[e] * s;
      for (int j = 0; j < k; ++j) dl[sel[j]] += a * p[sel[j]] * dg[j];
    }
  } else {
    if (c.renorm) {
      // g_j = a * s_j / S, S = sum of the selected sigmoids
      double S = 0, cc = 0;
      for (int j = 0; j < k; ++j) S += sigm(l[sel[j]]);
      for (int j = 0; j < k; ++j) cc += dg[j] * g[j] / a;
      for (int j = 0; j < k; ++j) {
        const double s = sigm(l[sel[j]]);
        const double ds = (a / S) * (dg[j] - cc);
        dl[sel[j]] = ds * s * (1.0 - s);
      }
    } else {
      for (int j = 0; j < k; ++j) {
        const double s = sigm(l[sel[j]]);
        dl[sel[j]] = a * dg[j] * s * (1.0 - s);
      }
    }
  }
}

// One SwiGLU expert applied to one token.  w13: [2F,H] (gate rows then up rows),
// w2: [H,F].  Outputs (all length as named): gr,ur (F) = stored pre-activations,
// ar (F) = stored activation, yr (H) = stored expert output.
// gate: multiplies the activation before the down projection (gated mode; 1 otherwise)
void expert_fwd(const ora_cfg& c, int F, const uint16_t* w13, const uint16_t* w2, const double* x_in,
                double* gr, double* ur, double* ar, double* yr, double gate = 1.0) {
  const int H = c.H;
  // FP8: the token row enters FC1 as 1x128 blocks along H, the activation enters
  // FC2 as 1x128 blocks along F; the weights are passed already block-quantized.
  std::vector<double> xq, aq;
  const double* x = x_in;
  if (c.fp8) {
    xq.resize(H);
    qdq_blocks(x_in, xq.data(), H, 128);
    x = xq.data();
  }
  for (int f = 0; f < F; ++f) {
    double g = 0, u = 0;
    const uint16_t* wg = w13 + (size_t)f * H;
    const uint16_t* wu = w13 + (size_t)(F + f) * H;
    for (int h = 0; h < H; ++h) {
      g += bf(wg[h]) * x[h];
      u += bf(wu[h]) * x[h];
    }
    gr[f] = maybe_r(c, g);
    ur[f] = maybe_r(c, u);
    ar[f] = maybe_r(c, gate * (silu(g) * u));  // the activation is formed from the unrounded g, u
  }
  const double* a = ar;
  if (c.fp8) {
    aq.resize(F);
    qdq_blocks(ar, aq.data(), F, 128);
    a = aq.data();
  }
  for (int h = 0; h < H; ++h) {
    double y = 0;
    const uint16_t* w = w2 + (size_t)h * F;
    for (int f = 0; f < F; ++f) y += bf(w[f]) * a[f];
    yr[h] = maybe_r(c, y);
  }
}

// Backward of one expert for one token, given the upstream gradient dyp (H) of
// its output.  Produces dG, dU (F, as stored) and dx (H, as stored).  Gated
// mode (dgate != null): dyp is the gradient of the gate-weighted output; the gate
// gradient <W2^T dyp, silu(g) u> goes to *dgate and the activation gradient is
// gate * W2^T dyp.
void expert_bwd(const ora_cfg& c, int F, const uint16_t* w13, const uint16_t* w2, const double* gr,
                const double* ur, const double* dyp_in, double* dG, double* dU, double* dx, double gate = 1.0,
                double* dgate = nullptr) {
  const int H = c.H;
  std::vector<double> dA(F, 0.0), dq;
  const double* dyp = dyp_in;
  if (c.fp8) {  // FC2 dgrad takes the output gradient as 1x128 blocks along H
    dq.resize(H);
    qdq_blocks(dyp_in, dq.data(), H, 128);
    dyp = dq.data();
  }
  for (int h = 0; h < H; ++h) {
    const uint16_t* w = w2 + (size_t)h * F;
    const double d = dyp[h];
    for (int f = 0; f < F; ++f) dA[f] += bf(w[f]) * d;
  }
  if (dgate) {
    double s = 0;
    for (int f = 0; f < F; ++f) s += dA[f] * (silu(gr[f]) * ur[f]);
    *dgate = s;
    for (int f = 0; f < F; ++f) dA[f] *= gate;
  }
  for (int f = 0; f < F; ++f) {
    dG[f] = maybe_r(c, dA[f] * ur[f] * dsilu(gr[f]));
    dU[f] = maybe_r(c, dA[f] * silu(gr[f]));
  }
  for (int h = 0; h < H; ++h) dx[h] = 0.0;
  std::vector<double> gq;
  if (c.fp8) {  // FC1 dgrad takes [dG | dU] as 1x128 blocks along 2F
    gq.resize(2 * (size_t)F);
    std::vector<double> cat(2 * (size_t)F);
    for (int f = 0; f < F; ++f) {
      cat[f] = dG[f];
      cat[F + f] = dU[f];
    }
    qdq_blocks(cat.data(), gq.data(), 2 * F, 128);
  }
  for (int f = 0; f < F; ++f) {
    const uint16_t* wg = w13 + (size_t)f * H;
    const uint16_t* wu = w13 + (size_t)(F + f) * H;
    const double a = c.fp8 ? gq[f] : dG[f], b = c.fp8 ? gq[F + f] : dU[f];
    for (int h = 0; h < H; ++h) dx[h] += bf(wg[h]) * a + bf(wu[h]) * b;
  }
  for (int h = 0; h < H; ++h) dx[h] = maybe_r(c, dx[h]);
}

}  // namespace

extern "C" {

// Router logits and scores for all tokens: logits = X W_r^T (+ logit_bias),
// scores = softmax over E (softmax mode) or sigmoid(logit) (sigmoid mode).
void ora_router(const ora_cfg* cp, const uint16_t* X, const float* Wr, const float* logit_bias,
                double* logits, double* scores) {
  const ora_cfg c = *cp;
  const int H = c.H, E = c.E;
  parallel_for(c.T, nthreads_of(c), [&](int64_t t) {
    double* l = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      double s = 0;
      for (int h = 0; h < H; ++h) s += bf(X[(size_t)t * H + h]) * (double)Wr[(size_t)e * H + h];
      l[e] = s + (logit_bias ? (double)logit_bias[e] : 0.0);
    }
    double* s = scores + (size_t)t * E;
    if (c.score_fn == 0) {
      double m = l[0];
      for (int e = 1; e < E; ++e) m = std::max(m, l[e]);
      double z = 0;
      for (int e = 0; e < E; ++e) z += (s[e] = std::exp(l[e] - m));
      for (int e = 0; e < E; ++e) s[e] /= z;
    } else {
      for (int e = 0; e < E; ++e) s[e] = sigm(l[e]);
    }
  });
}

// Selection on double logits/scores (pure oracle routing).
// key = logit (softmax) or score (sigmoid), plus sel_bias when given.
void ora_select_f64(const ora_cfg* cp, const double* logits, const double* scores, const float* sel_bias,
                    int32_t* topk_idx) {
  const ora_cfg c = *cp;
  parallel_for(c.T, nthreads_of(c), [&](int64_t t) {
    std::vector<double> key(c.E);
    const double* base = (c.score_fn == 0 ? logits : scores) + (size_t)t * c.E;
    for (int e = 0; e < c.E; ++e) key[e] = base[e] + (sel_bias ? (double)sel_bias[e] : 0.0);
    select_topk<double>(c, key.data(), topk_idx + (size_t)t * c.k);
  });
}

// Selection on float32 logits/scores, keys and group sums formed in float32.
// Used to run the oracle's selection on the exact scores another
// implementation produced, so that selections can be compared bit for bit.
void ora_select_f32(const ora_cfg* cp, const float* logits, const float* scores, const float* sel_bias,
                    int32_t* topk_idx) {
  const ora_cfg c = *cp;
  parallel_for(c.T, nthreads_of(c), [&](int64_t t) {
    std::vector<float> key(c.E);
    const float* base = (c.score_fn == 0 ? logits : scores) + (size_t)t * c.E;
    for (int e = 0; e < c.E; ++e) key[e] = base[e] + (sel_bias ? sel_bias[e] : 0.0f);
    select_topk<float>(c, key.data(), topk_idx + (size_t)t * c.k);
  });
}

// Gate values of all tokens from double logits and a given selection.
void ora_gates(const ora_cfg* cp, const double* logits, const int32_t* topk_idx, double* gates) {
  const ora_cfg c = *cp;
  parallel_for(c.T, nthreads_of(c), [&](int64_t t) {
    token_gates(c, logits + (size_t)t * c.E, topk_idx + (size_t)t * c.k, gates + (size_t)t * c.k);
  });
}

// Dispatch maps by a stable counting sort.  slot_src has R entries; entries at
// or beyond offsets[E] are left untouched.  Padding slots get -1.
int ora_dispatch_priority(const ora_cfg* cp, const int32_t* topk_idx, int32_t capacity, const double* priority,
                          int32_t* counts, int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map,
                          int32_t* slot_src, int64_t R);

int ora_dispatch(const ora_cfg* cp, const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                 int32_t* tile_offsets, int32_t* row_id_map, int32_t* slot_src, int64_t R) {
  return ora_dispatch_priority(cp, topk_idx, INT32_MAX, nullptr, counts, offsets, tile_offsets, row_id_map, slot_src,
                               R);
}

// Capacity-controlled token dropping ("Scalable Training of Mixture-of-Experts Models
// with Megatron Core", summary page, "Results": a production feature, no policy given;
// both policies below are readings).
// Position policy: expert e keeps its first `capacity`
// assignments in token order; a dropped assignment gets row_id_map = -1 and no row.
// counts are the kept counts.
int ora_dispatch_capacity(const ora_cfg* cp, const int32_t* topk_idx, int32_t capacity, int32_t* counts,
                          int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map, int32_t* slot_src,
                          int64_t R) {
  return ora_dispatch_priority(cp, topk_idx, capacity, nullptr, counts, offsets, tile_offsets, row_id_map, slot_src,
                               R);
}

// Capacity-controlled dropping, priority policy (priority [T,k], e.g. the gates): an
// expert with more than `capacity` assignments keeps the `capacity` of largest
// priority, equal priorities going to the earlier assignment in token order.  Kept
// assignments take their rows in token order.  priority == nullptr is the position
// policy.
int ora_dispatch_priority(const ora_cfg* cp, const int32_t* topk_idx, int32_t capacity, const double* priority,
                          int32_t* counts, int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map,
                          int32_t* slot_src, int64_t R) {
  const ora_cfg c = *cp;
  const int E = c.E, k = c.k;
  const int64_t n = (int64_t)c.T * k;
  // per expert, its assignments in token order (t-major, then j)
  std::vector<std::vector<int64_t>> mine(E);
  for (int64_t i = 0; i < n; ++i) mine[topk_idx[i]].push_back(i);
  std::vector<char> keep(n, 0);
  for (int e = 0; e < E; ++e) {
    std::vector<int64_t> order = mine[e];
    if (priority)  // stable: equal priorities stay in token order
      std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return priority[a] > priority[b]; });
    const size_t nk = std::min(order.size(), (size_t)std::max(capacity, 0));
    for (size_t q = 0; q < nk; ++q) keep[order[q]] = 1;
    counts[e] = (int32_t)nk;
  }
  offsets[0] = 0;
  tile_offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    const int32_t padded = (counts[e] + c.align - 1) / c.align * c.align;
    offsets[e + 1] = offsets[e] + padded;
    tile_offsets[e + 1] = tile_offsets[e] + (counts[e] + c.BM - 1) / c.BM;
  }
  if ((int64_t)offsets[E] > R) return -1;
  std::vector<int32_t> cursor(offsets, offsets + E);
  for (int64_t i = 0; i < n; ++i) {
    if (!keep[i]) {
      row_id_map[i] = -1;
      continue;
    }
    const int32_t slot = cursor[topk_idx[i]]++;
    row_id_map[i] = slot;
    slot_src[slot] = (int32_t)i;
  }
  for (int e = 0; e < E; ++e)
    for (int32_t s = offsets[e] + counts[e]; s < offsets[e + 1]; ++s) slot_src[s] = -1;
  return 0;
}

// Forward and backward of the listed tokens.  Per token t (index i in tok_list):
//   Y[i]      = sum_j gates[t,j] * expert_{e_tj}(x_t) + shared(x_t)          (H)
//   dgates[i] = <dY_t, expert_{e_tj}(x_t)>                                  (k)
//   dlogits[i]= exact gradient of the gates w.r.t. the logits, applied to dgates (E)
//   dX[i]     = sum_j d expert / dx + d shared / dx + dlogits W_r           (H)
// logits are the double router logits of all T tokens; gates the double gates.
// Any output may be null; dX/dgates/dlogits need dY.
void ora_tokens_kept(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                     const uint16_t* W13s, const uint16_t* W2s, const float* Wr, const int32_t* topk_idx,
                     const double* logits, const double* gates, const uint16_t* dY, int64_t ntok,
                     const int64_t* tok_list, double* Y, double* dX, double* dgates_out, double* dlogits_out,
                     const int32_t* kept);

void ora_tokens(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                const uint16_t* W13s, const uint16_t* W2s, const float* Wr, const int32_t* topk_idx,
                const double* logits, const double* gates, const uint16_t* dY, int64_t ntok,
                const int64_t* tok_list, double* Y, double* dX, double* dgates_out, double* dlogits_out) {
  ora_tokens_kept(cp, X, W13, W2, W13s, W2s, Wr, topk_idx, logits, gates, dY, ntok, tok_list, Y, dX, dgates_out,
                  dlogits_out, nullptr);
}

// Same, where kept[t*k+j] == 0 marks an assignment dropped by capacity: it adds
// nothing to Y and receives no gradient (its dgate is 0).
void ora_tokens_kept(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                     const uint16_t* W13s, const uint16_t* W2s, const float* Wr, const int32_t* topk_idx,
                     const double* logits, const double* gates, const uint16_t* dY, int64_t ntok,
                     const int64_t* tok_list, double* Y, double* dX, double* dgates_out, double* dlogits_out,
                     const int32_t* kept) {
  const ora_cfg c = *cp;
  const int H = c.H, F = c.F, Fs = c.F_shared, E = c.E, k = c.k;
  const bool bwd = dY && (dX || dgates_out || dlogits_out);
  parallel_for(ntok, nthreads_of(c), [&](int64_t i) {
    const int64_t t = tok_list[i];
    std::vector<double> x(H), y(H, 0.0), dx(H, 0.0), dy(H), dyp(H), ye(H), dxe(H);
    const int Fm = std::max(F, Fs);
    std::vector<double> gr(Fm), ur(Fm), ar(Fm), dG(Fm), dU(Fm);
    std::vector<double> dg(k, 0.0), dl(E, 0.0);
    for (int h = 0; h < H; ++h) x[h] = bf(X[(size_t)t * H + h]);
    if (dY)
      for (int h = 0; h < H; ++h) dy[h] = bf(dY[(size_t)t * H + h]);
    const int32_t* sel = topk_idx + (size_t)t * k;
    const double* gt = gates + (size_t)t * k;
    for (int j = 0; j < k; ++j) {
      if (kept && !kept[(size_t)t * k + j]) continue;
      const int e = sel[j];
      const uint16_t* w13 = W13 + (size_t)e * 2 * F * H;
      const uint16_t* w2 = W2 + (size_t)e * H * F;
      if (c.gated) {  // the expert's output is gate-weighted already
        expert_fwd(c, F, w13, w2, x.data(), gr.data(), ur.data(), ar.data(), ye.data(), gt[j]);
        for (int h = 0; h < H; ++h) y[h] += ye[h];
        if (bwd) {
          expert_bwd(c, F, w13, w2, gr.data(), ur.data(), dy.data(), dG.data(), dU.data(), dxe.data(), gt[j],
                     &dg[j]);
          for (int h = 0; h < H; ++h) dx[h] += dxe[h];
        }
        continue;
      }
      expert_fwd(c, F, w13, w2, x.data(), gr.data(), ur.data(), ar.data(), ye.data());
      for (int h = 0; h < H; ++h) y[h] += gt[j] * ye[h];
      if (bwd) {
        double s = 0;
        for (int h = 0; h < H; ++h) s += dy[h] * ye[h];
        dg[j] = s;
        for (int h = 0; h < H; ++h) dyp[h] = maybe_r(c, gt[j] * dy[h]);
        expert_bwd(c, F, w13, w2, gr.data(), ur.data(), dyp.data(), dG.data(), dU.data(), dxe.data());
        for (int h = 0; h < H; ++h) dx[h] += dxe[h];
      }
    }
    if (Fs > 0) {
      expert_fwd(c, Fs, W13s, W2s, x.data(), gr.data(), ur.data(), ar.data(), ye.data());
      for (int h = 0; h < H; ++h) y[h] += ye[h];
      if (bwd) {
        expert_bwd(c, Fs, W13s, W2s, gr.data(), ur.data(), dy.data(), dG.data(), dU.data(), dxe.data());
        for (int h = 0; h < H; ++h) dx[h] += dxe[h];
      }
    }
    if (Y)
      for (int h = 0; h < H; ++h) Y[(size_t)i * H + h] = maybe_r(c, y[h]);
    if (bwd) {
      token_dlogits(c, logits + (size_t)t * E, sel, gt, dg.data(), dl.data());
      for (int e = 0; e < E; ++e) {
        if (dl[e] == 0.0) continue;
        const float* w = Wr + (size_t)e * H;
        for (int h = 0; h < H; ++h) dx[h] += dl[e] * (double)w[h];
      }
      if (dX)
        for (int h = 0; h < H; ++h) dX[(size_t)i * H + h] = maybe_r(c, dx[h]);
      if (dgates_out)
        for (int j = 0; j < k; ++j) dgates_out[(size_t)i * k + j] = dg[j];
      if (dlogits_out)
        for (int e = 0; e < E; ++e) dlogits_out[(size_t)i * E + e] = dl[e];
    }
  });
}

// Weight gradients of one expert (expert = -1: the shared expert, which sees
// every token with gate 1).  dW13: [2F,H] (gate rows then up rows), dW2: [H,F].
void ora_expert_wgrad_kept(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                           const uint16_t* W13s, const uint16_t* W2s, const int32_t* topk_idx, const double* gates,
                           const uint16_t* dY, int32_t expert, double* dW13, double* dW2, const int32_t* c_kept);

void ora_expert_wgrad(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                      const uint16_t* W13s, const uint16_t* W2s, const int32_t* topk_idx,
                      const double* gates, const uint16_t* dY, int32_t expert, double* dW13, double* dW2) {
  ora_expert_wgrad_kept(cp, X, W13, W2, W13s, W2s, topk_idx, gates, dY, expert, dW13, dW2, nullptr);
}

// Weight gradients counting only kept assignments (c_kept may be null: all kept).
void ora_expert_wgrad_kept(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                           const uint16_t* W13s, const uint16_t* W2s, const int32_t* topk_idx, const double* gates,
                           const uint16_t* dY, int32_t expert, double* dW13, double* dW2, const int32_t* c_kept) {
  const ora_cfg c = *cp;
  const int H = c.H, k = c.k;
  const int F = expert < 0 ? c.F_shared : c.F;
  const uint16_t* w13 = expert < 0 ? W13s : W13 + (size_t)expert * 2 * F * H;
  const uint16_t* w2 = expert < 0 ? W2s : W2 + (size_t)expert * H * F;
  // the (token, gate) pairs routed to this expert, in token order
  std::vector<int64_t> toks;
  std::vector<double> gsel;
  for (int64_t t = 0; t < c.T; ++t) {
    if (expert < 0) {
      toks.push_back(t);
      gsel.push_back(1.0);
      continue;
    }
    for (int j = 0; j < k; ++j)
      if (topk_idx[t * k + j] == expert && (!c_kept || c_kept[t * k + j])) {
        toks.push_back(t);
        gsel.push_back(gates[t * k + j]);
      }
  }
  std::fill(dW13, dW13 + (size_t)2 * F * H, 0.0);
  std::fill(dW2, dW2 + (size_t)H * F, 0.0);
  const int64_t n = (int64_t)toks.size();
  const int64_t chunk = 512;
  std::vector<double> xs, dyps, as, dGs, dUs;
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t m = std::min(chunk, n - c0);
    xs.assign((size_t)m * H, 0.0);
    dyps.assign((size_t)m * H, 0.0);
    as.assign((size_t)m * F, 0.0);
    dGs.assign((size_t)m * F, 0.0);
    dUs.assign((size_t)m * F, 0.0);
    parallel_for(m, nthreads_of(c), [&](int64_t i) {
      const int64_t t = toks[c0 + i];
      std::vector<double> gr(F), ur(F), ye(H), dxe(H);
      double* x = &xs[(size_t)i * H];
      double* dyp = &dyps[(size_t)i * H];
      for (int h = 0; h < H; ++h) x[h] = bf(X[(size_t)t * H + h]);
      expert_fwd(c, F, w13, w2, x, gr.data(), ur.data(), &as[(size_t)i * F], ye.data());
      if (c.gated && expert >= 0) {
        // the gradient of the gated output is dY itself; dW2 pairs it with the gated
        // activation recomputed from the stored g, u
        const double gj = gsel[c0 + i];
        double dgate;
        for (int h = 0; h < H; ++h) dyp[h] = bf(dY[(size_t)t * H + h]);
        for (int f = 0; f < F; ++f) as[(size_t)i * F + f] = maybe_r(c, gj * (silu(gr[f]) * ur[f]));
        expert_bwd(c, F, w13, w2, gr.data(), ur.data(), dyp, &dGs[(size_t)i * F], &dUs[(size_t)i * F],
                   dxe.data(), gj, &dgate);
        return;
      }
      for (int h = 0; h < H; ++h) dyp[h] = maybe_r(c, gsel[c0 + i] * bf(dY[(size_t)t * H + h]));
      expert_bwd(c, F, w13, w2, gr.data(), ur.data(), dyp, &dGs[(size_t)i * F], &dUs[(size_t)i * F], dxe.data());
    });
    if (c.fp8) {
      // wgrad operands: 128x1 blocks along the expert's tokens (in token order, 128 per block)
      qdq_columns(dyps.data(), m, H);
      qdq_columns(as.data(), m, F);
      qdq_columns(xs.data(), m, H);
      std::vector<double> cat((size_t)m * 2 * F);
      for (int64_t i = 0; i < m; ++i)
        for (int f = 0; f < F; ++f) {
          cat[(size_t)i * 2 * F + f] = dGs[(size_t)i * F + f];
          cat[(size_t)i * 2 * F + F + f] = dUs[(size_t)i * F + f];
        }
      qdq_columns(cat.data(), m, 2 * F);
      for (int64_t i = 0; i < m; ++i)
        for (int f = 0; f < F; ++f) {
          dGs[(size_t)i * F + f] = cat[(size_t)i * 2 * F + f];
          dUs[(size_t)i * F + f] = cat[(size_t)i * 2 * F + F + f];
        }
    }
    // dW2[h,f] += dyp[h] a[f]; dWg[f,h] += dG[f] x[h]; dWu[f,h] += dU[f] x[h]
    parallel_for(H, nthreads_of(c), [&](int64_t h) {
      double* row = dW2 + (size_t)h * F;
      for (int64_t i = 0; i < m; ++i) {
        const double d = dyps[(size_t)i * H + h];
        const double* a = &as[(size_t)i * F];
        for (int f = 0; f < F; ++f) row[f] += d * a[f];
      }
    });
    parallel_for(2 * (int64_t)F, nthreads_of(c), [&](int64_t r) {
      double* row = dW13 + (size_t)r * H;
      const bool up = r >= F;
      const int f = (int)(up ? r - F : r);
      for (int64_t i = 0; i < m; ++i) {
        const double d = up ? dUs[(size_t)i * F + f] : dGs[(size_t)i * F + f];
        const double* x = &xs[(size_t)i * H];
        for (int h = 0; h < H; ++h) row[h] += d * x[h];
      }
    });
  }
  if (c.mirror) {
    for (size_t i = 0; i < (size_t)2 * F * H; ++i) dW13[i] = rbf(dW13[i]);
    for (size_t i = 0; i < (size_t)H * F; ++i) dW2[i] = rbf(dW2[i]);
  }
}

// The weight gradients of one expert restricted to a few FFN indices f = cols[0..ncols):
// rows f and F+f of dW13 (dW13_rows [2*ncols, H]: the gate rows of cols, then their up
// rows) and column f of dW2 (dW2_cols [H, ncols]).  Each entry is formed by the same
// operations, roundings and summation order as in ora_expert_wgrad_kept (the token rows of
// the expert in token order, the same 128-token FP8 column blocks), so it equals that
// function's value; this form costs O(rows * ncols * H) instead of O(rows * F * H), which
// makes experts with thousands of rows of a 7168-wide layer checkable.
void ora_expert_wgrad_cols(const ora_cfg* cp, const uint16_t* X, const uint16_t* W13, const uint16_t* W2,
                           const uint16_t* W13s, const uint16_t* W2s, const int32_t* topk_idx, const double* gates,
                           const uint16_t* dY, int32_t expert, int32_t ncols, const int32_t* cols,
                           double* dW13_rows, double* dW2_cols, const int32_t* c_kept) {
  const ora_cfg c = *cp;
  const int H = c.H, k = c.k, nc = ncols;
  const int F = expert < 0 ? c.F_shared : c.F;
  const uint16_t* w13 = expert < 0 ? W13s : W13 + (size_t)expert * 2 * F * H;
  const uint16_t* w2 = expert < 0 ? W2s : W2 + (size_t)expert * H * F;
  std::vector<int64_t> toks;
  std::vector<double> gsel;
  for (int64_t t = 0; t < c.T; ++t) {
    if (expert < 0) {
      toks.push_back(t);
      gsel.push_back(1.0);
      continue;
    }
    for (int j = 0; j < k; ++j)
      if (topk_idx[t * k + j] == expert && (!c_kept || c_kept[t * k + j])) {
        toks.push_back(t);
        gsel.push_back(gates[t * k + j]);
      }
  }
  std::fill(dW13_rows, dW13_rows + (size_t)2 * nc * H, 0.0);
  std::fill(dW2_cols, dW2_cols + (size_t)H * nc, 0.0);
  const int64_t n = (int64_t)toks.size();
  const int64_t chunk = 512;
  // per chunk: x and the expert-output gradient of every row (all H), the activation and
  // dG, dU of the sampled indices only
  std::vector<double> xs, dyps, as, dGs, dUs;
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t m = std::min(chunk, n - c0);
    xs.assign((size_t)m * H, 0.0);
    dyps.assign((size_t)m * H, 0.0);
    as.assign((size_t)m * nc, 0.0);
    dGs.assign((size_t)m * nc, 0.0);
    dUs.assign((size_t)m * nc, 0.0);
    parallel_for(m, nthreads_of(c), [&](int64_t i) {
      const int64_t t = toks[c0 + i];
      const double gj = gsel[c0 + i];
      const bool gated = c.gated && expert >= 0;
      double* x = &xs[(size_t)i * H];
      double* dyp = &dyps[(size_t)i * H];
      for (int h = 0; h < H; ++h) x[h] = bf(X[(size_t)t * H + h]);
      std::vector<double> xq, dq;
      const double* xin = x;
      if (c.fp8) {  // FC1 reads the token row as 1x128 blocks along H
        xq.resize(H);
        qdq_blocks(x, xq.data(), H, 128);
        xin = xq.data();
      }
      for (int h = 0; h < H; ++h) dyp[h] = gated ? bf(dY[(size_t)t * H + h]) : maybe_r(c, gj * bf(dY[(size_t)t * H + h]));
      const double* din = dyp;
      if (c.fp8) {  // FC2 dgrad reads the output gradient as 1x128 blocks along H
        dq.resize(H);
        qdq_blocks(dyp, dq.data(), H, 128);
        din = dq.data();
      }
      for (int q = 0; q < nc; ++q) {
        const int f = cols[q];
        double g = 0, u = 0;
        const uint16_t* wg = w13 + (size_t)f * H;
        const uint16_t* wu = w13 + (size_t)(F + f) * H;
        for (int h = 0; h < H; ++h) {
          g += bf(wg[h]) * xin[h];
          u += bf(wu[h]) * xin[h];
        }
        const double gr = maybe_r(c, g), ur = maybe_r(c, u);
        as[(size_t)i * nc + q] = gated ? maybe_r(c, gj * (silu(gr) * ur)) : maybe_r(c, 1.0 * (silu(g) * u));
        double dA = 0;
        for (int h = 0; h < H; ++h) dA += bf(w2[(size_t)h * F + f]) * din[h];
        if (gated) dA *= gj;
        dGs[(size_t)i * nc + q] = maybe_r(c, dA * ur * dsilu(gr));
        dUs[(size_t)i * nc + q] = maybe_r(c, dA * silu(gr));
      }
    });
    if (c.fp8) {  // wgrad operands: 128x1 blocks along the expert's tokens
      qdq_columns(dyps.data(), m, H);
      qdq_columns(as.data(), m, nc);
      qdq_columns(xs.data(), m, H);
      qdq_columns(dGs.data(), m, nc);
      qdq_columns(dUs.data(), m, nc);
    }
    parallel_for(H, nthreads_of(c), [&](int64_t h) {
      double* row = dW2_cols + (size_t)h * nc;
      for (int64_t i = 0; i < m; ++i) {
        const double d = dyps[(size_t)i * H + h];
        for (int q = 0; q < nc; ++q) row[q] += d * as[(size_t)i * nc + q];
      }
    });
    parallel_for(2 * (int64_t)nc, nthreads_of(c), [&](int64_t r) {
      double* row = dW13_rows + (size_t)r * H;
      const bool up = r >= nc;
      const int q = (int)(up ? r - nc : r);
      for (int64_t i = 0; i < m; ++i) {
        const double d = up ? dUs[(size_t)i * nc + q] : dGs[(size_t)i * nc + q];
        const double* x = &xs[(size_t)i * H];
        for (int h = 0; h < H; ++h) row[h] += d * x[h];
      }
    });
  }
  if (c.mirror) {
    for (size_t i = 0; i < (size_t)2 * nc * H; ++i) dW13_rows[i] = rbf(dW13_rows[i]);
    for (size_t i = 0; i < (size_t)H * nc; ++i) dW2_cols[i] = rbf(dW2_cols[i]);
  }
}

// Router logit gradients for given gate gradients (summary page, "Method": the router
// is differentiated through its gates): per token, the exact gradient of the gates with
// respect to the logits for the given selection (token_dlogits), applied to dgates.
// logits [T,E], gates [T,k], dgates [T,k], dlogits [T,E] (double); topk_idx [T,k].
void ora_router_dlogits(const ora_cfg* cp, const double* logits, const int32_t* topk_idx, const double* gates,
                        const double* dgates, double* dlogits) {
  const ora_cfg c = *cp;
  for (int64_t t = 0; t < c.T; ++t)
    token_dlogits(c, logits + (size_t)t * c.E, topk_idx + (size_t)t * c.k, gates + (size_t)t * c.k,
                  dgates + (size_t)t * c.k, dlogits + (size_t)t * c.E);
}

// Router weight gradients from the double dlogits of all T tokens:
// dW_r[e,h] = sum_t dl[t,e] x[t,h];  dlogit_bias[e] = sum_t dl[t,e].
void ora_router_wgrad(const ora_cfg* cp, const uint16_t* X, const double* dlogits, double* dWr,
                      double* dlogit_bias) {
  const ora_cfg c = *cp;
  const int H = c.H, E = c.E;
  parallel_for(E, nthreads_of(c), [&](int64_t e) {
    double* row = dWr + (size_t)e * H;
    for (int h = 0; h < H; ++h) row[h] = 0.0;
    double sb = 0;
    for (int64_t t = 0; t < c.T; ++t) {
      const double d = dlogits[(size_t)t * E + e];
      sb += d;
      if (d == 0.0) continue;
      for (int h = 0; h < H; ++h) row[h] += d * bf(X[(size_t)t * H + h]);
    }
    if (dlogit_bias) dlogit_bias[e] = sb;
  });
}

// 128x128 block quantization of nmat row-major [rows x cols] bf16 matrices; the
// dequantized values (exact in bf16) are written back as bf16 bit patterns.
void ora_qdq_weight_blocks(const uint16_t* W, int64_t nmat, int rows, int cols, uint16_t* out) {
  unsigned hc = std::thread::hardware_concurrency();
  parallel_for(nmat * ((rows + 127) / 128), hc ? (int)hc : 1, [&](int64_t job) {
    const int64_t mi = job / ((rows + 127) / 128);
    const int r0 = (int)(job % ((rows + 127) / 128)) * 128, r1 = std::min(rows, r0 + 128);
    const uint16_t* w = W + mi * rows * (int64_t)cols;
    uint16_t* o = out + mi * rows * (int64_t)cols;
    for (int c0 = 0; c0 < cols; c0 += 128) {
      const int c1 = std::min(cols, c0 + 128);
      double amax = 0;
      for (int r = r0; r < r1; ++r)
        for (int cc = c0; cc < c1; ++cc) amax = std::max(amax, std::fabs(bf(w[(int64_t)r * cols + cc])));
      const double sc = block_scale(amax);
      for (int r = r0; r < r1; ++r)
        for (int cc = c0; cc < c1; ++cc) {
          const double q = e4m3_rne(bf(w[(int64_t)r * cols + cc]) / sc) * sc;
          float f = (float)q;  // exact: 4 significant bits
          uint32_t u;
          std::memcpy(&u, &f, 4);
          o[(int64_t)r * cols + cc] = (uint16_t)(u >> 16);
        }
    }
  });
}

// E4M3 rounding and block quantization, exposed for their own tests.
void ora_e4m3(const double* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_rne(in[i]);
}
void ora_qdq_blocks(const double* in, double* out, int64_t n, int blk) { qdq_blocks(in, out, (int)n, blk); }

// bf16 rounding as used in mirror mode, exposed for its own test.
void ora_round_bf16(const double* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = rbf(in[i]);
}

}  // extern "C"
