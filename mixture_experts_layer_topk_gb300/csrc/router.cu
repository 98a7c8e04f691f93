// Route stage and its backward.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (summary
// page, "Method"): the router is a learned linear projection of the hidden
// states, kept in FP32, followed by softmax or sigmoid scoring and top-k
// selection.  With a workspace the projection runs on the tensor cores
// (router_tc.cu: exact bf16 split of W_r, block sums promoted to FP32 registers)
// and a routing pass (one warp per token: scores, optional group limit, top-k by
// warp reductions, gates, histogram) follows.  Without one, the projection runs
// on the CUDA cores: fused with the routing into one launch for E <= 32, a
// register-tiled split-K FP32 GEMM for larger E.  The backward's products (dW_r,
// dX_router) run on the tensor cores from bf16 splits for E > 32 (for small E they
// are HBM-bound either way, and the CUDA-core kernels take fewer launches).
//
// Selection rule: key = logit (+ sel_bias) for softmax, sigmoid(logit)
// (+ sel_bias) for sigmoid, formed in FP32; the k experts are listed in
// descending key order, exact ties going to the lower expert index.  With
// n_group > 1 the experts form contiguous groups; a group's score is the sum
// of its two largest keys (or its largest key), the topk_group best groups
// are kept (ties to the lower group id) and top-k runs inside them.
#include <float.h>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

struct RouteArgs {
  const uint16_t* X;
  const float* Wr;
  const float* logit_bias;
  const float* sel_bias;
  float* logits;
  float* scores;
  int32_t* topk_idx;
  float* gates;
  int32_t* counts;
  int T, H, E, k;
  int score_fn, renorm;
  float gate_scale;
  int n_group, topk_group, group_score;
  const int32_t* given;  // router replay: the selection to use instead of top-k (nullable)
  // k_route_rows: the product is logits + the nmore partial [T,E] sums at more (fixed order)
  const float* more;
  int nmore;
};

// Order-preserving map of an fp32 key to uint32: a < b as floats iff ord_key(a) <
// ord_key(b).  -0 is first turned into +0, so the two zeros tie as they do under
// float comparison.
__device__ __forceinline__ uint32_t ord_key(float v) {
  const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_val(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// (value, index) maximum over the warp; ties to the lower index: the warp-wide
// maximum of the ordered keys (one redux.sync), then the least index among the
// lanes that hold it (another).  Lanes with no candidate pass (-FLT_MAX, INT_MAX).
__device__ __forceinline__ void warp_argmax(float& v, int& e) {
  const uint32_t u = ord_key(v);
  const uint32_t m = __reduce_max_sync(0xffffffffu, u);
  e = (int)__reduce_min_sync(0xffffffffu, u == m ? (uint32_t)e : 0xffffffffu);
  v = ord_val(m);
}

// ---------------------------------------------------------------- exact bf16 splits
// w = hi + mid + lo exactly: each term is the leading 8 significant bits of what is
// left (truncation), and an fp32 has 24, so the third remainder fits in a bf16.
__device__ __forceinline__ void split3(float w, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
  hi = (uint16_t)(__float_as_uint(w) >> 16);
  const float r1 = __fsub_rn(w, __uint_as_float((uint32_t)hi << 16));
  mid = (uint16_t)(__float_as_uint(r1) >> 16);
  const float r2 = __fsub_rn(r1, __uint_as_float((uint32_t)mid << 16));
  lo = (uint16_t)(__float_as_uint(r2) >> 16);
}

// Scores, selection and gates of token t by one warp.  lrow: the token's E
// logits (bias included) in shared memory.  hist: per-CTA expert histogram.
template <int V>
__device__ void route_token(const RouteArgs& a, int t, const float* lrow, int* hist) {
  const int lane = threadIdx.x & 31;
  const int E = a.E;
  float l[V], key[V];
  uint32_t excl = 0;
  float lmax = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    const bool valid = e < E;
    l[i] = valid ? lrow[e] : -FLT_MAX;
    if (!valid) excl |= 1u << i;
    lmax = fmaxf(lmax, l[i]);
  }
  // scores
  float M = 0.f, Zinv = 0.f;
  if (a.score_fn == 0) {
    M = warp_max(lmax);
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (!(excl >> i & 1)) z += expf(l[i] - M);
    Zinv = 1.0f / warp_sum(z);
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float s = a.score_fn == 0 ? expf(l[i] - M) * Zinv : 1.0f / (1.0f + expf(-l[i]));
      a.logits[(size_t)t * E + e] = l[i];
      a.scores[(size_t)t * E + e] = s;
      const float base = a.score_fn == 0 ? l[i] : s;
      key[i] = a.sel_bias ? base + a.sel_bias[e] : base;
    } else {
      key[i] = -FLT_MAX;
    }
  }
  // group limit
  if (a.n_group > 1 && !a.given) {
    const int per = E / a.n_group;
    int gi[V];  // group of each of this lane's experts
#pragma unroll
    for (int i = 0; i < V; ++i) gi[i] = (lane + 32 * i) / per;
    float my_gs = -FLT_MAX;
    if (per == 32 && a.n_group == V) {
      // each group is one register of every lane (expert lane + 32 g): its best two by one
      // warp arg-max each, no scan over the lane's other registers
#pragma unroll
      for (int g = 0; g < V; ++g) {
        const bool ok = !(excl >> g & 1);
        const int eg = lane + 32 * g;
        float v1 = ok ? key[g] : -FLT_MAX;
        int e1 = ok ? eg : INT_MAX;
        warp_argmax(v1, e1);
        float gs = v1;
        if (a.group_score == 0) {
          const bool ok2 = ok && eg != e1;
          float v2 = ok2 ? key[g] : -FLT_MAX;
          int e2 = ok2 ? eg : INT_MAX;
          warp_argmax(v2, e2);
          gs = v1 + v2;
        }
        if (lane == g) my_gs = gs;
      }
    } else {
      for (int g = 0; g < a.n_group; ++g) {
        float v1 = -FLT_MAX;
        int e1 = INT_MAX;
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const int e = lane + 32 * i;
          if (!(excl >> i & 1) && gi[i] == g && (key[i] > v1 || (key[i] == v1 && e < e1))) {
            v1 = key[i];
            e1 = e;
          }
        }
        warp_argmax(v1, e1);
        float gs = v1;
        if (a.group_score == 0 && per > 1) {
          float v2 = -FLT_MAX;
          int e2 = INT_MAX;
#pragma unroll
          for (int i = 0; i < V; ++i) {
            const int e = lane + 32 * i;
            if (!(excl >> i & 1) && gi[i] == g && e != e1 && (key[i] > v2 || (key[i] == v2 && e < e2))) {
              v2 = key[i];
              e2 = e;
            }
          }
          warp_argmax(v2, e2);
          gs = v1 + v2;
        }
        if (lane == g) my_gs = gs;
      }
    }
    uint32_t keep = 0;
    for (int r = 0; r < a.topk_group; ++r) {
      float v = (lane < a.n_group && !(keep >> lane & 1)) ? my_gs : -FLT_MAX;
      int g = (lane < a.n_group && !(keep >> lane & 1)) ? lane : INT_MAX;
      warp_argmax(v, g);
      keep |= 1u << g;
    }
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(keep >> gi[i] & 1)) excl |= 1u << i;
    }
  }
  // top-k: lane j ends up holding the j-th selected expert (router replay: read it)
  int my_e = -1;
  if (a.given && lane < a.k) {
    my_e = a.given[(size_t)t * a.k + lane];
    if ((unsigned)my_e >= (unsigned)E) my_e = 0;  // ids are validated on the host side of replay callers
  }
  for (int j = 0; j < (a.given ? 0 : a.k); ++j) {
    float v = -FLT_MAX;
    int e = INT_MAX;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int ee = lane + 32 * i;
      if (!(excl >> i & 1) && (key[i] > v || (key[i] == v && ee < e))) {
        v = key[i];
        e = ee;
      }
    }
    warp_argmax(v, e);
    if (lane == j) my_e = e;
    if ((e & 31) == lane) excl |= 1u << (e >> 5);
  }
  // gates
  const bool act = lane < a.k;
  const float lj = act ? lrow[my_e] : -FLT_MAX;
  float g = 0.f;
  if (a.score_fn == 0) {
    if (a.renorm) {
      const float m = warp_max(lj);
      const float ex = act ? expf(lj - m) : 0.f;
      g = a.gate_scale * ex / warp_sum(ex);
    } else {
      g = act ? a.gate_scale * expf(lj - M) * Zinv : 0.f;
    }
  } else {
    const float s = act ? 1.0f / (1.0f + expf(-lj)) : 0.f;
    g = a.renorm ? a.gate_scale * s / warp_sum(s) : a.gate_scale * s;
  }
  if (act) {
    a.topk_idx[(size_t)t * a.k + lane] = my_e;
    a.gates[(size_t)t * a.k + lane] = g;
    atomicAdd(&hist[my_e], 1);
  }
}

// E <= 32: one warp per token (TPW tokens at a time), lanes split H.
// E <= 32: a CTA routes 8 * TPW tokens (TPW per warp).  W_r goes through shared memory
// in chunks of KC columns (EMAX * KC * 4 = 32 KB), loaded once per CTA; each warp
// streams its tokens' X over the chunk and accumulates from shared memory.
template <int EMAX, int TPW, int KC>
__global__ void __launch_bounds__(256) k_router_small(RouteArgs a) {
  __shared__ __align__(16) float wsm[EMAX * KC];
  __shared__ float lrows[8][TPW][EMAX];
  __shared__ int hist[EMAX];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < EMAX; i += blockDim.x) hist[i] = 0;
  const int H = a.H, E = a.E;
  for (int base = blockIdx.x * 8 * TPW; base < a.T; base += gridDim.x * 8 * TPW) {
    const int t0 = base + warp * TPW;
    float acc[TPW][EMAX];
#pragma unroll
    for (int u = 0; u < TPW; ++u)
#pragma unroll
      for (int e = 0; e < EMAX; ++e) acc[u][e] = 0.f;
    for (int k0 = 0; k0 < H; k0 += KC) {
      const int kc = H - k0 < KC ? H - k0 : KC;  // a multiple of 8
      __syncthreads();                            // the previous chunk is consumed
      for (int i = threadIdx.x; i < EMAX * (kc / 4); i += 256) {
        const int e = i / (kc / 4), j = i % (kc / 4);
        const float4 w = e < E ? __ldg(reinterpret_cast<const float4*>(a.Wr + (size_t)e * H + k0) + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(&wsm[e * KC + 4 * j]) = w;
      }
      __syncthreads();
      // all of this lane's X vectors of the chunk are loaded before any is used
      constexpr int IT = KC / 256;  // 16-byte vectors per lane per token and chunk
      uint4 xv[IT][TPW];
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int c = it * 32 + lane;
#pragma unroll
        for (int u = 0; u < TPW; ++u)
          xv[it][u] = c < kc / 8 && t0 + u < a.T
                          ? __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)(t0 + u) * H + k0) + c)
                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int c = it * 32 + lane;
        if (c >= kc / 8) continue;
        float x[TPW][8];
#pragma unroll
        for (int u = 0; u < TPW; ++u) unpack8(xv[it][u], x[u]);
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
          const float4 w0 = *reinterpret_cast<const float4*>(&wsm[e * KC + 8 * c]);
          const float4 w1 = *reinterpret_cast<const float4*>(&wsm[e * KC + 8 * c + 4]);
#pragma unroll
          for (int u = 0; u < TPW; ++u) {
            float sum = acc[u][e];
            sum = fmaf(x[u][0], w0.x, sum);
            sum = fmaf(x[u][1], w0.y, sum);
            sum = fmaf(x[u][2], w0.z, sum);
            sum = fmaf(x[u][3], w0.w, sum);
            sum = fmaf(x[u][4], w1.x, sum);
            sum = fmaf(x[u][5], w1.y, sum);
            sum = fmaf(x[u][6], w1.z, sum);
            sum = fmaf(x[u][7], w1.w, sum);
            acc[u][e] = sum;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < TPW; ++u)
#pragma unroll
      for (int e = 0; e < EMAX; ++e) acc[u][e] = warp_sum(acc[u][e]);
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < TPW; ++u)
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
          if (e < E) lrows[warp][u][e] = acc[u][e] + (a.logit_bias ? a.logit_bias[e] : 0.f);
    }
    __syncwarp();
    for (int u = 0; u < TPW; ++u)
      if (t0 + u < a.T) route_token<1>(a, t0 + u, lrows[warp][u], hist);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (hist[e]) atomicAdd(&a.counts[e], hist[e]);
}

// 32 < E <= EP: a CTA computes the logits of BT tokens for all experts with a
// register-tiled FP32 GEMM (TM tokens x 8 experts per thread), then its warps
// route the tokens.
// ---------------------------------------------------------------- E > 32
// Logits on the CUDA cores in two passes.  k_router_gemm: P = X W_r^T over one half
// of K (FP32 FMA, register-tiled: a CTA computes 128 tokens x BE experts, each of its
// 256 threads an 8 x BE/16 block), the two halves written to the logits and scores
// buffers.  k_route_rows: one warp per token sums the halves in a fixed order, adds
// the bias and routes the token (route_token), overwriting both rows.
constexpr int kRgBT = 128, kRgBK = 16;

template <int BE>
__global__ void __launch_bounds__(256, 2) k_router_gemm(const uint16_t* __restrict__ X, const float* __restrict__ Wr,
                                                        int T, int H, int E, float* __restrict__ P0,
                                                        float* __restrict__ P1) {
  constexpr int BT = kRgBT, BK = kRgBK, NE = BE / 16;
  constexpr int WV = BE * BK / 4 / 256;  // float4 W vectors per thread per K step
  __shared__ __align__(16) float Xs[2][BK][BT];
  __shared__ __align__(16) float Ws[2][BK][BE];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int t0 = blockIdx.x * BT, e0 = blockIdx.y * BE;
  const int half = H / BK / 2 * BK;  // K of the first pass
  const int kbeg = blockIdx.z ? half : 0, kend = blockIdx.z ? H : half;
  float* P = blockIdx.z ? P1 : P0;
  float acc[8][NE];
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int n = 0; n < NE; ++n) acc[m][n] = 0.f;
  // loaders: X as 16-byte vectors (8 bf16 along K) of token tid % 128, W as float4
  // (4 fp32 along K) of expert i % BE
  const int xt = tid & 127, xh = tid >> 7;
  const bool xok = t0 + xt < T;
  uint4 xr;
  float4 wr[WV];
  auto load = [&](int k0) {
    xr = xok ? __ldg(reinterpret_cast<const uint4*>(X + (size_t)(t0 + xt) * H + k0) + xh) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + 256 * v, e = i % BE, j = i / BE;
      wr[v] = e0 + e < E ? __ldg(reinterpret_cast<const float4*>(Wr + (size_t)(e0 + e) * H + k0) + j)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store = [&](int b) {
    float x[8];
    unpack8(xr, x);
#pragma unroll
    for (int q = 0; q < 8; ++q) Xs[b][xh * 8 + q][xt] = x[q];
#pragma unroll
    for (int v = 0; v < WV; ++v) {
      const int i = tid + 256 * v, e = i % BE, j = i / BE;
      Ws[b][4 * j + 0][e] = wr[v].x;
      Ws[b][4 * j + 1][e] = wr[v].y;
      Ws[b][4 * j + 2][e] = wr[v].z;
      Ws[b][4 * j + 3][e] = wr[v].w;
    }
  };
  if (kbeg < kend) {
    load(kbeg);
    store(0);
  }
  __syncthreads();
  int b = 0;
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    const bool more = k0 + BK < kend;
    if (more) load(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      // rows ty*4..+3 and 64+ty*4..+3; columns tx*4..+3 (and 64+tx*4..+3 when BE = 128)
      const float4 x0 = *reinterpret_cast<const float4*>(&Xs[b][kk][ty * 4]);
      const float4 x1 = *reinterpret_cast<const float4*>(&Xs[b][kk][64 + ty * 4]);
      const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      float wb[NE];
      const float4 w0 = *reinterpret_cast<const float4*>(&Ws[b][kk][tx * 4]);
      wb[0] = w0.x; wb[1] = w0.y; wb[2] = w0.z; wb[3] = w0.w;
      if constexpr (NE == 8) {
        const float4 w1 = *reinterpret_cast<const float4*>(&Ws[b][kk][64 + tx * 4]);
        wb[4] = w1.x; wb[5] = w1.y; wb[6] = w1.z; wb[7] = w1.w;
      }
#pragma unroll
      for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int n = 0; n < NE; ++n) acc[m][n] = fmaf(xa[m], wb[n], acc[m][n]);
    }
    if (more) store(b ^ 1);
    __syncthreads();
    b ^= 1;
  }
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int t = t0 + (m < 4 ? ty * 4 + m : 64 + ty * 4 + m - 4);
    if (t >= T) continue;
#pragma unroll
    for (int h = 0; h < NE / 4; ++h) {
      const int e = e0 + h * 64 + tx * 4;
      if (e < E)
        *reinterpret_cast<float4*>(P + (size_t)t * E + e) =
            make_float4(acc[m][4 * h], acc[m][4 * h + 1], acc[m][4 * h + 2], acc[m][4 * h + 3]);
    }
  }
}

template <int V>
__global__ void __launch_bounds__(256) k_route_rows(RouteArgs a) {
  __shared__ float lrows[8][32 * V];
  __shared__ int hist[32 * V];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * V; i += 256) hist[i] = 0;
  __syncthreads();
  const int E = a.E;
  for (int t = blockIdx.x * 8 + warp; t < a.T; t += gridDim.x * 8) {
    // the product is split over K: logits holds the first part, `more` the others
    for (int e = lane; e < E; e += 32) {
      float p = a.logits[(size_t)t * E + e];
      for (int s = 0; s < a.nmore; ++s) p += a.more[((size_t)s * a.T + t) * E + e];
      lrows[warp][e] = p + (a.logit_bias ? a.logit_bias[e] : 0.f);
    }
    __syncwarp();
    route_token<V>(a, t, lrows[warp], hist);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256)
    if (hist[e]) atomicAdd(&a.counts[e], hist[e]);
}

template <int V>
cudaError_t launch_route_rows(const RouteArgs& a, cudaStream_t st, int nsm) {
  // a token's routing is a chain of dependent warp reductions: many warps per SM hide it
  int g2 = (a.T + 7) / 8;
  g2 = g2 < 8 * nsm ? g2 : 8 * nsm;
  k_route_rows<V><<<g2, 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int BE, int V>
cudaError_t launch_two_pass(RouteArgs a, cudaStream_t st, int nsm) {
  dim3 g1((a.T + kRgBT - 1) / kRgBT, (a.E + BE - 1) / BE, 2);
  k_router_gemm<BE><<<g1, 256, 0, st>>>(a.X, a.Wr, a.T, a.H, a.E, a.logits, a.scores);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  a.more = a.scores;  // the second K half; each warp reads its token's row before overwriting it
  a.nmore = 1;
  return launch_route_rows<V>(a, st, nsm);
}

template <int EMAX, int TPW, int KC>
cudaError_t launch_small(const RouteArgs& a, cudaStream_t st, int nsm) {
  const int groups = (a.T + 8 * TPW - 1) / (8 * TPW);  // 8 * TPW tokens per CTA
  const int grid = groups < 8 * nsm ? groups : 8 * nsm;
  k_router_small<EMAX, TPW, KC><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward

struct RouteBwdArgs {
  const float* logits;
  const int32_t* topk_idx;
  const float* gates;
  const float* dgates;
  float* dl;  // [T,E]
  int T, E, k;
  int score_fn, renorm;
  float gate_scale;
  // optional exact bf16 splits of dl for the tensor-core router GEMMs
  uint16_t* dl_rows;  // [3*Tp, Ep]: rows t, Tp+t, 2Tp+t hold hi, mid, lo
  uint16_t* dl_cols;  // [T, 3*Ep]: column blocks hi, hi, mid
  int Tp, Ep;
};

// dlogits of one token per warp: the exact gradient of the gates with respect
// to the logits for the fixed selection, applied to dgates.
template <int V>
__global__ void __launch_bounds__(256) k_router_dlogits(RouteBwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int E = a.E, k = a.k;
  const float al = a.gate_scale;
  const bool act = lane < k;
  const int ej = act ? a.topk_idx[(size_t)t * k + lane] : 0;
  const float gj = act ? a.gates[(size_t)t * k + lane] : 0.f;
  const float dgj = act ? a.dgates[(size_t)t * k + lane] : 0.f;
  const float lj = act ? a.logits[(size_t)t * E + ej] : 0.f;
  const float* lrow = a.logits + (size_t)t * E;
  float dlj = 0.f;        // gradient at the selected expert held by lane j
  float dense_s = 0.f;    // softmax without renorm: sum_j dg_j p_j
  float M = 0.f, Zinv = 0.f;
  if (a.score_fn == 0) {
    if (a.renorm) {
      const float q = gj / al;
      const float s = warp_sum(act ? q * dgj : 0.f);
      dlj = al * q * (dgj - s);
    } else {
      float lmax = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane + 32 * i;
        if (e < E) lmax = fmaxf(lmax, lrow[e]);
      }
      M = warp_max(lmax);
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane + 32 * i;
        if (e < E) z += expf(lrow[e] - M);
      }
      Zinv = 1.0f / warp_sum(z);
      const float pj = act ? expf(lj - M) * Zinv : 0.f;
      dense_s = warp_sum(act ? dgj * pj : 0.f);
    }
  } else {
    const float sj = act ? 1.0f / (1.0f + expf(-lj)) : 0.f;
    if (a.renorm) {
      const float S = warp_sum(sj);
      const float c = warp_sum(act ? dgj * gj : 0.f) / al;
      dlj = (al / S) * (dgj - c) * sj * (1.0f - sj);
    } else {
      dlj = al * dgj * sj * (1.0f - sj);
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    float v = 0.f, dgm = 0.f;
    for (int j = 0; j < k; ++j) {
      const int ej2 = __shfl_sync(0xffffffffu, ej, j);
      const float d2 = __shfl_sync(0xffffffffu, dlj, j);
      const float g2 = __shfl_sync(0xffffffffu, dgj, j);
      if (ej2 == e) {
        v = d2;
        dgm = g2;
      }
    }
    if (a.score_fn == 0 && !a.renorm && e < E) {
      const float p = expf(lrow[e] - M) * Zinv;
      v = al * p * (dgm - dense_s);
    }
    if (e < E) a.dl[(size_t)t * E + e] = v;
    if (a.dl_rows && e < a.Ep) {
      uint16_t hi = 0, mid = 0, lo = 0;
      if (e < E) split3(v, hi, mid, lo);
      a.dl_rows[(size_t)t * a.Ep + e] = hi;
      a.dl_rows[((size_t)a.Tp + t) * a.Ep + e] = mid;
      a.dl_rows[((size_t)2 * a.Tp + t) * a.Ep + e] = lo;
      uint16_t* c = a.dl_cols + (size_t)t * 3 * a.Ep + e;
      c[0] = hi;
      c[a.Ep] = hi;
      c[2 * a.Ep] = mid;
    }
  }
}

// dlogit_bias[e] = sum_t dl[t,e]; one CTA per expert, fixed summation order.
__global__ void __launch_bounds__(256) k_colsum(const float* dl, int T, int E, float* out) {
  const int e = blockIdx.x;
  float s = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) s += dl[(size_t)t * E + e];
  __shared__ float red[8];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 0.f;
    for (int i = 0; i < 8; ++i) r += red[i];
    out[e] = r;
  }
}

// C[M,N] = sum_k A(m,k) B(k,n), FP32, 128x128 tiles, 8x8 per thread.
// A(m,k) = A[m*lda + k] (A_KM=false) or A[k*lda + m] (A_KM=true); B(k,n) = B[k*ldb + n].
// Split-K over blockIdx.z: split z covers k in [z*kps, (z+1)*kps) and writes C + z*c_zstride.
template <bool A_KM, typename TB>
__global__ void __launch_bounds__(256) k_sgemm(int M, int N, int K, const float* __restrict__ A, int64_t lda,
                                               const TB* __restrict__ B, int64_t ldb, float* __restrict__ Cm,
                                               int64_t ldc, int kps, int64_t c_zstride) {
  __shared__ __align__(16) float As[8][128 + 4];
  __shared__ __align__(16) float Bs[8][128 + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
  const int kbeg = blockIdx.z * kps;
  const int kend = min(K, kbeg + kps);
  Cm += blockIdx.z * c_zstride;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = tid + 256 * r;  // 0..1023
      int mm, kk;
      if (A_KM) {
        mm = i & 127;
        kk = i >> 7;
      } else {
        kk = i & 7;
        mm = i >> 3;
      }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < M && gk < kend) v = A_KM ? A[(int64_t)gk * lda + gm] : A[(int64_t)gm * lda + gk];
      As[kk][mm] = v;
      const int nn = i & 127, kb = i >> 7;
      const int gn = n0 + nn, gk2 = k0 + kb;
      float w = 0.f;
      if (gn < N && gk2 < kend) w = (float)B[(int64_t)gk2 * ldb + gn];
      Bs[kb][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      float av[8], bv[8];
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w;
      av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
      bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
      bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
      if (gn < N) Cm[(int64_t)gm * ldc + gn] = acc[i][j];
    }
  }
}

// Partial dW_r for E <= EM <= 32 over one token split: each thread owns two
// columns of H and all E rows; dlogits of 64 tokens at a time in shared memory.
template <int EM>
__global__ void __launch_bounds__(256) k_dwr_small(const float* __restrict__ dl, const uint16_t* __restrict__ X,
                                                   int T, int H, int E, int tps, float* __restrict__ part) {
  __shared__ float dls[64][EM];
  const int split = blockIdx.y;
  const int h0 = (blockIdx.x * 256 + threadIdx.x) * 2;
  const int t0 = split * tps, t1 = min(T, t0 + tps);
  float acc[EM][2];
#pragma unroll
  for (int e = 0; e < EM; ++e) acc[e][0] = acc[e][1] = 0.f;
  for (int tb = t0; tb < t1; tb += 64) {
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * EM; i += 256) {
      const int tt = i / EM, e = i % EM;
      dls[tt][e] = (tb + tt < t1 && e < E) ? dl[(size_t)(tb + tt) * E + e] : 0.f;
    }
    __syncthreads();
    if (h0 < H) {
      const int nt = min(64, t1 - tb);
      for (int tt = 0; tt < nt; ++tt) {
        const uint32_t xv = __ldg(reinterpret_cast<const uint32_t*>(X + (size_t)(tb + tt) * H + h0));
        const float x0 = bf16_lo(xv), x1 = bf16_hi(xv);
#pragma unroll
        for (int e = 0; e < EM; ++e) {
          acc[e][0] = fmaf(dls[tt][e], x0, acc[e][0]);
          acc[e][1] = fmaf(dls[tt][e], x1, acc[e][1]);
        }
      }
    }
  }
  if (h0 < H)
#pragma unroll
    for (int e = 0; e < EM; ++e)
      if (e < E)
        *reinterpret_cast<float2*>(part + ((size_t)split * E + e) * H + h0) = make_float2(acc[e][0], acc[e][1]);
}

// out[i] = sum over splits s (in order) of part[s*n + i].
__global__ void __launch_bounds__(256) k_reduce_splits(const float* __restrict__ part, int splits, int64_t n,
                                                       float* __restrict__ out) {
  for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    float s = 0.f;
    for (int z = 0; z < splits; ++z) s += part[(int64_t)z * n + i];
    out[i] = s;
  }
}

// W_r [E,H] fp32 -> fwd [3*Ep,H] (row blocks hi, mid, lo) and/or bwd [3*Ep,H] (row blocks
// hi, mid, hi); rows E..Ep-1 of each block zero.  Each thread splits 8 consecutive weights
// of one row (H is a multiple of 8): two 16-byte loads, 16-byte stores of each term.
__global__ void __launch_bounds__(256) k_split_wr(const float* __restrict__ Wr, int E, int H, int Ep,
                                                  uint16_t* __restrict__ fwd, uint16_t* __restrict__ bwd) {
  const int n = Ep * H, n8 = n / 8;  // Ep * H < 2^31 (E <= 256, H < 2^23)
  for (int i = blockIdx.x * 256 + threadIdx.x; i < n8; i += gridDim.x * 256) {
    const int e = i * 8 / H;
    float w[8];
    if (e < E) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(Wr) + 2 * i);
      const float4 b = __ldg(reinterpret_cast<const float4*>(Wr) + 2 * i + 1);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = 0.f;
    }
    uint32_t hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint16_t h0, m0, l0, h1, m1, l1;
      split3(w[2 * j], h0, m0, l0);
      split3(w[2 * j + 1], h1, m1, l1);
      hi[j] = (uint32_t)h0 | ((uint32_t)h1 << 16);
      mid[j] = (uint32_t)m0 | ((uint32_t)m1 << 16);
      lo[j] = (uint32_t)l0 | ((uint32_t)l1 << 16);
    }
    const uint4 vh = make_uint4(hi[0], hi[1], hi[2], hi[3]), vm = make_uint4(mid[0], mid[1], mid[2], mid[3]),
                vl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (fwd) {
      reinterpret_cast<uint4*>(fwd)[i] = vh;
      reinterpret_cast<uint4*>(fwd + n)[i] = vm;
      reinterpret_cast<uint4*>(fwd + 2 * (size_t)n)[i] = vl;
    }
    if (bwd) {
      reinterpret_cast<uint4*>(bwd)[i] = vh;
      reinterpret_cast<uint4*>(bwd + n)[i] = vm;
      reinterpret_cast<uint4*>(bwd + 2 * (size_t)n)[i] = vh;
    }
  }
}

}  // namespace

cudaError_t launch_router_topk(const moe_config& c, const uint16_t* X, const float* Wr, const float* logit_bias,
                               const float* sel_bias, float* logits, float* scores, int32_t* topk_idx, float* gates,
                               int32_t* counts, cudaStream_t st, int nsm, const int32_t* given,
                               const RouterFwdScratch* w) {
  RouteArgs a{X,       Wr,    logit_bias, sel_bias, logits, scores,  topk_idx,     gates,         counts,
              c.T,     c.H,   c.E,        c.k,      c.score_fn, c.renorm, c.gate_scale, c.n_group, c.topk_group,
              c.group_score, given, nullptr, 0};
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st);
  if (e != cudaSuccess) return e;
  if (c.T == 0) return cudaSuccess;
  // With a workspace: the logits on the tensor cores from the exact bf16 split of W_r,
  // block sums promoted to FP32 registers every 64 columns of K, the K splits' partial
  // sums added by the routing pass (one warp per token).
  if (w) {
    const int Ep = (c.E + 31) / 32 * 32;
    if ((int64_t)Ep * c.H >= (1LL << 31)) return cudaErrorInvalidValue;  // k_split_wr indexes in 32 bits
    int blocks = (int)(((int64_t)Ep * c.H / 8 + 255) / 256);
    blocks = blocks < 4 * nsm ? blocks : 4 * nsm;
    k_split_wr<<<blocks, 256, 0, st>>>(Wr, c.E, c.H, Ep, w->wsplit, nullptr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int splits = router_tc_splits(c.T, c.H, c.E, nsm, w->max_splits);
    if ((e = launch_router_logits_tc(c.T, c.H, c.E, Ep, X, w->wsplit, logits, w->part, splits, w->err, st)) !=
        cudaSuccess)
      return e;
    a.more = w->part;
    a.nmore = splits - 1;
    if (c.E <= 32) return launch_route_rows<1>(a, st, nsm);
    if (c.E <= 64) return launch_route_rows<2>(a, st, nsm);
    if (c.E <= 128) return launch_route_rows<4>(a, st, nsm);
    return launch_route_rows<8>(a, st, nsm);
  }
  // Without a workspace: E <= 32 in one fused launch (the projection on the CUDA cores,
  // W_r staged through shared memory); larger E as below.
  if (c.E <= 8) return launch_small<8, 2, 1024>(a, st, nsm);
  if (c.E <= 16) return launch_small<16, 2, 512>(a, st, nsm);
  if (c.E <= 32) return launch_small<32, 1, 256>(a, st, nsm);
  // Without a workspace: an FP32 register-tiled GEMM on the CUDA cores, then the
  // routing pass.
  if (c.E <= 64) return launch_two_pass<64, 2>(a, st, nsm);
  if (c.E <= 128) return launch_two_pass<128, 4>(a, st, nsm);
  return launch_two_pass<128, 8>(a, st, nsm);
}

cudaError_t launch_router_bwd(const moe_config& c, const uint16_t* X, const float* Wr, const float* logits,
                              const int32_t* topk_idx, const float* gates, const float* dgates, float* dW_r,
                              float* dlogit_bias, float* dX_router, const RouterBwdScratch& w, int* err, int nsm,
                              cudaStream_t st) {
  cudaError_t e;
  if (c.T == 0) {
    e = cudaMemsetAsync(dW_r, 0, sizeof(float) * c.E * c.H, st);
    if (e == cudaSuccess && dlogit_bias) e = cudaMemsetAsync(dlogit_bias, 0, sizeof(float) * c.E, st);
    return e;
  }
  const bool tc = c.E > 32;  // large E: the router-gradient products on the tensor cores
  RouteBwdArgs a{logits, topk_idx, gates, dgates, w.dl, c.T, c.E, c.k, c.score_fn, c.renorm, c.gate_scale,
                 tc ? w.dl_rows : nullptr, tc ? w.dl_cols : nullptr, w.Tp, w.Ep};
  if (tc) {
    // rows T..Tp-1 of each third of dl_rows must read as zero
    e = cudaMemsetAsync(w.dl_rows, 0, sizeof(uint16_t) * 3 * (size_t)w.Tp * w.Ep, st);
    if (e != cudaSuccess) return e;
  }
  const int grid = (c.T + 7) / 8;
  if (c.E <= 32)
    k_router_dlogits<1><<<grid, 256, 0, st>>>(a);
  else if (c.E <= 64)
    k_router_dlogits<2><<<grid, 256, 0, st>>>(a);
  else if (c.E <= 128)
    k_router_dlogits<4><<<grid, 256, 0, st>>>(a);
  else
    k_router_dlogits<8><<<grid, 256, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (dlogit_bias) {
    k_colsum<<<c.E, 256, 0, st>>>(w.dl, c.T, c.E, dlogit_bias);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (tc) {
    if ((int64_t)w.Ep * c.H >= (1LL << 31)) return cudaErrorInvalidValue;  // k_split_wr indexes in 32 bits
    int blocks = (int)(((int64_t)w.Ep * c.H / 8 + 255) / 256);
    blocks = blocks < 4 * nsm ? blocks : 4 * nsm;
    k_split_wr<<<blocks, 256, 0, st>>>(Wr, c.E, c.H, w.Ep, nullptr, w.wb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // dW_r = a reduction over 3*Tp rows into only ceil(E/128)*H/256 output tiles: split
    // the rows over w.splits partials, then sum them in a fixed order
    const int splits = w.splits;
    if ((e = launch_router_dwr_tc(c.T, w.Tp, c.H, c.E, w.Ep, w.dl_rows, X, splits > 1 ? w.part : dW_r, splits, err,
                                  nsm, st)) != cudaSuccess)
      return e;
    if (splits > 1) {
      const int64_t n = (int64_t)c.E * c.H;
      int blocks = (int)((n + 255) / 256);
      blocks = blocks < 2048 ? blocks : 2048;
      k_reduce_splits<<<blocks, 256, 0, st>>>(w.part, splits, n, dW_r);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return launch_router_dx_tc(c.T, c.H, w.Ep, w.dl_cols, w.wb, dX_router, err, nsm, st);
  }
  // small E: dW_r over token splits (fixed-order reduction), dX_r = dl W_r with K = E
  {
    const int splits = w.splits;
    const int tps = (c.T + splits - 1) / splits;
    float* dst = splits > 1 ? w.part : dW_r;
    if (c.E <= 8)
      k_dwr_small<8><<<dim3((c.H + 511) / 512, splits), 256, 0, st>>>(w.dl, X, c.T, c.H, c.E, tps, dst);
    else if (c.E <= 16)
      k_dwr_small<16><<<dim3((c.H + 511) / 512, splits), 256, 0, st>>>(w.dl, X, c.T, c.H, c.E, tps, dst);
    else
      k_dwr_small<32><<<dim3((c.H + 511) / 512, splits), 256, 0, st>>>(w.dl, X, c.T, c.H, c.E, tps, dst);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (splits > 1) {
      const int64_t n = (int64_t)c.E * c.H;
      int blocks = (int)((n + 255) / 256);
      blocks = blocks < 2048 ? blocks : 2048;
      k_reduce_splits<<<blocks, 256, 0, st>>>(w.part, splits, n, dW_r);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  dim3 grid3((c.H + 127) / 128, (c.T + 127) / 128);
  k_sgemm<false, float><<<grid3, 256, 0, st>>>(c.T, c.H, c.E, w.dl, c.E, Wr, c.H, dX_router, c.H, c.E, 0);
  return cudaGetLastError();
}

}  // namespace moe
