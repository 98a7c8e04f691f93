// FP8 E4M3 quantization of the expert GEMM operands.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (index
// page, "Abstract"; summary page, "Method" and "Key claims"): low-precision
// training with FP8 across the expert GEMMs while the router stays in higher
// precision.  Blocks of 128 share one scale: activations in 1x128 blocks along
// the GEMM's K, weights in 128x128 blocks, weight-gradient operands in 128x1
// blocks along the tokens.  A block's scale is the smallest power of two s with
// 448*s >= max|x| (s = 1 for an all-zero block), stored as its UE8M0 byte
// (exponent + 127); values are x/s rounded to nearest-even E4M3.  Power-of-two
// scales are exact to apply and to undo, and they are what the block-scaled
// tcgen05 MMA consumes directly.
#include <cuda_fp8.h>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// Exponent e of the block scale 2^e: the smallest e with 448 * 2^e >= amax.
__device__ __forceinline__ int block_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int e;
  frexpf(amax * (1.0f / 448.0f), &e);  // estimate; corrected by exact comparisons below
  while (e > -126 && ldexpf(448.0f, e - 1) >= amax) --e;
  while (ldexpf(448.0f, e) < amax) ++e;
  return e;
}

__device__ __forceinline__ float pow2(int e) { return __int_as_float((uint32_t)(127 + e) << 23); }

__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Row blocks: X [rows, K] bf16 -> q [rows, K] e4m3, sc [rows, K/128]; rows at or beyond
// *rows_valid (when given) are skipped.  A warp takes four consecutive (row, block) tasks:
// each half-warp owns one 128-element block per step (16 bytes per lane), two steps in
// flight, the block's maximum reduced within the half-warp.
__global__ void __launch_bounds__(256) k_quant_rows(const uint16_t* __restrict__ X, int64_t rows, int K,
                                                    const int32_t* __restrict__ rows_valid, uint8_t* __restrict__ q,
                                                    uint8_t* __restrict__ sc) {
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int nb = K / 128;
  const int64_t limit = rows_valid ? (int64_t)*rows_valid : rows;
  const int64_t tasks = limit * nb;
  const int64_t nwarps = (gridDim.x * 256LL) >> 5;
  for (int64_t w = (blockIdx.x * 256LL + threadIdx.x) >> 5; w * 4 < tasks; w += nwarps) {
    uint4 v[2];
    int64_t task[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      task[u] = w * 4 + 2 * u + half;
      if (task[u] < tasks) {
        const int64_t row = task[u] / nb;
        const int b = (int)(task[u] - row * nb);
        v[u] = __ldg(reinterpret_cast<const uint4*>(X + row * K + b * 128) + hl);
      } else {
        v[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float f[8];
      unpack8(v[u], f);
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int e = block_exp(m);
      const float inv = pow2(-e);
      const uint32_t lo = (uint32_t)e4m3x2(f[0] * inv, f[1] * inv) | ((uint32_t)e4m3x2(f[2] * inv, f[3] * inv) << 16);
      const uint32_t hi = (uint32_t)e4m3x2(f[4] * inv, f[5] * inv) | ((uint32_t)e4m3x2(f[6] * inv, f[7] * inv) << 16);
      if (task[u] < tasks) {
        const int64_t row = task[u] / nb;
        const int b = (int)(task[u] - row * nb);
        reinterpret_cast<uint2*>(q + row * K + b * 128)[hl] = make_uint2(lo, hi);
        if (hl == 0) sc[row * nb + b] = (uint8_t)(e + 127);
      }
    }
  }
}

// Column blocks along rows: X [rows, N] bf16 -> q [rows, N], sc [ceil(rows/128), N]; rows at
// or beyond *rows_valid (when given) are neither read nor written.  A CTA takes a tile of
// 128 rows x 64 columns: coalesced 16-byte loads (a warp reads four 128-byte row pieces),
// each column's maximum reduced through shared memory, then each thread quantizes the
// vectors it holds.
__global__ void __launch_bounds__(256) k_quant_cols(const uint16_t* __restrict__ X, int64_t rows, int N,
                                                    const int32_t* __restrict__ rows_valid, uint8_t* __restrict__ q,
                                                    uint8_t* __restrict__ sc) {
  __shared__ float cmax[4][64];
  __shared__ float cinv[64];
  const int64_t limit = rows_valid ? (int64_t)*rows_valid : rows;
  const int64_t rb = blockIdx.y;
  const int64_t r0 = rb * 128;
  if (r0 >= limit) return;
  const int c0 = blockIdx.x * 64;
  // vector i = threadIdx.x + 256 u (u < 4): tile row i / 8, columns 8 (i % 8) ..+7
  float f[4][8];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + 256 * u;
    const int64_t r = r0 + (i >> 3);
    uint4 x = make_uint4(0, 0, 0, 0);
    if (r < limit) x = __ldg(reinterpret_cast<const uint4*>(X + r * N + c0) + (i & 7));
    unpack8(x, f[u]);
  }
  // per-thread maxima of its 8 columns over its 4 rows; the 32 rows a warp covers per u
  // share columns every 8 lanes
  const int cg = threadIdx.x & 7;  // column group: columns 8 cg ..+7
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    m[k] = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) m[k] = fmaxf(m[k], fabsf(f[u][k]));
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) m[k] = fmaxf(m[k], __shfl_xor_sync(0xffffffffu, m[k], o));
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < 4 && lane < 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) cmax[warp][8 * cg + k] = m[k];
  }
  __syncthreads();
  if (warp >= 4 && lane < 8) {  // the second half of the warps folds into the first
#pragma unroll
    for (int k = 0; k < 8; ++k) atomicMax(reinterpret_cast<int*>(&cmax[warp & 3][8 * cg + k]), __float_as_int(m[k]));
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    const int c = threadIdx.x;
    const float mm = fmaxf(fmaxf(cmax[0][c], cmax[1][c]), fmaxf(cmax[2][c], cmax[3][c]));
    const int e = block_exp(mm);
    cinv[c] = pow2(-e);
    sc[rb * N + c0 + c] = (uint8_t)(e + 127);
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + 256 * u;
    const int64_t r = r0 + (i >> 3);
    if (r >= limit) continue;
    const float* iv = cinv + 8 * cg;
    const uint32_t lo = (uint32_t)e4m3x2(f[u][0] * iv[0], f[u][1] * iv[1]) |
                        ((uint32_t)e4m3x2(f[u][2] * iv[2], f[u][3] * iv[3]) << 16);
    const uint32_t hi = (uint32_t)e4m3x2(f[u][4] * iv[4], f[u][5] * iv[5]) |
                        ((uint32_t)e4m3x2(f[u][6] * iv[6], f[u][7] * iv[7]) << 16);
    reinterpret_cast<uint2*>(q + r * N + c0)[i & 7] = make_uint2(lo, hi);
  }
}

// 128x128 blocks of nmat matrices [rows, cols]: one CTA per block.
__global__ void __launch_bounds__(256) k_quant_weights(const uint16_t* __restrict__ W, int rows, int cols,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  const int nbr = rows / 128, nbc = cols / 128;
  const int64_t mat = blockIdx.z;
  const int br = blockIdx.y, bc = blockIdx.x;
  const uint16_t* base = W + (mat * rows + (int64_t)br * 128) * cols + bc * 128;
  // the block's 2048 16-byte vectors: vector i = threadIdx.x + 256 v is row i / 16, columns
  // 8 (i % 16) ..+7, so a warp reads (and later writes) two whole 128-column rows at a time
  float f[64];
  float m = 0.f;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const int i = threadIdx.x + 256 * v;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)(i >> 4) * cols) + (i & 15));
    unpack8(x, f + 8 * v);
  }
#pragma unroll
  for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(f[i]));
  __shared__ float red[8];
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  const int e = block_exp(m);
  const float inv = pow2(-e);
  uint8_t* qb = q + (mat * rows + (int64_t)br * 128) * cols + bc * 128;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const int i = threadIdx.x + 256 * v;
    const float* g = f + 8 * v;
    const uint32_t lo = (uint32_t)e4m3x2(g[0] * inv, g[1] * inv) | ((uint32_t)e4m3x2(g[2] * inv, g[3] * inv) << 16);
    const uint32_t hi = (uint32_t)e4m3x2(g[4] * inv, g[5] * inv) | ((uint32_t)e4m3x2(g[6] * inv, g[7] * inv) << 16);
    *reinterpret_cast<uint2*>(qb + (int64_t)(i >> 4) * cols + 8 * (i & 15)) = make_uint2(lo, hi);
  }
  if (threadIdx.x == 0) sc[(mat * nbr + br) * nbc + bc] = (uint8_t)(e + 127);
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t* X, int64_t rows, int K, const int32_t* rows_valid, uint8_t* q,
                              uint8_t* sc, int nsm, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int64_t tasks = rows * (K / 128);
  int64_t blocks = (tasks + 7) / 8;
  if (blocks > 16LL * nsm) blocks = 16LL * nsm;
  k_quant_rows<<<(int)blocks, 256, 0, st>>>(X, rows, K, rows_valid, q, sc);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols(const uint16_t* X, int64_t rows, int N, const int32_t* rows_valid, uint8_t* q,
                              uint8_t* sc, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (N % 64 != 0) return cudaErrorInvalidValue;
  dim3 grid(N / 64, (unsigned)((rows + 127) / 128));
  k_quant_cols<<<grid, 256, 0, st>>>(X, rows, N, rows_valid, q, sc);
  return cudaGetLastError();
}

cudaError_t launch_quant_weights(const uint16_t* W, int64_t nmat, int rows, int cols, uint8_t* q, uint8_t* sc,
                                 cudaStream_t st) {
  if (nmat <= 0) return cudaSuccess;
  dim3 grid(cols / 128, rows / 128, (unsigned)nmat);
  k_quant_weights<<<grid, 256, 0, st>>>(W, rows, cols, q, sc);
  return cudaGetLastError();
}

}  // namespace moe
