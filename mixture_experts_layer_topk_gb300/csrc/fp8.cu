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

// Row blocks: X [rows, K] bf16 -> q [rows, K] e4m3, sc [rows, K/128].  One warp per
// (row, block); rows at or beyond *rows_valid (when given) are skipped.
__global__ void __launch_bounds__(256) k_quant_rows(const uint16_t* __restrict__ X, int64_t rows, int K,
                                                    const int32_t* __restrict__ rows_valid, uint8_t* __restrict__ q,
                                                    uint8_t* __restrict__ sc) {
  const int lane = threadIdx.x & 31;
  const int nb = K / 128;
  const int64_t limit = rows_valid ? (int64_t)*rows_valid : rows;
  const int64_t tasks = limit * nb;
  for (int64_t w = (blockIdx.x * 256LL + threadIdx.x) >> 5; w < tasks; w += (gridDim.x * 256LL) >> 5) {
    const int64_t row = w / nb;
    const int b = (int)(w % nb);
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(X + row * K + b * 128) + lane);
    const float f0 = bf16_lo(v.x), f1 = bf16_hi(v.x), f2 = bf16_lo(v.y), f3 = bf16_hi(v.y);
    float m = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
    m = warp_max(m);
    const int e = block_exp(m);
    const float inv = pow2(-e);
    const uint32_t packed = (uint32_t)e4m3x2(f0 * inv, f1 * inv) | ((uint32_t)e4m3x2(f2 * inv, f3 * inv) << 16);
    reinterpret_cast<uint32_t*>(q + row * K + b * 128)[lane] = packed;
    if (lane == 0) sc[row * nb + b] = (uint8_t)(e + 127);
  }
}

// Column blocks along rows: X [rows, N] bf16 -> q [rows, N], sc [ceil(rows/128), N].
// One thread per column of a 128-row block; two passes (max, then quantize).
__global__ void __launch_bounds__(256) k_quant_cols(const uint16_t* __restrict__ X, int64_t rows, int N,
                                                    const int32_t* __restrict__ rows_valid, uint8_t* __restrict__ q,
                                                    uint8_t* __restrict__ sc) {
  const int64_t limit = rows_valid ? (int64_t)*rows_valid : rows;
  const int64_t rb = blockIdx.y;
  const int64_t r0 = rb * 128;
  if (r0 >= limit) return;
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= N) return;
  const int64_t r1 = min(limit, r0 + 128);
  float m = 0.f;
  for (int64_t r = r0; r < r1; ++r) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)__ldg(X + r * N + c) << 16)));
  const int e = block_exp(m);
  const float inv = pow2(-e);
  for (int64_t r = r0; r < r1; ++r) {
    const float f = __uint_as_float((uint32_t)__ldg(X + r * N + c) << 16) * inv;
    q[r * N + c] = (uint8_t)(e4m3x2(f, 0.f) & 0xFF);
  }
  sc[rb * N + c] = (uint8_t)(e + 127);
}

// 128x128 blocks of nmat matrices [rows, cols]: one CTA per block.
__global__ void __launch_bounds__(256) k_quant_weights(const uint16_t* __restrict__ W, int rows, int cols,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  const int nbr = rows / 128, nbc = cols / 128;
  const int64_t mat = blockIdx.z;
  const int br = blockIdx.y, bc = blockIdx.x;
  const uint16_t* base = W + (mat * rows + (int64_t)br * 128) * cols + bc * 128;
  // thread t: row (t / 2) of the block, 64 columns starting at (t & 1) * 64
  const int rr = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * 64;
  float f[64];
  float m = 0.f;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)rr * cols + c0) + v);
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
  uint8_t* qo = q + (mat * rows + (int64_t)br * 128 + rr) * cols + bc * 128 + c0;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 16 * v + 4 * j;
      w[j] = (uint32_t)e4m3x2(f[i] * inv, f[i + 1] * inv) | ((uint32_t)e4m3x2(f[i + 2] * inv, f[i + 3] * inv) << 16);
    }
    reinterpret_cast<uint4*>(qo)[v] = make_uint4(w[0], w[1], w[2], w[3]);
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
  dim3 grid((N + 255) / 256, (unsigned)((rows + 127) / 128));
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
