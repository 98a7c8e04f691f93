// Dispatch and Combine stages and their backwards.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (summary
// page, "Method"): the dispatcher permutes tokens so that the tokens of one
// expert are contiguous, which the grouped GEMM requires, and the last stage
// (Combine) sums each token's gate-weighted expert outputs.  The same section
// asks for sync-free execution of the dropless layer: here the expert sizes
// never leave the device.  A per-chunk histogram, a one-CTA scan and a
// scatter produce the permutation; the scan also writes the grouped GEMM's
// M-tile schedule (tile_offsets), so no host round trip is needed.
//
// Slot of assignment (t, j) routed to expert e:
//   offsets[e] + #{t' < t : e selected by t'}     (tokens keep their order)
// computed as chunk_base[c][e] + rank of the assignment among the chunk's
// assignments to e, the rank taken with warp match/ballot in token-major order.
#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// Per-chunk expert histogram: chunk_counts[c][e].
__global__ void __launch_bounds__(256) k_chunk_hist(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                                                    int32_t* __restrict__ chunk_counts) {
  __shared__ int hist[256];
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += 256) hist[e] = 0;
  __syncthreads();
  const int t0 = c * kChunk;
  const int t1 = min(T, t0 + kChunk);
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += 256) {
    const int e = topk_idx[i];
    if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1);  // ids outside [0,E) are dropped (and flagged by the scan)
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256) chunk_counts[(size_t)c * E + e] = hist[e];
}

// One CTA: offsets (aligned segments), tile_offsets, and the per-chunk bases.
// G threads per expert each own a contiguous range of chunks.
__global__ void __launch_bounds__(1024) k_scan(const int32_t* __restrict__ counts,
                                               const int32_t* __restrict__ chunk_counts, int nch, int E, int align,
                                               int32_t* __restrict__ offsets, int32_t* __restrict__ tile_offsets,
                                               int32_t* __restrict__ chunk_base, int* err) {
  __shared__ int part[1024];
  __shared__ int seg_start[257];
  const int G = 1024 / E >= 1 ? 1024 / E : 1;  // threads per expert
  const int tid = threadIdx.x;
  const int e = tid / G, g = tid % G;
  const int per = (nch + G - 1) / G;
  const int c0 = g * per, c1 = min(nch, c0 + per);
  int s = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) s += chunk_counts[(size_t)c * E + e];
  part[tid] = s;
  __syncthreads();
  if (g == 0 && e < E) {
    int tot = 0;
    for (int y = 0; y < G; ++y) tot += part[e * G + y];
    if (tot != counts[e]) set_device_error(err, MOE_ERR_DEVICE, 1000 + e);
    seg_start[e] = tot;
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0, tiles = 0;
    offsets[0] = 0;
    tile_offsets[0] = 0;
    for (int x = 0; x < E; ++x) {
      const int tot = seg_start[x];
      seg_start[x] = off;
      off += (tot + align - 1) / align * align;
      tiles += (tot + 127) / 128;
      offsets[x + 1] = off;
      tile_offsets[x + 1] = tiles;
    }
  }
  __syncthreads();
  if (e < E) {
    int base = seg_start[e];
    for (int y = 0; y < g; ++y) base += part[e * G + y];
    for (int c = c0; c < c1; ++c) {
      chunk_base[(size_t)c * E + e] = base;
      base += chunk_counts[(size_t)c * E + e];
    }
  }
}

// Chunk CTAs (blockIdx < nch): rank assignments and write the maps.  The chunk's
// assignments (token-major) are split into 8 contiguous runs, one per warp; a
// per-warp histogram and a scan over the warps give each run its starting slot per
// expert, then each warp ranks its run with match_any, so token order is kept.
// Padding CTAs (blockIdx >= nch): kPadSplit CTAs per expert zero its padding rows.
constexpr int kPadSplit = 8;
__global__ void __launch_bounds__(256) k_scatter(const uint16_t* __restrict__ X, const int32_t* __restrict__ topk_idx,
                                                 const int32_t* __restrict__ chunk_base,
                                                 const int32_t* __restrict__ counts,
                                                 const int32_t* __restrict__ offsets, int T, int H, int E, int k,
                                                 int nch, int32_t* __restrict__ row_id_map,
                                                 int32_t* __restrict__ slot_src, uint16_t* __restrict__ Xperm) {
  __shared__ int cursor[8][256];
  const int nvec = H / 8;
  if ((int)blockIdx.x >= nch) {
    const int p = blockIdx.x - nch;
    const int e = p / kPadSplit, part = p % kPadSplit;
    const int r1e = offsets[e + 1];
    const int r0e = min(max(offsets[e] + counts[e], offsets[e]), r1e);
    const int per = (r1e - r0e + kPadSplit - 1) / kPadSplit;
    const int r0 = r0e + part * per, r1 = min(r1e, r0 + per);
    for (int r = r0 + threadIdx.x; r < r1; r += 256) slot_src[r] = -1;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = (int64_t)r0 * nvec + threadIdx.x; i < (int64_t)r1 * nvec; i += 256)
      reinterpret_cast<uint4*>(Xperm)[i] = z;
    return;
  }
  const int c = blockIdx.x;
  const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
  const int n_items = (t1 - t0) * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int run = (n_items + 7) / 8;
  const int i0 = warp * run, i1 = min(n_items, i0 + run);
  for (int i = threadIdx.x; i < 8 * 256; i += 256) (&cursor[0][0])[i] = 0;
  __syncthreads();
  for (int i = i0 + lane; i < i1; i += 32) {
    const int e = topk_idx[(size_t)t0 * k + i];
    if ((unsigned)e < (unsigned)E) atomicAdd(&cursor[warp][e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 256) {
    int base = chunk_base[(size_t)c * E + e];
    for (int w = 0; w < 8; ++w) {
      const int n = cursor[w][e];
      cursor[w][e] = base;
      base += n;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    int e = i < i1 ? topk_idx[(size_t)t0 * k + i] : -1 - lane;
    const bool ok = i < i1 && (unsigned)e < (unsigned)E;
    if (i < i1 && !ok) {
      row_id_map[(size_t)t0 * k + i] = -1;  // an id outside [0,E): no slot
      e = -1 - lane;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt);
    int base = 0;
    if (ok) base = cursor[warp][e];
    __syncwarp();
    if (ok) {
      const int slot = base + rank;
      row_id_map[(size_t)t0 * k + i] = slot;
      slot_src[slot] = t0 * k + i;
      if (rank == 0) cursor[warp][e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

// Xperm[row_id_map[t,j]] = X[t]: 16-byte vectors over the whole grid, each
// token vector read once and written to its k rows.
__global__ void __launch_bounds__(256) k_copy_rows(const uint16_t* __restrict__ X,
                                                   const int32_t* __restrict__ row_id_map, int T, int H, int k,
                                                   uint16_t* __restrict__ Xperm) {
  const int nvec = H / 8;
  const int64_t total = (int64_t)T * nvec;
  for (int64_t v = blockIdx.x * 256LL + threadIdx.x; v < total; v += (int64_t)gridDim.x * 256) {
    const int t = (int)(v / nvec), c = (int)(v % nvec);
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(X + (size_t)t * H) + c);
    for (int j = 0; j < k; ++j) {
      const int slot = __ldg(row_id_map + (size_t)t * k + j);
      if (slot >= 0) reinterpret_cast<uint4*>(Xperm + (size_t)slot * H)[c] = x;
    }
  }
}

// Y[t] = sum_j g[t,j] Yperm[row_id_map[t,j]] (+ Yshared[t]); one warp per token.
__global__ void __launch_bounds__(256) k_combine(const uint16_t* __restrict__ Yperm,
                                                 const int32_t* __restrict__ row_id_map,
                                                 const float* __restrict__ gates, const uint16_t* __restrict__ Ysh,
                                                 uint16_t* __restrict__ Y, int T, int H, int k) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = lane < k ? row_id_map[(size_t)t * k + lane] : 0;
  const float my_g = lane < k ? gates[(size_t)t * k + lane] : 0.f;
  const int nvec = H / 8;
  // every lane runs every iteration (the shuffles need the full warp)
  for (int v0 = 0; v0 < nvec; v0 += 32) {
    const int v = v0 + lane;
    const bool ok = v < nvec;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      if (!ok || slot < 0) continue;
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(Yperm + (size_t)slot * H) + v);
      float f[8];
      unpack8(y, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, f[q], acc[q]);
    }
    if (!ok) continue;
    if (Ysh) {
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(Ysh + (size_t)t * H) + v), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    reinterpret_cast<uint4*>(Y + (size_t)t * H)[v] = pack8(acc);
  }
}

// dYperm[slot] = bf16(g dY[t]); dgates[t,j] = <dY[t], Yperm[slot]>.
// CTAs past the token range zero the padding rows, kPadSplit CTAs per expert.
__global__ void __launch_bounds__(256) k_combine_bwd(const uint16_t* __restrict__ dY,
                                                     const uint16_t* __restrict__ Yperm,
                                                     const int32_t* __restrict__ row_id_map,
                                                     const float* __restrict__ gates,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ counts, uint16_t* __restrict__ dYperm,
                                                     float* __restrict__ dgates, int T, int H, int k, int tok_blocks) {
  const int nvec = H / 8;
  if ((int)blockIdx.x >= tok_blocks) {
    const int p = blockIdx.x - tok_blocks;
    const int e = p / kPadSplit, part = p % kPadSplit;
    const int r1e = offsets[e + 1];
    const int r0e = min(max(offsets[e] + counts[e], offsets[e]), r1e);
    const int per = (r1e - r0e + kPadSplit - 1) / kPadSplit;
    const int r0 = r0e + part * per, r1 = min(r1e, r0 + per);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = (int64_t)r0 * nvec + threadIdx.x; i < (int64_t)r1 * nvec; i += 256)
      reinterpret_cast<uint4*>(dYperm)[i] = z;
    return;
  }
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = lane < k ? row_id_map[(size_t)t * k + lane] : 0;
  const float my_g = lane < k ? gates[(size_t)t * k + lane] : 0.f;
  float my_dot = 0.f;
  for (int j = 0; j < k; ++j) {
    const int slot = __shfl_sync(0xffffffffu, my_slot, j);
    const float g = __shfl_sync(0xffffffffu, my_g, j);
    float dot = 0.f;
    for (int v = lane; v < nvec && slot >= 0; v += 32) {
      float dy[8], y[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(dY + (size_t)t * H) + v), dy);
      unpack8(__ldg(reinterpret_cast<const uint4*>(Yperm + (size_t)slot * H) + v), y);
      float o[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        dot = fmaf(dy[q], y[q], dot);
        o[q] = g * dy[q];
      }
      reinterpret_cast<uint4*>(dYperm + (size_t)slot * H)[v] = pack8(o);
    }
    dot = warp_sum(dot);
    if (lane == j) my_dot = dot;
  }
  if (lane < k) dgates[(size_t)t * k + lane] = my_dot;
}

// dX[t] = sum_j dXperm[row_id_map[t,j]] + dX_router[t] + dX_shared[t].
__global__ void __launch_bounds__(256) k_permute_bwd(const uint16_t* __restrict__ dXperm,
                                                     const int32_t* __restrict__ row_id_map,
                                                     const float* __restrict__ dXr, const uint16_t* __restrict__ dXs,
                                                     uint16_t* __restrict__ dX, int T, int H, int k) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = lane < k ? row_id_map[(size_t)t * k + lane] : 0;
  const int nvec = H / 8;
  for (int v0 = 0; v0 < nvec; v0 += 32) {
    const int v = v0 + lane;
    const bool ok = v < nvec;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      if (!ok || slot < 0) continue;
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(dXperm + (size_t)slot * H) + v), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    if (!ok) continue;
    if (dXr) {
      const float4* r = reinterpret_cast<const float4*>(dXr + (size_t)t * H) + 2 * v;
      const float4 a = __ldg(r), b = __ldg(r + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    if (dXs) {
      float f[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(dXs + (size_t)t * H) + v), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
    reinterpret_cast<uint4*>(dX + (size_t)t * H)[v] = pack8(acc);
  }
}

}  // namespace

cudaError_t launch_permute(const moe_config& c, const uint16_t* X, const int32_t* topk_idx, const int32_t* counts,
                           int32_t* offsets, int32_t* tile_offsets, int32_t* row_id_map, int32_t* slot_src,
                           uint16_t* Xperm, int32_t* chunk_counts, int32_t* chunk_base, int* err, int nsm,
                           cudaStream_t st) {
  const int nch = (c.T + kChunk - 1) / kChunk;
  cudaError_t e;
  if (nch > 0) {
    k_chunk_hist<<<nch, 256, 0, st>>>(topk_idx, c.T, c.E, c.k, chunk_counts);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_scan<<<1, 1024, 0, st>>>(counts, chunk_counts, nch, c.E, c.align, offsets, tile_offsets, chunk_base, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_scatter<<<nch + c.E * kPadSplit, 256, 0, st>>>(X, topk_idx, chunk_base, counts, offsets, c.T, c.H, c.E, c.k,
                                                   nch, row_id_map, slot_src, Xperm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (c.T > 0) {
    const int64_t vec = (int64_t)c.T * (c.H / 8);
    int64_t blocks = (vec + 255) / 256;
    if (blocks > 8LL * nsm) blocks = 8LL * nsm;
    k_copy_rows<<<(int)blocks, 256, 0, st>>>(X, row_id_map, c.T, c.H, c.k, Xperm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_combine(const moe_config& c, const uint16_t* Yperm, const int32_t* row_id_map, const float* gates,
                           const uint16_t* Ysh, uint16_t* Y, cudaStream_t st) {
  if (c.T == 0) return cudaSuccess;
  k_combine<<<(c.T + 7) / 8, 256, 0, st>>>(Yperm, row_id_map, gates, Ysh, Y, c.T, c.H, c.k);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const moe_config& c, const uint16_t* dY, const uint16_t* Yperm,
                               const int32_t* row_id_map, const float* gates, const int32_t* offsets,
                               const int32_t* counts, uint16_t* dYperm, float* dgates, cudaStream_t st) {
  const int tb = (c.T + 7) / 8;
  k_combine_bwd<<<tb + c.E * kPadSplit, 256, 0, st>>>(dY, Yperm, row_id_map, gates, offsets, counts, dYperm, dgates, c.T, c.H,
                                           c.k, tb);
  return cudaGetLastError();
}

cudaError_t launch_permute_bwd(const moe_config& c, const uint16_t* dXperm, const int32_t* row_id_map,
                               const float* dXr, const uint16_t* dXs, uint16_t* dX, cudaStream_t st) {
  if (c.T == 0) return cudaSuccess;
  k_permute_bwd<<<(c.T + 7) / 8, 256, 0, st>>>(dXperm, row_id_map, dXr, dXs, dX, c.T, c.H, c.k);
  return cudaGetLastError();
}

}  // namespace moe
