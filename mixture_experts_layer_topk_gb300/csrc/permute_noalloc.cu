// moe_permute_noalloc: the dispatch permutation for callers that cannot
// allocate device memory.
//
// moe_permute needs a caller-provided workspace for its per-chunk expert
// histograms and per-chunk base offsets.  Some callers have no way to provide
// one: code that runs inside a memory arena sized once at start-up (a serving
// runtime that forbids device allocation after warm-up), a plugin handed only
// its inputs and outputs by a host framework, or a caller that is in the middle
// of recording a CUDA graph, where cudaMalloc is not allowed.  This variant
// keeps that scratch in a file-scope __device__ array instead, so the call
// itself allocates nothing.
//
// The scratch array (kNoAllocScratchInts 32-bit words, 512 KiB + 1.25 KiB) is
// part of the library image: every GPU that loads the library holds it until
// the process exits.  All calls share it, so calls whose kernels overlap on the
// GPU (different streams without ordering between them) race on it.
#include <mutex>

#include "common.cuh"
#include "moe_internal.h"

namespace {

// Layout: [0, 64) error word and detail; [64, 320) the rows each expert keeps (E <= 256);
// then chunk_counts[nch*E]; then chunk_base[nch*E], nch*E <= 65536.
constexpr int64_t kNoAllocMaxChunkExperts = 65536;
constexpr int64_t kNoAllocScratchInts = 64 + 256 + 2 * kNoAllocMaxChunkExperts;

__device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

std::mutex g_setup_mutex;
int32_t* g_scratch_ptr[64] = {nullptr};
int g_nsm[64] = {0};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).  nullptr on failure.
int32_t* scratch_on_current_device(int* nsm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return nullptr;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return nullptr;
    g_nsm[dev] = n;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *nsm = g_nsm[dev];
  return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, const moe_bf16* X, const int32_t* topk_idx,
                                          const int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
                                          int32_t* row_id_map, int32_t* slot_src, moe_bf16* Xperm, void* stream) {
  int64_t R = 0;
  const moe_status s = moe_max_rows(cfg, &R);  // validates the configuration
  if (s != MOE_OK) return s;
  const bool empty = cfg->T == 0;
  // Xperm NULL: the dispatch maps only (X is then not read), as in moe_permute
  if ((Xperm && !X && !empty) || (!topk_idx && !empty) || !counts || !offsets || !tile_offsets ||
      (!row_id_map && !empty) || !slot_src)
    return MOE_ERR_INVALID_ARG;
  if (Xperm && (!aligned16(X) || !aligned16(Xperm))) return MOE_ERR_INVALID_ARG;
  const int64_t nch = ((int64_t)cfg->T + moe::kChunk - 1) / moe::kChunk;
  if (nch * cfg->E > kNoAllocMaxChunkExperts) return MOE_ERR_WORKSPACE;  // beyond the built-in scratch
  int nsm = 0;
  int32_t* scratch = scratch_on_current_device(&nsm);
  if (!scratch) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the error word must start at zero; the histogram and base arrays are fully rewritten
  if (cudaMemsetAsync(scratch, 0, 64 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* kept = scratch + 64;
  int32_t* chunk_counts = kept + 256;
  int32_t* chunk_base = chunk_counts + nch * cfg->E;
  const cudaError_t e =
      moe::launch_permute(*cfg, X, topk_idx, counts, INT_MAX, nullptr, kept, offsets, tile_offsets, row_id_map,
                          slot_src, Xperm, chunk_counts, chunk_base, nullptr, nullptr, scratch, nsm, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
