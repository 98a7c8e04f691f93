// Dispatch and Combine stages and their backwards.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (summary
// page, "Method"): the dispatcher permutes tokens so that the tokens of one
// expert are contiguous, which the grouped GEMM requires, and the last stage
// (Combine) sums each token's gate-weighted expert outputs.  The same section
// asks for sync-free execution of the dropless layer: here the expert sizes
// never leave the device.  A per-chunk histogram, a one-CTA scan and a
// scatter produce the permutation; the scan also writes the grouped GEMM's
// M-tile schedule (tile_offsets), so no host round trip is needed.  A small
// dropless layer (T*k <= 16K, E <= 32) takes one launch in all when its token
// rows fit the copy CTAs' shared memory.
//
// Slot of assignment (t, j) routed to expert e:
//   offsets[e] + #{t' < t : e selected by t'}     (tokens keep their order)
// computed as chunk_base[c][e] + rank of the assignment among the chunk's
// assignments to e, the rank taken with warp match/ballot in token-major order.
//
// Capacity-controlled token dropping (summary page, "Results": listed among the
// production features, no policy given) reuses the same ranks: with a capacity C, an
// assignment whose position within its expert, in token order, is C or more gets
// no slot (row_id_map -1), and the segments are sized by the kept counts
// min(counts[e], C).  Dropless dispatch is the case C = INT_MAX.
//
// Dropping by priority (an over-full expert keeps the C assignments of largest
// priority, e.g. the gate; equal priorities to the earlier assignment): the
// scatter only groups each expert's assignments in token order (drop_order), and
// one CTA per expert finds the C-th largest priority by a 4-pass radix select on
// order-preserving 32-bit keys, breaks ties in token order with a block scan, and
// writes the kept assignments' rows, still in token order.
#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

// 16-byte vectors per lane per source row that the gather kernels load before using any
constexpr int kGatherUnroll = 4;

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

// One CTA: offsets (aligned segments), tile_offsets, the per-chunk bases, and kept[e], the
// rows expert e keeps (min of its histogram total and the capacity).  The later launches
// size each segment's padding from kept, so they agree with the slots handed out even when
// the caller's counts do not match topk_idx (which the scan flags in the error word).
// G threads per expert each own a contiguous range of chunks.  The chunk histogram
// is first copied into shared memory with coalesced loads when it fits
// (kScanStage entries); the per-expert prefix sums run on warp 0 (each lane a run
// of consecutive experts, then a shuffle scan across the lanes).
constexpr int kScanStage = 24576;
__global__ void __launch_bounds__(1024) k_scan(const int32_t* __restrict__ counts,
                                               const int32_t* __restrict__ chunk_counts, int nch, int E, int align,
                                               int cap, int32_t* __restrict__ kept,
                                               int32_t* __restrict__ offsets, int32_t* __restrict__ tile_offsets,
                                               int32_t* __restrict__ chunk_base, int32_t* __restrict__ drop_start,
                                               int* err) {
  extern __shared__ int cc_s[];
  __shared__ int part[1024];
  __shared__ int tot_s[256];
  __shared__ int seg_start[256];
  const bool staged = nch * E <= kScanStage;
  const int tid = threadIdx.x, lane = tid & 31;
  if (staged)
    for (int i = tid; i < nch * E; i += 1024) cc_s[i] = chunk_counts[i];
  __syncthreads();
  const int32_t* cc = staged ? cc_s : chunk_counts;
  const int G = 1024 / E >= 1 ? 1024 / E : 1;  // threads per expert
  const int e = tid / G, g = tid % G;
  const int per = (nch + G - 1) / G;
  const int c0 = g * per, c1 = min(nch, c0 + per);
  int s = 0;
  if (e < E)
    for (int c = c0; c < c1; ++c) s += cc[c * E + e];
  part[tid] = s;
  __syncthreads();
  if (g == 0 && e < E) {
    int tot = 0;
    for (int y = 0; y < G; ++y) tot += part[e * G + y];
    if (tot != counts[e]) set_device_error(err, MOE_ERR_DEVICE, 1000 + e);
    tot_s[e] = tot;
  }
  __syncthreads();
  if (tid < 32) {
    const int pl = (E + 31) / 32;
    const int x0 = lane * pl, x1 = min(E, x0 + pl);
    int sa = 0, sb = 0, sd = 0;  // aligned rows, M tiles, rows before capacity
    for (int x = x0; x < x1; ++x) {
      const int kt = min(tot_s[x], cap);
      sa += (kt + align - 1) / align * align;
      sb += (kt + 127) / 128;
      sd += tot_s[x];
    }
    int ia = sa, ib = sb, id = sd;  // inclusive scans across the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ta = __shfl_up_sync(0xffffffffu, ia, o), tb = __shfl_up_sync(0xffffffffu, ib, o),
                td = __shfl_up_sync(0xffffffffu, id, o);
      if (lane >= o) {
        ia += ta;
        ib += tb;
        id += td;
      }
    }
    int oa = ia - sa, ob = ib - sb, od = id - sd;
    for (int x = x0; x < x1; ++x) {
      const int tot = tot_s[x], kt = min(tot, cap);
      if (drop_start) drop_start[x] = od;
      od += tot;
      kept[x] = kt;
      seg_start[x] = oa;
      oa += (kt + align - 1) / align * align;
      ob += (kt + 127) / 128;
      offsets[x + 1] = oa;
      tile_offsets[x + 1] = ob;
    }
    if (lane == 0) {
      offsets[0] = 0;
      tile_offsets[0] = 0;
    }
    if (lane == 31 && drop_start) drop_start[E] = id;
  }
  __syncthreads();
  if (e < E) {
    int base = seg_start[e];
    for (int y = 0; y < g; ++y) base += part[e * G + y];
    for (int c = c0; c < c1; ++c) {
      chunk_base[(size_t)c * E + e] = base;
      base += cc[c * E + e];
    }
  }
}

// Chunk CTAs (blockIdx < nch): rank assignments and write the maps.  The chunk's
// assignments (token-major) are split into 8 contiguous runs, one per warp; a
// per-warp histogram and a scan over the warps give each run its starting slot per
// expert, then each warp ranks its run with match_any, so token order is kept.
// Padding CTAs (blockIdx >= nch): kPadSplit CTAs per expert mark its padding rows in
// slot_src (-1); k_copy_rows zeroes their rows of Xperm.
constexpr int kPadSplit = 8;
__global__ void __launch_bounds__(256) k_scatter(const int32_t* __restrict__ topk_idx,
                                                 const int32_t* __restrict__ chunk_base,
                                                 const int32_t* __restrict__ kept,
                                                 const int32_t* __restrict__ offsets, int T, int E, int k,
                                                 int nch, int cap, int32_t* __restrict__ row_id_map,
                                                 int32_t* __restrict__ slot_src, int32_t* __restrict__ drop_order,
                                                 const int32_t* __restrict__ drop_start) {
  __shared__ int cursor[8][256];
  if ((int)blockIdx.x >= nch) {
    const int p = blockIdx.x - nch;
    const int e = p / kPadSplit, part = p % kPadSplit;
    const int r1e = offsets[e + 1];
    const int r0e = min(max(offsets[e] + kept[e], offsets[e]), r1e);
    const int per = (r1e - r0e + kPadSplit - 1) / kPadSplit;
    const int r0 = r0e + part * per, r1 = min(r1e, r0 + per);
    for (int r = r0 + threadIdx.x; r < r1; r += 256) slot_src[r] = -1;  // (k_copy_rows zeroes their Xperm rows)
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
      if (drop_order) {
        drop_order[drop_start[e] + (slot - offsets[e])] = t0 * k + i;  // rows are assigned by k_drop_select
      } else if (slot - offsets[e] < cap) {
        row_id_map[(size_t)t0 * k + i] = slot;
        slot_src[slot] = t0 * k + i;
      } else {
        row_id_map[(size_t)t0 * k + i] = -1;  // beyond the expert's capacity: dropped
      }
      if (rank == 0) cursor[warp][e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

// Dispatch maps of a small layer in one launch (dropless, T*k <= kSmallAssign, E <= 32,
// T*k*E <= kSmallWork): the chunked path's histogram, scan and scatter are three short
// dependent launches, which dominate when the layer moves only ~100 MB.  Here CTA c takes
// tokens [c*kSmallTok, (c+1)*kSmallTok) and
//   1. counts, from all of topk_idx, each expert's assignments before its first token and
//      in total (warp ballots, one per expert per 32 assignments; lane e keeps expert e;
//      each warp loads its ids before counting any; 32 warps share the passes),
//   2. derives the aligned segment starts and the M-tile schedule from the totals,
//   3. ranks its own assignments in token order (match_any within warp 0, running
//      per-expert cursors across the passes) and writes row_id_map and slot_src,
//   4. marks the padding rows of expert c (c < E) in slot_src.
// The grid has max(token CTAs, E) CTAs.  CTA 0 writes offsets, tile_offsets and kept, and
// checks the totals against counts.  The slots are those of the chunked path: offsets[e] +
// #{earlier assignments to e}; the row copy (k_copy_rows, which also zeroes the padding
// rows) follows.
constexpr int kSmallTok = 128;
constexpr int kSmallAssign = 16384;
constexpr int kSmallMaxE = 32;
constexpr int64_t kSmallWork = 131072;  // T*k*E: each warp makes at most 128 ballots
constexpr int kSmallThreads = 1024;

__global__ void __launch_bounds__(kSmallThreads) k_dispatch_small(const int32_t* __restrict__ topk_idx,
                                                                  const int32_t* __restrict__ counts, int T, int E,
                                                                  int k, int align, int tok_blocks,
                                                                  int32_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ tile_offsets,
                                                                  int32_t* __restrict__ kept,
                                                                  int32_t* __restrict__ row_id_map,
                                                                  int32_t* __restrict__ slot_src, int* err) {
  constexpr int NW = kSmallThreads / 32;
  __shared__ int s_cnt[2][NW][kSmallMaxE];  // per warp: [0] before this CTA's tokens, [1] in total
  __shared__ int s_off[kSmallMaxE + 1];     // aligned segment starts
  __shared__ int s_tot[kSmallMaxE];
  __shared__ int s_mine[kSmallTok * 32];    // this CTA's assignments (k <= 32)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = T * k;
  const bool tok_cta = (int)blockIdx.x < tok_blocks;
  const int t0 = tok_cta ? (int)blockIdx.x * kSmallTok : T;
  const int a0 = t0 * k;  // this CTA's first assignment
  if (tok_cta)  // this CTA's own assignments, for the ranking below
    for (int i = threadIdx.x; i < min(kSmallTok, T - t0) * k; i += kSmallThreads) s_mine[i] = __ldg(topk_idx + a0 + i);
  // warp w counts assignments w*32 + 32*NW*p (+ lane), loading all of its ids first
  constexpr int NP = kSmallAssign / (32 * NW);  // passes per warp at most
  int before = 0, total = 0;
  int ids[NP];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int i = q * 32 * NW + warp * 32 + lane;
    ids[q] = i < S ? __ldg(topk_idx + i) : -1;
  }
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int i0 = q * 32 * NW + warp * 32;
    if (i0 >= S) break;
    const int nb = a0 - i0;  // lanes of this pass that come before a0
    const unsigned bmask = nb >= 32 ? 0xffffffffu : (nb <= 0 ? 0u : (1u << nb) - 1u);
    for (int x = 0; x < E; ++x) {
      const unsigned m = __ballot_sync(0xffffffffu, ids[q] == x);
      if (lane == x) {
        total += __popc(m);
        before += __popc(m & bmask);
      }
    }
  }
  s_cnt[0][warp][lane] = before;
  s_cnt[1][warp][lane] = total;
  __syncthreads();
  if (warp == 0) {
    int bsum = 0, tsum = 0;
    for (int w = 0; w < NW; ++w) {
      bsum += s_cnt[0][w][lane];
      tsum += s_cnt[1][w][lane];
    }
    if (lane >= E) bsum = tsum = 0;
    // exclusive scans over the experts (lanes) of the aligned rows and the M tiles
    const int rows = (tsum + align - 1) / align * align, tiles = (tsum + 127) / 128;
    int ir = rows, it = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, ir, o), b = __shfl_up_sync(0xffffffffu, it, o);
      if (lane >= o) {
        ir += a;
        it += b;
      }
    }
    if (lane < E) {
      s_off[lane + 1] = ir;
      s_tot[lane] = tsum;
    }
    if (lane == 0) s_off[0] = 0;
    if (blockIdx.x == 0) {
      if (lane < E) {
        offsets[lane + 1] = ir;
        tile_offsets[lane + 1] = it;
        kept[lane] = tsum;
        if (tsum != counts[lane]) set_device_error(err, MOE_ERR_DEVICE, 1000 + lane);
      }
      if (lane == 0) offsets[0] = tile_offsets[0] = 0;
    }
    if (tok_cta) {
      // rank this CTA's assignments; lane e holds the next slot of expert e
      int cursor = lane < E ? ir - rows + bsum : 0;
      const int n = min(kSmallTok, T - t0) * k;
      const unsigned lt = (1u << lane) - 1u;
      for (int b = 0; b < n; b += 32) {
        const int i = b + lane;
        int e = i < n ? s_mine[i] : -1 - lane;
        const bool ok = i < n && (unsigned)e < (unsigned)E;
        if (i < n && !ok) e = -1 - lane;  // an id outside [0,E): no slot
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int base = __shfl_sync(0xffffffffu, cursor, ok ? e : 0);
        const int slot = ok ? base + __popc(peers & lt) : -1;
        if (i < n) {
          row_id_map[a0 + i] = slot;
          if (ok) slot_src[slot] = a0 + i;
        }
        // each expert's cursor advances by its assignments in this pass
        for (int x = 0; x < E; ++x) {
          const unsigned m = __ballot_sync(0xffffffffu, ok && e == x);
          if (lane == x) cursor += __popc(m);
        }
      }
    }
  }
  const int e = blockIdx.x;
  if (e >= E) return;
  __syncthreads();
  // the padding rows of expert e: slot_src -1 (k_copy_rows zeroes their Xperm rows)
  for (int r = s_off[e] + s_tot[e] + threadIdx.x; r < s_off[e + 1]; r += kSmallThreads) slot_src[r] = -1;
}

// The whole dispatch of a small dropless layer with its row copy, in one launch
// (T*k <= kSmallAssign, E <= 32, each CTA's token rows fit in shared memory).  On such a
// layer the copy moves ~100 MB and the maps kernel's latency, paid before the copy can
// start, is what keeps the stage off the memory roofline.  Here CTA c owns tokens
// [c*tpc, (c+1)*tpc) and
//   1. one thread starts bulk copies of the CTA's X rows (contiguous in X) into shared
//      memory, in 16 KB pieces on one mbarrier, before any other load of the CTA;
//   2. while they are in flight all threads count, from all of topk_idx, each expert's
//      assignments before the CTA's first assignment and in total: each thread adds its
//      ids into packed 16-bit counters (two experts per 32-bit word), each warp sums the
//      words with one redux.sync apiece, and its lanes add them into shared counters;
//   3. warp 0 derives the aligned segments (CTA 0 writes offsets, tile_offsets and kept
//      and checks the totals against counts) and ranks the CTA's assignments, staged in
//      shared memory during the count, in token order, into shared memory;
//   4. once the rows have arrived, each warp takes its share of the CTA's assignments:
//      it writes row_id_map and slot_src and copies the row from shared memory to its
//      slot of Xperm (16-byte stores); then it zeroes its share of the CTA's part of all
//      experts' padding rows (slot_src -1).
// Reads and writes each keep HBM busy in turn (all CTAs load, then all store): a probe of
// the phases on the Mixtral-style token shape found the rows arriving ~6 us after launch
// whatever the order of the pieces, so per-piece barriers gained nothing.
// The slots are those of the chunked path: offsets[e] + #{earlier assignments to e}.
constexpr int kFusedThreads = 1024;
constexpr int kFusedMaxAssign = 1024;               // tpc*k: the CTA's slots kept in shared memory
constexpr int kFusedRowBytes = 219 * 1024;          // tpc*H*2: the CTA's rows
constexpr uint32_t kFusedPiece = 16384;             // bytes per bulk copy of the rows
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// EW: packed 32-bit counter words per thread, two experts each (4, for E <= 8), or 0 for
// the ballot count (E <= 32).
template <int EW>
__global__ void __launch_bounds__(kFusedThreads, 1) k_dispatch_copy_small(
    const uint16_t* __restrict__ X, const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ counts, int T,
    int H, int E, int k, int align, int tpc, int32_t* __restrict__ offsets, int32_t* __restrict__ tile_offsets,
    int32_t* __restrict__ kept, int32_t* __restrict__ row_id_map, int32_t* __restrict__ slot_src,
    uint16_t* __restrict__ Xperm, int* err, uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t s_rows[];  // the CTA's token rows of X
  __shared__ uint64_t bar;
  __shared__ int s_h[64];  // [e]: assignments to e before this CTA's first; [32 + e]: from it on
  __shared__ int s_off[kSmallMaxE + 1], s_tot[kSmallMaxE], s_pad[kSmallMaxE + 1];
  __shared__ int s_slot[kFusedMaxAssign];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = T * k;
  const int t0 = (int)blockIdx.x * tpc, nt = min(tpc, T - t0);
  const int a0 = t0 * k, n = nt * k;
  const uint32_t row_bytes = (uint32_t)H * 2u;
  if (threadIdx.x < 64) s_h[threadIdx.x] = 0;
  if (threadIdx.x == kFusedThreads - 32) {
    // before this thread's first load: the release fence of the barrier's initialisation
    // then has no load of its own to wait for
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint32_t bytes = row_bytes * (uint32_t)nt;
    mbar_arrive_expect_tx(&bar, bytes);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(X + (size_t)t0 * H);
    for (uint32_t o = 0; o < bytes; o += kFusedPiece)
      bulk_load_1d(s_rows + o, src + o, bytes - o < kFusedPiece ? bytes - o : kFusedPiece, &bar);
  }
  // the caller's totals, for the check by CTA 0 (loaded now, compared after the count)
  const int cnt_in = blockIdx.x == 0 && (int)threadIdx.x < E ? __ldg(counts + threadIdx.x) : 0;
  // 2. counts: each thread loads its ids of all passes first, then adds each into packed
  // counters (expert x: word x/2, bits 16*(x%2); a field never carries, a warp sees at
  // most 32 * NP = 512 ids), or (EW == 0) counts them with ballots; the CTA's own ids go
  // to s_slot.
  constexpr int NP = kSmallAssign / kFusedThreads;
  int ids[NP];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const int i = q * kFusedThreads + (int)threadIdx.x;
    ids[q] = i < S ? __ldg(topk_idx + i) : -1;
  }
  uint32_t mt = 0u, mb = 0u;  // packed: lane w, experts 2w and 2w+1 (EW > 0)
  int before = 0, total = 0;   // lane x, expert x (EW == 0)
  if constexpr (EW > 0) {
    uint32_t tot[EW], bef[EW];
#pragma unroll
    for (int w = 0; w < EW; ++w) tot[w] = bef[w] = 0u;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      if (q * kFusedThreads >= S) break;  // CTA-uniform
      const int i = q * kFusedThreads + (int)threadIdx.x;
      const int id = ids[q];
      if (i >= a0 && i < a0 + n) s_slot[i - a0] = id;
      const bool ok = (unsigned)id < (unsigned)E;  // (ids past S are -1)
      const uint32_t inc = ok ? 1u << ((id & 1) << 4) : 0u, incb = i < a0 ? inc : 0u;
      const int w0 = id >> 1;
#pragma unroll
      for (int w = 0; w < EW; ++w) {
        tot[w] += w0 == w ? inc : 0u;
        bef[w] += w0 == w ? incb : 0u;
      }
    }
    // warp sums; lane w keeps word w (totals, and those before the CTA)
#pragma unroll
    for (int w = 0; w < EW; ++w) {
      const uint32_t st = __reduce_add_sync(0xffffffffu, tot[w]), sb = __reduce_add_sync(0xffffffffu, bef[w]);
      if (lane == w) {
        mt = st;
        mb = sb;
      }
    }
  } else {
    // one ballot per expert per pass, lane x of the warp keeping expert x
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const int i0 = q * kFusedThreads + warp * 32;
      if (i0 >= S) break;  // warp-uniform
      const int i = i0 + lane;
      if (i >= a0 && i < a0 + n) s_slot[i - a0] = ids[q];
      const int nb = a0 - i0;  // lanes of this pass before the CTA's first assignment
      const unsigned bmask = nb >= 32 ? 0xffffffffu : (nb <= 0 ? 0u : (1u << nb) - 1u);
      for (int x = 0; x < E; ++x) {
        const unsigned m = __ballot_sync(0xffffffffu, ids[q] == x);
        if (lane == x) {
          total += __popc(m);
          before += __popc(m & bmask);
        }
      }
    }
  }
  __syncthreads();  // s_h is zeroed and s_slot holds the CTA's ids
  if constexpr (EW > 0) {
    if (lane < EW && mt != 0u) {
      atomicAdd(&s_h[2 * lane], (int)(mb & 0xffffu));
      atomicAdd(&s_h[2 * lane + 1], (int)(mb >> 16));
      atomicAdd(&s_h[32 + 2 * lane], (int)((mt - mb) & 0xffffu));
      atomicAdd(&s_h[32 + 2 * lane + 1], (int)((mt - mb) >> 16));
    }
  } else if (lane < E && total > 0) {
    atomicAdd(&s_h[lane], before);
    atomicAdd(&s_h[32 + lane], total - before);
  }
  __syncthreads();
  // 3. segments and this CTA's ranks
  if (warp == 0) {
    const int before_e = lane < E ? s_h[lane] : 0;
    const int tsum = lane < E ? before_e + s_h[32 + lane] : 0;
    const int rows = (tsum + align - 1) / align * align, tiles = (tsum + 127) / 128, pad = rows - tsum;
    int ir = rows, it = tiles, ip = pad;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, ir, o), b = __shfl_up_sync(0xffffffffu, it, o),
                c = __shfl_up_sync(0xffffffffu, ip, o);
      if (lane >= o) {
        ir += a;
        it += b;
        ip += c;
      }
    }
    if (lane < E) {
      s_off[lane + 1] = ir;
      s_tot[lane] = tsum;
      s_pad[lane + 1] = ip;
    }
    if (lane == 0) s_off[0] = s_pad[0] = 0;
    if (blockIdx.x == 0) {
      if (lane < E) {
        offsets[lane + 1] = ir;
        tile_offsets[lane + 1] = it;
        kept[lane] = tsum;
        if (tsum != cnt_in) set_device_error(err, MOE_ERR_DEVICE, 1000 + lane);
      }
      if (lane == 0) offsets[0] = tile_offsets[0] = 0;
    }
    // ranks in token order: lane x holds expert x's next slot; one ballot per expert per 32
    int cursor = lane < E ? ir - rows + before_e : 0;
    const unsigned lt = (1u << lane) - 1u;
    for (int b = 0; b < n; b += 32) {
      const int i = b + lane;
      const int e = i < n ? s_slot[i] : -1;
      const bool ok = i < n && (unsigned)e < (unsigned)E;  // an id outside [0,E): no slot
      int rank = 0, cnt = 0;
      for (int x = 0; x < E; ++x) {
        const unsigned m = __ballot_sync(0xffffffffu, ok && e == x);
        if (ok && e == x) rank = __popc(m & lt);
        if (lane == x) cnt = __popc(m);
      }
      const int base = __shfl_sync(0xffffffffu, cursor, ok ? e : 0);
      cursor += cnt;
      if (i < n) s_slot[i] = ok ? base + rank : -1;  // the lane's own entry, read above by this lane only
    }
  }
  __syncthreads();
  // 4. once the rows have arrived (every thread observes the barrier, within the library's
  // wait limit), warp w takes assignments w, w + 32, ...: their maps and their rows
  bool ok = mbar_wait(&bar, 0, wait_ns);
  const int nvec = H / 8;
  constexpr int NW = kFusedThreads / 32;
  for (int i = warp; i < n && ok; i += NW) {
    const int slot = s_slot[i];
    if (lane == 0) {
      row_id_map[a0 + i] = slot;
      if (slot >= 0) slot_src[slot] = a0 + i;
    }
    if (slot < 0) continue;
    const uint4* in = reinterpret_cast<const uint4*>(s_rows + (size_t)(i / k) * row_bytes);
    uint4* out = reinterpret_cast<uint4*>(Xperm + (size_t)slot * H);
    for (int v0 = 0; v0 < nvec; v0 += 4 * 32) {
      uint4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < nvec) x[u] = in[v];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < nvec) out[v] = x[u];
      }
    }
  }
  if (!ok) {
    // the wait ran out: record it, and let the copies still in flight land before the CTA exits
    if (threadIdx.x == 0) set_device_error(err, MOE_ERR_TIMEOUT, 20);
    mbar_wait(&bar, 0);
  }
  // this CTA's share of all experts' padding rows, one warp per row
  const int P = s_pad[E];
  const int p0 = (int)((int64_t)P * blockIdx.x / gridDim.x), p1 = (int)((int64_t)P * (blockIdx.x + 1) / gridDim.x);
  for (int p = p0 + warp; p < p1; p += NW) {
    int e = 0;
    while (s_pad[e + 1] <= p) ++e;
    const int row = s_off[e] + s_tot[e] + (p - s_pad[e]);
    uint4* out = reinterpret_cast<uint4*>(Xperm + (size_t)row * H);
    for (int v = lane; v < nvec; v += 32) out[v] = make_uint4(0, 0, 0, 0);
    if (lane == 0) slot_src[row] = -1;
  }
}

// Order-preserving key of a priority: a larger float gives a larger key; -0 and +0
// give the same key.
__device__ __forceinline__ uint32_t priority_key(float f) {
  const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix count of `flag` over the 1024 threads of the block, in thread
// order; *total receives the block's count.  Every thread must call it.
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) warp_tot[warp] = __popc(b);
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < 32; ++w) {
    const int n = warp_tot[w];
    before += w < warp ? n : 0;
    all += n;
  }
  __syncthreads();
  *total = all;
  return before + __popc(b & ((1u << lane) - 1u));
}

// One CTA per expert: keep the cap assignments of largest priority (ties to the
// earlier assignment in token order) and give them rows in token order.
__global__ void __launch_bounds__(1024) k_drop_select(const float* __restrict__ priority,
                                                      const int32_t* __restrict__ drop_order,
                                                      const int32_t* __restrict__ drop_start,
                                                      const int32_t* __restrict__ offsets,
                                                      const int32_t* __restrict__ kept, int cap,
                                                      int32_t* __restrict__ row_id_map,
                                                      int32_t* __restrict__ slot_src, int* err) {
  __shared__ int hist[256];
  __shared__ int warp_tot[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x, tid = threadIdx.x;
  const int s0 = drop_start[e], n = drop_start[e + 1] - s0;
  const int row0 = offsets[e];
  const int32_t* ord = drop_order + s0;
  if (n <= cap) {  // nothing to drop
    for (int i = tid; i < n; i += 1024) {
      const int src = ord[i];
      row_id_map[src] = row0 + i;
      slot_src[row0 + i] = src;
    }
    return;
  }
  if (cap == 0) {
    for (int i = tid; i < n; i += 1024) row_id_map[ord[i]] = -1;
    return;
  }
  // radix select, 8 bits per pass from the top: prefix = the cap-th largest key,
  // need = how many keys equal to it are kept
  uint32_t prefix = 0;
  int need = cap;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = tid; b < 256; b += 1024) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += 1024) {
      const uint32_t key = priority_key(__ldg(priority + ord[i]));
      if (pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8))) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int above = 0, b = 255;
      for (; b > 0; --b) {
        if (above + hist[b] >= need) break;
        above += hist[b];
      }
      s_prefix = prefix | ((uint32_t)b << shift);
      s_need = need - above;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
  }
  // token-order pass: keep key > prefix, and the first `need` keys equal to it
  int eq_run = 0, kept_run = 0;
  for (int r0 = 0; r0 < n; r0 += 1024) {
    const int i = r0 + tid;
    const bool valid = i < n;
    const int src = valid ? ord[i] : 0;
    const uint32_t key = valid ? priority_key(__ldg(priority + src)) : 0u;
    int eq_tot, kept_tot;
    const bool eq = valid && key == prefix;
    const int eq_rank = eq_run + block_excl_count(eq, warp_tot, &eq_tot);
    const bool keep = valid && (key > prefix || (eq && eq_rank < need));
    const int krank = kept_run + block_excl_count(keep, warp_tot, &kept_tot);
    if (keep) {
      row_id_map[src] = row0 + krank;
      slot_src[row0 + krank] = src;
    } else if (valid) {
      row_id_map[src] = -1;
    }
    eq_run += eq_tot;
    kept_run += kept_tot;
  }
  if (tid == 0 && kept_run != kept[e]) set_device_error(err, MOE_ERR_DEVICE, 3000 + e);
}

// Xperm[row_id_map[t,j]] = X[t]: one warp per token, its k destination rows read once;
// each lane loads U 16-byte vectors of the row before storing them to every kept row.
// CTAs past the token range zero the padding rows, kPadSplit CTAs per expert, in the
// same launch (their writes stream alongside the copy).
__global__ void __launch_bounds__(256) k_copy_rows(const uint16_t* __restrict__ X,
                                                   const int32_t* __restrict__ row_id_map,
                                                   const int32_t* __restrict__ offsets,
                                                   const int32_t* __restrict__ kept, int T, int H, int k,
                                                   int tok_blocks, uint16_t* __restrict__ Xperm) {
  constexpr int U = kGatherUnroll;
  if ((int)blockIdx.x >= tok_blocks) {
    const int64_t nvec = H / 8;
    const int p = blockIdx.x - tok_blocks;
    const int e = p / kPadSplit, part = p % kPadSplit;
    const int r1e = offsets[e + 1];
    const int r0e = min(max(offsets[e] + kept[e], offsets[e]), r1e);
    const int per = (r1e - r0e + kPadSplit - 1) / kPadSplit;
    const int r0 = r0e + part * per, r1 = min(r1e, r0 + per);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = (int64_t)r0 * nvec + threadIdx.x; i < (int64_t)r1 * nvec; i += 256)
      reinterpret_cast<uint4*>(Xperm)[i] = z;
    return;
  }
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = lane < k ? row_id_map[(size_t)t * k + lane] : -1;
  const int nvec = H / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)t * H);
  for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u + lane;
      x[u] = v < nvec ? __ldg(xr + v) : make_uint4(0, 0, 0, 0);
    }
    for (int j = 0; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      if (slot < 0) continue;  // dropped by capacity: no row
      uint4* out = reinterpret_cast<uint4*>(Xperm + (size_t)slot * H);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < nvec) out[v] = x[u];
      }
    }
  }
}

// Y[t] = sum_j g[t,j] Yperm[row_id_map[t,j]] (+ Yshared[t]); one warp per token.
// gates == nullptr: unit weights (the rows are gated already).
__global__ void __launch_bounds__(256) k_combine(const uint16_t* __restrict__ Yperm,
                                                 const int32_t* __restrict__ row_id_map,
                                                 const float* __restrict__ gates, const uint16_t* __restrict__ Ysh,
                                                 uint16_t* __restrict__ Y, int T, int H, int k) {
  constexpr int U = kGatherUnroll;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = lane < k ? row_id_map[(size_t)t * k + lane] : 0;
  const float my_g = lane < k ? (gates ? gates[(size_t)t * k + lane] : 1.0f) : 0.f;
  const int nvec = H / 8;
  // U vectors per lane per source row are loaded before any is used; every lane runs
  // every iteration (the shuffles need the full warp)
  for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      if (slot < 0) continue;  // the same for the whole warp
      const uint4* src = reinterpret_cast<const uint4*>(Yperm + (size_t)slot * H);
      uint4 y[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u + lane;
        y[u] = v < nvec ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[8];
        unpack8(y[u], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[u][q] = fmaf(g, f[q], acc[u][q]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u + lane;
      if (v >= nvec) continue;
      if (Ysh) {
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(Ysh + (size_t)t * H) + v), f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[u][q] += f[q];
      }
      reinterpret_cast<uint4*>(Y + (size_t)t * H)[v] = pack8(acc[u]);
    }
  }
}

// dYperm[slot] = bf16(g dY[t]); dgates[t,j] = <dY[t], Yperm[slot]>.
// One warp per assignment a = t*k + j, so that the k assignments of a token stream
// independently; they sit in consecutive warps, so dY[t] comes from DRAM once.
// CTAs past the assignment range zero the padding rows, kPadSplit CTAs per expert.
// gates == nullptr: g = 1 (gated rows); dgates == nullptr: no gate gradient.
__global__ void __launch_bounds__(256) k_combine_bwd(const uint16_t* __restrict__ dY,
                                                     const uint16_t* __restrict__ Yperm,
                                                     const int32_t* __restrict__ row_id_map,
                                                     const float* __restrict__ gates,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ counts, uint16_t* __restrict__ dYperm,
                                                     float* __restrict__ dgates, int T, int H, int k, int asg_blocks) {
  const int nvec = H / 8;
  if ((int)blockIdx.x >= asg_blocks) {
    const int p = blockIdx.x - asg_blocks;
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
  const int64_t a = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (a >= (int64_t)T * k) return;
  const int slot = row_id_map[a];
  float dot = 0.f;
  if (slot >= 0) {  // a dropped assignment (capacity) has no row and a zero gate gradient
    const int t = (int)(a / k);
    const float g = gates ? gates[a] : 1.0f;
    constexpr int U = kGatherUnroll;
    const uint4* dyr = reinterpret_cast<const uint4*>(dY + (size_t)t * H);
    const uint4* yr = reinterpret_cast<const uint4*>(Yperm + (size_t)slot * H);
    uint4* outr = reinterpret_cast<uint4*>(dYperm + (size_t)slot * H);
    for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
      uint4 dy[U], y[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u + lane;
        dy[u] = v < nvec ? __ldg(dyr + v) : make_uint4(0, 0, 0, 0);
        y[u] = dgates && v < nvec ? __ldg(yr + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v >= nvec) continue;
        if (dgates || g != 1.0f) {
          float df[8], yf[8], o[8];
          unpack8(dy[u], df);
          unpack8(y[u], yf);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            dot = fmaf(df[q], yf[q], dot);
            o[q] = g * df[q];
          }
          outr[v] = pack8(o);
        } else {
          outr[v] = dy[u];  // a unit gate: the row is a copy
        }
      }
    }
  }
  if (dgates) {
    dot = warp_sum(dot);
    if (lane == 0) dgates[a] = dot;
  }
}

// dX[t] = sum_j dXperm[row_id_map[t,j]] + dX_router[t] + dX_shared[t].
__global__ void __launch_bounds__(256) k_permute_bwd(const uint16_t* __restrict__ dXperm,
                                                     const int32_t* __restrict__ row_id_map,
                                                     const float* __restrict__ dXr, const uint16_t* __restrict__ dXs,
                                                     uint16_t* __restrict__ dX, int T, int H, int k) {
  constexpr int U = kGatherUnroll;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = lane < k ? row_id_map[(size_t)t * k + lane] : 0;
  const int nvec = H / 8;
  for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
    // the router and shared-expert terms are loaded first, so that they are in flight
    // with the expert rows (two rows per step); the sum keeps the order rows, router, shared
    float4 ra[U], rb[U];
    uint4 sx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u + lane;
      const bool in = v < nvec;
      if (dXr && in) {
        const float4* rr = reinterpret_cast<const float4*>(dXr + (size_t)t * H) + 2 * v;
        ra[u] = __ldg(rr);
        rb[u] = __ldg(rr + 1);
      } else {
        ra[u] = rb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      sx[u] = dXs && in ? __ldg(reinterpret_cast<const uint4*>(dXs + (size_t)t * H) + v) : make_uint4(0, 0, 0, 0);
    }
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
    for (int j = 0; j < k; j += 2) {
      const int s0 = __shfl_sync(0xffffffffu, my_slot, j);
      const int s1 = j + 1 < k ? __shfl_sync(0xffffffffu, my_slot, j + 1) : -1;
      uint4 x0[U], x1[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u + lane;
        x0[u] = s0 >= 0 && v < nvec ? __ldg(reinterpret_cast<const uint4*>(dXperm + (size_t)s0 * H) + v)
                                    : make_uint4(0, 0, 0, 0);
        x1[u] = s1 >= 0 && v < nvec ? __ldg(reinterpret_cast<const uint4*>(dXperm + (size_t)s1 * H) + v)
                                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[8];
        if (s0 >= 0) {  // a dropped assignment (capacity) adds nothing
          unpack8(x0[u], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[u][q] += f[q];
        }
        if (s1 >= 0) {
          unpack8(x1[u], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[u][q] += f[q];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u + lane;
      if (v >= nvec) continue;
      if (dXr) {
        acc[u][0] += ra[u].x; acc[u][1] += ra[u].y; acc[u][2] += ra[u].z; acc[u][3] += ra[u].w;
        acc[u][4] += rb[u].x; acc[u][5] += rb[u].y; acc[u][6] += rb[u].z; acc[u][7] += rb[u].w;
      }
      if (dXs) {
        float f[8];
        unpack8(sx[u], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[u][q] += f[q];
      }
      reinterpret_cast<uint4*>(dX + (size_t)t * H)[v] = pack8(acc[u]);
    }
  }
}

// Gated path: dgates[t,j] = sum over n of part[row][n] (fixed order), row =
// row_id_map[t,j]; 0 for a dropped assignment.
__global__ void __launch_bounds__(256) k_dgates_reduce(const int32_t* __restrict__ row_id_map,
                                                       const float* __restrict__ part, int ntile, int64_t n,
                                                       float* __restrict__ dgates) {
  for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const int row = row_id_map[i];
    float s = 0.f;
    if (row >= 0)
      for (int c = 0; c < ntile; ++c) s += part[(int64_t)row * ntile + c];
    dgates[i] = s;
  }
}

}  // namespace

cudaError_t launch_dgates_reduce(const moe_config& c, const int32_t* row_id_map, const float* part, int ntile,
                                 float* dgates, int nsm, cudaStream_t st) {
  const int64_t n = (int64_t)c.T * c.k;
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4LL * nsm) blocks = 4LL * nsm;
  k_dgates_reduce<<<(int)blocks, 256, 0, st>>>(row_id_map, part, ntile, n, dgates);
  return cudaGetLastError();
}

cudaError_t launch_permute(const moe_config& c, const uint16_t* X, const int32_t* topk_idx, const int32_t* counts,
                           int cap, const float* priority, int32_t* kept, int32_t* offsets, int32_t* tile_offsets,
                           int32_t* row_id_map, int32_t* slot_src, uint16_t* Xperm, int32_t* chunk_counts,
                           int32_t* chunk_base, int32_t* drop_order, int32_t* drop_start, int* err, int nsm,
                           cudaStream_t st) {
  if (!kept || (priority && (!drop_order || !drop_start))) return cudaErrorInvalidValue;
  if (!priority) drop_order = drop_start = nullptr;
  const int nch = (c.T + kChunk - 1) / kChunk;
  cudaError_t e;
  // (every CTA counts all assignments with E ballots per 32 of them: bounded by kSmallWork)
  if (cap == INT_MAX && c.T > 0 && (int64_t)c.T * c.k <= kSmallAssign && c.E <= kSmallMaxE &&
      (int64_t)c.T * c.k * c.E <= kSmallWork) {
    // a small dropless layer: the whole dispatch, with the row copy when each CTA's rows
    // fit in shared memory, in one launch
    const int g0 = nsm < c.T ? nsm : c.T;
    const int tpc = (c.T + g0 - 1) / g0;
    if (Xperm && (int64_t)tpc * c.H * 2 <= kFusedRowBytes && tpc * c.k <= kFusedMaxAssign) {
      const int grid = (c.T + tpc - 1) / tpc;
      const size_t smem = (size_t)tpc * c.H * 2;
      if (smem > 48 * 1024) {
        static std::atomic<uint64_t> attr{0};
        static std::atomic<uint64_t> attr0{0};
        if ((e = c.E <= 8 ? raise_smem_limit(attr, k_dispatch_copy_small<4>, kFusedRowBytes)
                          : raise_smem_limit(attr0, k_dispatch_copy_small<0>, kFusedRowBytes)) != cudaSuccess)
          return e;
      }
      if (c.E <= 8)
        k_dispatch_copy_small<4><<<grid, kFusedThreads, smem, st>>>(X, topk_idx, counts, c.T, c.H, c.E, c.k, c.align,
                                                                    tpc, offsets, tile_offsets, kept, row_id_map,
                                                                    slot_src, Xperm, err, pipeline_wait_ns());
      else
        k_dispatch_copy_small<0><<<grid, kFusedThreads, smem, st>>>(X, topk_idx, counts, c.T, c.H, c.E, c.k,
                                                                     c.align, tpc, offsets, tile_offsets, kept,
                                                                     row_id_map, slot_src, Xperm, err,
                                                                     pipeline_wait_ns());
      return cudaGetLastError();
    }
    const int tb = (c.T + kSmallTok - 1) / kSmallTok;
    k_dispatch_small<<<tb > c.E ? tb : c.E, kSmallThreads, 0, st>>>(topk_idx, counts, c.T, c.E, c.k, c.align, tb,
                                                                     offsets, tile_offsets, kept, row_id_map,
                                                                     slot_src, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (Xperm) {
      const int cb = (c.T + 7) / 8;
      k_copy_rows<<<cb + c.E * kPadSplit, 256, 0, st>>>(X, row_id_map, offsets, kept, c.T, c.H, c.k, cb, Xperm);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (nch > 0) {
    k_chunk_hist<<<nch, 256, 0, st>>>(topk_idx, c.T, c.E, c.k, chunk_counts);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t scan_smem = nch * c.E <= kScanStage ? sizeof(int) * (size_t)nch * c.E : 0;
  if (scan_smem > 48 * 1024) {
    static std::atomic<uint64_t> attr{0};
    if ((e = raise_smem_limit(attr, k_scan, sizeof(int) * kScanStage)) != cudaSuccess) return e;
  }
  k_scan<<<1, 1024, scan_smem, st>>>(counts, chunk_counts, nch, c.E, c.align, cap, kept, offsets, tile_offsets,
                                     chunk_base, drop_start, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the padding CTAs size each segment's tail from the kept rows the scan counted
  k_scatter<<<nch + c.E * kPadSplit, 256, 0, st>>>(topk_idx, chunk_base, kept, offsets, c.T, c.E, c.k, nch, cap,
                                                   row_id_map, slot_src, drop_order, drop_start);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (priority) {
    k_drop_select<<<c.E, 1024, 0, st>>>(priority, drop_order, drop_start, offsets, kept, cap, row_id_map, slot_src,
                                        err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (Xperm) {  // no Xperm: the maps only (the grouped GEMM gathers the rows)
    const int tb = (c.T + 7) / 8;
    k_copy_rows<<<tb + c.E * kPadSplit, 256, 0, st>>>(X, row_id_map, offsets, kept, c.T, c.H, c.k, tb, Xperm);
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
  const int ab = (int)(((int64_t)c.T * c.k + 7) / 8);
  k_combine_bwd<<<ab + c.E * kPadSplit, 256, 0, st>>>(dY, Yperm, row_id_map, gates, offsets, counts, dYperm, dgates, c.T,
                                                      c.H, c.k, ab);
  return cudaGetLastError();
}

cudaError_t launch_permute_bwd(const moe_config& c, const uint16_t* dXperm, const int32_t* row_id_map,
                               const float* dXr, const uint16_t* dXs, uint16_t* dX, cudaStream_t st) {
  if (c.T == 0) return cudaSuccess;
  k_permute_bwd<<<(c.T + 7) / 8, 256, 0, st>>>(dXperm, row_id_map, dXr, dXs, dX, c.T, c.H, c.k);
  return cudaGetLastError();
}

}  // namespace moe
