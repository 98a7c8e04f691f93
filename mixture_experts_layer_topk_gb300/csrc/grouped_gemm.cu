// Compute stage: the experts' SwiGLU MLPs as persistent grouped GEMMs on the
// sm_100-family tensor cores (tcgen05.mma, accumulators in tensor memory,
// operands staged by TMA), forward and backward.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (summary
// page, "Method"): all local experts run in a single grouped GEMM call; the
// compute recipes are grouped GEMM, kernel fusion and sync-free execution.
// Here each of the six expert GEMMs of a training step is one launch over all
// experts; the expert segments and the M-tile schedule are read on the device
// (offsets / tile_offsets written by the dispatch), so nothing goes back to
// the host.  SwiGLU ("GLU Variants Improve Transformer", cited on the index
// page) is fused into the FC1 epilogue, and its backward into the FC2-dgrad
// epilogue.
//
// One CTA per SM, 6 warps: warp 0 issues TMA loads into a ring of shared
// memory stages, warp 1 allocates tensor memory and issues tcgen05.mma from
// one thread, warps 2-5 drain the double-buffered accumulator (tcgen05.ld),
// apply the epilogue and stage bf16 outputs for TMA bulk stores.  bf16 tiles
// that are 256 wide run on CTA pairs (a cluster of two): one tcgen05.mma
// cta_group::2 computes a 256 x 256 x 16 step from both CTAs' shared memory,
// each CTA holding 128 rows of A and half of B, and each CTA's tensor memory
// holding its 128 rows of the accumulator.  Narrower bf16 tiles and the FP8
// tiles (128 x 128 x 128, block-scaled) run one CTA per tile.  Every wait is
// bounded; a wait that runs out records MOE_ERR_TIMEOUT in the device error
// word and the CTA unwinds.
//
// The three operand layouts:
//   FWD   D[m,n] = sum_k A[m,k] B[n,k]  A K-major (rows of a permuted buffer), B K-major (weights)
//   DGRAD D[m,n] = sum_k A[m,k] B[k,n]  A K-major, B MN-major (weights used transposed)
//   WGRAD D[m,n] = sum_r A[r,m] B[r,n]  both MN-major, K = the expert's rows (ragged)
#include <cudaTypedefs.h>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BM = 128;
// every stage holds 128 bytes of K per row: 64 bf16 or 128 FP8 elements
template <bool FP8>
struct Geo {
  static constexpr int EB = FP8 ? 1 : 2;          // element bytes
  static constexpr int BKE = 128 / EB;            // K elements per stage
  static constexpr int MN_INNER = 128 / EB;       // elements of one 128-byte MN-major row
  static constexpr int KSTEP = FP8 ? 32 : 16;     // K of one MMA instruction
};
constexpr int kStagingBytes = 16384;  // per epilogue warpgroup
// bf16 weight gradients: token rows per stage (both operands MN-major, 128-byte rows of
// 64 columns); 8 MMAs per stage wait and commit
constexpr int kWgradRows = 128;
// FP8: k-blocks whose scale words the scale-factor warps hold in registers ahead of use
constexpr int kSfAhead = 4;
constexpr int kEpiBarrier = 1;  // named barrier of the first epilogue warpgroup (the second uses 2)

// Threads of a launch: 6 warps, plus 4 scale-factor warps (FP8) or a second epilogue
// warpgroup (NEPI = 2).
template <bool FP8, int NEPI>
constexpr int threads_of() { return FP8 || NEPI == 2 ? 320 : 192; }

enum { MODE_FWD = 0, MODE_DGRAD = 1, MODE_WGRAD = 2 };
enum { EPI_STORE = 0, EPI_SWIGLU = 1, EPI_DSWIGLU = 2, EPI_F32 = 3 };

struct GemmArgs {
  int E;
  int K;           // FWD / DGRAD: reduction length
  int n_tiles;     // tiles along N
  int m_tiles;     // WGRAD: tiles along M of one expert's output
  int dense_rows;  // > 0: a single dense segment of this many rows (the shared expert)
  const int32_t* seg_off;   // [E+1] segment starts in the permuted buffers
  const int32_t* tile_off;  // [E+1] prefix of M tiles per expert
  const int32_t* counts;    // [E] rows per expert
  uint16_t* D;
  int64_t ldd;
  int64_t d_estride;        // WGRAD: elements between experts' outputs
  uint16_t* D2;             // EPI_SWIGLU: activation output
  int64_t ldd2;
  const uint16_t* GU;       // EPI_DSWIGLU: saved pre-activations
  int64_t ldgu;
  int F;                    // SWIGLU / DSWIGLU: column offset of the "up" half
  int n_valid;              // > 0: output columns at or beyond n_valid are not stored
  int ksplit_rows;          // WGRAD dense: > 0 splits the rows into chunks of this many ("experts")
  int kwrap;                // K-major A (FWD/DGRAD): the K coordinate wraps modulo kwrap;
                            // WGRAD: B's row coordinate wraps modulo kwrap (0: no wrap)
  int n_fast;               // WGRAD: tiles walk N fastest (else M fastest) within an expert
  // gated rows (the memory-efficient path): row r carries gate gates[slot_src[r]], 0 for
  // a padding row.  SWIGLU: the activation output is gate * silu(g) * u.  DSWIGLU: the
  // accumulator is the gradient of the gated activation; the epilogue recomputes
  // a = silu(g) * u from GU, writes gate * a to a_out, the per-tile partial of
  // <accumulator row, a> to dg_part[row * n_tiles + tile], and backpropagates gate * acc.
  const int32_t* slot_src;
  const float* gates;
  float* dg_part;
  uint16_t* a_out;
  int64_t lda_out;
  // gathered rows (CTA pairs; FWD: the A rows, WGRAD: the B rows along K): permuted row
  // r is row gather_src[r] / gather_k of the mapped tensor, or past it (zeros) when
  // gather_src[r] < 0; the map has one-row boxes.  gather_rows bounds r.
  const int32_t* gather_src;
  int gather_k, gather_oob;
  int64_t gather_rows;
  // FP8 block scales (UE8M0 bytes): A and B, addressed per mode (see the SF warps)
  const uint8_t* sfa;
  int64_t sfa_ld;
  const uint8_t* sfb;
  int sfb_r, sfb_c;
  int64_t sfb_ld;
  int* err;
  uint64_t wait_ns;  // limit of each pipeline wait (0: one non-blocking test)
};

struct Tile {
  int e, m0, n0, k0, kb;
  bool valid;  // CTA pairs: this CTA's half of the 256-row tile exists
  int krem;    // weight gradients: rows of K in the last k-block (else BK)
};

template <int MODE, int EPI, int BN, int BK>
__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& g, const int* s_seg, const int* s_tile,
                                            const int* s_cnt) {
  Tile r;
  r.krem = BK;
  if constexpr (MODE != MODE_WGRAD) {
    int e = 0, m, n;
    if (g.dense_rows > 0) {
      const int mt = (g.dense_rows + BM - 1) / BM;
      n = t / mt;
      m = t % mt;
      r.m0 = m * BM;
    } else {
      int lo = 0, hi = g.E;  // s_tile[lo]*nt <= t < s_tile[hi]*nt
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tile[mid] * g.n_tiles <= t)
          lo = mid;
        else
          hi = mid;
      }
      e = lo;
      const int local = t - s_tile[e] * g.n_tiles;
      const int mt = s_tile[e + 1] - s_tile[e];
      n = local / mt;
      m = local % mt;
      r.m0 = s_seg[e] + m * BM;
    }
    r.e = e;
    r.n0 = n * (EPI == EPI_SWIGLU ? BN / 2 : BN);
    r.k0 = 0;
    r.kb = g.K / BK;
    r.valid = true;
  } else {
    const int per = g.m_tiles * g.n_tiles;
    const int e = t / per, local = t % per;
    r.e = e;
    r.m0 = (g.n_fast ? local / g.n_tiles : local % g.m_tiles) * BM;
    r.n0 = (g.n_fast ? local % g.n_tiles : local / g.m_tiles) * BN;
    int rows;
    if (g.dense_rows > 0 && g.ksplit_rows > 0) {
      r.k0 = e * g.ksplit_rows;
      rows = g.dense_rows - r.k0 < g.ksplit_rows ? g.dense_rows - r.k0 : g.ksplit_rows;
      r.kb = rows > 0 ? (rows + BK - 1) / BK : 0;
    } else if (g.dense_rows > 0) {
      r.k0 = 0;
      rows = g.dense_rows;
      r.kb = (g.dense_rows + BK - 1) / BK;
    } else {
      r.k0 = s_seg[e];
      rows = s_cnt[e];
      r.kb = (s_cnt[e] + BK - 1) / BK;
    }
    // rows past the count in the last block are zero (segment padding, or past the dense
    // tensor, read as zeros): their MMA steps are skipped.  A split of the dense rows ends
    // on a block boundary unless it is the last one.
    if (r.kb > 0) r.krem = rows - (r.kb - 1) * BK;
    r.valid = true;
  }
  return r;
}

// CTA pairs: tile t is a 256-row pair of M tiles (2*mp and 2*mp+1 of one expert);
// CTA `rank` owns M tile 2*mp + rank, which may not exist when an expert has an odd
// number of M tiles (its A rows then point past the tensor and read as zeros).
template <int MODE, int EPI, int BN, int BK>
__device__ __forceinline__ Tile decode_pair_tile(int t, const GemmArgs& g, const int* s_seg, const int* s_tile,
                                                 const int* s_ptile, const int* s_cnt, int rank, int64_t oob_row) {
  Tile r;
  r.krem = BK;
  if constexpr (MODE != MODE_WGRAD) {
    int e = 0, n, mp, mt;
    if (g.dense_rows > 0) {
      mt = (g.dense_rows + BM - 1) / BM;
      const int pm = (mt + 1) / 2;
      n = t / pm;
      mp = t % pm;
    } else {
      int lo = 0, hi = g.E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_ptile[mid] * g.n_tiles <= t)
          lo = mid;
        else
          hi = mid;
      }
      e = lo;
      const int local = t - s_ptile[e] * g.n_tiles;
      const int pm = s_ptile[e + 1] - s_ptile[e];
      n = local / pm;
      mp = local % pm;
      mt = s_tile[e + 1] - s_tile[e];
    }
    const int m = 2 * mp + rank;
    r.valid = m < mt;
    r.m0 = g.dense_rows > 0 ? m * BM : (r.valid ? s_seg[e] + m * BM : (int)oob_row);
    r.e = e;
    r.n0 = n * (EPI == EPI_SWIGLU ? BN / 2 : BN);
    r.k0 = 0;
    r.kb = g.K / BK;
  } else {
    const int mpairs = (g.m_tiles + 1) / 2;
    const int per = mpairs * g.n_tiles;
    const int e = t / per, local = t % per;
    const int m = 2 * (g.n_fast ? local / g.n_tiles : local % mpairs) + rank;
    r.e = e;
    r.valid = m < g.m_tiles;
    r.m0 = m * BM;  // past M when invalid: the MN-major A box reads zeros
    r.n0 = (g.n_fast ? local % g.n_tiles : local / mpairs) * BN;
    const int rows = g.dense_rows > 0 ? g.dense_rows : s_cnt[e];
    r.k0 = g.dense_rows > 0 ? 0 : s_seg[e];
    r.kb = (rows + BK - 1) / BK;
    // the rows past the expert's count in its last block are zero (padding rows of the
    // 128-aligned segment): their MMA steps add nothing and are skipped
    if (r.kb > 0) r.krem = rows - (r.kb - 1) * BK;
  }
  return r;
}

// Weight-gradient epilogue without staging: stores one 32-row x 32-column chunk of bf16
// outputs held one row per lane (acc: the lane's 32 fp32 accumulator values, from
// tcgen05.ld 32x32b).  A 4x4 transpose of 16-byte units inside each group of four lanes
// (two butterfly exchanges, over lane bits 0 and 1) leaves lane 4j+l holding unit l of
// rows 4j..4j+3, so each of the four store instructions writes 8 rows x 64 contiguous
// bytes (whole 32-byte sectors) with no shared memory, proxy fence or barrier.
// row0: this warp's first output row at the chunk's first column; ldd: row pitch.
__device__ __forceinline__ void store_chunk_direct(uint16_t* row0, int64_t ldd, int lane, const uint32_t* acc) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
  const bool l0 = lane & 1, l1 = lane & 2;
  // lanes l and l^1 swap the units whose index bit 0 differs from the lane's bit 0
#pragma unroll
  for (int s1 = 0; s1 < 2; ++s1)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = 8 * s1 + q, b = 8 * s1 + 4 + q;  // units (s1, 0) and (s1, 1)
      const uint32_t y = __shfl_xor_sync(0xffffffffu, l0 ? w[a] : w[b], 1);
      if (l0)
        w[a] = y;
      else
        w[b] = y;
    }
  // lanes l and l^2 swap the units whose index bit 1 differs from the lane's bit 1
#pragma unroll
  for (int s0 = 0; s0 < 2; ++s0)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = 4 * s0 + q, b = 8 + 4 * s0 + q;  // units (0, s0) and (1, s0)
      const uint32_t y = __shfl_xor_sync(0xffffffffu, l1 ? w[a] : w[b], 2);
      if (l1)
        w[a] = y;
      else
        w[b] = y;
    }
  const int j = lane >> 2, l = lane & 3;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<uint4*>(row0 + (int64_t)(4 * j + u) * ldd + 8 * l) =
        make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
}

__device__ __forceinline__ void store32(uint16_t* dst, const float* v) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = pack8(v + 8 * i);
}

// Exit path of a producer: every TMA load this CTA issued has landed before the CTA may
// leave.  `issued` counts the producer's stage loads (issue i went to stage i % ST with
// phase parity (i / ST) & 1); only the producer's thread calls this.
//
// One CTA: wait for the last issue of every stage.  CTA pairs: the loads of both CTAs
// complete on the leader's barriers, which the leader arms for both halves, and after a
// timeout the two producers may have stopped after different numbers of issues (one
// passed a wait the other gave up on).  The peer therefore sends its count to the
// leader (a store into the leader's shared memory, then a release-arrive on peer_done);
// the leader arms the issues only the peer made for the peer's half alone (once the
// stage's previous phase has completed, so the arrival counts in the right phase),
// counts the missing half of the issues only it made as arrived (mbarrier.complete_tx),
// and then waits for the last issue of every stage.  Either count exceeds the other by
// at most ST: an issue needs the MMA to have consumed the stage's previous issue, which
// needs both halves of it.  The peer stays alive until the closing cluster barrier,
// which the leader reaches only after this.
template <int ST, bool PAIR>
__device__ __forceinline__ void drain_loads(uint64_t* full, int issued, int rank, uint32_t* peer_issued,
                                            uint64_t* peer_done, uint32_t half_bytes, int* err) {
  int n = issued;
  if constexpr (PAIR) {
    if (rank != 0) {
      st_shared_cluster(mapa_shared(smem_u32(peer_issued), 0), (uint32_t)issued);
      mbar_arrive_cluster(mapa_shared(smem_u32(peer_done), 0));
      return;
    }
    int np = issued;
    if (mbar_wait_cluster(peer_done, 0))
      np = (int)*peer_issued;
    else
      set_device_error(err, MOE_ERR_TIMEOUT, 8);
    for (int i = issued; i < np; ++i) {  // issued by the peer alone
      if (i >= ST && !mbar_wait(&full[i % ST], ((i - ST) / ST) & 1)) set_device_error(err, MOE_ERR_TIMEOUT, 9);
      mbar_arrive_expect_tx(&full[i % ST], half_bytes);
    }
    for (int i = np; i < issued; ++i) mbar_complete_tx(&full[i % ST], half_bytes);  // issued by the leader alone
    n = np > issued ? np : issued;
  }
  for (int i = n > ST ? n - ST : 0; i < n; ++i)
    if (!mbar_wait(&full[i % ST], (i / ST) & 1)) set_device_error(err, MOE_ERR_TIMEOUT, 2);
}

template <int MODE, int EPI, int BN, int ST, bool FP8, bool PAIR, int NEPI>
__global__ void __launch_bounds__(threads_of<FP8, NEPI>(), 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapD, const GemmArgs g) {
  using G = Geo<FP8>;
  // K per stage: 128 bytes of each K-major row, or (bf16 weight gradients) kWgradRows token
  // rows of the MN-major operands
  constexpr bool WROWS = MODE == MODE_WGRAD && EPI == EPI_STORE && !FP8;
  constexpr int BK = WROWS ? kWgradRows : G::BKE;
  constexpr int kThreads = threads_of<FP8, NEPI>();
  constexpr int ROWB = BK * G::EB;          // bytes per operand row (MN-major: per MN atom row x rows)
  constexpr int A_BYTES = BM * ROWB;
  constexpr int BNL = PAIR ? BN / 2 : BN;  // B rows (N) held by this CTA
  constexpr int B_BYTES = BNL * ROWB;
  constexpr int STAGE = A_BYTES + B_BYTES;
  constexpr int MNB = 128 * BK;            // bytes of one MN-major box: 128-byte rows x BK rows
  constexpr uint32_t TMEM_COLS = FP8 ? 512 : 2 * BN;  // FP8: accumulators + per-stage scale columns
  constexpr uint32_t SFC = 2 * BN;                    // first scale-factor column (FP8): 8 per stage
  constexpr uint32_t IDESC = FP8 ? idesc_mxf8(BM, BN, MODE == MODE_WGRAD, MODE != MODE_FWD)
                                 : idesc_bf16(PAIR ? 2 * BM : BM, BN, MODE == MODE_WGRAD, MODE != MODE_FWD);
  static_assert(!(PAIR && FP8), "CTA pairs are built for the bf16 path only");
  // bf16 weight gradients leave straight from registers (store_chunk_direct); the other
  // stored outputs through the staging buffer and TMA stores
  constexpr bool DIRECT = MODE == MODE_WGRAD && EPI == EPI_STORE;
  constexpr bool TMA_OUT = EPI != EPI_SWIGLU && !DIRECT;
  constexpr int STAGING = DIRECT ? 0 : NEPI * kStagingBytes;
  static_assert(NEPI == 1 || (NEPI == 2 && MODE == MODE_WGRAD && EPI == EPI_STORE && !FP8),
                "two epilogue warpgroups are built for the bf16 weight gradients");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  // per epilogue warpgroup two 8 KB halves, each one [128 rows x 32 bf16] box in the
  // 64-byte swizzle layout
  uint8_t* staging = smem + ST * STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + STAGING);
  uint64_t* empty = full + ST;
  uint64_t* sf_full = empty + ST;  // FP8: this stage's scale factors are in tensor memory
  uint64_t* acc_full = sf_full + ST;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* done_bar = acc_empty + 2;
  uint64_t* peer_done = done_bar + 1;  // CTA pairs: the peer's producer has stopped (leader's copy)
  // [0] tensor-memory base, [1]/[2] epilogue flags of warpgroups 0/1, [3] the peer's issue count
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(peer_done + 1);
  int* s_seg = reinterpret_cast<int*>(tmem_holder + 4);
  int* s_tile = s_seg + 260;
  int* s_cnt = s_tile + 260;
  int* s_ptile = s_cnt + 260;  // CTA pairs: prefix of ceil(M tiles / 2) per expert

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  if (g.dense_rows <= 0) {
    for (int i = threadIdx.x; i <= g.E; i += kThreads) {
      s_seg[i] = g.seg_off[i];
      if (MODE != MODE_WGRAD) s_tile[i] = g.tile_off[i];
      if (MODE == MODE_WGRAD && i < g.E) s_cnt[i] = g.counts[i];
    }
    if (PAIR && MODE != MODE_WGRAD) {
      __syncthreads();
      if (threadIdx.x == 0) {
        s_ptile[0] = 0;
        for (int e = 0; e < g.E; ++e) s_ptile[e + 1] = s_ptile[e] + (s_tile[e + 1] - s_tile[e] + 1) / 2;
      }
    }
  }
  // rows of the A tensor map: a coordinate at or past it reads zeros
  const int64_t oob_row = 1LL << 30;
  auto decode = [&](int t) {
    if constexpr (PAIR)
      return decode_pair_tile<MODE, EPI, BN, BK>(t, g, s_seg, s_tile, s_ptile, s_cnt, rank, oob_row);
    else
      return decode_tile<MODE, EPI, BN, BK>(t, g, s_seg, s_tile, s_cnt);
  };
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], (PAIR ? 8 : 4) * NEPI);  // pairs: both CTAs' epilogue warps release
    }
    mbar_init(done_bar, 1);
    mbar_init(peer_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
    if (TMA_OUT) tma_prefetch_desc(&mapD);
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // one warp of each CTA of the pair allocates together
      tmem_alloc_pair(tmem_holder, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  int total;
  if constexpr (MODE != MODE_WGRAD) {
    if constexpr (PAIR) {
      const int mt = g.dense_rows > 0 ? (g.dense_rows + BM - 1) / BM : 0;
      total = (g.dense_rows > 0 ? (mt + 1) / 2 : s_ptile[g.E]) * g.n_tiles;
    } else {
      const int mt = g.dense_rows > 0 ? (g.dense_rows + BM - 1) / BM : s_tile[g.E];
      total = mt * g.n_tiles;
    }
  } else {
    const int mtl = PAIR ? (g.m_tiles + 1) / 2 : g.m_tiles;
    total = (g.dense_rows > 0 && g.ksplit_rows <= 0 ? 1 : g.E) * mtl * g.n_tiles;
  }
  const int t_first = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int t_step = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;

  if (warp == 0 && PAIR && (MODE == MODE_FWD || MODE == MODE_WGRAD) && g.gather_src) {
    // ------------------------------------------------------------ TMA producer, gathered rows
    // Every lane gathers four of the operand's rows per stage (tile::gather4); lane 0
    // waits for the stage, arms the barrier and loads the other operand.
    auto src_row = [&](int64_t r) -> int {
      if (r < 0 || r >= g.gather_rows) return g.gather_oob;
      const int sr = __ldg(g.gather_src + r);
      return sr >= 0 ? sr / g.gather_k : g.gather_oob;
    };
    constexpr int NH = MODE == MODE_FWD ? 1 : BK / 64;  // WGRAD: 64-row halves of a stage's B rows
    int idx[NH][4];
    auto rows_of = [&](const Tile& tt, int k_b) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int64_t base = MODE == MODE_FWD ? (int64_t)tt.m0 + 4 * lane
                                              : (int64_t)tt.k0 + (int64_t)k_b * BK + 64 * h + 4 * (lane & 15);
#pragma unroll
        for (int i = 0; i < 4; ++i) idx[h][i] = src_row(base + i);
      }
    };
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    bool ok = true;
    int t = t_first;
    Tile tl;
    auto next_work = [&]() {  // the next tile with k-blocks, and its first rows
      while (t < total) {
        tl = decode(t);
        if (tl.kb > 0) break;
        t += t_step;
      }
      if (t < total) rows_of(tl, 0);
    };
    next_work();
    while (t < total && ok) {
      for (int kb = 0; kb < tl.kb; ++kb) {
        const int w_ok =
            __shfl_sync(0xffffffffu, lane == 0 ? (int)mbar_wait(&empty[stage], phase ^ 1, g.wait_ns) : 0, 0);
        if (!w_ok) {
          if (lane == 0) set_device_error(g.err, MOE_ERR_TIMEOUT, 1);
          ok = false;
          break;
        }
        uint8_t* sa = tiles + stage * STAGE;
        uint8_t* sb = sa + A_BYTES;
        uint64_t* bar = &full[stage];
        const int kc = kb * BK;
        if (lane == 0 && rank == 0) mbar_arrive_expect_tx(bar, 2 * STAGE);
        const uint32_t cbar = mapa_shared(smem_u32(bar), 0);
        if constexpr (MODE == MODE_FWD) {
          tma_gather4_pair(sa + lane * 512, &mapA, cbar, kc, idx[0][0], idx[0][1], idx[0][2], idx[0][3]);
          if (lane == 0) {
            const int brow = EPI == EPI_SWIGLU ? (rank ? g.F + tl.n0 : tl.n0) : tl.n0 + rank * BNL;
            tma_load_3d_pair(sb, &mapB, cbar, kc, brow, tl.e);
          }
        } else {
          if (lane == 0) {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              tma_load_2d_pair(sa + j * MNB, &mapA, cbar, tl.m0 + 64 * j, tl.k0 + kc);
          }
          // B: two 64-column MN-major boxes of BK rows; each lane gathers four rows of every
          // 64-row half of its box
          const int j = lane >> 4, q = lane & 15;
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tma_gather4_pair(sb + j * MNB + (64 * h + 4 * q) * 128, &mapB, cbar, tl.n0 + rank * BNL + 64 * j,
                             idx[h][0], idx[h][1], idx[h][2], idx[h][3]);
        }
        ++issued;
        if (++stage == ST) {
          stage = 0;
          phase ^= 1;
        }
        if (MODE == MODE_WGRAD && kb + 1 < tl.kb) rows_of(tl, kb + 1);
      }
      if (!ok) break;
      t += t_step;
      next_work();
    }
    if (lane == 0) drain_loads<ST, PAIR>(full, issued, rank, tmem_holder + 3, peer_done, STAGE, g.err);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = t_first; t < total && ok; t += t_step) {
        const Tile tl = decode(t);
        for (int kb = 0; kb < tl.kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, g.wait_ns)) {
            set_device_error(g.err, MOE_ERR_TIMEOUT, 1);
            ok = false;
            break;
          }
          uint8_t* sa = tiles + stage * STAGE;
          uint8_t* sb = sa + A_BYTES;
          uint64_t* bar = &full[stage];
          const int kc = kb * BK;
          if constexpr (PAIR) {
            // both CTAs' copies land on the leader's barrier, which expects both
            if (rank == 0) mbar_arrive_expect_tx(bar, 2 * STAGE);
            const uint32_t cbar = mapa_shared(smem_u32(bar), 0);
            if constexpr (MODE == MODE_WGRAD) {
#pragma unroll
              for (int j = 0; j < BM / 64; ++j) tma_load_2d_pair(sa + j * MNB, &mapA, cbar, tl.m0 + 64 * j, tl.k0 + kc);
#pragma unroll
              for (int j = 0; j < BNL / 64; ++j)
                tma_load_2d_pair(sb + j * MNB, &mapB, cbar, tl.n0 + rank * BNL + 64 * j, tl.k0 + kc);
            } else {
              tma_load_2d_pair(sa, &mapA, cbar, kc, tl.m0);
              if constexpr (MODE == MODE_FWD) {
                const int brow = EPI == EPI_SWIGLU ? (rank ? g.F + tl.n0 : tl.n0) : tl.n0 + rank * BNL;
                tma_load_3d_pair(sb, &mapB, cbar, kc, brow, tl.e);
              } else {
#pragma unroll
                for (int j = 0; j < BNL / 64; ++j)
                  tma_load_3d_pair(sb + j * MNB, &mapB, cbar, tl.n0 + rank * BNL + 64 * j, kc, tl.e);
              }
            }
          } else {
          mbar_arrive_expect_tx(bar, STAGE);
          if constexpr (MODE == MODE_WGRAD) {
#pragma unroll
            for (int j = 0; j < BM / G::MN_INNER; ++j)
              tma_load_2d(sa + j * MNB, &mapA, bar, tl.m0 + G::MN_INNER * j, tl.k0 + kc);
            const int kb_row = g.kwrap > 0 ? (tl.k0 + kc) % g.kwrap : tl.k0 + kc;
#pragma unroll
            for (int j = 0; j < BN / G::MN_INNER; ++j)
              tma_load_2d(sb + j * MNB, &mapB, bar, tl.n0 + G::MN_INNER * j, kb_row);
          } else {
            tma_load_2d(sa, &mapA, bar, g.kwrap > 0 ? kc % g.kwrap : kc, tl.m0);
            if constexpr (MODE == MODE_FWD) {
              if constexpr (EPI == EPI_SWIGLU) {
                tma_load_3d(sb, &mapB, bar, kc, tl.n0, tl.e);
                tma_load_3d(sb + B_BYTES / 2, &mapB, bar, kc, g.F + tl.n0, tl.e);
              } else {
                tma_load_3d(sb, &mapB, bar, kc, tl.n0, tl.e);
              }
            } else {
#pragma unroll
              for (int j = 0; j < BN / G::MN_INNER; ++j)
                tma_load_3d(sb + j * MNB, &mapB, bar, tl.n0 + G::MN_INNER * j, kc, tl.e);
            }
          }
          }
          ++issued;
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // nothing may still be landing in shared memory when the CTA exits
      drain_loads<ST, PAIR>(full, issued, rank, tmem_holder + 3, peer_done, STAGE, g.err);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the leader CTA of a pair)
    if (lane == 0 && (!PAIR || rank == 0)) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = t_first; t < total && ok; t += t_step) {
        const Tile tl = decode(t);
        if (tl.kb == 0) continue;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, g.wait_ns)) {
          set_device_error(g.err, MOE_ERR_TIMEOUT, 3);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < tl.kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, g.wait_ns) || (FP8 && !mbar_wait(&sf_full[stage], phase, g.wait_ns))) {
            set_device_error(g.err, MOE_ERR_TIMEOUT, 4);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + stage * STAGE);
          const uint32_t sb = sa + A_BYTES;
          // K-major operands step 32 bytes per instruction inside the 128-byte swizzle row;
          // MN-major operands step KSTEP rows of 128 bytes, with MN atoms MNB bytes apart
          constexpr uint32_t MN_STEP = G::KSTEP * 128;
          // weight gradients: the last block's K steps past the expert's rows are skipped
          const int nkk = MODE == MODE_WGRAD && kb + 1 == tl.kb ? (tl.krem + G::KSTEP - 1) / G::KSTEP : BK / G::KSTEP;
#pragma unroll
          for (int kk = 0; kk < BK / G::KSTEP; ++kk) {
            if (kk >= nkk) break;
            const uint64_t ad = MODE == MODE_WGRAD ? smem_desc_sw128(sa + kk * MN_STEP, MNB, 1024)
                                                   : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = MODE == MODE_FWD ? smem_desc_sw128(sb + kk * 32, 16, 1024)
                                                 : smem_desc_sw128(sb + kk * MN_STEP, MNB, 1024);
            if constexpr (PAIR)
              umma_f16_pair(d, ad, bd, IDESC, (kb | kk) != 0);
            else if constexpr (FP8)
              umma_mxf8(d, ad, bd, IDESC, tmem + SFC + 8 * stage, tmem + SFC + 8 * stage + 4, (kb | kk) != 0);
            else
              umma_f16(d, ad, bd, IDESC, (kb | kk) != 0);
          }
          if constexpr (PAIR)
            umma_commit_pair(&empty[stage]);
          else
            umma_commit(&empty[stage]);
          if (++stage == ST) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(&acc_full[acc]);
        else
          umma_commit(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // every issued MMA has finished before tensor memory is released
      if constexpr (PAIR)
        umma_commit_pair(done_bar);
      else
        umma_commit(done_bar);
      if (!mbar_wait(done_bar, 0)) set_device_error(g.err, MOE_ERR_TIMEOUT, 5);
    }
  } else if (warp < 2 + 4 * NEPI) {
    // ------------------------------------------------------------ epilogue
    // NEPI = 2: warps 2-5 drain the even 32-column chunks of an accumulator and warps
    // 6-9 the odd ones, each group with its own staging buffer, barrier and leader.
    const int grp = NEPI == 2 && warp >= 6 ? 1 : 0;
    uint8_t* const stg = staging + grp * kStagingBytes;
    const int ebar = kEpiBarrier + grp;
    const int q = warp & 3;
    const int r = q * 32 + lane;  // row within the tile = tensor-memory lane
    const bool leader = warp == 2 + 4 * grp && lane == 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    int half = 0;  // staging half used by the next box
    // Writes this thread's 32 values into staging half h (64-byte swizzle: 16-byte
    // unit j of row r sits at unit j ^ ((r >> 1) & 3)).
    auto stage_row = [&](int h, const float* v) {
      uint8_t* base = stg + h * 8192 + r * 64;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(base + ((j ^ ((r >> 1) & 3)) << 4)) = pack8(v + 8 * j);
    };
    // fp32 variant: one [128 rows x 32 fp32] box filling the whole staging buffer in
    // the 128-byte swizzle layout (16-byte unit j of row r sits at unit j ^ (r & 7)).
    auto stage_row_f32 = [&](const float* v) {
      uint8_t* base = stg + r * 128;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(base + ((j ^ (r & 7)) << 4)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    };
    // Hands staged boxes to TMA: all threads fence + barrier, the leader stores
    // (nothing is stored for the missing half of a CTA pair's tile).
    auto publish = [&](int nbox, const int* hx, const int* xs, int y, int z, bool store) {
      fence_proxy_async_smem();
      named_bar_sync(ebar, 128);
      if (leader && store) {
        for (int b = 0; b < nbox; ++b) tma_store_3d(&mapD, stg + hx[b] * 8192, xs[b], y, z);
        bulk_commit_group();
      }
    };
    // Before overwriting a staging half: its previous store must have read it.
    auto reserve = [&](bool both) {
      if (leader) {
        if (both)
          bulk_wait_group_read<0>();
        else
          bulk_wait_group_read<1>();
      }
      named_bar_sync(ebar, 128);
    };
    // The accumulator goes back to the MMA issuer: the leader CTA's barrier, which
    // in a pair also counts the peer's epilogue warps.
    auto release = [&](int b) {
      if constexpr (PAIR) {
        if (rank == 0)
          mbar_arrive_relaxed(&acc_empty[b]);
        else
          mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&acc_empty[b]), 0));
      } else {
        mbar_arrive_relaxed(&acc_empty[b]);
      }
    };
    for (int t = t_first; t < total; t += t_step) {
      const Tile tl = decode(t);
      if constexpr (DIRECT) {
        // each warp: its 32 rows of the tile; group grp: the chunks grp, grp + NEPI, ...
        uint16_t* const dwarp = g.D + (int64_t)tl.e * g.d_estride + (int64_t)(tl.m0 + q * 32) * g.ldd + tl.n0;
        if (tl.kb == 0) {
          // an expert without rows: its weight gradient is zero, written as whole rows
          // (this group's BN/NEPI columns of a row by LPR lanes, 16 bytes each)
          if (tl.valid) {
            constexpr int LPR = BN * 2 / NEPI / 16, RPI = 32 / LPR;
            uint16_t* const z0 = dwarp + grp * (BN / NEPI) + 8 * (lane % LPR);
#pragma unroll 4
            for (int r0 = 0; r0 < 32; r0 += RPI)
              *reinterpret_cast<uint4*>(z0 + (int64_t)(r0 + lane / LPR) * g.ldd) = make_uint4(0, 0, 0, 0);
          }
          continue;
        }
        const uint32_t w_ok = lane == 0 ? (mbar_wait(&acc_full[acc], acc_phase, g.wait_ns) ? 1u : 0u) : 0u;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
          if (lane == 0) set_device_error(g.err, MOE_ERR_TIMEOUT, 6);
          break;
        }
        mbar_wait(&acc_full[acc], acc_phase);  // already complete: acquires the accumulator for this thread
        tc_fence_after();
        // the accumulator goes back as soon as this warp's last tensor-memory load has completed
        auto release_now = [&]() {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release(acc);
        };
        if (tl.valid) {
          // two register buffers: the next chunk's tensor-memory load is in flight while
          // the current one is converted and stored
          constexpr int NC = BN / 32 / NEPI;
          const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN + 32 * grp;
          uint32_t ra[32], rb[32];
          tmem_ld32(tb, ra);
#pragma unroll
          for (int i = 0; i < NC; i += 2) {
            tmem_ld_wait();
            if (i + 1 < NC)
              tmem_ld32(tb + 32 * NEPI * (i + 1), rb);
            else
              release_now();
            store_chunk_direct(dwarp + 32 * (grp + NEPI * i), g.ldd, lane, ra);
            if (i + 1 < NC) {
              tmem_ld_wait();
              if (i + 2 < NC)
                tmem_ld32(tb + 32 * NEPI * (i + 2), ra);
              else
                release_now();
              store_chunk_direct(dwarp + 32 * (grp + NEPI * (i + 1)), g.ldd, lane, rb);
            }
          }
        } else {
          release_now();  // the missing half of a pair tile: nothing to read
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        continue;
      }
      const int64_t row = tl.m0 + r;
      if constexpr (EPI == EPI_DSWIGLU) {
        // pull this row's saved pre-activations into L2 while the accumulator fills
        if (tl.valid && (g.dense_rows <= 0 || row < g.dense_rows)) {
          const uint16_t* gp = g.GU + row * g.ldgu + tl.n0;
#pragma unroll
          for (int i = 0; i < BN * 2; i += 128) {
            prefetch_l2(reinterpret_cast<const uint8_t*>(gp) + i);
            prefetch_l2(reinterpret_cast<const uint8_t*>(gp + g.F) + i);
          }
        }
      }
      if (tl.kb == 0) {
        // an expert without rows: its weight gradient is zero
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
        for (int c = grp; c < BN / 32; c += NEPI) {
          if constexpr (EPI == EPI_F32) {
            reserve(true);
            stage_row_f32(z);
            const int hx[1] = {0}, xs[1] = {tl.n0 + 32 * c};
            publish(1, hx, xs, tl.m0, tl.e, tl.valid);
          } else {
            reserve(false);
            stage_row(half, z);
            const int hx[1] = {half}, xs[1] = {tl.n0 + 32 * c};
            publish(1, hx, xs, tl.m0, tl.e, tl.valid);
            half ^= 1;
          }
        }
        continue;
      }
      // one thread waits (bounded) and shares the outcome, so that all four warps
      // take the same path through the named barriers below
      if (leader) tmem_holder[1 + grp] = mbar_wait(&acc_full[acc], acc_phase, g.wait_ns) ? 1u : 0u;
      named_bar_sync(ebar, 128);
      const bool acc_ready = tmem_holder[1 + grp] != 0u;
      named_bar_sync(ebar, 128);  // everyone has read the flag before it is reused
      if (!acc_ready) {
        if (leader) set_device_error(g.err, MOE_ERR_TIMEOUT, 6);
        break;
      }
      mbar_wait(&acc_full[acc], acc_phase);  // already complete: acquires the accumulator for this thread
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      const bool valid = tl.valid && (g.dense_rows <= 0 || MODE == MODE_WGRAD || row < g.dense_rows);
      float rg = 1.0f;  // the row's gate on the gated path
      if (EPI != EPI_STORE && EPI != EPI_F32 && g.gates && valid) {
        const int sr = g.slot_src[row];
        rg = sr >= 0 ? g.gates[sr] : 0.0f;
      }
      if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t gr[32], ur[32];
          tmem_ld32(tbase + c * 32, gr);
          tmem_ld32(tbase + BN / 2 + c * 32, ur);
          tmem_ld_wait();
          if (valid) {
            float gv[32], uv[32], av[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              gv[i] = __uint_as_float(gr[i]);
              uv[i] = __uint_as_float(ur[i]);
              // silu(g) * u with the fast reciprocal (outputs are bf16; exp(-g) = inf gives 0)
              av[i] = rg * (__fdividef(gv[i], 1.0f + __expf(-gv[i])) * uv[i]);
            }
            const int col = tl.n0 + c * 32;
            store32(g.D + row * g.ldd + col, gv);
            store32(g.D + row * g.ldd + g.F + col, uv);
            store32(g.D2 + row * g.ldd2 + col, av);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release(acc);
      } else if constexpr (EPI == EPI_DSWIGLU) {
        const bool gated = g.gates != nullptr;
        float dot = 0.0f;  // gated: <accumulator row, silu(g) * u> over this tile's columns
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t dr[32];
          tmem_ld32(tbase + c * 32, dr);
          tmem_ld_wait();
          if (c == BN / 32 - 1) {  // the accumulator is no longer needed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(acc);
          }
          const int col = tl.n0 + c * 32;
          float dg[32], du[32];
          if (valid) {
            const uint4* gp = reinterpret_cast<const uint4*>(g.GU + row * g.ldgu + col);
            const uint4* up = reinterpret_cast<const uint4*>(g.GU + row * g.ldgu + g.F + col);
            float ag[32];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float gf[8], uf[8];
              unpack8(gp[v], gf);
              unpack8(up[v], uf);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float acc_v = __uint_as_float(dr[8 * v + i]);
                const float s = __fdividef(1.0f, 1.0f + __expf(-gf[i]));  // sigmoid, fast reciprocal
                const float sl = gf[i] * s;
                const float a = sl * uf[i];
                dot = fmaf(acc_v, a, dot);
                ag[8 * v + i] = rg * a;
                const float da = rg * acc_v;
                dg[8 * v + i] = da * uf[i] * (s * (1.0f + gf[i] * (1.0f - s)));
                du[8 * v + i] = da * sl;
              }
            }
            if (gated) store32(g.a_out + row * g.lda_out + col, ag);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) dg[i] = du[i] = 0.f;
          }
          reserve(true);
          stage_row(0, dg);
          stage_row(1, du);
          const int hx[2] = {0, 1}, xs[2] = {col, g.F + col};
          publish(2, hx, xs, tl.m0, 0, tl.valid);
        }
        if (gated && valid) g.dg_part[row * g.n_tiles + tl.n0 / BN] = dot;
      } else {
        int nch = BN / 32;
        if (g.n_valid > 0) {
          const int left = (g.n_valid - tl.n0 + 31) / 32;
          nch = left < nch ? (left > 1 ? left : 1) : nch;
        }
        if (grp >= nch) {  // no chunk for this group: hand the accumulator back at once
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release(acc);
        }
        for (int c = grp; c < nch; c += NEPI) {
          uint32_t vr[32];
          tmem_ld32(tbase + c * 32, vr);
          tmem_ld_wait();
          if (c + NEPI >= nch) {  // this group's last read of the accumulator
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(acc);
          }
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(vr[i]);
          const int hx[1] = {EPI == EPI_F32 ? 0 : half}, xs[1] = {tl.n0 + 32 * c};
          if constexpr (EPI == EPI_F32) {
            reserve(true);
            stage_row_f32(v);
          } else {
            reserve(false);
            stage_row(half, v);
            half ^= 1;
          }
          publish(1, hx, xs, tl.m0, MODE == MODE_WGRAD ? tl.e : 0, tl.valid);
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    // every store has finished before the CTA (and its shared memory) goes away
    if (TMA_OUT && leader) bulk_wait_group<0>();
  } else if constexpr (FP8) {
    // ------------------------------------------------------------ scale-factor warps (FP8)
    // The block-scaled MMA reads the scales of a 128-row operand as 32 lanes x 4 columns:
    // row m at lane m % 32, column m / 32, one byte per 32-wide K step (the byte chosen
    // by the scale-factor id).  Every lane quarter holds the same copy, so each of the four
    // warps writes it into its own 32 lanes.  Our blocks span 128 of K, so all four bytes
    // of a word carry the same UE8M0 scale.  A uses columns SFC+8s..+3, B SFC+8s+4..+7.
    const int q = warp & 3;
    int stage = 0;
    uint32_t phase = 0;
    auto wait_free = [&]() {  // the stage's previous MMAs have finished with its scale columns
      const bool w_ok =
          __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(&empty[stage], phase ^ 1, g.wait_ns) : false, 0);
      if (!w_ok && lane == 0) set_device_error(g.err, MOE_ERR_TIMEOUT, 7);
      return w_ok;
    };
    constexpr uint32_t R4 = 0x01010101u;  // a scale byte in all four bytes of its word
    // writes the words into this warp's lanes of the stage's scale columns
    auto put = [&](const uint32_t* wa, const uint32_t* wb) {
      const uint32_t sf_addr = tmem + ((uint32_t)(q * 32) << 16) + SFC + 8 * stage;
      tmem_st4(sf_addr, wa[0], wa[1], wa[2], wa[3]);
      tmem_st4(sf_addr + 4, wb[0], wb[1], wb[2], wb[3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_full[stage]);
      if (++stage == ST) {
        stage = 0;
        phase ^= 1;
      }
    };
    if constexpr (MODE == MODE_FWD) {
      // The forward GEMMs load each k-block's words once its stage is free: loading them
      // ahead, as the other modes do, measured slower there.
      bool ok = true;
      for (int t = t_first; t < total && ok; t += t_step) {
        const Tile tl = decode(t);
        for (int kb = 0; kb < tl.kb; ++kb) {
          if (!wait_free()) {
            ok = false;
            break;
          }
          uint32_t wa[4], wb[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = lane + 32 * j;  // tile row of this word
            const int64_t row = tl.m0 + r;
            // weights [E][N rows][K]: block (n/128, kb)
            const int nrow = EPI == EPI_SWIGLU ? (r < BN / 2 ? tl.n0 + r : g.F + tl.n0 + r - BN / 2) : tl.n0 + r;
            uint32_t a = 127;
            if (g.dense_rows <= 0 || row < g.dense_rows) a = g.sfa[row * g.sfa_ld + kb];
            wa[j] = a * R4;
            wb[j] = g.sfb[((int64_t)tl.e * g.sfb_r + nrow / 128) * g.sfb_c + kb] * R4;
          }
          put(wa, wb);
        }
      }
    } else {
      // The dgrads and weight gradients load the words of the next kSfAhead k-blocks into
      // registers before their stages come free, so the loads' latency overlaps the waits
      // instead of adding to every k-block (the weight gradients have one to a few k-blocks
      // per tile).
      // the bytes only: nothing here waits for the loads
      auto load_words = [&](const Tile& tl, int kb, uint32_t* wa, uint32_t* wb) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane + 32 * j;  // tile row of this word
          if constexpr (MODE == MODE_WGRAD) {
            const int64_t blk = tl.k0 / 128 + kb;  // 128-row block of the token dimension
            wa[j] = g.sfa[blk * g.sfa_ld + tl.m0 + r];
            wb[j] = g.sfb[blk * g.sfb_ld + tl.n0 + r];
          } else {  // weights [E][K rows][N]: block (kb, n/128)
            const int64_t row = tl.m0 + r;
            wa[j] = g.dense_rows <= 0 || row < g.dense_rows ? g.sfa[row * g.sfa_ld + kb] : 127;
            wb[j] = g.sfb[((int64_t)tl.e * g.sfb_r + kb) * g.sfb_c + (tl.n0 + r) / 128];
          }
        }
      };
      // the k-blocks in the order the producer and the MMA issuer walk them
      int t = t_first, kb = 0;
      Tile tl{};
      auto seek = [&]() {  // from tile t on, the first tile with a k-block
        for (; t < total; t += t_step) {
          tl = decode(t);
          if (tl.kb > 0) return true;
        }
        return false;
      };
      bool more = seek();
      auto fetch = [&](uint32_t* wa, uint32_t* wb) {  // loads the next k-block's words
        load_words(tl, kb, wa, wb);
        if (++kb == tl.kb) {
          kb = 0;
          t += t_step;
          more = seek();
        }
      };
      uint32_t wa[kSfAhead][4], wb[kSfAhead][4];
      bool have[kSfAhead];
#pragma unroll
      for (int d = 0; d < kSfAhead; ++d) {
        have[d] = more;
        if (more) fetch(wa[d], wb[d]);
      }
      for (bool go = true; go;) {
#pragma unroll
        for (int d = 0; d < kSfAhead; ++d) {  // slot d holds the k-blocks d, d + kSfAhead, ...
          if (!have[d] || !wait_free()) {
            go = false;
            break;
          }
          uint32_t ra[4], rb[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ra[j] = wa[d][j] * R4;
            rb[j] = wb[d][j] * R4;
          }
          put(ra, rb);
          have[d] = more;
          if (more) fetch(wa[d], wb[d]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int MODE, int EPI, int BN, bool FP8, bool PAIR = false, int NEPI = 1>
struct Kern {
  static constexpr int BNL = PAIR ? BN / 2 : BN;
  static constexpr bool WROWS = MODE == MODE_WGRAD && EPI == EPI_STORE && !FP8;
  static constexpr int STAGE = (BM + BNL) * (WROWS ? kWgradRows * 2 : 128);
  // bf16 weight gradients store from registers and need no staging buffer
  static constexpr bool DIRECT = MODE == MODE_WGRAD && EPI == EPI_STORE;
  static constexpr int STAGING = DIRECT ? 0 : NEPI * kStagingBytes;
  // a second epilogue warpgroup's staging buffer takes the room of one operand stage
  static constexpr int ST = STAGE > 49152 ? 3 : (STAGE > 32768 ? 4 : (NEPI == 2 && !DIRECT ? 5 : 6));
  static constexpr size_t smem = 1024 + (size_t)ST * STAGE + STAGING + (3 * ST + 6) * 8 + 16 + 4 * 260 * 4;
};

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 tensor map.  dims/strides innermost first (strides in elements).
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_elems,
              uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t esz = dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : dt == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bd[3] = {box0, box1, 1}, es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) gd[i] = dims[i];
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_elems[i] * esz;
  CUresult r = fn(m, dt, rank, const_cast<void*>(base), gd, gs, bd, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// operand maps: 128-byte swizzle, the layout the MMA descriptors expect
bool map2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t b0, uint32_t b1) {
  const uint64_t dims[2] = {inner, outer}, st[1] = {inner};
  return make_map(m, base, 2, dims, st, b0, b1, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer, uint32_t b0,
           uint32_t b1) {
  const uint64_t dims[3] = {inner, mid, outer}, st[2] = {inner, inner * mid};
  return make_map(m, base, 3, dims, st, b0, b1, CU_TENSOR_MAP_SWIZZLE_128B);
}
// output map: [outer][mid][inner] bf16, boxes of 32 columns x 128 rows, 64-byte swizzle
// (the staging layout the epilogue writes)
bool map_out(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer) {
  const uint64_t dims[3] = {inner, mid, outer}, st[2] = {inner, inner * mid};
  return make_map(m, base, 3, dims, st, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B);
}

// FP8 operand maps (bytes), 128-byte swizzle
bool map2d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t b0, uint32_t b1) {
  const uint64_t dims[2] = {inner, outer}, st[1] = {inner};
  return make_map(m, base, 2, dims, st, b0, b1, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}
bool map3d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer, uint32_t b0,
              uint32_t b1) {
  const uint64_t dims[3] = {inner, mid, outer}, st[2] = {inner, inner * mid};
  return make_map(m, base, 3, dims, st, b0, b1, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// fp32 output map: boxes of 32 columns x 128 rows, 128-byte swizzle
bool map_out_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer) {
  const uint64_t dims[3] = {inner, mid, outer}, st[2] = {inner, inner * mid};
  return make_map(m, base, 3, dims, st, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

template <int MODE, int EPI, int BN, bool FP8 = false, bool PAIR = false, int NEPI = 1>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& d, const GemmArgs& g, int max_tiles,
                   int nsm, cudaStream_t st) {
  using K = Kern<MODE, EPI, BN, FP8, PAIR, NEPI>;
  static std::atomic<uint64_t> attr{0};
  auto kern = k_grouped_gemm<MODE, EPI, BN, K::ST, FP8, PAIR, NEPI>;
  if (cudaError_t e = raise_smem_limit(attr, kern, K::smem); e != cudaSuccess) return e;
  if (max_tiles <= 0) return cudaSuccess;
  GemmArgs ga = g;
  ga.wait_ns = pipeline_wait_ns();
  if constexpr (PAIR) {
    // max_tiles counts 256-row pair tiles here; two CTAs (one cluster) per pair tile
    const int pairs = max_tiles < nsm / 2 ? max_tiles : nsm / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(threads_of<FP8, NEPI>());
    cfg.dynamicSmemBytes = K::smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, b, d, ga);
  } else {
    const int grid = max_tiles < nsm ? max_tiles : nsm;
    kern<<<grid, threads_of<FP8, NEPI>(), K::smem, st>>>(a, b, d, ga);
    return cudaGetLastError();
  }
}

inline int pick_bn(int n) { return n % 256 == 0 ? 256 : 128; }

// 256-wide bf16 tiles run on CTA pairs (cta_group::2): each CTA stages only half of
// B, halving its shared-memory operand traffic per MMA.
constexpr bool use_pairs() { return true; }

// Weight-gradient tile order.  Both operands of an expert's wgrad are its token rows:
// A spans the M columns, B the N columns.  Walking the smaller dimension fastest keeps
// that operand (all of its slices) resident in L2 while one slice of the larger
// operand is shared by the concurrent tiles, so each byte of the larger one is read
// from DRAM once.
inline int wgrad_n_fast(int m, int n) { return m > n ? 1 : 0; }

// Weight gradients whose experts hold few rows (K of a few 64-row blocks per tile) are
// bound by their epilogue, which writes a 256x256 tile per handful of MMAs: they run
// with a second epilogue warpgroup (and one operand stage fewer).  Long-K ones keep six
// operand stages.
inline bool wgrad_two_epilogues(const GemmShape& s) {
  return s.dense_rows <= 0 && s.E > 0 && s.rows / s.E < 512;
}

// pair tiles of a ragged launch: sum over experts of ceil(m tiles / 2) <= max_mtiles / 2 + E
inline int pair_tiles(const GemmShape& s, int n_tiles) {
  const int mt = s.dense_rows > 0 ? (s.dense_rows + 127) / 128 : s.max_mtiles;
  return (s.dense_rows > 0 ? (mt + 1) / 2 : mt / 2 + s.E) * n_tiles;
}

}  // namespace

int fc2_dgrad_tile_n(int F) { return pick_bn(F); }

// X1 = rows of A [rows, K] (Xperm or X), W13 [E, 2F, K]: GU [rows, 2F], A [rows, F].
cudaError_t launch_fc1_fwd(const GemmShape& s, const uint16_t* X1, const uint16_t* W13, uint16_t* GU, uint16_t* Aact,
                           int* err, cudaStream_t st, const Gating* gate, const RowGather* gather) {
  CUtensorMap ma, mb;
  // gathered rows: X1 is the token matrix [gather->src_rows, H], read a row at a time
  const bool ok_a = gather ? map2d(&ma, X1, s.H, gather->src_rows, 64, 1) : map2d(&ma, X1, s.H, s.rows, 64, 128);
  if (!ok_a || !map3d(&mb, W13, s.H, 2 * (uint64_t)s.F, s.E, 64, 128)) return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = s.H; g.n_tiles = s.F / 128; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = GU; g.ldd = 2 * (int64_t)s.F; g.D2 = Aact; g.ldd2 = s.F; g.F = s.F; g.err = err;
  if (gate) {
    g.slot_src = gate->slot_src;
    g.gates = gate->gates;
  }
  if (gather) {
    g.gather_src = gather->slot_src;
    g.gather_k = gather->k;
    g.gather_oob = (int)gather->src_rows;
    g.gather_rows = s.rows;
    return launch<MODE_FWD, EPI_SWIGLU, 256, false, true>(ma, mb, ma, g, pair_tiles(s, g.n_tiles), s.nsm, st);
  }
  if (use_pairs()) return launch<MODE_FWD, EPI_SWIGLU, 256, false, true>(ma, mb, ma, g, pair_tiles(s, g.n_tiles), s.nsm, st);
  return launch<MODE_FWD, EPI_SWIGLU, 256>(ma, mb, ma, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

// A [rows, F], W2 [E, H, F]: Y [rows, H].
cudaError_t launch_fc2_fwd(const GemmShape& s, const uint16_t* Aact, const uint16_t* W2, uint16_t* Y, int* err,
                           cudaStream_t st) {
  const int bn = pick_bn(s.H);
  const bool pairs = bn == 256 && use_pairs();
  CUtensorMap ma, mb, md;
  if (!map2d(&ma, Aact, s.F, s.rows, 64, 128) || !map3d(&mb, W2, s.F, s.H, s.E, 64, pairs ? bn / 2 : bn) ||
      !map_out(&md, Y, s.H, s.rows, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = s.F; g.n_tiles = s.H / bn; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = Y; g.ldd = s.H; g.err = err;
  if (pairs) return launch<MODE_FWD, EPI_STORE, 256, false, true>(ma, mb, md, g, pair_tiles(s, g.n_tiles), s.nsm, st);
  return bn == 256 ? launch<MODE_FWD, EPI_STORE, 256>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st)
                   : launch<MODE_FWD, EPI_STORE, 128>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

// dY [rows, H], W2 [E, H, F], GU [rows, 2F]: dGU [rows, 2F].
cudaError_t launch_fc2_dgrad(const GemmShape& s, const uint16_t* dYp, const uint16_t* W2, const uint16_t* GU,
                             uint16_t* dGU, int* err, cudaStream_t st, const Gating* gate) {
  const int bn = pick_bn(s.F);
  CUtensorMap ma, mb, md;
  if (!map2d(&ma, dYp, s.H, s.rows, 64, 128) || !map3d(&mb, W2, s.F, s.H, s.E, 64, 64) ||
      !map_out(&md, dGU, 2 * (uint64_t)s.F, s.rows, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = s.H; g.n_tiles = s.F / bn; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dGU; g.ldd = 2 * (int64_t)s.F; g.GU = GU; g.ldgu = 2 * (int64_t)s.F; g.F = s.F; g.err = err;
  if (gate) {
    g.slot_src = gate->slot_src;
    g.gates = gate->gates;
    g.dg_part = gate->dg_part;
    g.a_out = gate->a_out;
    g.lda_out = s.F;
  }
  if (bn == 256 && use_pairs())
    return launch<MODE_DGRAD, EPI_DSWIGLU, 256, false, true>(ma, mb, md, g, pair_tiles(s, g.n_tiles), s.nsm, st);
  return bn == 256 ? launch<MODE_DGRAD, EPI_DSWIGLU, 256>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st)
                   : launch<MODE_DGRAD, EPI_DSWIGLU, 128>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

// dGU [rows, 2F], W13 [E, 2F, H]: dX [rows, H].
cudaError_t launch_fc1_dgrad(const GemmShape& s, const uint16_t* dGU, const uint16_t* W13, uint16_t* dX1, int* err,
                             cudaStream_t st) {
  const int bn = pick_bn(s.H);
  CUtensorMap ma, mb, md;
  if (!map2d(&ma, dGU, 2 * (uint64_t)s.F, s.rows, 64, 128) || !map3d(&mb, W13, s.H, 2 * (uint64_t)s.F, s.E, 64, 64) ||
      !map_out(&md, dX1, s.H, s.rows, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = 2 * s.F; g.n_tiles = s.H / bn; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dX1; g.ldd = s.H; g.err = err;
  if (bn == 256 && use_pairs())
    return launch<MODE_DGRAD, EPI_STORE, 256, false, true>(ma, mb, md, g, pair_tiles(s, g.n_tiles), s.nsm, st);
  return bn == 256 ? launch<MODE_DGRAD, EPI_STORE, 256>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st)
                   : launch<MODE_DGRAD, EPI_STORE, 128>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

// dW2 [E, H, F] = dY^T A per expert.
cudaError_t launch_fc2_wgrad(const GemmShape& s, const uint16_t* dYp, const uint16_t* Aact, uint16_t* dW2, int* err,
                             cudaStream_t st) {
  const int bn = pick_bn(s.F);
  CUtensorMap ma, mb, md;
  if (!map2d(&ma, dYp, s.H, s.rows, 64, kWgradRows) || !map2d(&mb, Aact, s.F, s.rows, 64, kWgradRows) ||
      !map_out(&md, dW2, s.F, s.H, s.dense_rows > 0 ? 1 : s.E))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.m_tiles = s.H / 128; g.n_tiles = s.F / bn; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dW2; g.ldd = s.F; g.d_estride = (int64_t)s.H * s.F; g.err = err;
  g.n_fast = wgrad_n_fast(s.H, s.F);
  const int tiles = (s.dense_rows > 0 ? 1 : s.E) * g.m_tiles * g.n_tiles;
  if (bn == 256 && use_pairs()) {
    const int pair_tiles = (s.dense_rows > 0 ? 1 : s.E) * ((g.m_tiles + 1) / 2) * g.n_tiles;
    if (wgrad_two_epilogues(s))
      return launch<MODE_WGRAD, EPI_STORE, 256, false, true, 2>(ma, mb, md, g, pair_tiles, s.nsm, st);
    return launch<MODE_WGRAD, EPI_STORE, 256, false, true>(ma, mb, md, g, pair_tiles, s.nsm, st);
  }
  return bn == 256 ? launch<MODE_WGRAD, EPI_STORE, 256>(ma, mb, md, g, tiles, s.nsm, st)
                   : launch<MODE_WGRAD, EPI_STORE, 128>(ma, mb, md, g, tiles, s.nsm, st);
}

// dW13 [E, 2F, H] = dGU^T X per expert.
cudaError_t launch_fc1_wgrad(const GemmShape& s, const uint16_t* dGU, const uint16_t* X1, uint16_t* dW13, int* err,
                             cudaStream_t st, const RowGather* gather) {
  const int bn = pick_bn(s.H);
  if (gather && bn != 256) return cudaErrorInvalidValue;  // gathered rows need the CTA-pair kernel
  CUtensorMap ma, mb, md;
  const bool ok_b =
      gather ? map2d(&mb, X1, s.H, gather->src_rows, 64, 1) : map2d(&mb, X1, s.H, s.rows, 64, kWgradRows);
  if (!map2d(&ma, dGU, 2 * (uint64_t)s.F, s.rows, 64, kWgradRows) || !ok_b ||
      !map_out(&md, dW13, s.H, 2 * (uint64_t)s.F, s.dense_rows > 0 ? 1 : s.E))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.m_tiles = 2 * s.F / 128; g.n_tiles = s.H / bn; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dW13; g.ldd = s.H; g.d_estride = 2 * (int64_t)s.F * s.H; g.err = err;
  g.n_fast = wgrad_n_fast(2 * s.F, s.H);
  if (gather) {
    g.gather_src = gather->slot_src;
    g.gather_k = gather->k;
    g.gather_oob = (int)gather->src_rows;
    g.gather_rows = s.rows;
  }
  const int tiles = (s.dense_rows > 0 ? 1 : s.E) * g.m_tiles * g.n_tiles;
  if (bn == 256 && use_pairs()) {
    const int pair_tiles = (s.dense_rows > 0 ? 1 : s.E) * ((g.m_tiles + 1) / 2) * g.n_tiles;
    if (wgrad_two_epilogues(s))
      return launch<MODE_WGRAD, EPI_STORE, 256, false, true, 2>(ma, mb, md, g, pair_tiles, s.nsm, st);
    return launch<MODE_WGRAD, EPI_STORE, 256, false, true>(ma, mb, md, g, pair_tiles, s.nsm, st);
  }
  return bn == 256 ? launch<MODE_WGRAD, EPI_STORE, 256>(ma, mb, md, g, tiles, s.nsm, st)
                   : launch<MODE_WGRAD, EPI_STORE, 128>(ma, mb, md, g, tiles, s.nsm, st);
}

// ---------------------------------------------------------------- FP8 expert GEMMs
// E4M3 operands with UE8M0 block scales; 128 x 128 x 128 tiles on kind::mxf8f6f4.

cudaError_t launch_fc1_fwd_fp8(const GemmShape& s, const Fp8Op& X1, const Fp8Op& W13, uint16_t* GU, uint16_t* Aact,
                               int* err, cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!map2d_u8(&ma, X1.q, s.H, s.rows, 128, 128) || !map3d_u8(&mb, W13.q, s.H, 2 * (uint64_t)s.F, s.E, 128, 64))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = s.H; g.n_tiles = s.F / 64; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = GU; g.ldd = 2 * (int64_t)s.F; g.D2 = Aact; g.ldd2 = s.F; g.F = s.F; g.err = err;
  g.sfa = X1.sc; g.sfa_ld = s.H / 128; g.sfb = W13.sc; g.sfb_r = 2 * s.F / 128; g.sfb_c = s.H / 128;
  return launch<MODE_FWD, EPI_SWIGLU, 128, true>(ma, mb, ma, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

cudaError_t launch_fc2_fwd_fp8(const GemmShape& s, const Fp8Op& A1, const Fp8Op& W2, uint16_t* Y, int* err,
                               cudaStream_t st) {
  CUtensorMap ma, mb, md;
  if (!map2d_u8(&ma, A1.q, s.F, s.rows, 128, 128) || !map3d_u8(&mb, W2.q, s.F, s.H, s.E, 128, 128) ||
      !map_out(&md, Y, s.H, s.rows, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = s.F; g.n_tiles = s.H / 128; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = Y; g.ldd = s.H; g.err = err;
  g.sfa = A1.sc; g.sfa_ld = s.F / 128; g.sfb = W2.sc; g.sfb_r = s.H / 128; g.sfb_c = s.F / 128;
  return launch<MODE_FWD, EPI_STORE, 128, true>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

cudaError_t launch_fc2_dgrad_fp8(const GemmShape& s, const Fp8Op& dY1, const Fp8Op& W2, const uint16_t* GU,
                                 uint16_t* dGU, int* err, cudaStream_t st) {
  CUtensorMap ma, mb, md;
  if (!map2d_u8(&ma, dY1.q, s.H, s.rows, 128, 128) || !map3d_u8(&mb, W2.q, s.F, s.H, s.E, 128, 128) ||
      !map_out(&md, dGU, 2 * (uint64_t)s.F, s.rows, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = s.H; g.n_tiles = s.F / 128; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dGU; g.ldd = 2 * (int64_t)s.F; g.GU = GU; g.ldgu = 2 * (int64_t)s.F; g.F = s.F; g.err = err;
  g.sfa = dY1.sc; g.sfa_ld = s.H / 128; g.sfb = W2.sc; g.sfb_r = s.H / 128; g.sfb_c = s.F / 128;
  return launch<MODE_DGRAD, EPI_DSWIGLU, 128, true>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

cudaError_t launch_fc1_dgrad_fp8(const GemmShape& s, const Fp8Op& dGU1, const Fp8Op& W13, uint16_t* dX1, int* err,
                                 cudaStream_t st) {
  CUtensorMap ma, mb, md;
  if (!map2d_u8(&ma, dGU1.q, 2 * (uint64_t)s.F, s.rows, 128, 128) ||
      !map3d_u8(&mb, W13.q, s.H, 2 * (uint64_t)s.F, s.E, 128, 128) || !map_out(&md, dX1, s.H, s.rows, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.K = 2 * s.F; g.n_tiles = s.H / 128; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dX1; g.ldd = s.H; g.err = err;
  g.sfa = dGU1.sc; g.sfa_ld = 2 * s.F / 128; g.sfb = W13.sc; g.sfb_r = 2 * s.F / 128; g.sfb_c = s.H / 128;
  return launch<MODE_DGRAD, EPI_STORE, 128, true>(ma, mb, md, g, s.max_mtiles * g.n_tiles, s.nsm, st);
}

// Column-quantized operands: q [rows, cols], scales [rows/128, cols].
cudaError_t launch_fc2_wgrad_fp8(const GemmShape& s, const Fp8Op& dYc, const Fp8Op& Ac, uint16_t* dW2, int* err,
                                 cudaStream_t st) {
  CUtensorMap ma, mb, md;
  if (!map2d_u8(&ma, dYc.q, s.H, s.rows, 128, 128) || !map2d_u8(&mb, Ac.q, s.F, s.rows, 128, 128) ||
      !map_out(&md, dW2, s.F, s.H, s.dense_rows > 0 ? 1 : s.E))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.m_tiles = s.H / 128; g.n_tiles = s.F / 128; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dW2; g.ldd = s.F; g.d_estride = (int64_t)s.H * s.F; g.err = err;
  g.sfa = dYc.sc; g.sfa_ld = s.H; g.sfb = Ac.sc; g.sfb_ld = s.F;
  const int tiles = (s.dense_rows > 0 ? 1 : s.E) * g.m_tiles * g.n_tiles;
  return launch<MODE_WGRAD, EPI_STORE, 128, true>(ma, mb, md, g, tiles, s.nsm, st);
}

cudaError_t launch_fc1_wgrad_fp8(const GemmShape& s, const Fp8Op& dGUc, const Fp8Op& Xc, uint16_t* dW13, int* err,
                                 cudaStream_t st) {
  CUtensorMap ma, mb, md;
  if (!map2d_u8(&ma, dGUc.q, 2 * (uint64_t)s.F, s.rows, 128, 128) || !map2d_u8(&mb, Xc.q, s.H, s.rows, 128, 128) ||
      !map_out(&md, dW13, s.H, 2 * (uint64_t)s.F, s.dense_rows > 0 ? 1 : s.E))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = s.E; g.m_tiles = 2 * s.F / 128; g.n_tiles = s.H / 128; g.dense_rows = s.dense_rows;
  g.seg_off = s.offsets; g.tile_off = s.tile_offsets; g.counts = s.counts;
  g.D = dW13; g.ldd = s.H; g.d_estride = 2 * (int64_t)s.F * s.H; g.err = err;
  g.sfa = dGUc.sc; g.sfa_ld = 2 * s.F; g.sfb = Xc.sc; g.sfb_ld = s.H;
  const int tiles = (s.dense_rows > 0 ? 1 : s.E) * g.m_tiles * g.n_tiles;
  return launch<MODE_WGRAD, EPI_STORE, 128, true>(ma, mb, md, g, tiles, s.nsm, st);
}

// ---------------------------------------------------------------- router GEMMs on tensor cores
// FP32-grade products from bf16 operands: every FP32 operand is split exactly into
// three bf16 terms (hi + mid + lo), each bf16 x bf16 product is exact in the FP32
// accumulator, and the terms are laid out along K so one GEMM sums them.

// dW_r[E,H] (fp32) = sum over the 3*Tp rows of dlsplit[3Tp,Ep] (hi rows, mid rows, lo rows,
// each block zero beyond T) times X rows taken modulo Tp (rows >= T read as zero).
cudaError_t launch_router_dwr_tc(int T, int Tp, int H, int E, int Ep, const uint16_t* dlsplit, const uint16_t* X,
                                 float* dWr, int splits, int* err, int nsm, cudaStream_t st) {
  const int bn = H % 256 == 0 ? 256 : 128;
  CUtensorMap ma, mb, md;
  if (!map2d(&ma, dlsplit, Ep, 3 * (uint64_t)Tp, 64, 64) || !map2d(&mb, X, H, T, 64, 64) ||
      !map_out_f32(&md, dWr, H, E, splits))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = splits; g.m_tiles = (E + 127) / 128; g.n_tiles = H / bn; g.dense_rows = 3 * Tp; g.kwrap = Tp; g.err = err;
  // split s covers rows [s*ksplit_rows, ...) of the 3*Tp and writes the s-th [E,H] partial
  g.ksplit_rows = (3 * Tp / splits + 63) / 64 * 64;
  g.d_estride = (int64_t)E * H;
  const int tiles = splits * g.m_tiles * g.n_tiles;
  return bn == 256 ? launch<MODE_WGRAD, EPI_F32, 256>(ma, mb, md, g, tiles, nsm, st)
                   : launch<MODE_WGRAD, EPI_F32, 128>(ma, mb, md, g, tiles, nsm, st);
}

// dX_r[T,H] (fp32) = dlA[T,3Ep] . WB[3Ep,H]: the products hi.hi + hi.mid + mid.hi of the bf16
// splits of dlogits and W_r (relative error ~2^-16; dX_r is added into a bf16 dX).  K runs to
// the next multiple of 64; the maps read zeros past 3*Ep.
cudaError_t launch_router_dx_tc(int T, int H, int Ep, const uint16_t* dlA, const uint16_t* WB, float* dXr, int* err,
                                int nsm, cudaStream_t st) {
  const int bn = H % 256 == 0 ? 256 : 128;
  CUtensorMap ma, mb, md;
  if (!map2d(&ma, dlA, 3 * (uint64_t)Ep, T, 64, 128) || !map3d(&mb, WB, H, 3 * (uint64_t)Ep, 1, 64, 64) ||
      !map_out_f32(&md, dXr, H, T, 1))
    return cudaErrorInvalidValue;
  GemmArgs g{};
  g.E = 1; g.K = (3 * Ep + 63) / 64 * 64; g.n_tiles = H / bn; g.dense_rows = T; g.err = err;
  const int tiles = ((T + 127) / 128) * g.n_tiles;
  return bn == 256 ? launch<MODE_DGRAD, EPI_F32, 256>(ma, mb, md, g, tiles, nsm, st)
                   : launch<MODE_DGRAD, EPI_F32, 128>(ma, mb, md, g, tiles, nsm, st);
}

}  // namespace moe
