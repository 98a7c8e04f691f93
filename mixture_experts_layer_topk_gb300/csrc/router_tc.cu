// Router logits on the tensor cores (every E, when the call has a workspace).
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (summary
// page, "Method"): the router projection is kept in FP32.  Here P = X W_r^T is
// formed from the exact three-term bf16 split of W_r (W_r = hi + mid + lo, each
// term the leading 8 significant bits of what the previous terms leave), so
// every product x * w_part is exact inside the tensor core.  What the tensor
// core does not keep exact is its FP32 accumulation: summed over the whole of
// K in tensor memory the error grows linearly with K (about 4e-5 relative at
// K = 3 x 4096, above the 1e-5 logit bound).  So the accumulator restarts for
// every 64-column block of X: a block's 12 MMAs (3 split terms x 4 steps of 16)
// accumulate in tensor memory, and the epilogue warps read the block sum out
// (tcgen05.ld) and add it into FP32 registers with round-to-nearest adds.  The
// in-MMA error is then that of a 64-term partial, and the running sum is an
// ordinary FP32 sum over H/64 blocks.
//
// One CTA per 128-token x BN-expert tile (BN = 32, 64 or 128 by E) and K split (up
// to 8 splits when the tiles alone would leave SMs idle; split s writes its own
// partial [T,E] sum, added in a fixed order by the routing pass), 6 warps: warp 0
// issues the TMA loads of X and the three W_r splits into a ring of stages, warp 1
// allocates tensor memory (four or eight BN-column block accumulators) and issues the MMAs
// from one thread, warps 2-5 drain the block sums, one token row per thread.
// Every wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT in the device
// error word and the CTA unwinds.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRtBM = 128;                  // tokens per tile (MMA M, tensor-memory lanes)
constexpr int kRtBK = 64;                   // X columns per stage: 128 bytes of bf16
constexpr int kRtA = kRtBM * 128;           // X tile bytes
constexpr int kRtThreads = 192;

// BN experts per tile (MMA N); a stage holds the X tile and the three splits' W tiles
template <int BN>
struct RtGeo {
  static constexpr int B = BN * 128;                    // bytes of one split's W tile
  static constexpr int STAGE = kRtA + 3 * B;            // 28, 40 or 64 KB
  static constexpr int ST = BN == 128 ? 3 : (BN == 64 ? 4 : 6);
  // block-sum accumulators in tensor memory: the MMAs run up to NACC blocks ahead of the
  // read-out (NACC * BN columns: 256 for BN 32, 256 for 64, 512 for 128)
  static constexpr int NACC = BN == 32 ? 8 : 4;
  static constexpr size_t SMEM = 1024 + (size_t)ST * STAGE + 256;
  static_assert((2 * ST + 2 * NACC + 1) * 8 + 4 <= 256, "barriers and the tensor-memory address fit");
};

struct RouterTcArgs {
  int T, E, Ep;
  int nkb;      // 64-column blocks of X in all of K
  int kb_per;   // blocks per K split
  float* P0;    // split 0 (or the whole product): [T,E]
  float* Pn;    // splits 1..: [splits-1][T,E]
  int* err;
  uint64_t wait_ns;  // limit of each pipeline wait (0: one non-blocking test)
};

template <int BN>
__global__ void __launch_bounds__(kRtThreads, 1)
    k_router_logits_tc(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
                       const RouterTcArgs a) {
  using G = RtGeo<BN>;
  constexpr int kRtBN = BN, kRtST = G::ST, kRtB = G::B, kRtStage = G::STAGE;
  constexpr uint32_t IDESC = idesc_bf16(kRtBM, kRtBN, 0, 0);
  constexpr int NACC = G::NACC;
  constexpr uint32_t TMEM_COLS = NACC * kRtBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + kRtST * kRtStage);
  uint64_t* empty = full + kRtST;
  uint64_t* acc_full = empty + kRtST;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* done_bar = acc_empty + NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done_bar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kRtBM, e0 = blockIdx.y * kRtBN;
  const int kb0 = blockIdx.z * a.kb_per;
  const int kb1 = kb0 + a.kb_per < a.nkb ? kb0 + a.kb_per : a.nkb;
  const int nk = kb1 > kb0 ? kb1 - kb0 : 0;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kRtST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(done_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&mapX);
    tma_prefetch_desc(&mapW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, used = 0, last_par = 0;
      for (int i = 0; i < nk; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1, a.wait_ns)) {
          set_device_error(a.err, MOE_ERR_TIMEOUT, 11);
          break;
        }
        uint8_t* sa = tiles + stage * kRtStage;
        const int x = (kb0 + i) * kRtBK;
        mbar_arrive_expect_tx(&full[stage], kRtStage);
        tma_load_2d(sa, &mapX, &full[stage], x, m0);
#pragma unroll
        for (int s = 0; s < 3; ++s) tma_load_2d(sa + kRtA + s * kRtB, &mapW, &full[stage], x, s * a.Ep + e0);
        used |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kRtST) {
          stage = 0;
          phase ^= 1;
        }
      }
      // nothing may still be landing in shared memory when the CTA exits
      for (int s = 0; s < kRtST; ++s)
        if (used >> s & 1)
          if (!mbar_wait(&full[s], last_par >> s & 1)) set_device_error(a.err, MOE_ERR_TIMEOUT, 12);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0; i < nk; ++i) {
        const int b = i % NACC;
        if (!mbar_wait(&acc_empty[b], ((i / NACC) & 1) ^ 1, a.wait_ns) || !mbar_wait(&full[stage], phase, a.wait_ns)) {
          set_device_error(a.err, MOE_ERR_TIMEOUT, 13);
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(tiles + stage * kRtStage);
        const uint32_t d = tmem + b * kRtBN;
        // a fresh block sum: the first of the block's 12 MMAs overwrites the accumulator
#pragma unroll
        for (int s = 0; s < 3; ++s)
#pragma unroll
          for (int kk = 0; kk < kRtBK / 16; ++kk)
            umma_f16(d, smem_desc_sw128(sa + kk * 32, 16, 1024),
                     smem_desc_sw128(sa + kRtA + s * kRtB + kk * 32, 16, 1024), IDESC, (s | kk) != 0);
        umma_commit(&empty[stage]);
        umma_commit(&acc_full[b]);
        if (++stage == kRtST) {
          stage = 0;
          phase ^= 1;
        }
      }
      // every issued MMA has finished before tensor memory is released
      umma_commit(done_bar);
      if (!mbar_wait(done_bar, 0)) set_device_error(a.err, MOE_ERR_TIMEOUT, 14);
    }
  } else {
    // ------------------------------------------------------------ block sums -> FP32 registers
    const int q = warp & 3;           // this warp's quarter of the tensor-memory lanes
    const int r = q * 32 + lane;      // token row within the tile
    float acc[kRtBN];
#pragma unroll
    for (int c = 0; c < kRtBN; ++c) acc[c] = 0.f;
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int b = i % NACC;
      if (!mbar_wait(&acc_full[b], (i / NACC) & 1, a.wait_ns)) {
        set_device_error(a.err, MOE_ERR_TIMEOUT, 15);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + b * kRtBN;
#pragma unroll
      for (int j = 0; j < kRtBN / 32; ++j) {
        uint32_t v[32];
        tmem_ld32(base + 32 * j, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[32 * j + c] = __fadd_rn(acc[32 * j + c], __uint_as_float(v[c]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
    const int t = m0 + r;
    if (ok && t < a.T) {
      float* P = (blockIdx.z ? a.Pn + (size_t)(blockIdx.z - 1) * a.T * a.E : a.P0) + (size_t)t * a.E;
      if ((a.E & 3) == 0) {
#pragma unroll
        for (int c = 0; c < kRtBN; c += 4)
          if (e0 + c < a.E)
            *reinterpret_cast<float4*>(P + e0 + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < kRtBN; ++c)
          if (e0 + c < a.E) P[e0 + c] = acc[c];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// 2D bf16 tensor map over a row-major [rows, cols] matrix, boxes of 64 columns x
// box_rows rows in the 128-byte swizzle layout the MMA descriptors expect.
bool map_rows_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t gd[2] = {cols, rows}, gs[1] = {cols * 2};
  cuuint32_t bd[2] = {(cuuint32_t)kRtBK, box_rows}, es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gd, gs, bd, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_bn(int T, int H, int E, int Ep, const uint16_t* X, const uint16_t* wsplit, float* P0, float* Pn,
                      int splits, int* err, cudaStream_t st) {
  using G = RtGeo<BN>;
  static std::atomic<uint64_t> attr{0};
  if (cudaError_t e = raise_smem_limit(attr, k_router_logits_tc<BN>, G::SMEM); e != cudaSuccess) return e;
  CUtensorMap mx, mw;
  if (!map_rows_bf16(&mx, X, H, T, kRtBM) || !map_rows_bf16(&mw, wsplit, H, 3 * (uint64_t)Ep, BN))
    return cudaErrorInvalidValue;
  RouterTcArgs a{};
  a.T = T; a.E = E; a.Ep = Ep;
  a.nkb = (H + kRtBK - 1) / kRtBK;
  a.kb_per = (a.nkb + splits - 1) / splits;
  a.P0 = P0; a.Pn = Pn; a.err = err;
  a.wait_ns = pipeline_wait_ns();
  dim3 grid((T + kRtBM - 1) / kRtBM, (E + BN - 1) / BN, splits);
  k_router_logits_tc<BN><<<grid, kRtThreads, G::SMEM, st>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

int router_tc_splits(int T, int H, int E, int nsm, int max_splits) {
  const int bn = E <= 32 ? 32 : (E <= 64 ? 64 : 128);
  const int tiles = ((T + kRtBM - 1) / kRtBM) * ((E + bn - 1) / bn);
  int s = tiles > 0 ? nsm / tiles : 1;
  const int nkb = (H + kRtBK - 1) / kRtBK;
  s = s < max_splits ? s : max_splits;
  s = s < nkb ? s : nkb;
  s = s < 1 ? 1 : s;
  // every split gets at least one block: ceil(nkb / s) * (s - 1) < nkb
  while (s > 1 && ((nkb + s - 1) / s) * (s - 1) >= nkb) --s;
  return s;
}

cudaError_t launch_router_logits_tc(int T, int H, int E, int Ep, const uint16_t* X, const uint16_t* wsplit, float* P0,
                                    float* Pn, int splits, int* err, cudaStream_t st) {
  if (E <= 32) return launch_bn<32>(T, H, E, Ep, X, wsplit, P0, Pn, splits, err, st);
  if (E <= 64) return launch_bn<64>(T, H, E, Ep, X, wsplit, P0, Pn, splits, err, st);
  return launch_bn<128>(T, H, E, Ep, X, wsplit, P0, Pn, splits, err, st);
}

}  // namespace moe
