// tcgen05 GEMM on 2-CTA clusters (cta_group::2) for the dense contractions
// with 256-wide tiles and a TMA-loaded A (the encode's QKV, out-projection,
// MLP and second merger linears): out = epi(A B^T + bias) in 256 x 256 tiles,
// the same epilogues as the one-CTA kernel (gemm.cu).
//
// A tile's 256 rows are split between the two CTAs of the pair (128 each) and
// so are its 256 B rows: each CTA stages by TMA its own 128 x 64 A and 128 x 64
// B blocks per K step (32 KB, so six stages fit), and the even CTA (the
// leader) issues tcgen05.mma.cta_group::2 with M = 256, N = 256, which reads
// both CTAs' shared memory at the same offsets and writes each CTA's TMEM
// with its own 128 accumulator rows.  Barriers:
//   full[s]   (leader)  the leader arrives expecting both CTAs' bytes; both
//                       CTAs' TMA loads complete it;
//   empty[s]  (each)    tcgen05.commit multicast to both CTAs frees a stage;
//   tfull[a]  (each)    commit multicast: accumulator a holds a finished tile;
//   tempty[a] (leader)  all 16 epilogue warps of the pair have read it;
//   drain     (each)    the leader's last MMAs are done (TMEM, operands free).
// The pair meets at cluster barriers after the barrier initialisation and
// before the collective TMEM release.  No arrival inside the loops carries a
// cluster-scope release: one per stage halved the kernel's speed, one per
// tile cost microseconds.  Every mbarrier wait is bounded.
#include "internal.h"
#include "ptx.cuh"

#include <cudaTypedefs.h>

#include <map>
#include <mutex>

namespace dsvit {

namespace {

#include "gemm_common.cuh"

// RESID: the residual epilogue of a short-K GEMM (the out-projection, K =
// 1024): its eight warps each load the tile's residual rows by TMA into four
// staging chunks (32 rows x 32 columns, the store layout) and write the result
// back in place; that buffer takes the room of one operand stage.  Per-thread
// residual loads issued at a tile's start (4096 per SM) held up the TMA
// producer for about 2 us per tile; with two tiles per pair that was a sixth
// of the kernel.  Long-K GEMMs (FC2, K = 4096) keep six stages, which their
// main loop needs more, and load the residual into registers.
template <bool RESID>
struct PairCfgT {
  static constexpr int BM = 128;                               // rows per CTA
  static constexpr int TILE_M = 256;                           // rows per tile
  static constexpr int BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = 128 * BK * 2;                 // this CTA's half of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = RESID ? 5 : 6;
  static constexpr int EPI_WARPS = 8;
  static constexpr int STG_BYTES = 32 * 32 * 2;
  static constexpr int STG_PER_WARP = RESID ? 4 : 2;           // chunks of one tile / double buffer
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;
  static constexpr int OFF_BIAS = OFF_STG + EPI_WARPS * STG_PER_WARP * STG_BYTES;
  static constexpr int OFF_BAR = OFF_BIAS + 2 * 256 * 2;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr int TMEM_COLS = 512;                        // two 256-column accumulators
  static constexpr int THREADS = (EPI_WARPS + 2) * 32;
  static constexpr int BAR_RESID = 2 * STAGES + 5;             // one residual barrier per epilogue warp
};
using PairCfg = PairCfgT<false>;
static_assert(PairCfgT<false>::SMEM_BYTES <= 232448, "shared memory");
static_assert(PairCfgT<true>::SMEM_BYTES <= 232448, "shared memory");
static_assert(PairCfgT<false>::BAR_RESID <= 31 && PairCfgT<true>::BAR_RESID + 8 <= 31, "barrier slots");

template <int EPI, bool RESID_TMA>
__global__ void __launch_bounds__(PairCfg::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  static_assert(!RESID_TMA || EPI == kEpiBiasResid, "TMA residual with the residual epilogue only");
  using C = PairCfgT<RESID_TMA>;
  constexpr int BN = 256;
  constexpr uint32_t kAccs = 2;
  constexpr bool kResidTma = RESID_TMA;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 31);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4);
  auto stage_a = [&](int s) { return smem_u32(smem + s * C::STAGE_BYTES); };
  auto stage_b = [&](int s) { return smem_u32(smem + s * C::STAGE_BYTES + C::A_BYTES); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (p.M + C::TILE_M - 1) / C::TILE_M;
  const int num_n = p.N / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = p.K / C::BK;
  const uint32_t rank = cluster_rank();                 // 0: the leader
  const int pair = static_cast<int>(blockIdx.x >> 1), pairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    if constexpr (kResidTma)
      for (int w = 0; w < C::EPI_WARPS; ++w) mbar_init(bar0 + 8u * (C::BAR_RESID + w), 1);
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();   // the peer's barriers exist before either CTA signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_launch();
  grid_dep_wait();

  __shared__ int consumed_fills, issued_s;
  int issued_fills = 0;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = pair; tile < num_tiles; tile += pairs) {
        const int mb = tile_mb(tile, num_m, num_n, p.n_fast), nb = tile_nb(tile, num_m, num_n, p.n_fast);
        // SwiGLU: gate rows nb*128.. in the leader, the matching up rows
        // N/2 + nb*128.. in the peer (accumulator columns 0..127 / 128..255).
        const int brow = EPI == kEpiSwiglu ? (rank ? p.N / 2 : 0) + nb * (BN / 2)
                                           : nb * BN + static_cast<int>(rank) * (BN / 2);
        const int arow = mb * C::TILE_M + static_cast<int>(rank) * C::BM;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          // The leader alone arrives, expecting both CTAs' bytes.  The peer's
          // bytes may land first (the transaction count dips below zero); the
          // phase cannot complete before the leader's arrival, and the peer
          // refills a stage only after the MMAs of its previous phase, that is
          // after that phase completed.
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (rank == 0) mbar_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
          tma_load_2d_pair(stage_a(stage), &tmA, fb, kb * C::BK, arow);
          tma_load_2d_pair(stage_b(stage), &tmB, fb, kb * C::BK, brow);
          ++issued_fills;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(C::TILE_M, BN, false, false);
      const uint64_t da0 = sdesc_sw128(stage_a(0), 16, 1024);
      const uint64_t db0 = sdesc_sw128(stage_b(0), 16, 1024);
      int stage = 0, fills = 0;
      uint32_t phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += pairs) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t off = static_cast<uint64_t>(stage * (C::STAGE_BYTES >> 4));
#pragma unroll
          for (int k = 0; k < C::BK / 16; ++k)
            umma_bf16_pair(d_tmem, da0 + off + 2 * k, db0 + off + 2 * k, idesc, (kb | k) != 0);
          umma_commit_pair(empty_bar(stage));   // frees the stage in both CTAs
          ++fills;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      consumed_fills = fills;
      umma_commit_pair(drain_bar);
      mbar_wait(drain_bar, 0, p.status);
    } else if (lane == 0) {
      // The peer: its TMEM and operands are in use until the leader's MMAs drain.
      consumed_fills = 0;
      mbar_wait(drain_bar, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
#define GEMM_FIRST_TILE pair
#define GEMM_TILE_STEP pairs
#define GEMM_ROW0 mb * C::TILE_M + static_cast<int>(rank) * C::BM + quad * 32
#define GEMM_RELEASE_ACC mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0))
#include "gemm_epilogue.inc"
#undef GEMM_FIRST_TILE
#undef GEMM_TILE_STEP
#undef GEMM_ROW0
#undef GEMM_RELEASE_ACC
  }

  if (warp == 8 && lane == 0) issued_s = issued_fills;
  tc_fence_before();
  cluster_sync();
  if (warp == 8 && lane == 0 && rank == 0 && status_failed(p.status)) {
    // After a timeout: the peer's loads complete the leader's barriers, so the
    // leader waits (bounded) for the fills either CTA issued, and no TMA write
    // lands in shared memory after the pair has exited.
    int peer;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer) : "r"(mapa_shared(smem_u32(&issued_s), 1))
                 : "memory");
    const int upto = peer > issued_fills ? peer : issued_fills;
    for (int f = consumed_fills; f < upto; ++f) {
      const int s = f % C::STAGES;
      if (!mbar_wait(full_bar(s), (f / C::STAGES) & 1, nullptr)) break;
    }
  }
  cluster_sync();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

// Clusters of two CTAs of `kernel` that fit on the device at once (0 if none
// or the query fails); cached per kernel and device.
int max_active_pairs(const void* kernel, int smem_bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_sms());
  cfg.blockDim = dim3(PairCfg::THREADS);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

template <int EPI, bool RESID_TMA = false>
int launch_pair_t(const CUtensorMap& tmA, const CUtensorMap& tmB128, const CUtensorMap& tmC, const GemmParams& p,
                  cudaStream_t stream) {
  using C = PairCfgT<RESID_TMA>;
  const void* kfn = reinterpret_cast<const void*>(gemm_pair_kernel<EPI, RESID_TMA>);
  if (allow_smem(kfn, C::SMEM_BYTES) != cudaSuccess) return DS_VIT_ECUDA;
  const int max_pairs = max_active_pairs(kfn, C::SMEM_BYTES);
  if (max_pairs <= 0) return kGemmNoPair;
  // As few pairs as give the same number of rounds over the tiles: the same
  // time with less contention for L2 and power.
  const int tiles = ((p.M + C::TILE_M - 1) / C::TILE_M) * (p.N / 256);
  const int rounds = (tiles + max_pairs - 1) / max_pairs;
  const int pairs = (tiles + rounds - 1) / rounds;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<EPI, RESID_TMA>, tmA, tmB128, tmC, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

}  // namespace

int launch_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB128, const CUtensorMap& tmC, int M, int N,
                     int K, const bf16* bias, bf16* out, int epi, const int* rowpos, const float* rope_cs,
                     int* status, cudaStream_t stream) {
  if (M <= 0 || K <= 0 || K % 64 != 0 || N % 256 != 0) return DS_VIT_EINVAL;
  const GemmParams p{M, N, K, out, bias, rowpos, rope_cs, status, tile_order(M, K)};
  switch (epi) {
    case kEpiBias: return launch_pair_t<kEpiBias>(tmA, tmB128, tmC, p, stream);
    case kEpiBiasGelu: return launch_pair_t<kEpiBiasGelu>(tmA, tmB128, tmC, p, stream);
    case kEpiBiasResid:
      return K <= 1024 ? launch_pair_t<kEpiBiasResid, true>(tmA, tmB128, tmC, p, stream)
                       : launch_pair_t<kEpiBiasResid>(tmA, tmB128, tmC, p, stream);
    case kEpiQkvRope: return launch_pair_t<kEpiQkvRope>(tmA, tmB128, tmC, p, stream);
    case kEpiSwiglu: return launch_pair_t<kEpiSwiglu>(tmA, tmB128, tmC, p, stream);
    case kEpiQkvRope72: return launch_pair_t<kEpiQkvRope72>(tmA, tmB128, tmC, p, stream);
    default: return DS_VIT_EINVAL;
  }
}

}  // namespace dsvit
