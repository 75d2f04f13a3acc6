// tcgen05 GEMM for the encode's dense contractions: out = epi(A B^T + bias).
//
// A [M, K] (activations) and B [N, K] (nn.Linear weights) are both K-major
// bf16, staged by TMA into 128-byte-swizzled shared-memory tiles; one thread
// issues tcgen05.mma (M = 128, N = BN, K = 16 per instruction) into a TMEM
// accumulator; eight epilogue warps read it back with tcgen05.ld and apply the
// fused epilogue:
//   bias                 — patch projection ("Multimodal basics": a patch
//                          projection maps pixel rows into the vision hidden
//                          space) and the second merger linear;
//   bias + GELU(erf)     — MLP up-projection and the first merger linear
//                          ("End-to-end results and their limits": erf GELU);
//   bias + residual      — attention output projection and MLP down-projection
//                          (pre-norm block, residual stream stored in bf16);
//   bias + 2D RoPE       — QKV projection: q and k rotated per head, dims 0..31
//                          by the patch row and 32..63 by the patch column with
//                          the half-vector pairing (j, j+16) ("Step 3: Height and
//                          width occupy blocks in 2D RoPE").
// All from "DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision".
//
// Structure: persistent CTAs (one per SM), 10 warps: warps 0-7 epilogue (TMEM
// lane quadrant = warp % 4; warps 0-3 take the even 32-column chunks of a tile,
// warps 4-7 the odd ones), warp 8 TMA producer, warp 9 MMA issuer.  A ring of
// STAGES shared-memory stages (full/empty mbarriers) feeds the MMA; two TMEM
// accumulators (tfull/tempty mbarriers) let the epilogue of one tile overlap
// the main loop of the next.  The tile's bias is staged once in shared memory;
// each 32x32 output chunk goes through a 64-byte-swizzled shared staging tile
// (two per warp) and leaves by TMA store, which also clips rows past M.
// 320-wide tiles (the merger linears, N = 5120, at sizes where 256-wide tiles
// need a second, almost empty round) and 288-wide tiles (widths of 1152, which
// otherwise take 128-wide tiles) issue two MMAs per K step (N = 256 and
// N = 64 or 32 into adjacent TMEM columns), load B as a 256-row and a 64- or
// 32-row box, and keep one accumulator (320 or 288 of the 512 columns).
// Where 256-wide tiles are chosen and A comes by TMA, the 2-CTA-cluster
// kernel runs instead (gemm_pair.cu, 256 x 256 tiles, same epilogue source);
// this kernel keeps 128-wide tiles, the produced-A GEMMs and devices where no
// pair of its CTAs fits.
#include "internal.h"
#include "ptx.cuh"

#include <cudaTypedefs.h>

#include <map>
#include <mutex>

namespace dsvit {

namespace {

#include "gemm_common.cuh"

template <int BN, int ASRC = kATma>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // The pixel producer's raw-byte ring and LUT take the room of one stage.
  static constexpr int STAGES = (BN > 256 ? 3 : BN == 256 ? 4 : 6) - (ASRC == kAPixels ? 1 : 0);
  static constexpr int EPI_WARPS = 8;
  static constexpr int STG_BYTES = 32 * 32 * 2;                // one 32x32 bf16 chunk
  static constexpr int OFF_STG = STAGES * STAGE_BYTES;         // 2 staging chunks per warp
  static constexpr int OFF_BIAS = OFF_STG + EPI_WARPS * 2 * STG_BYTES;
  // kAPixels: RAW_SLOTS pixel rows in flight per producer thread, 44 bytes
  // (11 words: a 42-byte patch row and its 4-byte alignment) per row and slot;
  // an odd word stride keeps the 32 rows a warp reads in distinct banks.
  static constexpr int RAW_SLOTS = 4;
  static constexpr int RAW_ROW = 44;
  static constexpr int OFF_RAW = OFF_BIAS + 2 * BN * 2;        // bias, double-buffered by tile
  static constexpr int OFF_LUT = OFF_RAW + RAW_SLOTS * BM * RAW_ROW;
  static constexpr int OFF_BAR = ASRC == kAPixels ? OFF_LUT + 3 * 256 * 2 : OFF_RAW;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;      // + barriers + alignment slack
  static constexpr int ACCS = 2 * BN <= 512 ? 2 : 1;           // TMEM accumulators
  static constexpr int TMEM_COLS = ACCS == 2 ? 2 * BN : 512;
  // Warps 0-7 epilogue, 8 TMA, 9 MMA; with a produced A, warps 10-13 build the A
  // tiles (one row per thread) and 14-15 idle: 16 warps keep every SM
  // sub-partition within 4 x 32 x 128 registers.
  static constexpr int THREADS = (ASRC == kATma ? EPI_WARPS + 2 : 16) * 32;
  static constexpr int BAR_RESID = 0;                          // the residual comes in registers here
};
static_assert(GemmCfg<256>::SMEM_BYTES <= 232448, "shared memory");
static_assert(GemmCfg<128>::SMEM_BYTES <= 232448, "shared memory");
static_assert(GemmCfg<256, kAPixels>::SMEM_BYTES <= 232448, "shared memory");
static_assert(GemmCfg<128, kAPixels>::SMEM_BYTES <= 232448, "shared memory");
static_assert(GemmCfg<320>::SMEM_BYTES <= 232448, "shared memory");
static_assert(GemmCfg<320, kAMerge>::SMEM_BYTES <= 232448, "shared memory");
static_assert(GemmCfg<288>::SMEM_BYTES <= 232448, "shared memory");
static_assert(3 * GemmCfg<128>::STAGES + 5 <= 31, "barrier slots");

// Image of packed row `row` (offsets `off`, n images) and the row's index in it.
__device__ __forceinline__ int find_image(const int64_t* off, int n, int64_t row, int* local) {
  int i = 0;
  while (i + 1 < n && off[i + 1] <= row) ++i;
  *local = static_cast<int>(row - off[i]);
  return i;
}

// A producer, kAMerge.  A row = merged token (my, mx) of image i; column
// p*1024 + c holds z[(3my + dy)*gw + 3mx + dx, c] with p = dy*3 + dx, or 0 where
// the 3x3 window leaves the grid ("Step 4: The aligner pads a two-dimensional
// grid").  A K block is one 128-byte run of one z row per A row, copied by
// cp.async straight into the 128-byte-swizzled stage (16-byte unit u of row R
// at unit u ^ (R & 7)); eight consecutive threads copy the eight units of one
// row, so a warp moves four whole 128-byte lines per instruction.  Thread t
// serves rows q*16 + t/8 (q = 0..7).  Its arrival on the stage's A barrier
// fires once its copies have landed, so up to STAGES blocks are in flight.
template <class C>
__device__ __forceinline__ void produce_a_merge(const AGenParams& g, const GemmParams& p, uint8_t* smem,
                                                uint32_t afull0, uint32_t empty0, int num_m,
                                                int num_n, int num_tiles, int num_kb, int t) {
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  const int u = t & 7;
  for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
    // Per served row: z row of window position (0, 0), and gw << 9 | mask of
    // the window positions inside the grid (bit p).
    int base[8];
    uint32_t geo[8];
    const int64_t row0 = static_cast<int64_t>(tile_mb(tile, num_m, num_n, p.n_fast)) * C::BM;
    for (int q = 0; q < 8; ++q) {
      const int64_t row = row0 + q * 16 + (t >> 3);
      base[q] = 0;
      geo[q] = 0;
      if (row < p.M) {
        int local = 0;
        const int i = find_image(g.batch.tok_off, g.batch.n, row, &local);
        const int gh = g.batch.gh[i], gw = g.batch.gw[i];
        const int w = (gw + 2) / 3, my = local / w, mx = local % w;
        uint32_t mask = 0;
#pragma unroll
        for (int pw = 0; pw < 9; ++pw)
          if (3 * my + pw / 3 < gh && 3 * mx + pw % 3 < gw) mask |= 1u << pw;
        base[q] = static_cast<int>(g.batch.row_off[i]) + 3 * my * gw + 3 * mx;
        geo[q] = (static_cast<uint32_t>(gw) << 9) | mask;
      }
    }
    for (int kb = 0; kb < num_kb; ++kb) {
      const int pw = kb >> 4, c0 = (kb & 15) * 64;
      const int dy = pw / 3, dx = pw % 3;
      if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, p.status)) {
        ok = false;
        break;
      }
      const uint32_t dst0 = smem_u32(smem + stage * C::STAGE_BYTES);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int R = q * 16 + (t >> 3);
        const bool in = (geo[q] >> pw) & 1u;
        const int64_t zr = static_cast<int64_t>(base[q]) + dy * static_cast<int>(geo[q] >> 9) + dx;
        const bf16* src = in ? g.z + zr * 1024 + c0 + u * 8 : g.z;
        cp_async_16(dst0 + R * 128 + ((u ^ (R & 7)) << 4), src, in ? 16u : 0u);
      }
      cp_async_arrive(afull0 + 8u * stage);
      if (++stage == C::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  cp_async_wait<0>();   // no copy lands after the CTA has exited
}

// Source of one patch: its top-left pixel's first byte and the image pitch.
struct PatchSrc {
  const uint8_t* p;
  int pitch;            // bytes per pixel row (W * 3)
  int gy, gx;
  bool valid;
};

__device__ __forceinline__ PatchSrc patch_src(const AGenParams& g, int64_t row, int64_t M) {
  PatchSrc s{g.batch.pix[0], 0, 0, 0, false};
  if (row >= M) return s;
  int local = 0;
  const int i = find_image(g.batch.row_off, g.batch.n, row, &local);
  const int gw = g.batch.gw[i];
  s.gy = local / gw;
  s.gx = local % gw;
  s.pitch = gw * 14 * 3;
  s.p = g.batch.pix[i] + static_cast<int64_t>(s.gy) * 14 * s.pitch + s.gx * 42;
  s.valid = true;
  return s;
}

// A producer, kAPixels ("Step 1" items 5-6, "Step 5": 14x14 patches of
// bf16((v/255 - mean_c)/std_c)).  Thread r builds row r (one patch) of every
// A tile; K block y holds the patch's pixel row y: its 42 bytes (x*3 + c order,
// as they lie in the image) normalised through a per-CTA table, then 22 zero
// columns.  The 42 bytes start on an even address (the image is 4-byte
// aligned, rows and patches are multiples of 42 bytes apart): they are copied
// as 11 aligned words by cp.async into a per-thread ring RAW_SLOTS rows deep,
// so pixel loads run ahead of the conversion.
template <class C>
__device__ __forceinline__ void produce_a_pixels(const AGenParams& g, const GemmParams& p, uint8_t* smem,
                                                 uint32_t afull0, uint32_t empty0, int num_m,
                                                 int num_n, int num_tiles, int r) {
  constexpr int KB = 14;   // one patch row per K block
  uint16_t* lut = reinterpret_cast<uint16_t*>(smem + C::OFF_LUT);
  for (int j = r; j < 3 * 256; j += C::BM) lut[j] = reinterpret_cast<const uint16_t*>(g.lut)[j];
  named_barrier(2, C::BM);
  const uint32_t raw_row = smem_u32(smem + C::OFF_RAW) + r * C::RAW_ROW;
  const int total = (num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                    static_cast<int>(gridDim.x) * KB;

  // Issue the raw copy of fill f (tile f / KB of this CTA, pixel row f % KB).
  PatchSrc is{};
  auto issue = [&](int f) {
    if (f < total) {
      const int t = f / KB, y = f % KB;
      if (y == 0) {
        const int tile = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
        const int64_t row = static_cast<int64_t>(tile_mb(tile, num_m, num_n, p.n_fast)) * C::BM + r;
        is = patch_src(g, row, p.M);
      }
      const uintptr_t s = reinterpret_cast<uintptr_t>(is.p) + static_cast<uintptr_t>(y) * is.pitch;
      const uint8_t* a = reinterpret_cast<const uint8_t*>(s & ~static_cast<uintptr_t>(3));
      const uint32_t last = (s & 3) ? 4u : 2u;   // the run ends 2 bytes into word 10 when aligned
      const uint32_t dst = raw_row + (f % C::RAW_SLOTS) * (C::BM * C::RAW_ROW);
#pragma unroll
      for (int j = 0; j < 11; ++j)
        cp_async_4(dst + 4 * j, is.valid ? a + 4 * j : is.p, is.valid ? (j < 10 ? 4u : last) : 0u);
    }
    cp_async_commit();
  };

  for (int f = 0; f < C::RAW_SLOTS - 1; ++f) issue(f);
  int stage = 0;
  uint32_t phase = 0;
  PatchSrc cs{};
  for (int f = 0; f < total; ++f) {
    issue(f + C::RAW_SLOTS - 1);
    cp_async_wait<C::RAW_SLOTS - 1>();    // fill f's raw row has landed
    const int t = f / KB, y = f % KB;
    const int tile = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
    if (y == 0) {
      const int64_t row = static_cast<int64_t>(tile_mb(tile, num_m, num_n, p.n_fast)) * C::BM + r;
      cs = patch_src(g, row, p.M);
      if (cs.valid && tile_nb(tile, num_m, num_n, p.n_fast) == 0) g.rowpos[row] = (cs.gy << 16) | cs.gx;
    }
    uint32_t w[12];
    const uint32_t src = raw_row + (f % C::RAW_SLOTS) * (C::BM * C::RAW_ROW);
#pragma unroll
    for (int j = 0; j < 11; ++j) asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[j]) : "r"(src + 4 * j));
    w[11] = 0;
    // Start the byte sequence at the run: shift by 2 bytes when it began mid-word.
    const bool odd_half = ((reinterpret_cast<uintptr_t>(cs.p) + static_cast<uintptr_t>(y) * cs.pitch) & 3) != 0;
#pragma unroll
    for (int j = 0; j < 11; ++j) w[j] = odd_half ? __funnelshift_r(w[j], w[j + 1], 16) : w[j];
    uint32_t out[32];
#pragma unroll
    for (int j = 0; j < 21; ++j) {
      const uint32_t b0 = (w[j >> 1] >> ((j & 1) * 16)) & 0xffu;
      const uint32_t b1 = (w[j >> 1] >> ((j & 1) * 16 + 8)) & 0xffu;
      const uint32_t v0 = lut[((2 * j) % 3) * 256 + b0];
      const uint32_t v1 = lut[((2 * j + 1) % 3) * 256 + b1];
      out[j] = cs.valid ? (v0 | (v1 << 16)) : 0u;
    }
#pragma unroll
    for (int j = 21; j < 32; ++j) out[j] = 0u;
    if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, p.status)) break;
    const uint32_t dst = smem_u32(smem + stage * C::STAGE_BYTES) + r * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + ((u ^ (r & 7)) << 4)),
                   "r"(out[4 * u]), "r"(out[4 * u + 1]), "r"(out[4 * u + 2]), "r"(out[4 * u + 3])
                   : "memory");
    fence_proxy_async_smem();
    mbar_arrive(afull0 + 8u * stage);
    if (++stage == C::STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  }
  cp_async_wait<0>();   // no copy lands after the CTA has exited
}

template <int BN, int EPI, int ASRC>
__global__ void __launch_bounds__(GemmCfg<BN, ASRC>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB64,
                const GemmParams p, const __grid_constant__ AGenParams g) {
  using C = GemmCfg<BN, ASRC>;
  constexpr uint32_t kAccs = C::ACCS;
  constexpr bool kResidTma = false;
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
  // Produced A: the stage's A tile is complete when all BM producer threads
  // have arrived (the B tile still completes full_bar by its TMA bytes).
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + 5 + s); };
  auto stage_a = [&](int s) { return smem_u32(smem + s * C::STAGE_BYTES); };
  auto stage_b = [&](int s) { return smem_u32(smem + s * C::STAGE_BYTES + C::A_BYTES); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (p.M + C::BM - 1) / C::BM;
  const int num_n = p.N / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = p.K / C::BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      if constexpr (ASRC != kATma) mbar_init(afull_bar(s), C::BM);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), C::EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    if constexpr (ASRC == kATma) prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
    if constexpr (BN > 256) prefetch_tensormap(&tmB64);
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_launch();
  grid_dep_wait();

  __shared__ int consumed_fills;
  int issued_fills = 0;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int mb = tile_mb(tile, num_m, num_n, p.n_fast), nb = tile_nb(tile, num_m, num_n, p.n_fast);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full_bar(stage), ASRC == kATma ? C::STAGE_BYTES : C::B_BYTES);
          if constexpr (ASRC == kATma)
            tma_load_2d(stage_a(stage), &tmA, full_bar(stage), kb * C::BK, mb * C::BM);
          if constexpr (EPI == kEpiSwiglu) {
            // Gate rows nb*128.. and the matching up rows N/2 + nb*128.. fill
            // the two halves of the B stage (128-row boxes).
            tma_load_2d(stage_b(stage), &tmB, full_bar(stage), kb * C::BK, nb * (BN / 2));
            tma_load_2d(stage_b(stage) + (BN / 2) * C::BK * 2, &tmB, full_bar(stage), kb * C::BK,
                        p.N / 2 + nb * (BN / 2));
          } else if constexpr (BN > 256) {
            // Rows nb*BN .. +255 and the remaining BN - 256 rows (tmB64: a box
            // of exactly that many rows).
            tma_load_2d(stage_b(stage), &tmB, full_bar(stage), kb * C::BK, nb * BN);
            tma_load_2d(stage_b(stage) + 256 * C::BK * 2, &tmB64, full_bar(stage), kb * C::BK, nb * BN + 256);
          } else {
            tma_load_2d(stage_b(stage), &tmB, full_bar(stage), kb * C::BK, nb * BN);
          }
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN > 256 ? 256 : BN, false, false);
      constexpr uint32_t idesc_rest = idesc_bf16_f32(128, BN > 256 ? BN - 256 : 64, false, false);
      // Descriptors are built once; a stage or K step only advances the start
      // address field (byte offset >> 4).
      const uint64_t da0 = sdesc_sw128(stage_a(0), 16, 1024);
      const uint64_t db0 = sdesc_sw128(stage_b(0), 16, 1024);
      int stage = 0, fills = 0;
      uint32_t phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, p.status)) {
            ok = false;
            break;
          }
          if constexpr (ASRC != kATma) {
            if (!mbar_wait(afull_bar(stage), phase, p.status)) {
              ok = false;
              break;
            }
            fence_proxy_async_smem();   // producer-written A -> tensor core reads
          }
          tc_fence_after();
          const uint64_t off = static_cast<uint64_t>(stage * (C::STAGE_BYTES >> 4));
#pragma unroll
          for (int k = 0; k < C::BK / 16; ++k) {
            umma_bf16(d_tmem, da0 + off + 2 * k, db0 + off + 2 * k, idesc, (kb | k) != 0);
            // Rows 256..BN-1 of B (32 KB on) into accumulator columns 256..BN-1.
            if constexpr (BN > 256)
              umma_bf16(d_tmem + 256, da0 + off + 2 * k, db0 + off + ((256 * 128) >> 4) + 2 * k, idesc_rest,
                        (kb | k) != 0);
          }
          umma_commit(empty_bar(stage));
          ++fills;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
        if (++acc == kAccs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      consumed_fills = fills;
      // All MMAs of this CTA complete before TMEM is released.
      umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, p.status);
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ A producers (warps 10-13)
    if constexpr (ASRC != kATma) {
      if constexpr (ASRC == kAMerge) {
        if (warp < 14)
          produce_a_merge<C>(g, p, smem, afull_bar(0), empty_bar(0), num_m, num_n, num_tiles, num_kb,
                             threadIdx.x - 320);
      } else {
        if (warp < 14)
          produce_a_pixels<C>(g, p, smem, afull_bar(0), empty_bar(0), num_m, num_n, num_tiles,
                              threadIdx.x - 320);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-7)
#define GEMM_FIRST_TILE blockIdx.x
#define GEMM_TILE_STEP gridDim.x
#define GEMM_ROW0 mb * C::BM + quad * 32
#define GEMM_RELEASE_ACC mbar_arrive(tempty_bar(acc))
#include "gemm_epilogue.inc"
#undef GEMM_FIRST_TILE
#undef GEMM_TILE_STEP
#undef GEMM_ROW0
#undef GEMM_RELEASE_ACC
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8 && lane == 0 && status_failed(p.status)) {
    // After a timeout: wait (bounded) for the tile loads still in flight, so no
    // TMA write lands in shared memory after the CTA has exited.
    for (int f = consumed_fills; f < issued_fills; ++f) {
      const int s = f % C::STAGES;
      if (!mbar_wait(full_bar(s), (f / C::STAGES) & 1, nullptr)) break;
    }
  }
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int EPI, int ASRC = kATma>
int launch_gemm_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                  const GemmParams& p, cudaStream_t stream, const AGenParams* g = nullptr,
                  const CUtensorMap* tmB64 = nullptr) {
  using C = GemmCfg<BN, ASRC>;
  if (allow_smem(reinterpret_cast<const void*>(gemm_kernel<BN, EPI, ASRC>), C::SMEM_BYTES) != cudaSuccess)
    return DS_VIT_ECUDA;
  const int tiles = ((p.M + 127) / 128) * (p.N / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  static const AGenParams none{};
  const cudaError_t e = launch_pdl(gemm_kernel<BN, EPI, ASRC>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES,
                                   stream, tmA, tmB, tmC, tmB64 ? *tmB64 : tmB, p, g ? *g : none);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encode;
}

bool encode_tmap(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode || !base || rows == 0 || cols == 0) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * 2) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t allow_smem(const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, cudaError_t> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  const auto it = done.find(key);
  if (it != done.end()) return it->second;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) cudaGetLastError();
  done[key] = e;
  return e;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  return encode_tmap(map, base, rows, cols, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_bf16_tail16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows) {
  return encode_tmap(map, base, rows, cols, 16, box_rows, CU_TENSOR_MAP_SWIZZLE_32B);
}

bool make_tmap_store_bf16(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols) {
  return encode_tmap(map, base, rows, cols, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

int gemm_bn(int M, int N) {
  const int tiles256 = ((M + 127) / 128) * (N / 256);
  return 4 * tiles256 < 3 * num_sms() ? 128 : 256;
}

bool make_weight_map(WeightMap* m, const void* w, uint64_t n, uint64_t k) {
  return make_tmap_bf16(&m->bn256, w, n, k, 256) && make_tmap_bf16(&m->bn128, w, n, k, 128) &&
         make_tmap_bf16(&m->bn64, w, n, k, 64) && make_tmap_bf16(&m->bn32, w, n, k, 32);
}

// 320-wide tiles where they fit one round and the 256-wide choice needs two
// or more (the merger linears at about a thousand tokens: 128 tiles against
// 160 one-CTA or 80 paired 256-wide ones on 152 SMs).
bool prefer_bn320(int M, int N) {
  if (N % 320 != 0 || gemm_bn(M, N) != 256) return false;
  const int sms = num_sms();
  const int tiles320 = ((M + 127) / 128) * (N / 320);
  const int tiles_pair = ((M + 255) / 256) * (N / 256);
  return tiles320 <= sms && tiles_pair > sms / 2;
}

// 288-wide tiles for widths that are a multiple of 288 but not of 256 (1152)
// where they fit one round: 128 tiles against 288 128-wide ones (two rounds)
// at 4096 rows, with 11 instead of 15 KB of operands per MFLOP.
bool prefer_bn288(int M, int N) {
  if (N % 288 != 0 || N % 256 == 0) return false;
  return ((M + 127) / 128) * (N / 288) <= num_sms();
}

int launch_gemm(const CUtensorMap& tmA, const WeightMap& B, const CUtensorMap& tmC, int M, int N,
                int K, const bf16* bias, bf16* out, int epi, const int* rowpos,
                const float* rope_cs, int* status, cudaStream_t stream) {
  if (M <= 0 || K <= 0 || K % 64 != 0 || N % 128 != 0) return DS_VIT_EINVAL;
  if ((epi == kEpiBias || epi == kEpiBiasGelu) && prefer_bn320(M, N)) {
    const GemmParams p{M, N, K, out, bias, rowpos, rope_cs, status, tile_order(M, K)};
    return epi == kEpiBias ? launch_gemm_t<320, kEpiBias>(tmA, B.bn256, tmC, p, stream, nullptr, &B.bn64)
                           : launch_gemm_t<320, kEpiBiasGelu>(tmA, B.bn256, tmC, p, stream, nullptr, &B.bn64);
  }
  // Where 256-wide tiles keep the SMs busy: 256 x 256 tiles on 2-CTA clusters
  // (a third less operand traffic per stage, six stages).
  if (N % 256 == 0 && gemm_bn(M, N) == 256) {
    const int rc = launch_gemm_pair(tmA, B.bn128, tmC, M, N, K, bias, out, epi, rowpos, rope_cs, status, stream);
    if (rc != kGemmNoPair) return rc;
  }
  GemmParams p{M, N, K, out, bias, rowpos, rope_cs, status, tile_order(M, K)};
  // SwiGLU pairs the gate and up halves of one 256-column tile (two 128-row B boxes).
  if (epi == kEpiSwiglu) {
    if (N % 256 != 0) return DS_VIT_EINVAL;
    return launch_gemm_t<256, kEpiSwiglu>(tmA, B.bn128, tmC, p, stream);
  }
  if ((epi == kEpiBias || epi == kEpiBiasGelu || epi == kEpiBiasResid) && prefer_bn288(M, N)) {
    switch (epi) {
      case kEpiBias: return launch_gemm_t<288, kEpiBias>(tmA, B.bn256, tmC, p, stream, nullptr, &B.bn32);
      case kEpiBiasGelu: return launch_gemm_t<288, kEpiBiasGelu>(tmA, B.bn256, tmC, p, stream, nullptr, &B.bn32);
      default: return launch_gemm_t<288, kEpiBiasResid>(tmA, B.bn256, tmC, p, stream, nullptr, &B.bn32);
    }
  }
  // Widths that are a multiple of 128 but not of 256 (1152) take 128-wide tiles.
  if (N % 256 != 0 || gemm_bn(M, N) == 128) {
    const CUtensorMap& tmB = B.bn128;
    switch (epi) {
      case kEpiBias: return launch_gemm_t<128, kEpiBias>(tmA, tmB, tmC, p, stream);
      case kEpiBiasGelu: return launch_gemm_t<128, kEpiBiasGelu>(tmA, tmB, tmC, p, stream);
      case kEpiBiasResid: return launch_gemm_t<128, kEpiBiasResid>(tmA, tmB, tmC, p, stream);
      case kEpiQkvRope: return launch_gemm_t<128, kEpiQkvRope>(tmA, tmB, tmC, p, stream);
      case kEpiQkvRope72: return launch_gemm_t<128, kEpiQkvRope72>(tmA, tmB, tmC, p, stream);
      default: return DS_VIT_EINVAL;
    }
  }
  const CUtensorMap& tmB = B.bn256;
  switch (epi) {
    case kEpiBias: return launch_gemm_t<256, kEpiBias>(tmA, tmB, tmC, p, stream);
    case kEpiBiasGelu: return launch_gemm_t<256, kEpiBiasGelu>(tmA, tmB, tmC, p, stream);
    case kEpiBiasResid: return launch_gemm_t<256, kEpiBiasResid>(tmA, tmB, tmC, p, stream);
    case kEpiQkvRope: return launch_gemm_t<256, kEpiQkvRope>(tmA, tmB, tmC, p, stream);
    case kEpiQkvRope72: return launch_gemm_t<256, kEpiQkvRope72>(tmA, tmB, tmC, p, stream);
    default: return DS_VIT_EINVAL;
  }
}

int launch_gemm_agen(int asrc, const AGenParams& g, const WeightMap& B, const CUtensorMap& tmC,
                     int M, int N, int K, const bf16* bias, bf16* out, int epi, int* status,
                     cudaStream_t stream) {
  if (M <= 0 || K % 64 != 0 || N % 256 != 0) return DS_VIT_EINVAL;
  if (!(asrc == kAPixels && K == kPatchK && epi == kEpiBias) &&
      !(asrc == kAMerge && K == 9216 && epi == kEpiBiasGelu))
    return DS_VIT_EINVAL;
  GemmParams p{M, N, K, out, bias, nullptr, nullptr, status, tile_order(M, K)};
  if (asrc == kAMerge && prefer_bn320(M, N))
    return launch_gemm_t<320, kEpiBiasGelu, kAMerge>(B.bn256, B.bn256, tmC, p, stream, &g, &B.bn64);
  const bool narrow = gemm_bn(M, N) == 128;
  const CUtensorMap& tmB = narrow ? B.bn128 : B.bn256;
  if (asrc == kAPixels)
    return narrow ? launch_gemm_t<128, kEpiBias, kAPixels>(tmB, tmB, tmC, p, stream, &g)
                  : launch_gemm_t<256, kEpiBias, kAPixels>(tmB, tmB, tmC, p, stream, &g);
  return narrow ? launch_gemm_t<128, kEpiBiasGelu, kAMerge>(tmB, tmB, tmC, p, stream, &g)
                : launch_gemm_t<256, kEpiBiasGelu, kAMerge>(tmB, tmB, tmC, p, stream, &g);
}

}  // namespace dsvit
