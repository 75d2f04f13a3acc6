// Bidirectional varlen flash attention on tcgen05 (head_dim 64).
//
// Each image's patches attend to every patch of the same image and to nothing
// else ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision",
// "Multimodal basics": attention gives each patch information from the whole
// image); images are packed row-wise and separated by their row offsets.
// Softmax scale 1/sqrt(64), no mask inside an image, no QK norm (ds4-learning
// glossary "vision", family table).
//
// One CTA = one (image, 256 query rows, head), as two 128-row query tiles A
// and B that share every K/V tile.  Warps 0-7 run the softmax of tile A and
// warps 8-15 that of tile B: a warp takes 16 query rows (TMEM lanes) with two
// threads per row, one per 64-key half of the score tile, read with one
// tcgen05.ld.red of the 16x32bx2 shape (threads t and t + 16 on the same
// lane, 64 columns apart) that also returns the half-row maximum; the two
// halves exchange their maxima and sums by warp shuffle.  Every SM
// sub-partition runs four softmax warps.  Warp 16 loads Q once and streams K/V
// tiles of 128 rows through a 4-stage TMA ring; warp 17 issues the MMAs of
// tile A and warp 18 those of tile B, so the two tiles proceed independently
// on the tensor core:
//   S_X = Q_X K_j^T     (M 128, N 128, K 64)  smem x smem -> TMEM
//   O_X += P_X V_j      (M 128, N 64,  K 128) TMEM x smem -> TMEM
// The softmax threads of a tile read S_X from TMEM and hand the buffer back at
// once, so the next S_X is computed while they work.  The exponents of the
// two tiles take turns (A of step j, B of step j, A of step j+1, ...: an
// mbarrier per tile and TMEM lane quadrant, so each SM sub-partition hands
// over on its own), so each sub-partition runs one tile's exponents at full
// rate while the tensor core works on the other tile; left to run together the
// two tiles fall into step and their math serialises with the MMAs (1.5x
// slower).  Only the exponents take the turn: the row maximum and rescale
// decision come before it, the row sums and bf16 packs after its hand-off.
// The running row maximum m
// (exp2 domain) is raised only when a tile's maximum exceeds it by more than
// 8, so P = exp2(s - m) stays below 2^8 and O is rescaled (in TMEM, by
// exp2(m_old - m_new)) rarely; the final O / l uses the same m, so the result
// is the exact softmax.  P is written as bf16 pairs into TMEM, where the PV
// MMA reads its A operand.
#include "internal.h"
#include "ptx.cuh"


namespace dsvit {

namespace {

constexpr int kTile = 128;     // rows of a query tile and of a K/V tile
constexpr int kHd = 64;        // head dim
constexpr int kStages = 4;     // K/V ring depth
constexpr int kQBytes = kTile * kHd * 2;              // 16 KB per query tile
constexpr int kKVBytes = kTile * kHd * 2;             // 16 KB each for K and V
constexpr int kOffQ = 0;                              // Q_A, Q_B
constexpr int kOffK = kOffQ + 2 * kQBytes;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffBar = kOffV + kStages * kKVBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,320), O_B [320,384),
// P_A [384,448), P_B [448,512) (P as packed bf16 pairs).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;
constexpr int kThreads = 608;         // 16 softmax warps, TMA warp, 2 MMA warps
constexpr int kWarpTma = 16;
constexpr int kWarpMma = 17;          // 17: tile A, 18: tile B
constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays below 2^8

// Barrier slots (8 bytes each).
enum : int {
  kBarQ = 0, kBarKvFull = 1, kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages,   // [2]
  kBarSFree = kBarSFull + 2,           // [2]
  kBarPFull = kBarSFree + 2,           // [2]
  kBarPvDone = kBarPFull + 2,          // [2]
  kBarDrain = kBarPvDone + 2,          // [2]
  kBarTurn = kBarDrain + 2,            // [2 tiles][4 quadrants]: the quadrant's warps of tile X
                                       // finished the math of a step
  kBarCount = kBarTurn + 8
};
static_assert(kBarCount <= 30, "barrier area");

struct AttnParams {
  AttnBatch b;
  bf16* out;
  int* status;
  float scale_log2;  // log2(e) / sqrt(64)
};

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Registers are split per SM sub-partition: with 19 warps five of them share
// one sub-partition's 16K registers, which caps a thread at 96 (allocation in
// units of 8).
__global__ void __maxnreg__(96)
    attn_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 31);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto sQ = [&](int x) { return smem_u32(smem + kOffQ + x * kQBytes); };
  auto sK = [&](int s) { return smem_u32(smem + kOffK + s * kKVBytes); };
  auto sV = [&](int s) { return smem_u32(smem + kOffV + s * kKVBytes); };

  // Which image / 256-row query block this CTA owns (launch order from the host).
  int slot = 0;
  while (slot + 1 < p.b.n_images && p.b.tile_start[slot + 1] <= static_cast<int>(blockIdx.x)) ++slot;
  const int img = p.b.order[slot];
  const int row0 = p.b.cu[img];
  const int len = p.b.cu[img + 1] - row0;
  const int q0 = row0 + (static_cast<int>(blockIdx.x) - p.b.tile_start[slot]) * (2 * kTile);
  const int n_kv = (len + kTile - 1) / kTile;
  const int head = blockIdx.y;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 2);      // released by both MMA warps
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kBarSFull + x), 1);
      mbar_init(bar(kBarSFree + x), 256);
      mbar_init(bar(kBarPFull + x), 256);
      mbar_init(bar(kBarPvDone + x), 1);
      mbar_init(bar(kBarDrain + x), 1);
      for (int q = 0; q < 4; ++q) mbar_init(bar(kBarTurn + 4 * x + q), 64);
    }
    fence_barrier_init();
  }
  if (warp == kWarpTma && lane == 0) prefetch_tensormap(&tm);
  if (warp == kWarpTma) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_launch();
  grid_dep_wait();

  __shared__ int kv_consumed[2];
  int kv_issued = 0;
  bool q_issued = false;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(kBarQ), 2 * kQBytes);
      tma_load_2d(sQ(0), &tm, bar(kBarQ), head * kHd, q0);
      tma_load_2d(sQ(1), &tm, bar(kBarQ), head * kHd, q0 + kTile);
      q_issued = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(bar(kBarKvEmpty + s), ((j / kStages) & 1) ^ 1, p.status)) break;
        mbar_expect_tx(bar(kBarKvFull + s), 2 * kKVBytes);
        tma_load_2d(sK(s), &tm, bar(kBarKvFull + s), 1024 + head * kHd, row0 + j * kTile);
        tma_load_2d(sV(s), &tm, bar(kBarKvFull + s), 2048 + head * kHd, row0 + j * kTile);
        ++kv_issued;
      }
    }
  } else if (warp >= kWarpMma) {
    // ------------------------------------------------------------ MMA issuer of tile X
    const int x = warp - kWarpMma;
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_o = idesc_bf16_f32(128, 64, false, true);   // V is MN-major
      const uint32_t tS = tmem + x * 128, tO = tmem + kTmemO + x * 64, tP = tmem + kTmemP + x * 64;
      int consumed = 0;
      // Descriptors are built once; a stage or K step only advances the start
      // address field (byte offset >> 4).
      const uint64_t dq = sdesc_sw128(sQ(x), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sK(0), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sV(0), kKVBytes, 1024);
      auto issue_s = [&](int j) {
        const uint64_t dk = dk0 + static_cast<uint64_t>((j % kStages) * (kKVBytes >> 4));
#pragma unroll
        for (int k = 0; k < kHd / 16; ++k) umma_bf16(tS, dq + 2 * k, dk + 2 * k, id_s, k != 0);
        umma_commit(bar(kBarSFull + x));
      };
      bool ok = mbar_wait(bar(kBarQ), 0, p.status) && mbar_wait(bar(kBarKvFull), 0, p.status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const uint32_t par = j & 1;
        if (j + 1 < n_kv) {
          // The next scores as soon as the softmax has read the current ones.
          if (!mbar_wait(bar(kBarKvFull + (j + 1) % kStages), ((j + 1) / kStages) & 1, p.status)) break;
          if (!mbar_wait(bar(kBarSFree + x), par, p.status)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(bar(kBarPFull + x), par, p.status)) break;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>((j % kStages) * (kKVBytes >> 4));
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          umma_bf16_ts(tO, tP + k * 8, dv + 128 * k, id_o, (j | k) != 0);   // 16 rows = 2048 B
        umma_commit(bar(kBarPvDone + x));
        umma_commit(bar(kBarKvEmpty + j % kStages));
        consumed = j + 1;
      }
      kv_consumed[x] = consumed;
      // All MMAs of this warp complete before TMEM is released.
      umma_commit(bar(kBarDrain + x));
      mbar_wait(bar(kBarDrain + x), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-15)
    const int x = warp >> 3;                 // query tile A (0) or B (1)
    const int qd = warp & 3;                 // TMEM lane quadrant
    const int base = qd * 32 + ((warp >> 2) & 1) * 16;   // the warp's first row
    const int h = lane >> 4;                 // 64-key half of the score tile
    const int r = base + (lane & 15);        // row inside the tile == TMEM lane
    // Addresses of the first half; the 16x32bx2 accesses put threads 16-31
    // on the second (64 score columns, 32 O and P columns further on).
    const uint32_t lane_sel = static_cast<uint32_t>(base) << 16;
    const uint32_t tS = tmem + x * 128 + lane_sel;
    const uint32_t tO = tmem + kTmemO + x * 64 + lane_sel;
    const uint32_t tP = tmem + kTmemP + x * 64 + lane_sel;
    const float c = p.scale_log2;
    const uint64_t c2 = f2(c, c);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const uint32_t par = j & 1;
      if (!mbar_wait(bar(kBarSFull + x), par, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      // One load of the 64 scores that also reduces them to their maximum.
      float m_half = tmem_ld64_max_x2<64>(tS, sr);
      tmem_wait_ld();
      m_half = tmem_after_wait(m_half);
      tc_fence_before();
      mbar_arrive(bar(kBarSFree + x));       // the MMA may overwrite S_X now
      const int kv_valid = len - j * kTile - h * 64;
      if (kv_valid < 64) {
        // Keys past the image: masked, and the maximum taken over the rest.
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          if (i >= kv_valid) sr[i] = __float_as_uint(-INFINITY);
          mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(sr[i]));
        }
        m_half = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
      }
      // The row's maximum (a shuffle with the other half's thread) and the
      // rescale decision need no turn: only the exponent loop takes turns.
      const float m_other = __shfl_xor_sync(0xFFFFFFFFu, m_half, 16);
      // Both threads of the row derive the same m_new and alpha.
      const float m_tile = fmaxf(m_half, m_other) * c;
      float m_new = m, alpha = 1.f;
      if (m_tile > m + kRescaleThreshold) {   // always true on the first tile (m = -inf)
        m_new = m_tile;
        alpha = ex2_approx(m - m_new);
      }
      // Take turns: A's step j after B's step j-1, B's step j after A's step j.
      if (x == 1 || j > 0) {
        if (!mbar_wait(bar(kBarTurn + 4 * (x ^ 1) + qd), (x == 1 ? j : j - 1) & 1, p.status)) {
          ok = false;
          break;
        }
      }
      const uint64_t nm2 = f2(-m_new, -m_new);
      // Only the exponents take the turn; the sums and bf16 packs follow it.
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint64_t t = f2_fma(f2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), c2, nm2);
        float t0, t1;
        f2_split(t, t0, t1);
        sr[2 * i] = __float_as_uint(ex2_approx(t0));
        sr[2 * i + 1] = __float_as_uint(ex2_approx(t1));
      }
      mbar_arrive(bar(kBarTurn + 4 * x + qd));   // the other tile's turn on this sub-partition
      uint64_t acc[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = __uint_as_float(sr[2 * i]), p1 = __uint_as_float(sr[2 * i + 1]);
        acc[i & 3] = f2_add(acc[i & 3], f2(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      const uint64_t s2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      float s0, s1;
      f2_split(s2, s0, s1);
      l = l * alpha + (s0 + s1);              // this half's share of the row sum
      if (j > 0) {
        // PV_X of the previous tile must be done: it read P_X, and O_X is rescaled below.
        if (!mbar_wait(bar(kBarPvDone + x), par ^ 1, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32_x2<32>(tP, pk);
      if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        uint32_t o[32];
        tmem_ld32_x2<32>(tO, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32_x2<32>(tO, o);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + x));
      m = m_new;
    }
    const float l_other = __shfl_xor_sync(0xFFFFFFFFu, l, 16);
    if (ok && mbar_wait(bar(kBarPvDone + x), (n_kv - 1) & 1, p.status)) {
      tc_fence_after();
      const float inv_l = 1.f / (l + l_other);
      uint32_t o[32];
      tmem_ld32_x2<32>(tO, o);
      tmem_wait_ld();
      const int qrow = q0 + x * kTile + r;
      if (qrow < row0 + len) {
        uint4* dst =
            reinterpret_cast<uint4*>(p.out + static_cast<size_t>(qrow) * 1024 + head * kHd + h * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dst[q] = make_uint4(
              pack_bf16x2(__uint_as_float(o[q * 8 + 0]) * inv_l, __uint_as_float(o[q * 8 + 1]) * inv_l),
              pack_bf16x2(__uint_as_float(o[q * 8 + 2]) * inv_l, __uint_as_float(o[q * 8 + 3]) * inv_l),
              pack_bf16x2(__uint_as_float(o[q * 8 + 4]) * inv_l, __uint_as_float(o[q * 8 + 5]) * inv_l),
              pack_bf16x2(__uint_as_float(o[q * 8 + 6]) * inv_l, __uint_as_float(o[q * 8 + 7]) * inv_l));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpTma && lane == 0 && status_failed(p.status)) {
    // After a timeout: wait (bounded) for the loads still in flight, so no TMA
    // write lands in shared memory after the CTA has exited.
    if (q_issued) mbar_wait(bar(kBarQ), 0, nullptr);
    const int done = kv_consumed[0] < kv_consumed[1] ? kv_consumed[0] : kv_consumed[1];
    for (int j = done; j < kv_issued; ++j)
      if (!mbar_wait(bar(kBarKvFull + j % kStages), (j / kStages) & 1, nullptr)) break;
  }
  __syncthreads();
  if (warp == kWarpTma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_attention(const CUtensorMap& tm_qkv, const AttnBatch& batch, bf16* out, int* status,
                     cudaStream_t stream) {
  if (allow_smem(reinterpret_cast<const void*>(attn_kernel), kSmemBytes) != cudaSuccess) return DS_VIT_ECUDA;
  AttnParams p;
  p.b = batch;
  p.out = out;
  p.status = status;
  p.scale_log2 = 1.4426950408889634f * 0.125f;
  const int ctas = batch.tile_start[batch.n_images];
  if (ctas <= 0) return DS_VIT_OK;
  const cudaError_t e = launch_pdl(attn_kernel, dim3(ctas, 16), dim3(kThreads), kSmemBytes, stream, tm_qkv, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

}  // namespace dsvit
