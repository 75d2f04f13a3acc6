// Bidirectional attention of the Qwen3-VL-style tower ("DeepSeek V4.1 Flash
// Engineering, Part 3: Integrating Vision", comparison table: hidden 1,152,
// 16 heads -> head_dim 72) on tcgen05.
//
// The QKV projection writes every head 80 columns wide (dims 72..79 zero:
// the MMA's N and K come in steps of 16).  A Q or K head tile of 128 rows is
// loaded as two TMA boxes: columns 0..63 as a 128-byte-swizzled atom (16 KB)
// and columns 64..79 as a 32-byte-swizzled tail atom (4 KB).  A V tile is two
// 128-byte-swizzled atoms of 64 columns: the second holds dims 64..79 and the
// next head's first 48 columns (zero fill past the last head), of which the
// MMA reads only the first 16:
//   S_X = Q_X K_j^T  (M 128, N 128, K 80: four K steps in the atom, one in the tail)
//   O_X += P_X V_j   (M 128, N 80 across the two V atoms, K 128; P from TMEM,
//                     V MN-major)
// (Measured on GB300: a separate N = 16 MMA for dims 64..79 cost as much as
// a third of the kernel; one N = 80 MMA per K step does not.)
//
// The schedule is the head-64 kernel's: one CTA = (256 query rows, head) as
// two 128-row tiles A and B that share every K/V tile; warps 0-7 run the
// softmax of tile A and warps 8-15 that of tile B, each warp 16 query rows
// with two threads per row (one per 64-key half, threads t and t + 16 through
// the 16x32bx2 TMEM shape, half-row maxima and sums exchanged by warp
// shuffle); the exponent math of the two tiles takes turns; warp 16 loads Q
// once and streams K/V through a 3-stage TMA ring; warps 17 and 18 issue the
// MMAs of tiles A and B.  The running maximum is raised only when it grows by
// more than 8 (log2 units); the final O / l uses the same maximum, so the
// result is the exact softmax.  Softmax scale 1/sqrt(72).
//
// TMEM: S_A [0,128), S_B [128,256), O_A [256,336), O_B [384,464), and one P
// buffer (bf16 pairs) that the two tiles share: keys 0..63 at [336,368), keys
// 64..127 at [464,496).  Two 80-wide O accumulators leave no room for a P per
// tile, but the tiles' exponent math already takes turns (A0 B0 A1 B1 ...),
// so each tile writes P after the other tile's PV MMA that read the previous
// P has completed; the scores stay double-buffered against the softmax as in
// the head-64 kernel (the MMA computes S_X(j+1) once the softmax has loaded
// S_X(j)).  The output keeps the 72 real dims: out[row, head*72 + d].
#include "internal.h"
#include "ptx.cuh"


namespace dsvit {

namespace {

constexpr int kTile = 128;
constexpr int kHdPad = 80;                         // head width in qkv
constexpr int kHd = 72;                            // real head dims
constexpr int kHeads = 16;
constexpr int kStages = 3;
constexpr int kAtomBytes = kTile * 64 * 2;         // 16 KB: 128 rows x 64 bf16
constexpr int kTailBytes = kTile * 16 * 2;         // 4 KB: 128 rows x 16 bf16
constexpr int kTileBytes = kAtomBytes + kTailBytes;  // Q or K tile
constexpr int kVBytes = 2 * kAtomBytes;            // V tile
constexpr int kOffQ = 0;                           // Q_A, Q_B
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kVBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kTileBytes % 1024 == 0, "tiles stay 1024-byte aligned");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;                   // O_X at 256 + 128 X
constexpr uint32_t kTmemP0 = 336, kTmemP1 = 464;   // P keys 0..63, 64..127
constexpr int kThreads = 608;                      // 16 softmax warps, TMA warp, 2 MMA warps
constexpr int kWarpTma = 16;
constexpr int kWarpMma = 17;                       // 17: tile A, 18: tile B
constexpr float kRescaleThreshold = 8.f;

enum : int {
  kBarQ = 0, kBarKvFull = 1, kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages,   // [2]
  kBarSFree = kBarSFull + 2,           // [2]
  kBarPFull = kBarSFree + 2,           // [2]
  kBarPvDone = kBarPFull + 2,          // [2]
  kBarDrain = kBarPvDone + 2,          // [2]
  kBarTurn = kBarDrain + 2,            // [2]
  kBarCount = kBarTurn + 2
};
static_assert(kBarCount <= 30, "barrier area");

struct QwenAttnParams {
  int n;            // rows of the image
  bf16* out;        // [n, 16 * 72]
  int* status;
  float scale_log2;
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

// 19 warps: five share one SM sub-partition's 16K registers, so 96 a thread.
__global__ void __maxnreg__(96)
    attn_hd72_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tm_tail,
                     const __grid_constant__ QwenAttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 31);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto sQ = [&](int x) { return smem_u32(smem + kOffQ + x * kTileBytes); };
  auto sK = [&](int s) { return smem_u32(smem + kOffK + s * kTileBytes); };
  auto sV = [&](int s) { return smem_u32(smem + kOffV + s * kVBytes); };

  const int q0 = static_cast<int>(blockIdx.x) * (2 * kTile);
  const int head = blockIdx.y;
  const int len = p.n;
  const int n_kv = (len + kTile - 1) / kTile;
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
      mbar_init(bar(kBarTurn + x), 256);
    }
    fence_barrier_init();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tensormap(&tm);
    prefetch_tensormap(&tm_tail);
  }
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
  const int colq = head * kHdPad, colk = (kHeads + head) * kHdPad, colv = (2 * kHeads + head) * kHdPad;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(bar(kBarQ), 2 * kTileBytes);
      for (int x = 0; x < 2; ++x) {
        tma_load_2d(sQ(x), &tm, bar(kBarQ), colq, q0 + x * kTile);
        tma_load_2d(sQ(x) + kAtomBytes, &tm_tail, bar(kBarQ), colq + 64, q0 + x * kTile);
      }
      q_issued = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(bar(kBarKvEmpty + s), ((j / kStages) & 1) ^ 1, p.status)) break;
        mbar_expect_tx(bar(kBarKvFull + s), kTileBytes + kVBytes);
        tma_load_2d(sK(s), &tm, bar(kBarKvFull + s), colk, j * kTile);
        tma_load_2d(sK(s) + kAtomBytes, &tm_tail, bar(kBarKvFull + s), colk + 64, j * kTile);
        tma_load_2d(sV(s), &tm, bar(kBarKvFull + s), colv, j * kTile);
        tma_load_2d(sV(s) + kAtomBytes, &tm, bar(kBarKvFull + s), colv + 64, j * kTile);
        ++kv_issued;
      }
    }
  } else if (warp >= kWarpMma) {
    // ------------------------------------------------------------ MMA issuer of tile X
    const int x = warp - kWarpMma;
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_o = idesc_bf16_f32(128, 80, false, true);   // V is MN-major
      const uint32_t tS = tmem + x * 128, tO = tmem + kTmemO + x * 128;
      int consumed = 0;
      // Descriptors are built once; a stage or K step only advances the start
      // address field (byte offset >> 4).
      const uint64_t dq = sdesc_sw128(sQ(x), 16, 1024);
      const uint64_t dq_tail = sdesc_sw32(sQ(x) + kAtomBytes, 16, 256);
      const uint64_t dk0 = sdesc_sw128(sK(0), 16, 1024);
      const uint64_t dk0_tail = sdesc_sw32(sK(0) + kAtomBytes, 16, 256);
      // V: 8-key groups 1024 B apart, the two 64-column atoms kAtomBytes apart.
      const uint64_t dv0 = sdesc_sw128(sV(0), kAtomBytes, 1024);
      auto issue_s = [&](int j) {
        const uint64_t st = static_cast<uint64_t>((j % kStages) * (kTileBytes >> 4));
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_bf16(tS, dq + 2 * k, dk0 + st + 2 * k, id_s, k != 0);
        umma_bf16(tS, dq_tail, dk0_tail + st, id_s, 1u);
        umma_commit(bar(kBarSFull + x));
      };
      bool ok = mbar_wait(bar(kBarQ), 0, p.status) && mbar_wait(bar(kBarKvFull), 0, p.status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          // The next scores as soon as the softmax has read the current ones.
          if (!mbar_wait(bar(kBarKvFull + (j + 1) % kStages), ((j + 1) / kStages) & 1, p.status)) break;
          if (!mbar_wait(bar(kBarSFree + x), j & 1, p.status)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(bar(kBarPFull + x), j & 1, p.status)) break;
        tc_fence_after();
        const uint64_t sv = static_cast<uint64_t>((j % kStages) * (kVBytes >> 4));
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          // Keys 16k..16k+15 (2048 B of each V atom): columns 8 (k % 4) of P half k / 4.
          const uint32_t a = tmem + (k < 4 ? kTmemP0 : kTmemP1) + (k & 3) * 8;
          umma_bf16_ts(tO, a, dv0 + sv + 128 * k, id_o, (j | k) != 0);
        }
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
    const int r = base + (lane & 15);
    // Addresses of the first half; the 16x32bx2 accesses put threads 16-31 on
    // the second: scores 64 columns on, P 128 (kTmemP1 - kTmemP0), O 40 (the
    // first half owns O columns 0..39, the second 40..71; 72..79 stay zero).
    const uint32_t lane_sel = static_cast<uint32_t>(base) << 16;
    const uint32_t tS = tmem + x * 128 + lane_sel;
    const uint32_t tO = tmem + kTmemO + x * 128 + lane_sel;
    const uint32_t tP = tmem + kTmemP0 + lane_sel;
    static_assert(kTmemP1 - kTmemP0 == 128, "P halves 128 columns apart");
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
      // Take turns: A's step j after B's step j-1, B's step j after A's step j.
      if (x == 1 || j > 0) {
        if (!mbar_wait(bar(kBarTurn + (x ^ 1)), (x == 1 ? j : j - 1) & 1, p.status)) {
          ok = false;
          break;
        }
      }
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
      const float m_other = __shfl_xor_sync(0xFFFFFFFFu, m_half, 16);
      const float m_tile = fmaxf(m_half, m_other) * c;
      float m_new = m, alpha = 1.f;
      if (m_tile > m + kRescaleThreshold) {   // always true on the first tile (m = -inf)
        m_new = m_tile;
        alpha = ex2_approx(m - m_new);
      }
      const uint64_t nm2 = f2(-m_new, -m_new);
      uint64_t acc[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint64_t t = f2_fma(f2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), c2, nm2);
        float t0, t1;
        f2_split(t, t0, t1);
        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
        acc[i & 3] = f2_add(acc[i & 3], f2(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      mbar_arrive(bar(kBarTurn + x));         // the other tile's turn
      const uint64_t s2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      float s0, s1;
      f2_split(s2, s0, s1);
      l = l * alpha + (s0 + s1);              // this half's share of the row sum
      // O_X is rescaled below: its previous PV MMA must be done.  P is
      // rewritten: the PV MMA that read the last P (B's step j-1 before A's
      // step j, A's step j before B's step j) must be done.
      if (j > 0 && !mbar_wait(bar(kBarPvDone + x), par ^ 1, p.status)) {
        ok = false;
        break;
      }
      if ((x == 1 || j > 0) && !mbar_wait(bar(kBarPvDone + (x ^ 1)), (x == 1 ? j : j - 1) & 1, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32_x2<128>(tP, pk);
      if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        // Half h rescales O columns [40 h, 40 h + 32) and then [40 h + 32,
        // 40 h + 40) (for h = 1 columns 72..79, which stay zero).
        uint32_t o[32];
        tmem_ld32_x2<40>(tO, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32_x2<40>(tO, o);
        uint32_t o8[8];
        tmem_ld8_x2<40>(tO + 32, o8);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) o8[i] = __float_as_uint(__uint_as_float(o8[i]) * alpha);
        tmem_st8_x2<40>(tO + 32, o8);
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
      // Thread h = 0 writes dims 0..39, h = 1 dims 40..71: 32 columns, then
      // (h = 0) the 8 columns 32..39.
      const int qrow = q0 + x * kTile + r;
      uint4* dst =
          reinterpret_cast<uint4*>(p.out + static_cast<size_t>(qrow) * (kHeads * kHd) + head * kHd + h * 40);
      auto put8 = [&](uint4* d, const uint32_t* o) {
        *d = make_uint4(pack_bf16x2(__uint_as_float(o[0]) * inv_l, __uint_as_float(o[1]) * inv_l),
                        pack_bf16x2(__uint_as_float(o[2]) * inv_l, __uint_as_float(o[3]) * inv_l),
                        pack_bf16x2(__uint_as_float(o[4]) * inv_l, __uint_as_float(o[5]) * inv_l),
                        pack_bf16x2(__uint_as_float(o[6]) * inv_l, __uint_as_float(o[7]) * inv_l));
      };
      {
        uint32_t o[32];
        tmem_ld32_x2<40>(tO, o);
        tmem_wait_ld();
        if (qrow < len) {
#pragma unroll
          for (int q = 0; q < 4; ++q) put8(dst + q, o + 8 * q);
        }
      }
      {
        uint32_t o[8];
        tmem_ld8_x2<40>(tO + 32, o);         // h = 1: columns 72..79, not written
        tmem_wait_ld();
        if (h == 0 && qrow < len) put8(dst + 4, o);
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

int launch_attention_hd72(const CUtensorMap& tm_qkv, const CUtensorMap& tm_qkv_tail, int n, bf16* out,
                          int* status, cudaStream_t stream) {
  if (allow_smem(reinterpret_cast<const void*>(attn_hd72_kernel), kSmemBytes) != cudaSuccess) return DS_VIT_ECUDA;
  if (n <= 0) return DS_VIT_OK;
  QwenAttnParams p;
  p.n = n;
  p.out = out;
  p.status = status;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / 8.48528137423857);   // log2(e) / sqrt(72)
  const cudaError_t e = launch_pdl(attn_hd72_kernel, dim3((n + 2 * kTile - 1) / (2 * kTile), kHeads),
                                   dim3(kThreads), kSmemBytes, stream, tm_qkv, tm_qkv_tail, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

}  // namespace dsvit
