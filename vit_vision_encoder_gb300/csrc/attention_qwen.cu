// Bidirectional attention of the Qwen3-VL-style tower ("DeepSeek V4.1 Flash
// Engineering, Part 3: Integrating Vision", comparison table: hidden 1,152,
// 16 heads -> head_dim 72) on tcgen05.
//
// The QKV projection writes every head padded to 128 columns (dims 72..127
// zero), so each Q/K/V head tile is two 128-byte-swizzled 64-column atoms and
// the MMAs use the same descriptor forms as the head-64 kernel:
//   S = Q K^T   (M 128, N 128, K 80: four K steps in atom 0, one in atom 1;
//                dims 80..127 are zero and skipped)
//   O += P V    (M 128, N 64 per atom, K 128: P from TMEM, V MN-major)
// One CTA = (128 query rows, head); warps 0-7 softmax with two threads per
// row (one per 64-key half, half-row maxima and sums exchanged through shared
// memory), warp 8 loads Q once and streams K/V through a 2-stage TMA ring,
// warp 9 issues the MMAs.  TMEM: S [0,128), O [128,256), P [256,320).
// Softmax scale 1/sqrt(72); the running maximum is raised only when it grows
// by more than 8 (log2 units), as in the head-64 kernel.  The output keeps
// the 72 real dims: out[row, head*72 + d].
#include "internal.h"
#include "ptx.cuh"

#include <mutex>

namespace dsvit {

namespace {

constexpr int kTile = 128;
constexpr int kHdPad = 128;                        // padded head width in qkv
constexpr int kHd = 72;                            // real head dims
constexpr int kStages = 2;
constexpr int kAtomBytes = kTile * 64 * 2;         // 16 KB: 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kAtomBytes;         // Q, K or V tile of one head
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 128;
constexpr uint32_t kTmemP = 256;
constexpr int kThreads = 320;                      // 8 softmax warps, TMA warp, MMA warp
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr float kRescaleThreshold = 8.f;

enum : int {
  kBarQ = 0, kBarKvFull = 1, kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages, kBarSFree, kBarPFull, kBarPvDone, kBarDrain,
  kBarXch,                                         // [4 quadrants]
  kBarCount = kBarXch + 4
};
static_assert(kBarCount <= 30, "barrier area");

struct QwenAttnParams {
  int n;            // rows of the image
  int qkv_cols;     // 3 * 16 * 128
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
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_pad128_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ QwenAttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 31);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  const uint32_t sQ = smem_u32(smem + kOffQ);
  auto sK = [&](int s) { return smem_u32(smem + kOffK + s * kTileBytes); };
  auto sV = [&](int s) { return smem_u32(smem + kOffV + s * kTileBytes); };

  const int q0 = static_cast<int>(blockIdx.x) * kTile;
  const int head = blockIdx.y;
  const int len = p.n;
  const int n_kv = (len + kTile - 1) / kTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 256);
    mbar_init(bar(kBarPFull), 256);
    mbar_init(bar(kBarPvDone), 1);
    mbar_init(bar(kBarDrain), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(kBarXch + q), 64);
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

  __shared__ int kv_consumed;
  __shared__ float xch[2][2][kTile];     // [parity][half][row]
  int kv_issued = 0;
  bool q_issued = false;
  const int colq = head * kHdPad, colk = 16 * kHdPad + head * kHdPad, colv = 32 * kHdPad + head * kHdPad;

  if (warp == kWarpTma) {
    if (lane == 0) {
      mbar_expect_tx(bar(kBarQ), kTileBytes);
      tma_load_2d(sQ, &tm, bar(kBarQ), colq, q0);
      tma_load_2d(sQ + kAtomBytes, &tm, bar(kBarQ), colq + 64, q0);
      q_issued = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(bar(kBarKvEmpty + s), ((j / kStages) & 1) ^ 1, p.status)) break;
        mbar_expect_tx(bar(kBarKvFull + s), 2 * kTileBytes);
        tma_load_2d(sK(s), &tm, bar(kBarKvFull + s), colk, j * kTile);
        tma_load_2d(sK(s) + kAtomBytes, &tm, bar(kBarKvFull + s), colk + 64, j * kTile);
        tma_load_2d(sV(s), &tm, bar(kBarKvFull + s), colv, j * kTile);
        tma_load_2d(sV(s) + kAtomBytes, &tm, bar(kBarKvFull + s), colv + 64, j * kTile);
        ++kv_issued;
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_o = idesc_bf16_f32(128, 64, false, true);   // V is MN-major
      const uint32_t tS = tmem, tO = tmem + kTmemO, tP = tmem + kTmemP;
      int consumed = 0;
      auto issue_s = [&](int j) {
        const uint32_t kb = sK(j % kStages);
        // K steps of 16 dims: 0..3 in atom 0, step 4 (dims 64..79) in atom 1.
#pragma unroll
        for (int k = 0; k < 5; ++k) {
          const uint32_t off = (k < 4 ? k * 32 : kAtomBytes);
          umma_bf16(tS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), id_s, k != 0);
        }
        umma_commit(bar(kBarSFull));
      };
      bool ok = mbar_wait(bar(kBarQ), 0, p.status) && mbar_wait(bar(kBarKvFull), 0, p.status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const uint32_t par = j & 1;
        if (j + 1 < n_kv) {
          if (!mbar_wait(bar(kBarKvFull + (j + 1) % kStages), ((j + 1) / kStages) & 1, p.status)) break;
          if (!mbar_wait(bar(kBarSFree), par, p.status)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(bar(kBarPFull), par, p.status)) break;
        tc_fence_after();
        const uint32_t vb = sV(j % kStages);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)     // 16 keys = 2048 B of an atom
            umma_bf16_ts(tO + 64 * a, tP + k * 8, sdesc_sw128(vb + a * kAtomBytes + 2048 * k, kAtomBytes, 1024),
                         id_o, (j | k) != 0);
        }
        umma_commit(bar(kBarPvDone));
        umma_commit(bar(kBarKvEmpty + j % kStages));
        consumed = j + 1;
      }
      kv_consumed = consumed;
      umma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int qd = warp & 3;                 // TMEM lane quadrant
    const int h = warp >> 2;                 // 64-key half of the score tile
    const int r = qd * 32 + lane;
    const uint32_t lane_sel = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t tS = tmem + h * 64 + lane_sel;
    const uint32_t tO = tmem + kTmemO + h * 64 + lane_sel;
    const uint32_t tP = tmem + kTmemP + h * 32 + lane_sel;
    const uint32_t xbar = bar(kBarXch + qd);
    auto exchange = [&](float v, int e, float* other) {
      xch[e & 1][h][r] = v;
      mbar_arrive(xbar);
      if (!mbar_wait(xbar, e & 1, p.status)) return false;
      *other = xch[e & 1][h ^ 1][r];
      return true;
    };
    const float c = p.scale_log2;
    const uint64_t c2 = f2(c, c);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const uint32_t par = j & 1;
      if (!mbar_wait(bar(kBarSFull), par, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(sr));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(kBarSFree));
      const int kv_valid = len - j * kTile - h * 64;
      if (kv_valid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= kv_valid) sr[i] = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint32_t* v = sr + 16 * g;
        float a = max3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
        a = max3(a, __uint_as_float(v[3]), __uint_as_float(v[4]));
        a = max3(a, __uint_as_float(v[5]), __uint_as_float(v[6]));
        a = max3(a, __uint_as_float(v[7]), __uint_as_float(v[8]));
        a = max3(a, __uint_as_float(v[9]), __uint_as_float(v[10]));
        a = max3(a, __uint_as_float(v[11]), __uint_as_float(v[12]));
        a = max3(a, __uint_as_float(v[13]), __uint_as_float(v[14]));
        mx[g] = fmaxf(a, __uint_as_float(v[15]));
      }
      const float m_half = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
      float m_other;
      if (!exchange(m_half, j, &m_other)) {
        ok = false;
        break;
      }
      const float m_tile = fmaxf(m_half, m_other) * c;
      float m_new = m, alpha = 1.f;
      if (m_tile > m + kRescaleThreshold) {
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
      const uint64_t s2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      float s0, s1;
      f2_split(s2, s0, s1);
      l = l * alpha + (s0 + s1);
      if (j > 0) {
        if (!mbar_wait(bar(kBarPvDone), par ^ 1, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tP, pk);
      if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t o[32];
          tmem_ld32(tO + q * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + q * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
      m = m_new;
    }
    float l_other = 0.f;
    if (ok && exchange(l, n_kv, &l_other) && mbar_wait(bar(kBarPvDone), (n_kv - 1) & 1, p.status)) {
      tc_fence_after();
      const float inv_l = 1.f / (l + l_other);
      // Thread h = 0 writes dims 0..39, h = 1 dims 40..71.
      const uint32_t tOall = tmem + kTmemO + lane_sel;
      uint32_t o[40];
      if (h == 0) {
        tmem_ld32(tOall, *reinterpret_cast<uint32_t(*)[32]>(o));
        tmem_ld8(tOall + 32, *reinterpret_cast<uint32_t(*)[8]>(o + 32));
      } else {
        tmem_ld32(tOall + 40, *reinterpret_cast<uint32_t(*)[32]>(o));
      }
      tmem_wait_ld();
      const int qrow = q0 + r;
      if (qrow < len) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(qrow) * (16 * kHd) + head * kHd + h * 40);
        const int nq = h == 0 ? 5 : 4;
#pragma unroll
        for (int q = 0; q < 5; ++q) {
          if (q < nq)
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
    if (q_issued) mbar_wait(bar(kBarQ), 0, nullptr);
    for (int j = kv_consumed; j < kv_issued; ++j)
      if (!mbar_wait(bar(kBarKvFull + j % kStages), (j / kStages) & 1, nullptr)) break;
  }
  __syncthreads();
  if (warp == kWarpTma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_attention_pad128(const CUtensorMap& tm_qkv, int n, bf16* out, int* status, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_pad128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return DS_VIT_ECUDA;
  if (n <= 0) return DS_VIT_OK;
  QwenAttnParams p;
  p.n = n;
  p.qkv_cols = 48 * kHdPad;
  p.out = out;
  p.status = status;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / 8.48528137423857);   // log2(e) / sqrt(72)
  const cudaError_t e = launch_pdl(attn_pad128_kernel, dim3((n + kTile - 1) / kTile, 16), dim3(kThreads),
                                   kSmemBytes, stream, tm_qkv, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

}  // namespace dsvit
