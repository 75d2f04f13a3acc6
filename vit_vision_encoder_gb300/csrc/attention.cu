// Bidirectional varlen flash attention on tcgen05 (head_dim 64).
//
// Each image's patches attend to every patch of the same image and to nothing
// else ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision",
// "Multimodal basics": attention gives each patch information from the whole
// image); images are packed row-wise and separated by their row offsets.
// Softmax scale 1/sqrt(64), no mask inside an image, no QK norm (ds4-learning
// glossary "vision", family table).
//
// One CTA = one (image, 128-row query tile, head).  Warps 0-3 own one query
// row per thread (TMEM lane = row); warp 4 loads Q once and streams K/V tiles
// of 128 rows through a 3-stage TMA ring; warp 5 issues the MMAs:
//   S_j = Q K_j^T          (M 128, N 128, K 64)  -> TMEM, double-buffered
//   O  += P_j V_j          (M 128, N 64,  K 128) -> TMEM
// The softmax warps read S_j from TMEM, keep the running row max m and sum l
// in registers (exp2 domain), write P_j = exp2(s - m) as bf16 into a
// 128-byte-swizzled shared tile (the MMA's A operand), and rescale O in TMEM
// by exp2(m_old - m_new) when the max grows.  S_{j+1} is computed while the
// softmax of tile j runs.  Final O / l is written as bf16.
#include "internal.h"
#include "ptx.cuh"

#include <mutex>

namespace dsvit {

namespace {

constexpr int kTile = 128;     // query rows per CTA and key rows per K/V tile
constexpr int kHd = 64;        // head dim
constexpr int kStages = 3;     // K/V ring depth
constexpr int kQBytes = kTile * kHd * 2;              // 16 KB
constexpr int kKVBytes = kTile * kHd * 2;             // 16 KB each for K and V
constexpr int kPBytes = kTile * kTile * 2;            // 32 KB (two 64-column chunks)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffV = kOffK + kStages * kKVBytes;
constexpr int kOffP = kOffV + kStages * kKVBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kTmemCols = 512;   // S0 [0,128), S1 [128,256), O [256,320)
constexpr uint32_t kTmemO = 256;

struct AttnParams {
  AttnBatch b;
  bf16* out;
  int* status;
  float scale_log2;  // log2(e) / sqrt(64)
};

__global__ void __launch_bounds__(192, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + kStages + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (1 + 2 * kStages + b); };
  const uint32_t p_full = bar0 + 8u * (3 + 2 * kStages);
  const uint32_t pv_done = bar0 + 8u * (4 + 2 * kStages);
  const uint32_t drain = bar0 + 8u * (5 + 2 * kStages);
  const uint32_t sQ = smem_u32(smem + kOffQ);
  auto sK = [&](int s) { return smem_u32(smem + kOffK + s * kKVBytes); };
  auto sV = [&](int s) { return smem_u32(smem + kOffV + s * kKVBytes); };
  auto sP = [&](int b) { return smem_u32(smem + kOffP + b * kPBytes); };

  // Which image / query tile this CTA owns (launch order from the host).
  int slot = 0;
  while (slot + 1 < p.b.n_images && p.b.tile_start[slot + 1] <= static_cast<int>(blockIdx.x)) ++slot;
  const int img = p.b.order[slot];
  const int row0 = p.b.cu[img];
  const int len = p.b.cu[img + 1] - row0;
  const int q0 = row0 + (static_cast<int>(blockIdx.x) - p.b.tile_start[slot]) * kTile;
  const int q_valid = min(kTile, row0 + len - q0);
  const int n_kv = (len + kTile - 1) / kTile;
  const int head = blockIdx.y;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(s_full(0), 1);
    mbar_init(s_full(1), 1);
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) prefetch_tensormap(&tm);
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  __shared__ int kv_consumed;
  int kv_issued = 0;
  bool q_issued = false;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_expect_tx(q_full, kQBytes);
      tma_load_2d(sQ, &tm, q_full, head * kHd, q0);
      q_issued = true;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(kv_empty(s), ((j / kStages) & 1) ^ 1, p.status)) break;
        mbar_expect_tx(kv_full(s), 2 * kKVBytes);
        tma_load_2d(sK(s), &tm, kv_full(s), 1024 + head * kHd, row0 + j * kTile);
        tma_load_2d(sV(s), &tm, kv_full(s), 2048 + head * kHd, row0 + j * kTile);
        ++kv_issued;
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_o = idesc_bf16_f32(128, 64, false, true);   // V is MN-major
      int consumed = 0;
      auto issue_s = [&](int j) {
        const int s = j % kStages;
        const uint32_t d = tmem + (j & 1) * 128;
#pragma unroll
        for (int k = 0; k < kHd / 16; ++k)
          umma_bf16(d, sdesc_sw128(sQ + k * 32, 16, 1024), sdesc_sw128(sK(s) + k * 32, 16, 1024),
                    id_s, k != 0);
        umma_commit(s_full(j & 1));
      };
      bool ok = mbar_wait(q_full, 0, p.status) && mbar_wait(kv_full(0), 0, p.status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int s1 = (j + 1) % kStages;
          if (!mbar_wait(kv_full(s1), ((j + 1) / kStages) & 1, p.status)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(p_full, j & 1, p.status)) break;
        tc_fence_after();
        const int s = j % kStages;
        const uint32_t pa = sP(j & 1), vb = sV(s);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          const uint64_t a = sdesc_sw128(pa + (k >> 2) * (kPBytes / 2) + (k & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(vb + k * 16 * 128, kKVBytes, 1024);
          umma_bf16(tmem + kTmemO, a, b, id_o, (j | k) != 0);
        }
        umma_commit(pv_done);
        umma_commit(kv_empty(s));
        consumed = j + 1;
      }
      kv_consumed = consumed;
      // All MMAs of this CTA complete before TMEM is released.
      umma_commit(drain);
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int r = threadIdx.x;  // query row inside the tile == TMEM lane
    const uint32_t lane_sel = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      if (!mbar_wait(s_full(b), (j >> 1) & 1, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t* dst = sr + 32 * c;
        tmem_ld32(tmem + b * 128 + c * 32 + lane_sel, *reinterpret_cast<uint32_t(*)[32]>(dst));
      }
      tmem_wait_ld();
      const int kv_valid = min(kTile, len - j * kTile);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        const float x = (i < kv_valid) ? __uint_as_float(sr[i]) * p.scale_log2 : -INFINITY;
        sr[i] = __float_as_uint(x);
        mx = fmaxf(mx, x);
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = ex2_approx(m - m_new);
      float sum = 0.f;
      const uint32_t prow = sP(b) + r * 128;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2_approx(__uint_as_float(sr[u * 8 + 2 * e]) - m_new);
          const float p1 = ex2_approx(__uint_as_float(sr[u * 8 + 2 * e + 1]) - m_new);
          sum += p0 + p1;
          w[e] = pack_bf16x2(p0, p1);
        }
        const uint32_t addr = prow + (u >> 3) * (kPBytes / 2) + (((u & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      l = l * alpha + sum;
      fence_proxy_async_smem();
      if (j > 0) {
        if (!mbar_wait(pv_done, (j - 1) & 1, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, alpha < 1.f)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + kTmemO + c * 32 + lane_sel, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + kTmemO + c * 32 + lane_sel, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(p_full);
      m = m_new;
    }
    if (ok && n_kv > 0 && mbar_wait(pv_done, (n_kv - 1) & 1, p.status)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint32_t o[64];
      tmem_ld32(tmem + kTmemO + lane_sel, *reinterpret_cast<uint32_t(*)[32]>(o));
      tmem_ld32(tmem + kTmemO + 32 + lane_sel, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
      tmem_wait_ld();
      if (r < q_valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(q0 + r) * 1024 + head * kHd);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
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
  if (warp == 4 && lane == 0 && status_failed(p.status)) {
    if (q_issued) mbar_wait(q_full, 0, nullptr);
    for (int j = kv_consumed; j < kv_issued; ++j)
      if (!mbar_wait(kv_full(j % kStages), (j / kStages) & 1, nullptr)) break;
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

int launch_attention(const CUtensorMap& tm_qkv, const AttnBatch& batch, bf16* out, int* status,
                     cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return DS_VIT_ECUDA;
  AttnParams p;
  p.b = batch;
  p.out = out;
  p.status = status;
  p.scale_log2 = 1.4426950408889634f * 0.125f;
  const int tiles = batch.tile_start[batch.n_images];
  if (tiles <= 0) return DS_VIT_OK;
  attn_kernel<<<dim3(tiles, 16), 192, kSmemBytes, stream>>>(tm_qkv, p);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

}  // namespace dsvit
