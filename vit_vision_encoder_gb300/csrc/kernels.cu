// Memory-bound kernels of the encode: LayerNorm, the pixel normalisation
// table, the RoPE table, weight preparation and the overlay scatter.  Sources: "DeepSeek V4.1 Flash Engineering, Part 3:
// Integrating Vision" (cited per kernel).
#include "internal.h"
#include "ptx.cuh"

namespace dsvit {

namespace {

// ---------------------------------------------------------------- LayerNorm
// One warp per row of W values (1024 for the encode, 1152 for the Qwen-style
// tower); lane l holds the 16-byte chunks l, l+32, ... (coalesced across the
// warp), kept packed as bf16 pairs so a thread needs few registers and many
// rows stay in flight per SM.  fp32 statistics: mean, then the biased variance
// of the centred values; y = (x - mu) * (1/sqrt(var + eps)) * g + b rounded to
// bf16 ("Step 2": the final-norm boundary; block pre-norms).  gamma and beta
// are read after the statistics (they are hot in L1/L2).
// RMS mode (RMSNorm, page A's comparison table for the released tower): no
// centring and no beta, y = x * (1/sqrt(mean(x^2) + eps)) * g.
template <bool RMS, int W>
__global__ void __launch_bounds__(128) layernorm_kernel(const bf16* __restrict__ x,
                                                        const bf16* __restrict__ g,
                                                        const bf16* __restrict__ b,
                                                        bf16* __restrict__ y, int64_t M,
                                                        float eps) {
  constexpr int kChunks = W / 8;                  // 16-byte chunks per row
  constexpr int kPerLane = (kChunks + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  grid_dep_launch();
  grid_dep_wait();
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * W);
  uint32_t xw[4 * kPerLane];
#pragma unroll
  for (int q = 0; q < kPerLane; ++q) {
    const bool on = q * 32 + lane < kChunks;
    const uint4 u = on ? __ldg(xr + q * 32 + lane) : make_uint4(0, 0, 0, 0);
    xw[4 * q] = u.x;
    xw[4 * q + 1] = u.y;
    xw[4 * q + 2] = u.z;
    xw[4 * q + 3] = u.w;
  }
  float mu = 0.f;
  if constexpr (!RMS) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4 * kPerLane; ++i) {
      s0 += bf16lo(xw[i]);
      s1 += bf16hi(xw[i]);
    }
    float s = s0 + s1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    mu = __fdiv_rn(s, static_cast<float>(W));
  }
  float q0 = 0.f, q1 = 0.f;
#pragma unroll
  for (int q = 0; q < kPerLane; ++q) {
    if (q * 32 + lane < kChunks) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d0 = __fsub_rn(bf16lo(xw[4 * q + e]), mu), d1 = __fsub_rn(bf16hi(xw[4 * q + e]), mu);
        q0 = __fmaf_rn(d0, d0, q0);
        q1 = __fmaf_rn(d1, d1, q1);
      }
    }
  }
  float ss = q0 + q1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const float inv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(W)), eps)));
  const uint4* g4 = reinterpret_cast<const uint4*>(g);
  const uint4* b4 = reinterpret_cast<const uint4*>(b);
  uint4* yr = reinterpret_cast<uint4*>(y + row * W);
#pragma unroll
  for (int q = 0; q < kPerLane; ++q) {
    if (q * 32 + lane >= kChunks) continue;
    const uint4 gu = __ldg(g4 + q * 32 + lane);
    const uint4 bu = RMS ? make_uint4(0, 0, 0, 0) : __ldg(b4 + q * 32 + lane);
    const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
    const uint32_t bw[4] = {bu.x, bu.y, bu.z, bu.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t w = xw[4 * q + e];
      float y0, y1;
      if constexpr (RMS) {
        y0 = __fmul_rn(__fmul_rn(bf16lo(w), inv), bf16lo(gw[e]));
        y1 = __fmul_rn(__fmul_rn(bf16hi(w), inv), bf16hi(gw[e]));
      } else {
        y0 = __fadd_rn(__fmul_rn(__fmul_rn(__fsub_rn(bf16lo(w), mu), inv), bf16lo(gw[e])), bf16lo(bw[e]));
        y1 = __fadd_rn(__fmul_rn(__fmul_rn(__fsub_rn(bf16hi(w), mu), inv), bf16hi(gw[e])), bf16hi(bw[e]));
      }
      o[e] = pack_bf16x2(y0, y1);
    }
    yr[q * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------- pixel LUT
// lut[c*256 + v] = bf16((v/255 - mean_c)/std_c) in fp32 arithmetic ("Step 1"
// item 6 with the CLIP statistics); the patch-projection GEMM reads it while
// building its A tiles.
__global__ void pixel_lut_kernel(const __grid_constant__ PixelNorm norm, bf16* __restrict__ lut) {
  const int t = threadIdx.x + blockIdx.x * blockDim.x;
  if (t >= 768) return;
  const int c = t / 256, v = t % 256;
  lut[t] = __float2bfloat16_rn(__fdiv_rn(__fsub_rn(__fdiv_rn(static_cast<float>(v), 255.f), norm.mean[c]),
                                         norm.std[c]));
}

// ---------------------------------------------------------------- RoPE table
// [pos][i] = cos(pos * theta^(-i/16)), [pos][16+i] = sin(...), in double, cast
// to fp32 ("Step 3": height and width frequencies, 16 per 32-dim half).
__global__ void rope_table_kernel(float* table, int max_pos, double theta) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= max_pos * 16) return;
  const int pos = idx / 16, i = idx % 16;
  const double f = pow(theta, -static_cast<double>(i) / 16.0);
  const double a = static_cast<double>(pos) * f;
  table[pos * 32 + i] = static_cast<float>(cos(a));
  table[pos * 32 + 16 + i] = static_cast<float>(sin(a));
}

// q and k rows of W_qkv (and b_qkv) with head dims 16..31 and 32..47 swapped:
// the half-vector pairing (dim i with i + 32, angles [row f, col f]) becomes
// the axis-halves pairing the QKV epilogue applies, and q.k is unchanged
// because q and k take the same permutation.  One block per output row.
__global__ void permute_qk_rows_kernel(const bf16* __restrict__ w, const bf16* __restrict__ b,
                                       bf16* __restrict__ wp, bf16* __restrict__ bp, int hidden, int K) {
  const int r = blockIdx.x;                     // destination row
  int src = r;
  if (r < 2 * hidden) {
    const int d = r % 64, base = r - d;
    const int sd = (d >= 16 && d < 32) ? d + 16 : ((d >= 32 && d < 48) ? d - 16 : d);
    src = base + sd;
  }
  for (int k = threadIdx.x; k < K; k += blockDim.x)
    wp[static_cast<int64_t>(r) * K + k] = w[static_cast<int64_t>(src) * K + k];
  if (threadIdx.x == 0) bp[r] = b[src];
}

__global__ void permute_m1_kernel(const bf16* __restrict__ w, bf16* __restrict__ wp) {
  const int64_t o = blockIdx.x;
  for (int k = threadIdx.x; k < 9216; k += blockDim.x) {
    const int p = k / 1024, c = k % 1024;
    wp[o * 9216 + k] = w[o * 9216 + c * 9 + p];
  }
}

__global__ void pad_patch_w_kernel(const bf16* __restrict__ w, bf16* __restrict__ wp) {
  const int64_t o = blockIdx.x;
  for (int k = threadIdx.x; k < kPatchK; k += blockDim.x) {
    const int y = k / 64, j = k % 64, x = j / 3, c = j % 3;
    wp[o * kPatchK + k] = j < 42 ? w[o * 588 + c * 196 + y * 14 + x] : __float2bfloat16_rn(0.f);
  }
}

// ---------------------------------------------------------------- overlay
// Span row r of span s: r = 0 START, r = n-1 END, otherwise q = r-1,
// y = q / (w+1), x = q % (w+1): NEWLINE when x == w, else IMAGE with merged
// token y*w + x ("Connect the complete image-to-text path first").  IMAGE rows
// copy the aligner row, the others the learned vector.  One block per row,
// 16-byte vector copies.
__global__ void __launch_bounds__(128) overlay_kernel(bf16* __restrict__ hidden, int width,
                                                      const __grid_constant__ OverlaySpans spans,
                                                      const bf16* __restrict__ embeds,
                                                      const bf16* __restrict__ sentinel) {
  const int64_t g = blockIdx.x;
  int s = 0;
  while (s + 1 < spans.n && spans.row_start[s + 1] <= g) ++s;
  const int64_t r = g - spans.row_start[s];
  const int64_t n = spans.row_start[s + 1] - spans.row_start[s];
  const int w = spans.w[s];
  const bf16* src;
  if (r == 0) {
    src = sentinel;
  } else if (r == n - 1) {
    src = sentinel + 2 * static_cast<int64_t>(width);
  } else {
    const int64_t q = r - 1, y = q / (w + 1), x = q % (w + 1);
    src = (x == w) ? sentinel + width : embeds + (spans.embed_row[s] + y * w + x) * width;
  }
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(hidden + (spans.base_row[s] + r) * width);
  for (int k = threadIdx.x; k < width / 8; k += blockDim.x) d4[k] = s4[k];
}

// Chunked prefill: one block per chunk row g = chunk_begin + i.  The span that
// holds g (if any) gives the row's source as in overlay_kernel and its type
// code 1 + type; rows outside every span keep their contents, type 0.
__global__ void __launch_bounds__(128) overlay_chunk_kernel(bf16* __restrict__ chunk, int64_t chunk_begin,
                                                            int width,
                                                            const __grid_constant__ OverlaySpans spans,
                                                            const bf16* __restrict__ embeds,
                                                            const bf16* __restrict__ sentinel,
                                                            uint8_t* __restrict__ row_type) {
  const int64_t i = blockIdx.x;
  const int64_t g = chunk_begin + i;
  int s = -1;
  for (int k = 0; k < spans.n; ++k) {
    const int64_t n = spans.row_start[k + 1] - spans.row_start[k];
    if (g >= spans.base_row[k] && g < spans.base_row[k] + n) {
      s = k;
      break;
    }
  }
  if (s < 0) {
    if (row_type && threadIdx.x == 0) row_type[i] = 0;
    return;
  }
  const int64_t r = g - spans.base_row[s];
  const int64_t n = spans.row_start[s + 1] - spans.row_start[s];
  const int w = spans.w[s];
  const bf16* src;
  int type;
  if (r == 0) {
    src = sentinel;
    type = DS_VIT_TOK_START;
  } else if (r == n - 1) {
    src = sentinel + 2 * static_cast<int64_t>(width);
    type = DS_VIT_TOK_END;
  } else {
    const int64_t q = r - 1, y = q / (w + 1), x = q % (w + 1);
    if (x == w) {
      src = sentinel + width;
      type = DS_VIT_TOK_NEWLINE;
    } else {
      src = embeds + (spans.embed_row[s] + y * w + x) * width;
      type = DS_VIT_TOK_IMAGE;
    }
  }
  if (row_type && threadIdx.x == 0) row_type[i] = static_cast<uint8_t>(1 + type);
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(chunk + i * width);
  for (int k = threadIdx.x; k < width / 8; k += blockDim.x) d4[k] = s4[k];
}

// Overlay from caller-given per-row arrays (rows, type, src on the device).
// The entries are checked on the device before any row is written: the check
// kernel records the first error in *status, and the copy kernel, launched
// after it on the same stream, writes nothing while *status holds one.
__global__ void __launch_bounds__(256) overlay_rows_check_kernel(const int32_t* __restrict__ rows,
                                                                 const uint8_t* __restrict__ type,
                                                                 const int32_t* __restrict__ src, int64_t n,
                                                                 int64_t n_hidden, int64_t n_embeds,
                                                                 int* __restrict__ status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int t = type[i];
  int err = 0;
  if (t > DS_VIT_TOK_END)
    err = DS_VIT_EINVAL;
  else if (rows[i] < 0 || rows[i] >= n_hidden || (t == DS_VIT_TOK_IMAGE && (src[i] < 0 || src[i] >= n_embeds)))
    err = DS_VIT_ERANGE;
  if (err) atomicCAS(status, 0, err);
}

__global__ void __launch_bounds__(128) overlay_rows_kernel(bf16* __restrict__ hidden, int width,
                                                           const int32_t* __restrict__ rows,
                                                           const uint8_t* __restrict__ type,
                                                           const int32_t* __restrict__ src,
                                                           const bf16* __restrict__ embeds,
                                                           const bf16* __restrict__ sentinel,
                                                           const int* __restrict__ status) {
  if (*status != 0) return;
  const int64_t i = blockIdx.x;
  const int t = type[i];
  // Sentinel rows in the order START, NEWLINE, END.
  const bf16* from = t == DS_VIT_TOK_IMAGE ? embeds + static_cast<int64_t>(src[i]) * width
                     : sentinel + static_cast<int64_t>(t == DS_VIT_TOK_START ? 0 : t == DS_VIT_TOK_NEWLINE ? 1 : 2) * width;
  const uint4* s4 = reinterpret_cast<const uint4*>(from);
  uint4* d4 = reinterpret_cast<uint4*>(hidden + static_cast<int64_t>(rows[i]) * width);
  for (int k = threadIdx.x; k < width / 8; k += blockDim.x) d4[k] = s4[k];
}

}  // namespace

int launch_layernorm(const bf16* x, const bf16* g, const bf16* b, bf16* y, int64_t M, float eps,
                     cudaStream_t stream, bool rms, int width) {
  if (M <= 0) return DS_VIT_OK;
  const dim3 grid(static_cast<unsigned>((M + 3) / 4));
  cudaError_t e;
  if (width == 1152)
    e = launch_pdl(layernorm_kernel<false, 1152>, grid, dim3(128), 0, stream, x, g, b, y, M, eps);
  else if (width != 1024)
    return DS_VIT_EINVAL;
  else
    e = rms ? launch_pdl(layernorm_kernel<true, 1024>, grid, dim3(128), 0, stream, x, g, b, y, M, eps)
            : launch_pdl(layernorm_kernel<false, 1024>, grid, dim3(128), 0, stream, x, g, b, y, M, eps);
  if (e != cudaSuccess) cudaGetLastError();
  return e == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// completes, gives up after limit_ns of %globaltimer, records the timeout in
// *status as every kernel's bounded waits do, and stores how long it waited.
__global__ void selftest_wait_kernel(int* status, unsigned long long* elapsed, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  const unsigned long long t0 = global_timer();
  while (!mbar_try_wait(b, 0)) {
    if (global_timer() - t0 > limit_ns) {
      report_error(status, kErrTimeout);
      break;
    }
  }
  *elapsed = global_timer() - t0;
}

int launch_selftest_wait(int* status, unsigned long long* elapsed, unsigned long long limit_ns,
                         cudaStream_t stream) {
  selftest_wait_kernel<<<1, 1, 0, stream>>>(status, elapsed, limit_ns);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_pixel_lut(const PixelNorm& norm, bf16* lut, cudaStream_t stream) {
  pixel_lut_kernel<<<3, 256, 0, stream>>>(norm, lut);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_rope_table(float* table, int max_pos, float theta, cudaStream_t stream) {
  const int n = max_pos * 16;
  rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(table, max_pos, static_cast<double>(theta));
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_permute_qk_rows(const bf16* w, const bf16* b, bf16* w_perm, bf16* b_perm, int hidden, int K,
                           cudaStream_t stream) {
  permute_qk_rows_kernel<<<3 * hidden, 256, 0, stream>>>(w, b, w_perm, b_perm, hidden, K);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_permute_m1(const bf16* w, bf16* w_perm, int rows, cudaStream_t stream) {
  permute_m1_kernel<<<rows, 256, 0, stream>>>(w, w_perm);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_pad_patch_w(const bf16* w, bf16* w_pad, int rows, cudaStream_t stream) {
  pad_patch_w_kernel<<<rows, 128, 0, stream>>>(w, w_pad);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_overlay_chunk(bf16* chunk, int64_t chunk_begin, int64_t chunk_rows, int width,
                         const OverlaySpans& spans, const bf16* embeds, const bf16* sentinel,
                         uint8_t* row_type, cudaStream_t stream) {
  overlay_chunk_kernel<<<static_cast<unsigned>(chunk_rows), 128, 0, stream>>>(chunk, chunk_begin, width, spans,
                                                                              embeds, sentinel, row_type);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_overlay(bf16* hidden, int width, const OverlaySpans& spans, const bf16* embeds,
                   const bf16* sentinel, cudaStream_t stream) {
  const int64_t rows = spans.row_start[spans.n];
  if (rows <= 0) return DS_VIT_OK;
  overlay_kernel<<<static_cast<unsigned>(rows), 128, 0, stream>>>(hidden, width, spans, embeds, sentinel);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

int launch_overlay_rows(bf16* hidden, int64_t n_hidden, int width, const int32_t* rows, const uint8_t* type,
                        const int32_t* src, int64_t n, const bf16* embeds, int64_t n_embeds, const bf16* sentinel,
                        int* status, cudaStream_t stream) {
  if (n <= 0) return DS_VIT_OK;
  overlay_rows_check_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(rows, type, src, n, n_hidden,
                                                                                       n_embeds, status);
  if (cudaGetLastError() != cudaSuccess) return DS_VIT_ECUDA;
  overlay_rows_kernel<<<static_cast<unsigned>(n), 128, 0, stream>>>(hidden, width, rows, type, src, embeds, sentinel,
                                                                    status);
  return cudaGetLastError() == cudaSuccess ? DS_VIT_OK : DS_VIT_ECUDA;
}

}  // namespace dsvit
