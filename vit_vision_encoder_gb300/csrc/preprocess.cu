// Image preprocessing upstream of the encode: grid plan, PIL-"contain" resize
// with bicubic filtering, RGB 127 canvas ("DeepSeek V4.1 Flash Engineering,
// Part 3: Integrating Vision", "Step 1: Reproduce the discrete image-processing
// rules"; ds4-learning glossary "vision", V4.1 paragraph: minimum pixel budget
// 295,936, at most 1,024 image tokens, no aspect clamp; Lucebox "Image input":
// bicubic resizing that matches Pillow byte for byte).
//
// The plan is host integer/float64 code.  On the device: one kernel builds the
// per-output-index filter tables of both axes in float64 (every operation an
// explicitly rounded intrinsic, so no contraction changes a weight), one runs
// the horizontal pass (rows of the input -> Wr columns) and one the vertical
// pass, writing the canvas directly (gray outside the resized image).  Each
// pass rounds to uint8 as (2^21 + sum pixel * weight) >> 22, clamped.
#include "internal.h"

#include <algorithm>
#include <cmath>

namespace dsvit {

namespace {

constexpr int kUnit = 42;                // patch 14 x merge 3
constexpr int64_t kMinPixels = 295936;
constexpr int kPrecisionBits = 22;       // 32 - 8 - 2
constexpr uint8_t kGray = 127;
constexpr int kMaxSide = 65535;
constexpr int64_t kMaxPixels = int64_t{1} << 28;

size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }

// Keys' cubic convolution kernel, a = -0.5, in Horner form.
__device__ double keys(double x) {
  x = fabs(x);
  if (x < 1.0) return __dadd_rn(__dmul_rn(__dmul_rn(__dsub_rn(__dmul_rn(1.5, x), 2.5), x), x), 1.0);
  if (x < 2.0)
    return __dmul_rn(__dsub_rn(__dmul_rn(__dadd_rn(__dmul_rn(__dsub_rn(x, 5.0), x), 8.0), x), 4.0), -0.5);
  return 0.0;
}

// Filter tables of both axes, tap-major so that neighbouring output indices
// read neighbouring words: first[i] is output i's first input tap and
// w[k * n_out + i] its k-th fixed-point weight (zero past its taps).
struct ResizeAxes {
  int in_x, out_x, taps_x;   // width  W -> Wr
  int in_y, out_y, taps_y;   // height H -> Hr
  int* first_x;
  int* w_x;
  int* first_y;
  int* w_y;
};

// Taps of one output index never exceed ceil(support) * 2 + 1 nor the input size.
int max_taps(int n_in, int n_out) {
  const double scale = static_cast<double>(n_in) / n_out;
  const double support = 2.0 * (scale > 1.0 ? scale : 1.0);
  const int k = static_cast<int>(std::ceil(support)) * 2 + 1;
  return k < n_in ? k : n_in;
}

// One warp per output index: lanes evaluate the taps, lane 0 sums them in tap
// order, every lane normalises its own taps (float64 on the device is slow, so
// the taps run in parallel).  Same operations and order as a serial loop.
__device__ void build_index(int n_in, int n_out, int T, int i, int* first, int* wt, double* sw) {
  const int lane = threadIdx.x & 31;
  const double scale = __ddiv_rn(static_cast<double>(n_in), static_cast<double>(n_out));
  const double filterscale = scale > 1.0 ? scale : 1.0;
  const double support = __dmul_rn(2.0, filterscale);
  const double ss = __ddiv_rn(1.0, filterscale);
  const double center = __dmul_rn(__dadd_rn(static_cast<double>(i), 0.5), scale);
  int lo = static_cast<int>(__dadd_rn(__dsub_rn(center, support), 0.5));   // truncation
  if (lo < 0) lo = 0;
  int hi = static_cast<int>(__dadd_rn(__dadd_rn(center, support), 0.5));
  if (hi > n_in) hi = n_in;
  const int n = hi - lo;
  for (int x = lane; x < n; x += 32)
    sw[x] = keys(__dmul_rn(__dadd_rn(__dsub_rn(static_cast<double>(x + lo), center), 0.5), ss));
  __syncwarp();
  double total = 0.0;
  if (lane == 0)
    for (int x = 0; x < n; ++x) total = __dadd_rn(total, sw[x]);
  total = __shfl_sync(0xFFFFFFFFu, total, 0);
  if (lane == 0) first[i] = lo;
  for (int x = lane; x < T; x += 32) {
    int q = 0;
    if (x < n) {
      const double w = sw[x];
      const double k = total != 0.0 ? __ddiv_rn(w, total) : w;
      const double f = __dmul_rn(k, static_cast<double>(1 << kPrecisionBits));
      q = k >= 0.0 ? static_cast<int>(__dadd_rn(f, 0.5)) : static_cast<int>(__dsub_rn(f, 0.5));
    }
    wt[static_cast<size_t>(x) * n_out + i] = q;
  }
}

// Block of 32 threads per output index of either axis; `sw` holds its taps.
__global__ void resize_tables_kernel(const __grid_constant__ ResizeAxes a) {
  extern __shared__ double sw[];
  const int i = blockIdx.x;
  if (i < a.out_x)
    build_index(a.in_x, a.out_x, a.taps_x, i, a.first_x, a.w_x, sw);
  else
    build_index(a.in_y, a.out_y, a.taps_y, i - a.out_x, a.first_y, a.w_y, sw);
}

__device__ __forceinline__ uint8_t round_clamp(int acc) {
  const int v = acc >> kPrecisionBits;   // arithmetic shift: floor for negative sums
  return static_cast<uint8_t>(v < 0 ? 0 : (v > 255 ? 255 : v));
}

// Horizontal pass: in [H][W][3] -> out [H][Wr][3]; one thread per output pixel.
__global__ void resize_h_kernel(const uint8_t* __restrict__ in, int W, uint8_t* __restrict__ out, int Wr,
                                const int* __restrict__ first, const int* __restrict__ wt, int T) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  const int y = blockIdx.y;
  if (x >= Wr) return;
  const int lo = __ldg(first + x);
  const int n = T < W - lo ? T : W - lo;
  const uint8_t* src = in + (static_cast<size_t>(y) * W + lo) * 3;
  int a0 = 1 << (kPrecisionBits - 1), a1 = a0, a2 = a0;
  for (int k = 0; k < n; ++k) {
    const int w = __ldg(wt + static_cast<size_t>(k) * Wr + x);
    a0 += src[3 * k] * w;
    a1 += src[3 * k + 1] * w;
    a2 += src[3 * k + 2] * w;
  }
  uint8_t* dst = out + (static_cast<size_t>(y) * Wr + x) * 3;
  dst[0] = round_clamp(a0);
  dst[1] = round_clamp(a1);
  dst[2] = round_clamp(a2);
}

// Vertical pass into the canvas: src [H][Wr][3] (the horizontal pass's output,
// or the input when the width is unchanged) -> canvas [Hc][Wc][3]; rows of the
// resized image land at y0.., columns at x0..; gray elsewhere.  When the
// height is unchanged (H == Hr) the rows are copied.
__global__ void resize_v_canvas_kernel(const uint8_t* __restrict__ src, int H, int Wr, int Hr,
                                       const int* __restrict__ first, const int* __restrict__ wt, int T,
                                       uint8_t* __restrict__ canvas, int Wc, int y0, int x0) {
  const int X = blockIdx.x * blockDim.x + threadIdx.x;
  const int Y = blockIdx.y;
  if (X >= Wc) return;
  uint8_t p0 = kGray, p1 = kGray, p2 = kGray;
  const int yy = Y - y0, xx = X - x0;
  if (yy >= 0 && yy < Hr && xx >= 0 && xx < Wr) {
    if (H == Hr) {
      const uint8_t* s = src + (static_cast<size_t>(yy) * Wr + xx) * 3;
      p0 = s[0];
      p1 = s[1];
      p2 = s[2];
    } else {
      const int lo = __ldg(first + yy);
      const int n = T < H - lo ? T : H - lo;
      const uint8_t* s = src + (static_cast<size_t>(lo) * Wr + xx) * 3;
      const size_t pitch = static_cast<size_t>(Wr) * 3;
      int a0 = 1 << (kPrecisionBits - 1), a1 = a0, a2 = a0;
      for (int k = 0; k < n; ++k) {
        const int w = __ldg(wt + static_cast<size_t>(k) * Hr + yy);
        a0 += s[k * pitch] * w;
        a1 += s[k * pitch + 1] * w;
        a2 += s[k * pitch + 2] * w;
      }
      p0 = round_clamp(a0);
      p1 = round_clamp(a1);
      p2 = round_clamp(a2);
    }
  }
  uint8_t* d = canvas + (static_cast<size_t>(Y) * Wc + X) * 3;
  d[0] = p0;
  d[1] = p1;
  d[2] = p2;
}

struct PreLayout {
  size_t off_tmp, off_fx, off_wx, off_fy, off_wy, total;
  int taps_x, taps_y;
};

PreLayout pre_layout(const ds_vit_plan& p) {
  PreLayout L{};
  L.taps_x = max_taps(p.W, p.Wr);
  L.taps_y = max_taps(p.H, p.Hr);
  size_t o = 0;
  L.off_tmp = o;
  if (p.Wr != p.W) o += align256(static_cast<size_t>(p.H) * p.Wr * 3);
  L.off_fx = o;
  o += align256(static_cast<size_t>(p.Wr) * 4);
  L.off_wx = o;
  o += align256(static_cast<size_t>(p.Wr) * L.taps_x * 4);
  L.off_fy = o;
  o += align256(static_cast<size_t>(p.Hr) * 4);
  L.off_wy = o;
  o += align256(static_cast<size_t>(p.Hr) * L.taps_y * 4);
  L.total = o;
  return L;
}

bool same_plan(const ds_vit_plan& a, const ds_vit_plan& b) {
  return a.H == b.H && a.W == b.W && a.h == b.h && a.w == b.w && a.Hc == b.Hc && a.Wc == b.Wc &&
         a.Hr == b.Hr && a.Wr == b.Wr && a.y0 == b.y0 && a.x0 == b.x0;
}

}  // namespace

}  // namespace dsvit

using namespace dsvit;

extern "C" {

int ds_vit_plan_image(int32_t H, int32_t W, ds_vit_plan* out) {
  if (!out || H < 1 || W < 1 || H > kMaxSide || W > kMaxSide ||
      static_cast<int64_t>(H) * W > kMaxPixels)
    return DS_VIT_EINVAL;
  const int64_t area = static_cast<int64_t>(H) * W;
  double s = 1.0;
  if (area < kMinPixels) s = std::sqrt(static_cast<double>(kMinPixels) / static_cast<double>(area));
  const double He = static_cast<double>(H) * s, We = static_cast<double>(W) * s;
  int64_t h = static_cast<int64_t>(std::ceil(He / kUnit)), w = static_cast<int64_t>(std::ceil(We / kUnit));
  if (h * w > DS_VIT_MAX_TOKENS) {
    const double r = std::sqrt(static_cast<double>(DS_VIT_MAX_TOKENS * kUnit * kUnit) / (He * We));
    h = static_cast<int64_t>(std::floor(He * r / kUnit));
    w = static_cast<int64_t>(std::floor(We * r / kUnit));
    if (h < 1) h = 1;
    if (w < 1) w = 1;
    h = std::min<int64_t>(h, DS_VIT_MAX_TOKENS / w);
    if (h < 1) h = 1;
    w = std::min<int64_t>(w, DS_VIT_MAX_TOKENS / h);
  }
  ds_vit_plan p{};
  p.H = H;
  p.W = W;
  p.h = static_cast<int32_t>(h);
  p.w = static_cast<int32_t>(w);
  p.Hc = p.h * kUnit;
  p.Wc = p.w * kUnit;
  // PIL contain: compare aspect ratios, compute the other side with round (half to even).
  const double im_ratio = static_cast<double>(W) / H, dest_ratio = static_cast<double>(p.Wc) / p.Hc;
  p.Wr = p.Wc;
  p.Hr = p.Hc;
  if (im_ratio != dest_ratio) {
    if (im_ratio > dest_ratio) {
      const double v = std::nearbyint(static_cast<double>(H) / W * p.Wc);
      p.Hr = v < 1.0 ? 1 : static_cast<int32_t>(v);
    } else {
      const double v = std::nearbyint(static_cast<double>(W) / H * p.Hc);
      p.Wr = v < 1.0 ? 1 : static_cast<int32_t>(v);
    }
  }
  p.y0 = (p.Hc - p.Hr) / 2;
  p.x0 = (p.Wc - p.Wr) / 2;
  *out = p;
  return DS_VIT_OK;
}

int ds_vit_preprocess_workspace_bytes(const ds_vit_plan* plan, size_t* bytes) {
  if (!plan || !bytes) return DS_VIT_EINVAL;
  ds_vit_plan ref;
  if (ds_vit_plan_image(plan->H, plan->W, &ref) != DS_VIT_OK || !same_plan(ref, *plan)) return DS_VIT_EINVAL;
  *bytes = pre_layout(*plan).total;
  return DS_VIT_OK;
}

int ds_vit_preprocess(const ds_vit_plan* plan, const uint8_t* pixels, void* canvas, void* ws,
                      size_t ws_bytes, void* stream) {
  if (!plan || !pixels || !canvas || !ws) return DS_VIT_EINVAL;
  ds_vit_plan ref;
  if (ds_vit_plan_image(plan->H, plan->W, &ref) != DS_VIT_OK || !same_plan(ref, *plan)) return DS_VIT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return DS_VIT_EINVAL;
  const PreLayout L = pre_layout(ref);
  if (ws_bytes < L.total) return DS_VIT_ECAP;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  ResizeAxes a;
  a.in_x = ref.W;
  a.out_x = ref.Wr;
  a.taps_x = L.taps_x;
  a.in_y = ref.H;
  a.out_y = ref.Hr;
  a.taps_y = L.taps_y;
  a.first_x = reinterpret_cast<int*>(w8 + L.off_fx);
  a.w_x = reinterpret_cast<int*>(w8 + L.off_wx);
  a.first_y = reinterpret_cast<int*>(w8 + L.off_fy);
  a.w_y = reinterpret_cast<int*>(w8 + L.off_wy);
  const int max_t = L.taps_x > L.taps_y ? L.taps_x : L.taps_y;
  const size_t tab_smem = static_cast<size_t>(max_t) * sizeof(double);
  if (tab_smem > 48 * 1024 &&
      cudaFuncSetAttribute(resize_tables_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tab_smem)) != cudaSuccess) {
    cudaGetLastError();
    return DS_VIT_ECUDA;
  }
  resize_tables_kernel<<<ref.Wr + ref.Hr, 32, tab_smem, st>>>(a);
  const uint8_t* src = pixels;
  if (ref.Wr != ref.W) {
    uint8_t* tmp = w8 + L.off_tmp;
    resize_h_kernel<<<dim3((ref.Wr + 127) / 128, ref.H), 128, 0, st>>>(pixels, ref.W, tmp, ref.Wr, a.first_x,
                                                                         a.w_x, L.taps_x);
    src = tmp;
  }
  resize_v_canvas_kernel<<<dim3((ref.Wc + 127) / 128, ref.Hc), 128, 0, st>>>(
      src, ref.H, ref.Wr, ref.Hr, a.first_y, a.w_y, L.taps_y, static_cast<uint8_t*>(canvas), ref.Wc, ref.y0,
      ref.x0);
  if (cudaGetLastError() != cudaSuccess) return DS_VIT_ECUDA;
  return DS_VIT_OK;
}

}  // extern "C"
