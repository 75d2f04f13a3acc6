// Image preprocessing upstream of the encode: grid plan, PIL-"contain" resize
// with bicubic filtering, RGB 127 canvas ("DeepSeek V4.1 Flash Engineering,
// Part 3: Integrating Vision", "Step 1: Reproduce the discrete image-processing
// rules"; ds4-learning glossary "vision", V4.1 paragraph: minimum pixel budget
// 295,936, at most 1,024 image tokens, no aspect clamp; Lucebox "Image input":
// bicubic resizing that matches Pillow byte for byte).
//
// The plan is host integer/float64 code.  On the device: the filter tables of
// both axes in float64 (every operation an explicitly rounded intrinsic, so no
// contraction changes a weight; several output indices per warp), stored as
// tap-major ints and in byte planes for dp4a; the horizontal pass (rows of the
// input -> Wr columns, into rows padded to 16 bytes) and the vertical pass,
// writing the canvas directly (gray outside the resized image).  Each pass
// rounds to uint8 as (2^21 + sum pixel * weight) >> 22, clamped.  The planar
// passes take four taps' products per dp4a in each weight byte plane (exact
// in 32-bit integers): horizontally a block stages its input span split into
// R, G, B planes; vertically a thread transposes 4 rows x 8 bytes so that a
// word holds one output byte's four taps.  The horizontal pass builds the
// height's tables in leading blocks and stages its pixels before it waits for
// the width's tables (programmatic dependent launch).  The per-pixel kernels
// remain for wider filters and unaligned sources.
#include "internal.h"
#include "ptx.cuh"

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

// Scale, support and 1 / filterscale of an axis: single IEEE double
// operations, computed once on the host (the same doubles as on the device).
struct AxisScale {
  double scale, support, ss;
};

AxisScale axis_scale(int n_in, int n_out) {
  AxisScale s;
  s.scale = static_cast<double>(n_in) / static_cast<double>(n_out);
  const double filterscale = s.scale > 1.0 ? s.scale : 1.0;
  s.support = 2.0 * filterscale;
  s.ss = 1.0 / filterscale;
  return s;
}

// Filter tables of both axes.  Tap-major so that neighbouring output indices
// read neighbouring words: first[i] is output i's first input tap and
// w[k * n_out + i] its k-th fixed-point weight (zero past its taps).  The
// same weights in byte planes, for the dp4a passes: a weight w (|w| < 2^23)
// is b0 + 2^8 b1 + 2^16 b2 with b0, b1 unsigned bytes and b2 a signed byte;
// word (p * g4 + j) * n_out + i holds byte p of taps 4j .. 4j+3 of index i
// (g4 groups of four taps cover every nonzero tap; zero past them).
struct ResizeAxes {
  int in_x, out_x, taps_x, g4_x;   // width  W -> Wr
  int in_y, out_y, taps_y, g4_y;   // height H -> Hr
  AxisScale sx, sy;
  int* first_x;
  int* w_x;
  uint32_t* wp_x;
  int* first_y;
  int* w_y;
  uint32_t* wp_y;
};

// Taps of one output index never exceed ceil(support) * 2 + 1 nor the input size.
int max_taps(int n_in, int n_out) {
  const double scale = static_cast<double>(n_in) / n_out;
  const double support = 2.0 * (scale > 1.0 ? scale : 1.0);
  const int k = static_cast<int>(std::ceil(support)) * 2 + 1;
  return k < n_in ? k : n_in;
}

// Taps a filter of the axis can have nonzero: hi - lo <= floor(2 support) + 1
// (the ends are truncations of c -+ support + 1/2), and at most T.
int max_nonzero_taps(int n_in, int n_out, int T) {
  const double scale = static_cast<double>(n_in) / n_out;
  const int nb = static_cast<int>(std::floor(4.0 * (scale > 1.0 ? scale : 1.0) + 1e-6)) + 1;
  return nb < T ? nb : T;
}

int planar_groups(int n_in, int n_out) { return (max_nonzero_taps(n_in, n_out, max_taps(n_in, n_out)) + 3) / 4; }

// The float64 steps of one output index, shared by both table kernels so
// that they compute the same weights: its span [lo, hi) and centre, a tap's
// unnormalised weight, and the fixed-point weight after normalisation.
__device__ __forceinline__ void index_span(const AxisScale& s, int n_in, int i, double* center, int* lo,
                                           int* hi) {
  *center = __dmul_rn(__dadd_rn(static_cast<double>(i), 0.5), s.scale);
  int l = static_cast<int>(__dadd_rn(__dsub_rn(*center, s.support), 0.5));   // truncation
  if (l < 0) l = 0;
  int h = static_cast<int>(__dadd_rn(__dadd_rn(*center, s.support), 0.5));
  if (h > n_in) h = n_in;
  *lo = l;
  *hi = h;
}

__device__ __forceinline__ double tap_weight(const AxisScale& s, int x, int lo, double center) {
  return keys(__dmul_rn(__dadd_rn(__dsub_rn(static_cast<double>(x + lo), center), 0.5), s.ss));
}

__device__ __forceinline__ int quantise(double w, double total) {
  const double k = total != 0.0 ? __ddiv_rn(w, total) : w;
  const double f = __dmul_rn(k, static_cast<double>(1 << kPrecisionBits));
  return k >= 0.0 ? static_cast<int>(__dadd_rn(f, 0.5)) : static_cast<int>(__dsub_rn(f, 0.5));
}

// Tap k's weight q of index i into the byte planes (taps past 4 g4 are zero
// and not stored).
__device__ __forceinline__ void store_planes(uint32_t* wp, int g4, int n_out, int i, int k, int q) {
  if (wp == nullptr || k >= 4 * g4) return;
  uint8_t* b = reinterpret_cast<uint8_t*>(wp);
  const size_t col = static_cast<size_t>(k >> 2) * n_out + i;
  const size_t plane = static_cast<size_t>(g4) * n_out;
  b[col * 4 + (k & 3)] = static_cast<uint8_t>(q & 0xFF);
  b[(plane + col) * 4 + (k & 3)] = static_cast<uint8_t>((q >> 8) & 0xFF);
  b[(2 * plane + col) * 4 + (k & 3)] = static_cast<uint8_t>((q >> 16) & 0xFF);
}

// One warp per output index: lanes evaluate the taps, lane 0 sums them in tap
// order, every lane normalises its own taps (float64 on the device is slow, so
// the taps run in parallel).  Same operations and order as a serial loop.
__device__ void build_index(const AxisScale& s, int n_in, int n_out, int T, int g4, int i, int* first, int* wt,
                            uint32_t* wp, double* sw) {
  const int lane = threadIdx.x & 31;
  double center;
  int lo, hi;
  index_span(s, n_in, i, &center, &lo, &hi);
  const int n = hi - lo;
  for (int x = lane; x < n; x += 32) sw[x] = tap_weight(s, x, lo, center);
  __syncwarp();
  double total = 0.0;
  if (lane == 0)
    for (int x = 0; x < n; ++x) total = __dadd_rn(total, sw[x]);
  total = __shfl_sync(0xFFFFFFFFu, total, 0);
  if (lane == 0) first[i] = lo;
  const int kmax = T > 4 * g4 ? T : 4 * g4;
  for (int x = lane; x < kmax; x += 32) {
    const int q = x < n ? quantise(sw[x], total) : 0;
    if (x < T) wt[static_cast<size_t>(x) * n_out + i] = q;
    store_planes(wp, g4, n_out, i, x, q);
  }
}

// Block of 32 threads per output index of the axes it covers; `sw` holds its taps.
__global__ void resize_tables_kernel(const __grid_constant__ ResizeAxes a, int n_x) {
  extern __shared__ double sw[];
  const int i = blockIdx.x;
  if (i < n_x)
    build_index(a.sx, a.in_x, a.out_x, a.taps_x, a.g4_x, i, a.first_x, a.w_x, a.wp_x, sw);
  else
    build_index(a.sy, a.in_y, a.out_y, a.taps_y, a.g4_y, i - n_x, a.first_y, a.w_y, a.wp_y, sw);
}

// Axes with at most 32 taps: 32 / T output indices per warp (lane l takes
// tap l % T of index l / T), so a float64 warp instruction serves several
// indices; the sum in tap order is still one lane's serial loop.  Warp gw of
// [0, warps_x) covers the width, of [warps_x, warps_x + warps_y) the height;
// `sw` is the warp's 32 doubles of shared memory.
__device__ void packed_tables_warp(const ResizeAxes& a, int gw, int warps_x, int warps_y, double* sw) {
  if (gw >= warps_x + warps_y) return;   // whole warps
  const int lane = threadIdx.x & 31;
  const bool on_x = gw < warps_x;
  const AxisScale& s = on_x ? a.sx : a.sy;
  const int n_in = on_x ? a.in_x : a.in_y;
  const int n_out = on_x ? a.out_x : a.out_y;
  const int T = on_x ? a.taps_x : a.taps_y;
  const int g4 = on_x ? a.g4_x : a.g4_y;
  int* first = on_x ? a.first_x : a.first_y;
  int* wt = on_x ? a.w_x : a.w_y;
  uint32_t* wp = on_x ? a.wp_x : a.wp_y;
  const int G = 32 / T;
  const int g = lane / T, k = lane - g * T;
  const int i = (on_x ? gw : gw - warps_x) * G + g;
  const bool active = g < G && i < n_out;
  double center = 0.0;
  int lo = 0, hi = 0;
  if (active) {
    index_span(s, n_in, i, &center, &lo, &hi);
    if (k < hi - lo) sw[lane] = tap_weight(s, k, lo, center);
  }
  __syncwarp();
  double total = 0.0;
  if (active && k == 0)
    for (int x = 0; x < hi - lo; ++x) total = __dadd_rn(total, sw[lane + x]);
  total = __shfl_sync(0xFFFFFFFFu, total, active ? g * T : lane);
  if (!active) return;
  if (k == 0) first[i] = lo;
  const int q = k < hi - lo ? quantise(sw[lane], total) : 0;
  wt[static_cast<size_t>(k) * n_out + i] = q;
  store_planes(wp, g4, n_out, i, k, q);
  if (k == 0)
    for (int z = T; z < 4 * g4; ++z) store_planes(wp, g4, n_out, i, z, 0);
}

// One warp per block (the float64 pipe is the limit: small blocks spread
// the warps evenly over the SMs).  A dependent launch may start at once.
__global__ void __launch_bounds__(32) resize_tables_packed_kernel(const __grid_constant__ ResizeAxes a, int warps_x,
                                                                  int warps_y) {
  __shared__ double sw[32];
  grid_dep_launch();
  packed_tables_warp(a, blockIdx.x, warps_x, warps_y, sw);
}

__device__ __forceinline__ uint8_t round_clamp(int acc) {
  const int v = acc >> kPrecisionBits;   // arithmetic shift: floor for negative sums
  return static_cast<uint8_t>(v < 0 ? 0 : (v > 255 ? 255 : v));
}

// dp4a with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ uint32_t dp4a_us(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Horizontal pass: in [H][W][3] -> out [H][Wr][3] (rows `pitch` bytes apart);
// one thread per output pixel (filters of any width, any alignment).
__global__ void resize_h_kernel(const uint8_t* __restrict__ in, int W, uint8_t* __restrict__ out, int Wr,
                                size_t pitch, const int* __restrict__ first, const int* __restrict__ wt, int T) {
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
  uint8_t* dst = out + static_cast<size_t>(y) * pitch + static_cast<size_t>(x) * 3;
  dst[0] = round_clamp(a0);
  dst[1] = round_clamp(a1);
  dst[2] = round_clamp(a2);
}

// Vertical pass into the canvas: one thread per canvas pixel, gray outside
// the resized image; src rows `pitch` bytes apart (any filter width).
__global__ void resize_v_canvas_kernel(const uint8_t* __restrict__ src, size_t pitch, int H, int Wr, int Hr,
                                       const int* __restrict__ first, const int* __restrict__ wt, int T,
                                       uint8_t* __restrict__ canvas, int Wc, int y0, int x0) {
  const int X = blockIdx.x * blockDim.x + threadIdx.x;
  const int Y = blockIdx.y;
  if (X >= Wc) return;
  const int xx = X - x0, yy = Y - y0;
  uint8_t p0 = kGray, p1 = kGray, p2 = kGray;
  if (xx >= 0 && xx < Wr && yy >= 0 && yy < Hr) {
    if (H == Hr) {
      const uint8_t* s = src + static_cast<size_t>(yy) * pitch + static_cast<size_t>(xx) * 3;
      p0 = s[0];
      p1 = s[1];
      p2 = s[2];
    } else {
      const int lo = __ldg(first + yy);
      const int n = T < H - lo ? T : H - lo;
      const uint8_t* s = src + static_cast<size_t>(lo) * pitch + static_cast<size_t>(xx) * 3;
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

// Planar horizontal pass (input 16-byte aligned, G4 <= 4): 128 output pixels
// x 8 rows per block (tiles after `tab_blocks` leading blocks that build the
// height's filter tables meanwhile, on the float64 pipe).  The block stages its span as 16-pixel units (48 bytes
// from a 16-pixel boundary: three aligned 16-byte loads) split into R, G and
// B planes by byte permutes, so a channel's taps are consecutive bytes; a
// thread reads its window per channel as words, realigns it with funnel
// shifts and takes four taps' products per dp4a in each weight plane:
// sum p w = D0 + 2^8 D1 + 2^16 D2, exactly, in 32-bit integers.
constexpr int kRowsFast = 8;
constexpr int kPixFast = 128;
constexpr int kUnitPx = 16;

struct HPlanar {
  int nunits;         // 16-pixel units staged per row
  int plane_stride;   // bytes per staged plane
  uint32_t inv_units; // ceil(2^32 / nunits): umulhi(c, inv_units) = c / nunits for c < 2^16
};

// The span: 127 output steps of the reduction factor, the taps read, one
// pixel for the rounding of each end, two for the staging start below the
// first tap, and a lead of up to 15 pixels before it; 16 bytes of slack for
// the window's last word.
HPlanar h_planar(int W, int Wr, int G4) {
  const double scale = static_cast<double>(W) / Wr;
  const int span = static_cast<int>(std::ceil(scale * (kPixFast - 1))) + 4 * G4 + 4;
  HPlanar h;
  h.nunits = (span + 2 * (kUnitPx - 1)) / kUnitPx;
  h.plane_stride = h.nunits * kUnitPx + 16;
  h.inv_units = static_cast<uint32_t>(((uint64_t{1} << 32) + h.nunits - 1) / h.nunits);
  return h;
}

// A staging start at most the first tap of output xb and at most 2 below it,
// from integers: the table's lo is the truncation of c - support + 1/2, whose
// exact value is ((2 xb - 3) W + Wr) / (2 Wr) when W > Wr and
// ((2 xb + 1) W - 3 Wr) / (2 Wr) otherwise; the double it is computed in lies
// within 1e-9 of that, so its truncation (clamped at 0) is at least
// floor(exact) - 1.
__device__ __forceinline__ int staging_start(int xb, int W, int Wr) {
  const int64_t num = W > Wr ? (2 * static_cast<int64_t>(xb) - 3) * W + Wr
                             : (2 * static_cast<int64_t>(xb) + 1) * W - 3 * static_cast<int64_t>(Wr);
  const int64_t den = 2 * static_cast<int64_t>(Wr);
  const int64_t fl = num >= 0 ? num / den : -((-num + den - 1) / den);
  return fl - 1 > 0 ? static_cast<int>(fl - 1) : 0;
}

template <int G4>
__global__ void __launch_bounds__(kPixFast) resize_h_planar_kernel(const uint8_t* __restrict__ in, int W, int H,
                                                                   uint8_t* __restrict__ out, int Wr, size_t pitch,
                                                                   const __grid_constant__ ResizeAxes a,
                                                                   int tab_blocks, int warps_y, int nbx,
                                                                   HPlanar hp) {
  extern __shared__ __align__(16) uint8_t planes_s[];   // [kRowsFast][3][hp.plane_stride]
  if (static_cast<int>(blockIdx.x) < tab_blocks) {
    // The height's tables: independent of everything before this launch.
    packed_tables_warp(a, blockIdx.x * (kPixFast / 32) + (threadIdx.x >> 5), 0, warps_y,
                       reinterpret_cast<double*>(planes_s) + (threadIdx.x & ~31));
    return;
  }
  const int tile = blockIdx.x - tab_blocks;
  const int xb = (tile % nbx) * kPixFast;
  const int x = xb + threadIdx.x;
  const int yb = (tile / nbx) * kRowsFast;
  const int nrows = H - yb < kRowsFast ? H - yb : kRowsFast;
  const int* __restrict__ first = a.first_x;
  const uint32_t* __restrict__ wp = a.wp_x;
  // Staged before the width's tables are read: the span starts at s0 <= every
  // first tap of the block (the pixels were written before the tables'
  // launch, which this one follows).
  const int s0 = staging_start(xb, W, Wr);
  const size_t total = static_cast<size_t>(H) * W * 3;
  const int ps = hp.plane_stride;
  // Two units per thread and pass, all six loads issued before either is
  // split (a pass waits for its loads once).
  const int n_units = nrows * hp.nunits;
  for (int c0 = threadIdx.x; c0 < n_units; c0 += 2 * kPixFast) {
    uint32_t xw[2][12];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + h * kPixFast;
      const int r = static_cast<int>(__umulhi(static_cast<uint32_t>(c), hp.inv_units)), u = c - r * hp.nunits;
      const size_t g = (((static_cast<size_t>(yb + r) * W + s0) & ~size_t{kUnitPx - 1}) * 3) +
                       48 * static_cast<size_t>(u);
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const size_t gq = g + 16 * q;
        if (c < n_units && gq + 16 <= total) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(in + gq));
          xw[h][4 * q] = v.x;
          xw[h][4 * q + 1] = v.y;
          xw[h][4 * q + 2] = v.z;
          xw[h][4 * q + 3] = v.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t wv = 0;
            for (int b = 0; b < 4 && c < n_units; ++b) {
              const size_t o = gq + 4 * e + b;
              if (o < total) wv |= static_cast<uint32_t>(__ldg(in + o)) << (8 * b);
            }
            xw[h][4 * q + e] = wv;
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + h * kPixFast;
      if (c >= n_units) break;
      const int r = static_cast<int>(__umulhi(static_cast<uint32_t>(c), hp.inv_units)), u = c - r * hp.nunits;
      // Pixels 4m..4m+3 of the unit are bytes 12m..12m+11 (words 3m..3m+2).
      uint32_t pr[4], pg[4], pb[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t x0 = xw[h][3 * m], x1 = xw[h][3 * m + 1], x2 = xw[h][3 * m + 2];
        pr[m] = __byte_perm(__byte_perm(x0, x1, 0x0630u), x2, 0x5210u);
        pg[m] = __byte_perm(__byte_perm(x0, x1, 0x0741u), x2, 0x6210u);
        pb[m] = __byte_perm(__byte_perm(x0, x1, 0x0052u), x2, 0x7410u);
      }
      uint8_t* row = planes_s + (r * 3) * ps + kUnitPx * u;
      *reinterpret_cast<uint4*>(row) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
      *reinterpret_cast<uint4*>(row + ps) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
      *reinterpret_cast<uint4*>(row + 2 * ps) = make_uint4(pb[0], pb[1], pb[2], pb[3]);
    }
  }
  __syncthreads();
  grid_dep_launch();
  grid_dep_wait();   // the width's tables
  if (x >= Wr) return;
  const int lo = __ldg(first + x);
  uint32_t w0[G4], w1[G4], w2[G4];
  const size_t plane = static_cast<size_t>(G4) * Wr;
#pragma unroll
  for (int j = 0; j < G4; ++j) {
    w0[j] = __ldg(wp + static_cast<size_t>(j) * Wr + x);
    w1[j] = __ldg(wp + plane + static_cast<size_t>(j) * Wr + x);
    w2[j] = __ldg(wp + 2 * plane + static_cast<size_t>(j) * Wr + x);
  }
  for (int r = 0; r < nrows; ++r) {
    const int lead = static_cast<int>((static_cast<unsigned>(yb + r) * static_cast<unsigned>(W) +
                                       static_cast<unsigned>(s0)) & (kUnitPx - 1));
    const int pos = lead + (lo - s0);
    const uint8_t* row = planes_s + (r * 3) * ps + (pos & ~3);
    const uint32_t sh = static_cast<uint32_t>(pos & 3) * 8u;
    uint8_t* dst = out + static_cast<size_t>(yb + r) * pitch + static_cast<size_t>(x) * 3;
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) {
      const uint32_t* p = reinterpret_cast<const uint32_t*>(row + ch * ps);
      uint32_t t[G4 + 1];
#pragma unroll
      for (int j = 0; j <= G4; ++j) t[j] = p[j];
      uint32_t d0 = 1u << (kPrecisionBits - 1), d1 = 0, d2 = 0;
#pragma unroll
      for (int j = 0; j < G4; ++j) {
        const uint32_t v = __funnelshift_r(t[j], t[j + 1], sh);
        d0 = __dp4a(v, w0[j], d0);
        d1 = __dp4a(v, w1[j], d1);
        d2 = dp4a_us(v, w2[j], d2);
      }
      dst[ch] = round_clamp(static_cast<int>(d0 + (d1 << 8) + (d2 << 16)));
    }
  }
}

using HPlanarKernel = void (*)(const uint8_t*, int, int, uint8_t*, int, size_t, ResizeAxes, int, int, int,
                               HPlanar);

HPlanarKernel h_planar_kernel(int G4) {
  switch (G4) {
    case 1: return resize_h_planar_kernel<1>;
    case 2: return resize_h_planar_kernel<2>;
    case 3: return resize_h_planar_kernel<3>;
    case 4: return resize_h_planar_kernel<4>;
    default: return nullptr;
  }
}

// Planar vertical pass: src rows of `row_bytes` bytes, `pitch` apart (a
// multiple of 16, src 16-byte aligned) -> canvas rows y0 + yy at byte x0 * 3.
// A thread makes 8 consecutive bytes of an output row: per group of four
// taps it loads the four source rows' 8 bytes, transposes them with byte
// permutes (a word per output byte, holding its four taps) and takes dp4a in
// each weight plane (the row's weights, the same for every byte).  Rows past
// the input are read as its last row (their weights are zero).  G4T > 0
// unrolls the groups so that all loads are issued first; 0 loops over G4.
// The block's bytes go through shared memory so that the canvas is written
// in aligned 16-byte stores (the ragged ends bytewise).
constexpr int kVThreads = 256;
constexpr int kVPerThread = 8;
constexpr int kVBytes = kVPerThread * kVThreads;

template <int G4T>
__global__ void __launch_bounds__(kVThreads) resize_v_planar_kernel(const uint8_t* __restrict__ src, size_t pitch,
                                                                    int H, int row_bytes, int Hr,
                                                                    const int* __restrict__ first,
                                                                    const uint32_t* __restrict__ wp, int G4,
                                                                    uint8_t* __restrict__ canvas, int Wc, int y0,
                                                                    int x0) {
  __shared__ __align__(16) uint8_t out_s[kVBytes + 32];
  grid_dep_wait();   // the horizontal pass and the height's tables
  const int tid = threadIdx.x;
  const int per_block = static_cast<int>(blockDim.x) * kVPerThread;
  const int b0 = blockIdx.x * per_block + tid * kVPerThread;
  const int yy = blockIdx.y;
  if (G4T > 0) G4 = G4T;
  if (b0 < row_bytes) {
    const int lo = __ldg(first + yy);
    uint32_t d0[8], d1[8], d2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      d0[i] = 1u << (kPrecisionBits - 1);
      d1[i] = 0;
      d2[i] = 0;
    }
    const size_t plane = static_cast<size_t>(G4) * Hr;
    constexpr int kPre = G4T > 0 ? G4T : 1;   // groups whose rows are loaded together
    for (int j0 = 0; j0 < G4; j0 += kPre) {
      uint2 rw[kPre][4];
#pragma unroll
      for (int jj = 0; jj < kPre; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tap = lo + 4 * (j0 + jj) + e;
          const int row = tap < H ? tap : H - 1;
          rw[jj][e] = __ldg(reinterpret_cast<const uint2*>(src + static_cast<size_t>(row) * pitch + b0));
        }
#pragma unroll
      for (int jj = 0; jj < kPre; ++jj) {
        const int j = j0 + jj;
        const uint32_t w0 = __ldg(wp + static_cast<size_t>(j) * Hr + yy);
        const uint32_t w1 = __ldg(wp + plane + static_cast<size_t>(j) * Hr + yy);
        const uint32_t w2 = __ldg(wp + 2 * plane + static_cast<size_t>(j) * Hr + yy);
        const uint32_t ra[2] = {rw[jj][0].x, rw[jj][0].y}, rb[2] = {rw[jj][1].x, rw[jj][1].y};
        const uint32_t rc[2] = {rw[jj][2].x, rw[jj][2].y}, rd[2] = {rw[jj][3].x, rw[jj][3].y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t ab_lo = __byte_perm(ra[q], rb[q], 0x5140u), ab_hi = __byte_perm(ra[q], rb[q], 0x7362u);
          const uint32_t cd_lo = __byte_perm(rc[q], rd[q], 0x5140u), cd_hi = __byte_perm(rc[q], rd[q], 0x7362u);
          const uint32_t t[4] = {__byte_perm(ab_lo, cd_lo, 0x5410u), __byte_perm(ab_lo, cd_lo, 0x7632u),
                                 __byte_perm(ab_hi, cd_hi, 0x5410u), __byte_perm(ab_hi, cd_hi, 0x7632u)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            d0[4 * q + e] = __dp4a(t[e], w0, d0[4 * q + e]);
            d1[4 * q + e] = __dp4a(t[e], w1, d1[4 * q + e]);
            d2[4 * q + e] = dp4a_us(t[e], w2, d2[4 * q + e]);
          }
        }
      }
    }
    uint32_t o[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * q + e;
        word |= static_cast<uint32_t>(round_clamp(static_cast<int>(d0[i] + (d1[i] << 8) + (d2[i] << 16))))
                << (8 * e);
      }
      o[q] = word;
    }
    *reinterpret_cast<uint2*>(out_s + tid * kVPerThread) = make_uint2(o[0], o[1]);
  }
  __syncthreads();
  const int left = row_bytes - blockIdx.x * per_block;
  const int nb = left < per_block ? left : per_block;
  uint8_t* D = canvas + (static_cast<size_t>(y0 + yy) * Wc + x0) * 3 + static_cast<size_t>(blockIdx.x) * per_block;
  const int lead = static_cast<int>((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(D)) & 15u)) & 15u);
  if (lead >= nb) {
    if (tid < nb) D[tid] = out_s[tid];
    return;
  }
  const int nch = (nb - lead) >> 4;
  const int tail = lead + (nch << 4);
  if (tid < lead) D[tid] = out_s[tid];
  if (tid < nb - tail) D[tail + tid] = out_s[tail + tid];
  if (tid < nch) {
    const int s = lead + 16 * tid;
    const uint32_t* q = reinterpret_cast<const uint32_t*>(out_s + (s & ~3));
    const uint32_t sh = static_cast<uint32_t>(s & 3) * 8u;
    const uint32_t q0 = q[0], q1 = q[1], q2 = q[2], q3 = q[3], q4 = q[4];
    *reinterpret_cast<uint4*>(D + s) = make_uint4(__funnelshift_r(q0, q1, sh), __funnelshift_r(q1, q2, sh),
                                                  __funnelshift_r(q2, q3, sh), __funnelshift_r(q3, q4, sh));
  }
}

using VPlanarKernel = void (*)(const uint8_t*, size_t, int, int, int, const int*, const uint32_t*, int, uint8_t*, int,
                               int, int);

VPlanarKernel v_planar_kernel(int G4) {
  switch (G4) {
    case 1: return resize_v_planar_kernel<1>;
    case 2: return resize_v_planar_kernel<2>;
    case 3: return resize_v_planar_kernel<3>;
    case 4: return resize_v_planar_kernel<4>;
    default: return resize_v_planar_kernel<0>;
  }
}

struct PreLayout {
  size_t off_tmp, off_fx, off_wx, off_px, off_fy, off_wy, off_py, total;
  size_t pitch_tmp;   // horizontal pass output rows: Wr * 3 bytes rounded up to 16
  int taps_x, taps_y, g4_x, g4_y;
};

PreLayout pre_layout(const ds_vit_plan& p) {
  PreLayout L{};
  L.taps_x = max_taps(p.W, p.Wr);
  L.taps_y = max_taps(p.H, p.Hr);
  L.g4_x = planar_groups(p.W, p.Wr);
  L.g4_y = planar_groups(p.H, p.Hr);
  size_t o = 0;
  L.pitch_tmp = (static_cast<size_t>(p.Wr) * 3 + 15) & ~size_t{15};
  L.off_tmp = o;
  if (p.Wr != p.W) o += align256(static_cast<size_t>(p.H) * L.pitch_tmp);
  L.off_fx = o;
  o += align256(static_cast<size_t>(p.Wr) * 4);
  L.off_wx = o;
  o += align256(static_cast<size_t>(p.Wr) * L.taps_x * 4);
  L.off_px = o;
  o += align256(static_cast<size_t>(p.Wr) * 3 * L.g4_x * 4);
  L.off_fy = o;
  o += align256(static_cast<size_t>(p.Hr) * 4);
  L.off_wy = o;
  o += align256(static_cast<size_t>(p.Hr) * L.taps_y * 4);
  L.off_py = o;
  o += align256(static_cast<size_t>(p.Hr) * 3 * L.g4_y * 4);
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
  a.g4_x = L.g4_x;
  a.in_y = ref.H;
  a.out_y = ref.Hr;
  a.taps_y = L.taps_y;
  a.g4_y = L.g4_y;
  a.sx = axis_scale(ref.W, ref.Wr);
  a.sy = axis_scale(ref.H, ref.Hr);
  a.first_x = reinterpret_cast<int*>(w8 + L.off_fx);
  a.w_x = reinterpret_cast<int*>(w8 + L.off_wx);
  a.wp_x = reinterpret_cast<uint32_t*>(w8 + L.off_px);
  a.first_y = reinterpret_cast<int*>(w8 + L.off_fy);
  a.w_y = reinterpret_cast<int*>(w8 + L.off_wy);
  a.wp_y = reinterpret_cast<uint32_t*>(w8 + L.off_py);
  uint8_t* cv = static_cast<uint8_t*>(canvas);
  const bool border = ref.x0 > 0 || ref.y0 > 0 || ref.Wr < ref.Wc || ref.Hr < ref.Hc;
  const bool resize_h = ref.Wr != ref.W;
  // The passes to run: the planar horizontal pass for filters of at most 16
  // taps on a 16-byte aligned image; the planar vertical pass when the rows
  // it reads are 16-byte aligned.
  const HPlanarKernel hk = resize_h ? h_planar_kernel(L.g4_x) : nullptr;
  const HPlanar hp = hk ? h_planar(ref.W, ref.Wr, L.g4_x) : HPlanar{};
  const size_t h_smem = static_cast<size_t>(kRowsFast) * 3 * hp.plane_stride;
  const bool planar_h = hk && h_smem <= 48 * 1024 && (reinterpret_cast<uintptr_t>(pixels) & 15) == 0;
  const uint8_t* src = resize_h ? w8 + L.off_tmp : pixels;
  const size_t pitch = resize_h ? L.pitch_tmp : static_cast<size_t>(ref.W) * 3;
  const bool planar_v = ref.Hr != ref.H && (pitch & 15) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;

  // The gray border first: only the vertical pass writes the canvas after it.
  if (planar_v && border && cudaMemsetAsync(cv, kGray, static_cast<size_t>(ref.Hc) * ref.Wc * 3, st) != cudaSuccess) {
    cudaGetLastError();
    return DS_VIT_ECUDA;
  }
  // Tables: axes of at most 32 taps packed several indices per warp, wider
  // ones one index per warp; the height's packed tables are built inside the
  // planar horizontal pass.
  const bool pack_x = L.taps_x <= 32, pack_y = L.taps_y <= 32;
  const bool y_in_h = planar_h && pack_y;
  if (!pack_x || !pack_y) {
    const int max_t = std::max(pack_x ? 0 : L.taps_x, pack_y ? 0 : L.taps_y);
    const size_t tab_smem = static_cast<size_t>(max_t) * sizeof(double);
    if (tab_smem > 48 * 1024 &&
        cudaFuncSetAttribute(resize_tables_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tab_smem)) != cudaSuccess) {
      cudaGetLastError();
      return DS_VIT_ECUDA;
    }
    // Blocks [0, n_x) take the width when it is not packed, the rest the height.
    const int n_x = pack_x ? 0 : ref.Wr;
    const int n_y = pack_y ? 0 : ref.Hr;
    resize_tables_kernel<<<n_x + n_y, 32, tab_smem, st>>>(a, n_x);
  }
  const int warps_x = pack_x ? (ref.Wr + 32 / L.taps_x - 1) / (32 / L.taps_x) : 0;
  const int warps_y = pack_y ? (ref.Hr + 32 / L.taps_y - 1) / (32 / L.taps_y) : 0;
  if (warps_x + (y_in_h ? 0 : warps_y) > 0)
    resize_tables_packed_kernel<<<warps_x + (y_in_h ? 0 : warps_y), 32, 0, st>>>(a, warps_x,
                                                                                y_in_h ? 0 : warps_y);
  if (resize_h) {
    uint8_t* tmp = w8 + L.off_tmp;
    if (planar_h) {
      const int nbx = (ref.Wr + kPixFast - 1) / kPixFast;
      const int nby = (ref.H + kRowsFast - 1) / kRowsFast;
      const int tab_blocks = y_in_h ? (warps_y + kPixFast / 32 - 1) / (kPixFast / 32) : 0;
      if (launch_pdl(hk, dim3(tab_blocks + nbx * nby), dim3(kPixFast), h_smem, st, pixels, ref.W, ref.H, tmp,
                     ref.Wr, L.pitch_tmp, a, tab_blocks, y_in_h ? warps_y : 0, nbx, hp) != cudaSuccess) {
        cudaGetLastError();
        return DS_VIT_ECUDA;
      }
    } else {
      resize_h_kernel<<<dim3((ref.Wr + 127) / 128, ref.H), 128, 0, st>>>(pixels, ref.W, tmp, ref.Wr, L.pitch_tmp,
                                                                           a.first_x, a.w_x, L.taps_x);
    }
  }
  if (planar_v) {
    // Blocks sized to the row: as few blocks per row as 256 threads allow,
    // each with a whole number of warps.
    const int row_bytes = ref.Wr * 3;
    const int chunks = (row_bytes + kVPerThread - 1) / kVPerThread;
    const int nblk = (chunks + kVThreads - 1) / kVThreads;
    const int threads = ((chunks + nblk - 1) / nblk + 31) / 32 * 32;
    if (launch_pdl(v_planar_kernel(L.g4_y), dim3(nblk, ref.Hr), dim3(threads), 0, st, src, pitch, ref.H, row_bytes,
                   ref.Hr, static_cast<const int*>(a.first_y), static_cast<const uint32_t*>(a.wp_y), L.g4_y, cv,
                   ref.Wc, ref.y0, ref.x0) != cudaSuccess) {
      cudaGetLastError();
      return DS_VIT_ECUDA;
    }
  } else {
    resize_v_canvas_kernel<<<dim3((ref.Wc + 127) / 128, ref.Hc), 128, 0, st>>>(
        src, pitch, ref.H, ref.Wr, ref.Hr, a.first_y, a.w_y, L.taps_y, cv, ref.Wc, ref.y0, ref.x0);
  }
  if (cudaGetLastError() != cudaSuccess) return DS_VIT_ECUDA;
  return DS_VIT_OK;
}

}  // extern "C"
