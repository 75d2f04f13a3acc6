// The Qwen3-VL-style vision tower ("DeepSeek V4.1 Flash Engineering, Part 3:
// Integrating Vision": comparison table; "Patch order reflects the spatial
// reducer"; "Qwen3-VL has two layers of positional meaning"; "DeepStack means
// that 'vision output' is plural"): 16x16x2 patches in 2x2-merge-group order,
// an interpolated learned 48x48 position table, 27 pre-LayerNorm blocks of
// hidden 1152 with 16 heads of 72 and 2D RoPE, a 2x2 merger, and three
// DeepStack mergers on the outputs of blocks 8, 16 and 24.
//
// Kernels here: patchify (pixels -> [N, 1536] through the prepared pixel
// table), position-table interpolation (fp32, the same operation order as the
// oracle), the RoPE cos/sin tables (per position, then per patch row and pair
// slot), and the preparation copy of W_qkv with every head padded to 80 rows
// (q and k columns reordered so that the QKV GEMM's epilogue applies the
// rotation).  The GEMMs, LayerNorm and attention are the shared kernels
// (attention in its head-72 form).  Host code: the C ABI of the tower.
#include "internal.h"

#include <algorithm>
#include <cmath>

namespace dsvit {

int launch_attention_hd72(const CUtensorMap& tm_qkv, const CUtensorMap& tm_qkv_tail, int n, bf16* out,
                          int* status, cudaStream_t stream);

namespace {

constexpr int kD = 1152, kHeads = 16, kHd = 72, kHdPad = 80, kF = 4608, kOut = 5120;
constexpr int kQkvPad = 3 * kHeads * kHdPad;       // 3840
constexpr int kMaxRopePos = 2048;
constexpr int kTaps[3] = {8, 16, 24};

size_t align_up(size_t v) { return (v + 255) & ~size_t{255}; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Patch row r in merge-group order -> (gy, gx).
__device__ __forceinline__ void group_pos(int r, int gw, int* gy, int* gx) {
  const int g = r >> 2, in = r & 3, half = gw >> 1;
  *gy = 2 * (g / half) + (in >> 1);
  *gx = 2 * (g % half) + (in & 1);
}

// A[r, ((c*2 + t)*16 + y)*16 + x] = lut[c][pixel(16 gy + y, 16 gx + x, c)] for
// both temporal slots t (a still image fills both).  One block per row.
__global__ void qwen_patch_kernel(const uint8_t* __restrict__ pix, int W, int gw,
                                  const bf16* __restrict__ lut, bf16* __restrict__ A) {
  const int r = blockIdx.x;
  int gy, gx;
  group_pos(r, gw, &gy, &gx);
  const unsigned short* lu = reinterpret_cast<const unsigned short*>(lut);
  unsigned short* out = reinterpret_cast<unsigned short*>(A) + static_cast<size_t>(r) * 1536;
  for (int k = threadIdx.x; k < 1536; k += blockDim.x) {
    const int x = k & 15, y = (k >> 4) & 15, ct = k >> 8, c = ct >> 1;
    const uint8_t v = pix[(static_cast<size_t>(16 * gy + y) * W + 16 * gx + x) * 3 + c];
    out[k] = lu[c * 256 + v];
  }
}

// x[r] = bf16(bilinear sample of the 48x48 table at the align-corners position
// of patch (gy, gx)): y = gy*47/(gh-1) in float64, weights in fp32, products
// and sums rounded one at a time in the oracle's order.  One block of 144
// threads per row, 8 consecutive dims a thread (16-byte loads and stores).
constexpr int kPosThreads = kD / 8;
__global__ void __launch_bounds__(kPosThreads) qwen_pos_kernel(const bf16* __restrict__ table, int gh, int gw,
                                                               bf16* __restrict__ x) {
  const int r = blockIdx.x;
  int gy, gx;
  group_pos(r, gw, &gy, &gx);
  const double yv = gh == 1 ? 0.0 : __ddiv_rn(static_cast<double>(gy * 47), static_cast<double>(gh - 1));
  const double xv = gw == 1 ? 0.0 : __ddiv_rn(static_cast<double>(gx * 47), static_cast<double>(gw - 1));
  const int y0 = min(static_cast<int>(floor(yv)), 47), y1 = min(y0 + 1, 47);
  const int x0 = min(static_cast<int>(floor(xv)), 47), x1 = min(x0 + 1, 47);
  const float fy = static_cast<float>(__dsub_rn(yv, static_cast<double>(y0)));
  const float fx = static_cast<float>(__dsub_rn(xv, static_cast<double>(x0)));
  const float ofy = __fsub_rn(1.f, fy), ofx = __fsub_rn(1.f, fx);
  const int d = threadIdx.x;   // 16-byte word of the row
  auto row = [&](int ty, int tx) {
    return __ldg(reinterpret_cast<const uint4*>(table + static_cast<size_t>(ty * 48 + tx) * kD) + d);
  };
  const uint4 a00 = row(y0, x0), a01 = row(y0, x1), a10 = row(y1, x0), a11 = row(y1, x1);
  const uint32_t w00[4] = {a00.x, a00.y, a00.z, a00.w}, w01[4] = {a01.x, a01.y, a01.z, a01.w};
  const uint32_t w10[4] = {a10.x, a10.y, a10.z, a10.w}, w11[4] = {a11.x, a11.y, a11.z, a11.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float v[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      auto f = [&](uint32_t w) { return hh ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16); };
      const float top = __fadd_rn(__fmul_rn(f(w00[e]), ofx), __fmul_rn(f(w01[e]), fx));
      const float bot = __fadd_rn(__fmul_rn(f(w10[e]), ofx), __fmul_rn(f(w11[e]), fx));
      v[hh] = __fadd_rn(__fmul_rn(top, ofy), __fmul_rn(bot, fy));
    }
    __nv_bfloat162 pv = __floats2bfloat162_rn(v[0], v[1]);
    o[e] = *reinterpret_cast<uint32_t*>(&pv);
  }
  reinterpret_cast<uint4*>(x + static_cast<size_t>(r) * kD)[d] = make_uint4(o[0], o[1], o[2], o[3]);
}

// [pos][j] = cos(pos * theta^(-j/18)), [pos][18 + j] = sin(...), double -> fp32.
__global__ void qwen_rope_table_kernel(float* cs, int max_pos, double theta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= max_pos * 18) return;
  const int pos = i / 18, j = i % 18;
  const double a = static_cast<double>(pos) * pow(theta, -static_cast<double>(j) / 18.0);
  cs[pos * 36 + j] = static_cast<float>(cos(a));
  cs[pos * 36 + 18 + j] = static_cast<float>(sin(a));
}

// Column order inside an 80-wide q or k head: the 36 rotation pairs (dims
// (36 half + j, 36 half + 18 + j), half 0 at the patch row, half 1 at the
// patch column) fill pair slots s = 0..35 of five 16-column groups, slot
// s = 8 g + i holding its two dims at columns 16 g + i and 16 g + 8 + i; slots
// 36..39 are zero.  q and k share the order, so Q K^T is unchanged; the QKV
// GEMM epilogue rotates each pair inside one 32-column chunk.  V keeps the
// natural order.  Returns the source dim of column c, or -1 for a zero column.
__host__ __device__ constexpr int qk_source_dim(int c) {
  const int g = c / 16, w = c % 16, slot = 8 * g + (w % 8);
  return slot >= 36 ? -1 : 36 * (slot / 18) + slot % 18 + 18 * (w / 8);
}
// Every dim 0..71 appears exactly once among the 80 columns.
constexpr bool qk_order_is_permutation() {
  int seen[kHd] = {};
  for (int c = 0; c < kHdPad; ++c) {
    const int d = qk_source_dim(c);
    if (d >= kHd) return false;
    if (d >= 0) ++seen[d];
  }
  for (int d = 0; d < kHd; ++d)
    if (seen[d] != 1) return false;
  return true;
}
static_assert(qk_order_is_permutation(), "q/k column order");
static_assert(kQwenQkCols == 2 * kHeads * kHdPad, "q and k columns of the QKV output");

// rt[r][slot] = (cos, sin) of pair slot `slot` at patch row r (merge-group
// order): slots 0..17 at the patch row gy with frequency j = slot, 18..35 at
// the column gx with j = slot - 18, 36..39 (1, 0).  Built once per encode
// from the [pos][cos 0..17, sin 0..17] table.
__global__ void qwen_rope_rows_kernel(float2* __restrict__ rt, int n_rows, int gw, const float* __restrict__ cs) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * 40) return;
  const int r = i / 40, slot = i % 40;
  int gy, gx;
  group_pos(r, gw, &gy, &gx);
  float2 v = make_float2(1.f, 0.f);
  if (slot < 36) {
    const int pos = slot < 18 ? gy : gx, j = slot % 18;
    v = make_float2(cs[pos * 36 + j], cs[pos * 36 + 18 + j]);
  }
  rt[i] = v;
}

// W'[(s*16 + h)*80 + c] = W[(s*16 + h)*72 + d(c)] with d(c) = qk_source_dim(c)
// for q and k (s = 0, 1) and d(c) = c for v, zero rows where d(c) is -1 or
// >= 72; bias likewise.  One block per padded row.
__global__ void qwen_pad_qkv_kernel(const bf16* __restrict__ w, const bf16* __restrict__ b,
                                    bf16* __restrict__ wp, bf16* __restrict__ bp) {
  const int r = blockIdx.x;
  const int head = r / kHdPad, c = r % kHdPad;
  const int d = head < 2 * kHeads ? qk_source_dim(c) : c;
  const bool real = d >= 0 && d < kHd;
  const size_t src = static_cast<size_t>(head) * kHd + (real ? d : 0);
  for (int k = threadIdx.x; k < kD; k += blockDim.x)
    wp[static_cast<size_t>(r) * kD + k] = real ? w[src * kD + k] : __float2bfloat16_rn(0.f);
  if (threadIdx.x == 0) bp[r] = real ? b[src] : __float2bfloat16_rn(0.f);
}

int check_qwen_config(const ds_vit_config* c) {
  if (!c) return DS_VIT_EINVAL;
  if (c->n_layers < 1 || c->n_layers > DS_VIT_MAX_LAYERS || c->hidden != kD || c->heads != kHeads ||
      c->head_dim != kHd || c->mlp != kF || c->out_dim != kOut || c->patch != 16 || c->merge != 2 ||
      !(c->rope_theta > 0.f) || !(c->ln_eps > 0.f) || c->norm_kind != DS_VIT_NORM_LAYER ||
      c->mlp_kind != DS_VIT_MLP_GELU)
    return DS_VIT_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (!(c->std[i] != 0.f)) return DS_VIT_EINVAL;
  return DS_VIT_OK;
}

bool merger_ok(const ds_vit_qwen_merger& m) {
  const void* f[] = {m.ln_g, m.ln_b, m.w1, m.b1, m.w2, m.b2};
  for (const void* q : f)
    if (!q || !aligned16(q)) return false;
  return true;
}

int check_qwen_weights(const ds_vit_qwen_weights* w, int n_layers) {
  if (!w) return DS_VIT_EINVAL;
  const void* top[] = {w->patch_w, w->patch_b, w->pos_table};
  for (const void* q : top)
    if (!q || !aligned16(q)) return DS_VIT_EINVAL;
  for (int l = 0; l < n_layers; ++l) {
    const ds_vit_layer_weights& L = w->layers[l];
    const void* lw[] = {L.ln1_g, L.ln1_b, L.qkv_w, L.qkv_b, L.proj_w, L.proj_b,
                        L.ln2_g, L.ln2_b, L.fc1_w, L.fc1_b, L.fc2_w, L.fc2_b};
    for (const void* q : lw)
      if (!q || !aligned16(q)) return DS_VIT_EINVAL;
  }
  if (!merger_ok(w->merger)) return DS_VIT_EINVAL;
  for (int t = 0; t < 3; ++t)
    if (n_layers >= kTaps[t] && !merger_ok(w->deepstack[t])) return DS_VIT_EINVAL;
  return DS_VIT_OK;
}

struct QwenPlan {
  int64_t N, T;
  size_t off_x, off_y, off_o, off_qkv, off_h, off_rope, total;
};

int qwen_plan(int32_t H, int32_t W, QwenPlan* pl) {
  if (H <= 0 || W <= 0 || H % 32 != 0 || W % 32 != 0) return DS_VIT_EINVAL;
  const int64_t gh = H / 16, gw = W / 16, N = gh * gw, T = N / 4;
  if (T > DS_VIT_MAX_TOKENS || gh > kMaxRopePos || gw > kMaxRopePos) return DS_VIT_ERANGE;
  size_t o = 0;
  pl->N = N;
  pl->T = T;
  pl->off_x = o;   o += align_up(static_cast<size_t>(N) * kD * 2);
  pl->off_y = o;   o += align_up(static_cast<size_t>(N) * kD * 2);
  pl->off_o = o;   o += align_up(static_cast<size_t>(N) * kD * 2);
  pl->off_qkv = o; o += align_up(static_cast<size_t>(N) * kQkvPad * 2);   // also the merger hidden
  pl->off_h = o;   o += align_up(static_cast<size_t>(N) * kF * 2);        // also the patch matrix
  pl->off_rope = o; o += align_up(static_cast<size_t>(N) * 40 * 8);     // per-row cos/sin of the pair slots
  pl->total = o;
  return DS_VIT_OK;
}

}  // namespace

}  // namespace dsvit

using namespace dsvit;

struct ds_vit_qwen_prepared {
  ds_vit_config cfg;
  ds_vit_qwen_weights w;
  bf16* qkv_pad;      // per layer: W [3840, 1152] then b [3840]
  bf16* pix_lut;      // [3, 256]
  float* rope_cs;     // [kMaxRopePos, 36]
  int* status;
  WeightMap tm_patch, tm_qkv[DS_VIT_MAX_LAYERS], tm_proj[DS_VIT_MAX_LAYERS], tm_fc1[DS_VIT_MAX_LAYERS],
      tm_fc2[DS_VIT_MAX_LAYERS], tm_m1[4], tm_m2[4];
};

namespace {

constexpr size_t kPadStride = size_t{kQkvPad} * (kD + 1);
bf16* pad_w(const ds_vit_qwen_prepared* p, int l) { return p->qkv_pad + l * kPadStride; }
bf16* pad_b(const ds_vit_qwen_prepared* p, int l) { return pad_w(p, l) + size_t{kQkvPad} * kD; }

const ds_vit_qwen_merger& merger_of(const ds_vit_qwen_prepared* p, int m) {
  return m == 0 ? p->w.merger : p->w.deepstack[m - 1];
}

}  // namespace

#define QW_CUDA(call)           \
  do {                          \
    if ((call) != cudaSuccess) { \
      cudaGetLastError();       \
      return DS_VIT_ECUDA;      \
    }                           \
  } while (0)
#define QW_TRY(call)             \
  do {                           \
    const int rc_ = (call);      \
    if (rc_ != DS_VIT_OK) return rc_; \
  } while (0)

extern "C" {

int ds_vit_qwen_release(ds_vit_qwen_prepared* p) {
  if (!p) return DS_VIT_OK;
  cudaDeviceSynchronize();
  cudaFree(p->qkv_pad);
  cudaFree(p->pix_lut);
  cudaFree(p->rope_cs);
  cudaFree(p->status);
  delete p;
  return DS_VIT_OK;
}

int ds_vit_qwen_prepare(const ds_vit_config* cfg, const ds_vit_qwen_weights* w, ds_vit_qwen_prepared** out,
                        void* stream) {
  if (!out) return DS_VIT_EINVAL;
  *out = nullptr;
  QW_TRY(check_qwen_config(cfg));
  QW_TRY(check_qwen_weights(w, cfg->n_layers));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ds_vit_qwen_prepared* p = new (std::nothrow) ds_vit_qwen_prepared();
  if (!p) return DS_VIT_ENOMEM;
  p->cfg = *cfg;
  p->w = *w;
  auto fail = [&](int rc) {
    ds_vit_qwen_release(p);
    return rc;
  };
  if (cudaMalloc(&p->qkv_pad, static_cast<size_t>(cfg->n_layers) * kPadStride * 2) != cudaSuccess ||
      cudaMalloc(&p->pix_lut, 3 * 256 * 2) != cudaSuccess ||
      cudaMalloc(&p->rope_cs, static_cast<size_t>(kMaxRopePos) * 36 * 4) != cudaSuccess ||
      cudaMalloc(&p->status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return fail(DS_VIT_ENOMEM);
  }
  if (cudaMemsetAsync(p->status, 0, sizeof(int), st) != cudaSuccess) return fail(DS_VIT_ECUDA);
  for (int l = 0; l < cfg->n_layers; ++l)
    qwen_pad_qkv_kernel<<<kQkvPad, 256, 0, st>>>(static_cast<const bf16*>(w->layers[l].qkv_w),
                                                 static_cast<const bf16*>(w->layers[l].qkv_b), pad_w(p, l),
                                                 pad_b(p, l));
  qwen_rope_table_kernel<<<(kMaxRopePos * 18 + 255) / 256, 256, 0, st>>>(p->rope_cs, kMaxRopePos,
                                                                          static_cast<double>(cfg->rope_theta));
  PixelNorm norm;
  for (int c = 0; c < 3; ++c) {
    norm.mean[c] = cfg->mean[c];
    norm.std[c] = cfg->std[c];
  }
  if (cudaGetLastError() != cudaSuccess || launch_pixel_lut(norm, p->pix_lut, st) != DS_VIT_OK)
    return fail(DS_VIT_ECUDA);
  bool ok = make_weight_map(&p->tm_patch, w->patch_w, kD, 1536);
  for (int l = 0; ok && l < cfg->n_layers; ++l) {
    const ds_vit_layer_weights& L = w->layers[l];
    ok = make_weight_map(&p->tm_qkv[l], pad_w(p, l), kQkvPad, kD) &&
         make_weight_map(&p->tm_proj[l], L.proj_w, kD, kD) && make_weight_map(&p->tm_fc1[l], L.fc1_w, kF, kD) &&
         make_weight_map(&p->tm_fc2[l], L.fc2_w, kD, kF);
  }
  for (int m = 0; ok && m < 4; ++m) {
    if (m > 0 && cfg->n_layers < kTaps[m - 1]) continue;
    const ds_vit_qwen_merger& M = merger_of(p, m);
    ok = make_weight_map(&p->tm_m1[m], M.w1, 4 * kD, 4 * kD) && make_weight_map(&p->tm_m2[m], M.w2, kOut, 4 * kD);
  }
  if (!ok) return fail(DS_VIT_ECUDA);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return fail(DS_VIT_ECUDA);
  }
  *out = p;
  return DS_VIT_OK;
}

int ds_vit_qwen_workspace_bytes(int32_t H, int32_t W, size_t* bytes) {
  if (!bytes) return DS_VIT_EINVAL;
  QwenPlan pl;
  QW_TRY(qwen_plan(H, W, &pl));
  *bytes = pl.total;
  return DS_VIT_OK;
}

int ds_vit_qwen_encode(const ds_vit_qwen_prepared* p, const uint8_t* pixels, int32_t H, int32_t W, void* out,
                       void* deepstack, void* ws, size_t ws_bytes, void* blocks, void* stream) {
  if (!p || !pixels || !out || !ws) return DS_VIT_EINVAL;
  QwenPlan pl;
  QW_TRY(qwen_plan(H, W, &pl));
  if (!aligned16(out) || !aligned16(ws) || (deepstack && !aligned16(deepstack)) || (blocks && !aligned16(blocks)))
    return DS_VIT_EINVAL;
  if (ws_bytes < pl.total) return DS_VIT_ECAP;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ds_vit_config& cfg = p->cfg;
  const ds_vit_qwen_weights& w = p->w;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const int N = static_cast<int>(pl.N), T = static_cast<int>(pl.T), gh = H / 16, gw = W / 16;
  bf16* x = reinterpret_cast<bf16*>(wsb + pl.off_x);
  bf16* y = reinterpret_cast<bf16*>(wsb + pl.off_y);
  bf16* o = reinterpret_cast<bf16*>(wsb + pl.off_o);
  bf16* qkv = reinterpret_cast<bf16*>(wsb + pl.off_qkv);
  bf16* h = reinterpret_cast<bf16*>(wsb + pl.off_h);
  float2* rope_rows = reinterpret_cast<float2*>(wsb + pl.off_rope);
  bf16* dout = static_cast<bf16*>(out);
  bf16* ddeep = static_cast<bf16*>(deepstack);
  bf16* dblocks = static_cast<bf16*>(blocks);

  CUtensorMap tA_pix, tA_y, tA_o, tA_h, tA_m, tA_u, t_qkv, t_qkv_tail, tC_x, tC_qkv, tC_h, tC_u, tC_out[4];
  if (!make_tmap_bf16(&tA_pix, h, N, 1536, 128) || !make_tmap_bf16(&tA_y, y, N, kD, 128) ||
      !make_tmap_bf16(&tA_o, o, N, kD, 128) || !make_tmap_bf16(&tA_h, h, N, kF, 128) ||
      !make_tmap_bf16(&tA_m, y, T, 4 * kD, 128) || !make_tmap_bf16(&tA_u, qkv, T, 4 * kD, 128) ||
      !make_tmap_bf16(&t_qkv, qkv, N, kQkvPad, 128) || !make_tmap_bf16_tail16(&t_qkv_tail, qkv, N, kQkvPad, 128) ||
      !make_tmap_store_bf16(&tC_x, x, N, kD) ||
      !make_tmap_store_bf16(&tC_qkv, qkv, N, kQkvPad) || !make_tmap_store_bf16(&tC_h, h, N, kF) ||
      !make_tmap_store_bf16(&tC_u, qkv, T, 4 * kD) || !make_tmap_store_bf16(&tC_out[0], dout, T, kOut))
    return DS_VIT_ECUDA;
  for (int t = 0; t < 3; ++t)
    if (ddeep && cfg.n_layers >= kTaps[t] &&
        !make_tmap_store_bf16(&tC_out[1 + t], ddeep + static_cast<size_t>(t) * T * kOut, T, kOut))
      return DS_VIT_ECUDA;

  // Merger m (0 primary, 1..3 DeepStack) of the current x into `dst`.
  auto run_merger = [&](int m) -> int {
    const ds_vit_qwen_merger& M = merger_of(p, m);
    QW_TRY(launch_layernorm(x, static_cast<const bf16*>(M.ln_g), static_cast<const bf16*>(M.ln_b), y, N,
                            cfg.ln_eps, st, false, kD));
    QW_TRY(launch_gemm(tA_m, p->tm_m1[m], tC_u, T, 4 * kD, 4 * kD, static_cast<const bf16*>(M.b1), qkv,
                       kEpiBiasGelu, nullptr, nullptr, p->status, st));
    bf16* dst = m == 0 ? dout : ddeep + static_cast<size_t>(m - 1) * T * kOut;
    return launch_gemm(tA_u, p->tm_m2[m], tC_out[m], T, kOut, 4 * kD, static_cast<const bf16*>(M.b2), dst,
                       kEpiBias, nullptr, nullptr, p->status, st);
  };

  qwen_patch_kernel<<<N, 256, 0, st>>>(pixels, W, gw, p->pix_lut, h);
  qwen_rope_rows_kernel<<<(N * 40 + 255) / 256, 256, 0, st>>>(rope_rows, N, gw, p->rope_cs);
  qwen_pos_kernel<<<N, kPosThreads, 0, st>>>(static_cast<const bf16*>(w.pos_table), gh, gw, x);
  QW_CUDA(cudaGetLastError());
  QW_TRY(launch_gemm(tA_pix, p->tm_patch, tC_x, N, kD, 1536, static_cast<const bf16*>(w.patch_b), x,
                     kEpiBiasResid, nullptr, nullptr, p->status, st));
  if (dblocks) QW_CUDA(cudaMemcpyAsync(dblocks, x, static_cast<size_t>(N) * kD * 2, cudaMemcpyDeviceToDevice, st));
  for (int l = 0; l < cfg.n_layers; ++l) {
    const ds_vit_layer_weights& L = w.layers[l];
    QW_TRY(launch_layernorm(x, static_cast<const bf16*>(L.ln1_g), static_cast<const bf16*>(L.ln1_b), y, N,
                            cfg.ln_eps, st, false, kD));
    QW_TRY(launch_gemm(tA_y, p->tm_qkv[l], tC_qkv, N, kQkvPad, kD, pad_b(p, l), qkv, kEpiQkvRope72, nullptr,
                       reinterpret_cast<const float*>(rope_rows), p->status, st));
    QW_TRY(launch_attention_hd72(t_qkv, t_qkv_tail, N, o, p->status, st));
    QW_TRY(launch_gemm(tA_o, p->tm_proj[l], tC_x, N, kD, kD, static_cast<const bf16*>(L.proj_b), x,
                       kEpiBiasResid, nullptr, nullptr, p->status, st));
    QW_TRY(launch_layernorm(x, static_cast<const bf16*>(L.ln2_g), static_cast<const bf16*>(L.ln2_b), y, N,
                            cfg.ln_eps, st, false, kD));
    QW_TRY(launch_gemm(tA_y, p->tm_fc1[l], tC_h, N, kF, kD, static_cast<const bf16*>(L.fc1_b), h, kEpiBiasGelu,
                       nullptr, nullptr, p->status, st));
    QW_TRY(launch_gemm(tA_h, p->tm_fc2[l], tC_x, N, kD, kF, static_cast<const bf16*>(L.fc2_b), x, kEpiBiasResid,
                       nullptr, nullptr, p->status, st));
    if (dblocks)
      QW_CUDA(cudaMemcpyAsync(dblocks + static_cast<size_t>(l + 1) * N * kD, x, static_cast<size_t>(N) * kD * 2,
                              cudaMemcpyDeviceToDevice, st));
    for (int t = 0; t < 3; ++t)
      if (ddeep && l + 1 == kTaps[t]) QW_TRY(run_merger(1 + t));
  }
  return run_merger(0);
}

int ds_vit_qwen_layout(int32_t h, int32_t w, int32_t seq_start, int32_t* pos, int64_t cap, int32_t* rope_delta) {
  if (h < 1 || w < 1 || seq_start < 0 || !rope_delta) return DS_VIT_EINVAL;
  const int64_t n = static_cast<int64_t>(h) * w + 2;
  const int64_t q = static_cast<int64_t>(seq_start) + 1 + std::max(h, w);
  if (q > INT32_MAX - 1 || static_cast<int64_t>(seq_start) + n > INT32_MAX) return DS_VIT_ERANGE;
  if (pos && cap < 3 * n) return DS_VIT_ECAP;
  *rope_delta = static_cast<int32_t>((q + 1) - (seq_start + n));
  if (!pos) return DS_VIT_OK;
  for (int a = 0; a < 3; ++a) {
    pos[a * n] = seq_start;
    pos[a * n + n - 1] = static_cast<int32_t>(q);
  }
  for (int64_t i = 0; i < n - 2; ++i) {
    pos[0 * n + 1 + i] = seq_start + 1;
    pos[1 * n + 1 + i] = static_cast<int32_t>(seq_start + 1 + i / w);
    pos[2 * n + 1 + i] = static_cast<int32_t>(seq_start + 1 + i % w);
  }
  return DS_VIT_OK;
}

}  // extern "C"
