// C ABI of libdsvit: validation, weight preparation, the workspace plan and
// the sequence of kernel launches of one encode on one stream.
//
// Encode ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision"):
//   patch projection GEMM (+bias), its A tiles patchified and normalised
//   in shared memory            ("Step 1" items 5-6, "Step 5";
//                                 "Multimodal basics", second step)
//   n_layers x [LN1, QKV GEMM (+bias, 2D RoPE), attention, out-proj GEMM
//              (+bias, +residual), LN2, FC1 GEMM (+bias, GELU), FC2 GEMM
//              (+bias, +residual)]   ("Step 2" table, "Step 3")
//   final LN, merger GEMM1 (+bias, GELU) with the 3x3 merge-gather done
//   in its A producer, merger GEMM2 (+bias)
//                                 ("Step 4", comparison table)
// Layout and overlay: "Connect the complete image-to-text path first";
// ds4-learning glossary "vision", V4.1 paragraph.
#include "internal.h"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

using namespace dsvit;

struct ds_vit_prepared {
  ds_vit_config cfg;
  ds_vit_weights w;
  int device;
  bf16* patch_w_pad;   // [1024, kPatchK], patch-row-major K order
  bf16* m1_perm;       // [5120, 9216], column p*1024 + c
  float* rope_cs;      // [kMaxPos, 32]
  bf16* pix_lut;       // [3, 256] normalised value of each (channel, byte)
  bf16* qkv_perm;      // half-vector RoPE pairing: per layer W_qkv [3072, 1024] then b_qkv [3072]
  int* status;         // device status word
  WeightMap tm_patch, tm_m1, tm_m2;
  WeightMap tm_qkv[DS_VIT_MAX_LAYERS], tm_proj[DS_VIT_MAX_LAYERS];
  WeightMap tm_fc1[DS_VIT_MAX_LAYERS], tm_fc2[DS_VIT_MAX_LAYERS];
  // Optional per-launch timing (ds_vit_set_kernel_timer).
  cudaEvent_t* t_events;
  int32_t* t_kinds;
  int32_t t_slots;
  int32_t* t_count;
};

namespace {

// Layer l of the permuted QKV copy: W [3072, 1024] at l * stride, b [3072] after it.
constexpr size_t kQkvPermStride = size_t{3072} * 1025;
bf16* qkv_perm_w(const ds_vit_prepared* p, int l) { return p->qkv_perm + l * kQkvPermStride; }
bf16* qkv_perm_b(const ds_vit_prepared* p, int l) { return qkv_perm_w(p, l) + size_t{3072} * 1024; }

constexpr int kMaxPos = DS_VIT_MAX_PATCHES;   // a grid side can reach 9216 (a 1 x 9216 grid)
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

#define DSV_CUDA(call)                        \
  do {                                        \
    if ((call) != cudaSuccess) {              \
      cudaGetLastError();                     \
      return DS_VIT_ECUDA;                    \
    }                                         \
  } while (0)

#define DSV_TRY(call)                         \
  do {                                        \
    const int rc_ = (call);                   \
    if (rc_ != DS_VIT_OK) return rc_;         \
  } while (0)

struct Plan {
  int n;
  int64_t N, T;
  size_t off_x, off_y, off_o, off_qkv, off_h, off_rowpos, off_pix, off_out, total;
  std::vector<size_t> pix_off;   // host variant: per-image pixel staging offsets
};

int check_images(int n, const int32_t* H, const int32_t* W) {
  if (n < 1 || n > DS_VIT_MAX_IMAGES || !H || !W) return DS_VIT_EINVAL;
  for (int i = 0; i < n; ++i) {
    if (H[i] <= 0 || W[i] <= 0 || H[i] % 14 != 0 || W[i] % 14 != 0) return DS_VIT_EINVAL;
    const int64_t gh = H[i] / 14, gw = W[i] / 14;
    if (gh * gw > DS_VIT_MAX_PATCHES) return DS_VIT_ERANGE;
    if (((gh + 2) / 3) * ((gw + 2) / 3) > DS_VIT_MAX_TOKENS) return DS_VIT_ERANGE;
  }
  return DS_VIT_OK;
}

Plan make_plan(int n, const int32_t* H, const int32_t* W, bool host_io) {
  Plan pl{};
  pl.n = n;
  for (int i = 0; i < n; ++i) {
    const int64_t gh = H[i] / 14, gw = W[i] / 14;
    pl.N += gh * gw;
    pl.T += ((gh + 2) / 3) * ((gw + 2) / 3);
  }
  const size_t N = static_cast<size_t>(pl.N), T = static_cast<size_t>(pl.T);
  size_t o = 0;
  pl.off_x = o;      o += align_up(N * 1024 * 2);
  pl.off_y = o;      o += align_up(N * 1024 * 2);
  pl.off_o = o;      o += align_up(N * 1024 * 2);
  pl.off_qkv = o;    o += align_up(std::max(N * 3072, T * 5120) * 2);
  pl.off_h = o;      o += align_up(N * 4096 * 2);
  pl.off_rowpos = o; o += align_up(N * 4);
  if (host_io) {
    pl.off_pix = o;
    for (int i = 0; i < n; ++i) {
      pl.pix_off.push_back(o);
      o += align_up(static_cast<size_t>(H[i]) * W[i] * 3);
    }
    pl.off_out = o;
    o += align_up(T * 5120 * 2);
  }
  pl.total = o;
  return pl;
}

int check_config(const ds_vit_config* c) {
  if (!c) return DS_VIT_EINVAL;
  if (c->n_layers < 1 || c->n_layers > DS_VIT_MAX_LAYERS || c->hidden != 1024 || c->heads != 16 ||
      c->head_dim != 64 || c->mlp != 4096 || c->out_dim != 5120 || c->patch != 14 ||
      c->merge != 3 || !(c->rope_theta > 0.f) || !(c->ln_eps > 0.f) ||
      (c->norm_kind != DS_VIT_NORM_LAYER && c->norm_kind != DS_VIT_NORM_RMS) ||
      (c->mlp_kind != DS_VIT_MLP_GELU && c->mlp_kind != DS_VIT_MLP_SWIGLU) ||
      (c->rope_pairing != DS_VIT_ROPE_AXIS_HALVES && c->rope_pairing != DS_VIT_ROPE_HALF_VECTOR))
    return DS_VIT_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (!(c->std[i] != 0.f)) return DS_VIT_EINVAL;
  return DS_VIT_OK;
}

// Every weight pointer non-null and 16-byte aligned; the norm betas may be
// NULL under RMSNorm (unused there).
int check_weights(const ds_vit_weights* w, int n_layers, bool rms) {
  if (!w) return DS_VIT_EINVAL;
  auto bad = [](const void* q, bool optional) { return q ? !aligned16(q) : !optional; };
  const void* top[] = {w->patch_w, w->patch_b, w->lnm_g, w->m1_w, w->m1_b, w->m2_w, w->m2_b, w->sentinel};
  for (const void* q : top)
    if (bad(q, false)) return DS_VIT_EINVAL;
  if (bad(w->lnm_b, rms)) return DS_VIT_EINVAL;
  for (int l = 0; l < n_layers; ++l) {
    const ds_vit_layer_weights& L = w->layers[l];
    const void* lw[] = {L.ln1_g, L.qkv_w, L.qkv_b, L.proj_w, L.proj_b,
                        L.ln2_g, L.fc1_w, L.fc1_b, L.fc2_w, L.fc2_b};
    for (const void* q : lw)
      if (bad(q, false)) return DS_VIT_EINVAL;
    if (bad(L.ln1_b, rms) || bad(L.ln2_b, rms)) return DS_VIT_EINVAL;
  }
  return DS_VIT_OK;
}

// The sequence of launches of one (batched) encode.  Everything is validated
// and every tensor map is built before the first launch.
int run_encode(const ds_vit_prepared* p, int n, const uint8_t* const* pix, const int32_t* H,
               const int32_t* W, bf16* out, int64_t* tok_offsets, uint8_t* ws, const Plan& pl,
               bf16* dump_blocks, bf16* dump_final, cudaStream_t st) {
  const ds_vit_config& cfg = p->cfg;
  const ds_vit_weights& w = p->w;
  ImageBatch ib{};
  ib.n = n;
  AttnBatch ab{};
  ab.n_images = n;
  for (int i = 0; i < n; ++i) {
    ib.gh[i] = H[i] / 14;
    ib.gw[i] = W[i] / 14;
    ib.pix[i] = pix[i];
    ib.row_off[i + 1] = ib.row_off[i] + static_cast<int64_t>(ib.gh[i]) * ib.gw[i];
    ib.tok_off[i + 1] = ib.tok_off[i] + static_cast<int64_t>((ib.gh[i] + 2) / 3) * ((ib.gw[i] + 2) / 3);
    ab.cu[i + 1] = static_cast<int>(ib.row_off[i + 1]);
  }
  // Attention launch order: longest images first (their CTAs run longest).
  for (int i = 0; i < n; ++i) ab.order[i] = i;
  std::stable_sort(ab.order, ab.order + n, [&](int a, int b) {
    return (ab.cu[a + 1] - ab.cu[a]) > (ab.cu[b + 1] - ab.cu[b]);
  });
  for (int k = 0; k < n; ++k) {
    const int i = ab.order[k];
    ab.tile_start[k + 1] =
        ab.tile_start[k] + (ab.cu[i + 1] - ab.cu[i] + kAttnRowsPerCta - 1) / kAttnRowsPerCta;
  }
  const int64_t N = pl.N, T = pl.T;
  bf16* x = reinterpret_cast<bf16*>(ws + pl.off_x);
  bf16* y = reinterpret_cast<bf16*>(ws + pl.off_y);
  bf16* o = reinterpret_cast<bf16*>(ws + pl.off_o);
  bf16* qkv = reinterpret_cast<bf16*>(ws + pl.off_qkv);
  bf16* h = reinterpret_cast<bf16*>(ws + pl.off_h);
  int* rowpos = reinterpret_cast<int*>(ws + pl.off_rowpos);

  CUtensorMap tA_y, tA_o, tA_h, tA_u, t_qkv;
  if (!make_tmap_bf16(&tA_y, y, N, 1024, 128) || !make_tmap_bf16(&tA_o, o, N, 1024, 128) ||
      !make_tmap_bf16(&tA_h, h, N, 4096, 128) || !make_tmap_bf16(&tA_u, qkv, T, 5120, 128) ||
      !make_tmap_bf16(&t_qkv, qkv, N, 3072, 128))
    return DS_VIT_ECUDA;
  CUtensorMap tC_x, tC_qkv, tC_h, tC_u, tC_out;
  if (!make_tmap_store_bf16(&tC_x, x, N, 1024) || !make_tmap_store_bf16(&tC_qkv, qkv, N, 3072) ||
      !make_tmap_store_bf16(&tC_h, h, N, 4096) || !make_tmap_store_bf16(&tC_u, qkv, T, 5120) ||
      !make_tmap_store_bf16(&tC_out, out, T, 5120))
    return DS_VIT_ECUDA;
  for (int i = 0; i <= n; ++i) tok_offsets[i] = ib.tok_off[i];

  AGenParams ag{};
  ag.batch = ib;
  ag.lut = p->pix_lut;
  ag.z = y;
  ag.rowpos = rowpos;
  // Each launch goes through `timed`, which brackets it with the caller's
  // events when a kernel timer is attached.
  int n_timed = 0;
  auto tstart = [&]() {
    if (p->t_events && n_timed < p->t_slots) cudaEventRecord(p->t_events[2 * n_timed], st);
  };
  auto tstop = [&](int kind) {
    if (p->t_events && n_timed < p->t_slots) {
      cudaEventRecord(p->t_events[2 * n_timed + 1], st);
      p->t_kinds[n_timed] = kind;
    }
    ++n_timed;
  };
#define DSV_LAUNCH(kind, call) \
  do {                         \
    tstart();                  \
    const int rc_ = (call);    \
    tstop(kind);               \
    if (rc_ != DS_VIT_OK) return rc_; \
  } while (0)
  DSV_LAUNCH(DS_VIT_KERNEL_PATCH_GEMM,
             launch_gemm_agen(kAPixels, ag, p->tm_patch, tC_x, N, 1024, kPatchK,
                              static_cast<const bf16*>(w.patch_b), x, kEpiBias, p->status, st));
  if (dump_blocks) DSV_CUDA(cudaMemcpyAsync(dump_blocks, x, N * 1024 * 2, cudaMemcpyDeviceToDevice, st));
  const bool rms = cfg.norm_kind == DS_VIT_NORM_RMS;
  const bool swiglu = cfg.mlp_kind == DS_VIT_MLP_SWIGLU;
  for (int l = 0; l < cfg.n_layers; ++l) {
    const ds_vit_layer_weights& L = w.layers[l];
    // The half-vector pairing runs on W_qkv / b_qkv with q, k rows permuted at preparation.
    const bf16* qkv_b = p->qkv_perm ? qkv_perm_b(p, l) : static_cast<const bf16*>(L.qkv_b);
    DSV_LAUNCH(DS_VIT_KERNEL_LAYERNORM,
               launch_layernorm(x, static_cast<const bf16*>(L.ln1_g),
                                static_cast<const bf16*>(L.ln1_b), y, N, cfg.ln_eps, st, rms));
    DSV_LAUNCH(DS_VIT_KERNEL_QKV_GEMM,
               launch_gemm(tA_y, p->tm_qkv[l], tC_qkv, N, 3072, 1024, qkv_b,
                           qkv, kEpiQkvRope, rowpos, p->rope_cs, p->status, st));
    DSV_LAUNCH(DS_VIT_KERNEL_ATTENTION, launch_attention(t_qkv, ab, o, p->status, st));
    DSV_LAUNCH(DS_VIT_KERNEL_PROJ_GEMM,
               launch_gemm(tA_o, p->tm_proj[l], tC_x, N, 1024, 1024, static_cast<const bf16*>(L.proj_b),
                           x, kEpiBiasResid, nullptr, nullptr, p->status, st));
    DSV_LAUNCH(DS_VIT_KERNEL_LAYERNORM,
               launch_layernorm(x, static_cast<const bf16*>(L.ln2_g),
                                static_cast<const bf16*>(L.ln2_b), y, N, cfg.ln_eps, st, rms));
    DSV_LAUNCH(DS_VIT_KERNEL_FC1_GEMM,
               launch_gemm(tA_y, p->tm_fc1[l], tC_h, N, swiglu ? 8192 : 4096, 1024,
                           static_cast<const bf16*>(L.fc1_b), h, swiglu ? kEpiSwiglu : kEpiBiasGelu, nullptr,
                           nullptr, p->status, st));
    DSV_LAUNCH(DS_VIT_KERNEL_FC2_GEMM,
               launch_gemm(tA_h, p->tm_fc2[l], tC_x, N, 1024, 4096, static_cast<const bf16*>(L.fc2_b), x,
                           kEpiBiasResid, nullptr, nullptr, p->status, st));
    if (dump_blocks)
      DSV_CUDA(cudaMemcpyAsync(dump_blocks + (l + 1) * N * 1024, x, N * 1024 * 2,
                               cudaMemcpyDeviceToDevice, st));
  }
  DSV_LAUNCH(DS_VIT_KERNEL_LAYERNORM,
             launch_layernorm(x, static_cast<const bf16*>(w.lnm_g), static_cast<const bf16*>(w.lnm_b),
                              y, N, cfg.ln_eps, st, rms));
  if (dump_final) DSV_CUDA(cudaMemcpyAsync(dump_final, y, N * 1024 * 2, cudaMemcpyDeviceToDevice, st));
  DSV_LAUNCH(DS_VIT_KERNEL_MERGER_GEMM1,
             launch_gemm_agen(kAMerge, ag, p->tm_m1, tC_u, T, 5120, 9216,
                              static_cast<const bf16*>(w.m1_b), qkv, kEpiBiasGelu, p->status, st));
  DSV_LAUNCH(DS_VIT_KERNEL_MERGER_GEMM2,
             launch_gemm(tA_u, p->tm_m2, tC_out, T, 5120, 5120, static_cast<const bf16*>(w.m2_b), out,
                         kEpiBias, nullptr, nullptr, p->status, st));
#undef DSV_LAUNCH
  if (p->t_count) *p->t_count = n_timed < p->t_slots ? n_timed : p->t_slots;
  return DS_VIT_OK;
}

int encode_common(const ds_vit_prepared* p, int n, const uint8_t* const* pixels, const int32_t* H,
                  const int32_t* W, void* out, int64_t* tok_offsets, void* ws, size_t ws_bytes,
                  void* blocks, void* final_norm, void* stream) {
  if (!p || !pixels || !out || !tok_offsets || !ws) return DS_VIT_EINVAL;
  DSV_TRY(check_images(n, H, W));
  for (int i = 0; i < n; ++i)
    if (!pixels[i] || (reinterpret_cast<uintptr_t>(pixels[i]) & 3) != 0) return DS_VIT_EINVAL;
  if (!aligned16(out) || !aligned16(ws) || (blocks && !aligned16(blocks)) ||
      (final_norm && !aligned16(final_norm)))
    return DS_VIT_EINVAL;
  const Plan pl = make_plan(n, H, W, false);
  if (ws_bytes < pl.total) return DS_VIT_ECAP;
  return run_encode(p, n, pixels, H, W, static_cast<bf16*>(out), tok_offsets,
                    static_cast<uint8_t*>(ws), pl, static_cast<bf16*>(blocks),
                    static_cast<bf16*>(final_norm), static_cast<cudaStream_t>(stream));
}

// Validated device-side description of the spans of one overlay call.  Spans
// must have positive grids, embed rows inside [0, n_embeds), base_row >= 0,
// rows inside [0, n_hidden) when n_hidden >= 0, and must not overlap.
int build_spans(const ds_vit_span* spans, int n_spans, int64_t n_embeds, int64_t n_hidden,
                OverlaySpans* os) {
  if (!spans || n_spans < 1 || n_spans > DS_VIT_MAX_IMAGES || n_embeds < 0) return DS_VIT_EINVAL;
  os->n = n_spans;
  std::vector<std::pair<int64_t, int64_t>> ranges;
  for (int s = 0; s < n_spans; ++s) {
    const ds_vit_span& sp = spans[s];
    if (sp.gh <= 0 || sp.gw <= 0) return DS_VIT_EINVAL;
    const int64_t h = (sp.gh + 2) / 3, w = (sp.gw + 2) / 3, rows = 2 + h * (w + 1);
    if (sp.base_row < 0 || (n_hidden >= 0 && sp.base_row + rows > n_hidden)) return DS_VIT_ERANGE;
    if (sp.embed_row < 0 || sp.embed_row + h * w > n_embeds) return DS_VIT_ERANGE;
    os->base_row[s] = sp.base_row;
    os->embed_row[s] = sp.embed_row;
    os->h[s] = static_cast<int>(h);
    os->w[s] = static_cast<int>(w);
    os->row_start[s + 1] = os->row_start[s] + rows;
    ranges.emplace_back(sp.base_row, sp.base_row + rows);
  }
  std::sort(ranges.begin(), ranges.end());
  for (size_t i = 1; i < ranges.size(); ++i)
    if (ranges[i].first < ranges[i - 1].second) return DS_VIT_EINVAL;
  return DS_VIT_OK;
}

}  // namespace

int dsvit::prepared_device(const ds_vit_prepared* p) { return p->device; }

extern "C" {

const char* ds_vit_strerror(int code) {
  switch (code) {
    case DS_VIT_OK: return "ok";
    case DS_VIT_EINVAL: return "invalid argument (null pointer, bad size or unsupported config)";
    case DS_VIT_ERANGE: return "out of range (image over the patch/token limits, or a row outside the buffer)";
    case DS_VIT_ECAP: return "capacity too small (output array or workspace)";
    case DS_VIT_ECUDA: return "CUDA call failed";
    case DS_VIT_ETIMEOUT: return "a kernel's bounded wait timed out";
    case DS_VIT_ENOMEM: return "device allocation failed";
    default: return "unknown error";
  }
}

int ds_vit_prepare(const ds_vit_config* cfg, const ds_vit_weights* w, ds_vit_prepared** out,
                   void* stream) {
  if (!out) return DS_VIT_EINVAL;
  *out = nullptr;
  DSV_TRY(check_config(cfg));
  DSV_TRY(check_weights(w, cfg->n_layers, cfg->norm_kind == DS_VIT_NORM_RMS));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ds_vit_prepared* p = new (std::nothrow) ds_vit_prepared();
  if (!p) return DS_VIT_ENOMEM;
  p->cfg = *cfg;
  p->w = *w;
  cudaGetDevice(&p->device);
  auto fail = [&](int rc) {
    ds_vit_release(p);
    return rc;
  };
  if (cudaMalloc(&p->patch_w_pad, 1024 * kPatchK * 2) != cudaSuccess ||
      cudaMalloc(&p->m1_perm, static_cast<size_t>(5120) * 9216 * 2) != cudaSuccess ||
      cudaMalloc(&p->rope_cs, static_cast<size_t>(kMaxPos) * 32 * 4) != cudaSuccess ||
      cudaMalloc(&p->pix_lut, 3 * 256 * 2) != cudaSuccess ||
      cudaMalloc(&p->status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return fail(DS_VIT_ENOMEM);
  }
  if (cudaMemsetAsync(p->status, 0, sizeof(int), st) != cudaSuccess) return fail(DS_VIT_ECUDA);
  int rc = launch_pad_patch_w(static_cast<const bf16*>(w->patch_w), p->patch_w_pad, 1024, st);
  if (rc == DS_VIT_OK) rc = launch_permute_m1(static_cast<const bf16*>(w->m1_w), p->m1_perm, 5120, st);
  if (rc == DS_VIT_OK) rc = launch_rope_table(p->rope_cs, kMaxPos, cfg->rope_theta, st);
  if (rc == DS_VIT_OK) {
    PixelNorm norm;
    for (int c = 0; c < 3; ++c) {
      norm.mean[c] = cfg->mean[c];
      norm.std[c] = cfg->std[c];
    }
    rc = launch_pixel_lut(norm, p->pix_lut, st);
  }
  if (rc == DS_VIT_OK && cfg->rope_pairing == DS_VIT_ROPE_HALF_VECTOR) {
    if (cudaMalloc(&p->qkv_perm, static_cast<size_t>(cfg->n_layers) * kQkvPermStride * 2) != cudaSuccess) {
      cudaGetLastError();
      return fail(DS_VIT_ENOMEM);
    }
    for (int l = 0; rc == DS_VIT_OK && l < cfg->n_layers; ++l)
      rc = launch_permute_qk_rows(static_cast<const bf16*>(w->layers[l].qkv_w),
                                  static_cast<const bf16*>(w->layers[l].qkv_b), qkv_perm_w(p, l),
                                  qkv_perm_b(p, l), 1024, 1024, st);
  }
  if (rc != DS_VIT_OK) return fail(rc);
  bool ok = make_weight_map(&p->tm_patch, p->patch_w_pad, 1024, kPatchK) &&
            make_weight_map(&p->tm_m1, p->m1_perm, 5120, 9216) &&
            make_weight_map(&p->tm_m2, w->m2_w, 5120, 5120);
  for (int l = 0; ok && l < cfg->n_layers; ++l) {
    const ds_vit_layer_weights& L = w->layers[l];
    ok = make_weight_map(&p->tm_qkv[l], p->qkv_perm ? qkv_perm_w(p, l) : L.qkv_w, 3072, 1024) &&
         make_weight_map(&p->tm_proj[l], L.proj_w, 1024, 1024) &&
         make_weight_map(&p->tm_fc1[l], L.fc1_w, cfg->mlp_kind == DS_VIT_MLP_SWIGLU ? 8192 : 4096, 1024) &&
         make_weight_map(&p->tm_fc2[l], L.fc2_w, 1024, 4096);
  }
  if (!ok) return fail(DS_VIT_ECUDA);
  if (cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return fail(DS_VIT_ECUDA);
  }
  *out = p;
  return DS_VIT_OK;
}

int ds_vit_release(ds_vit_prepared* p) {
  if (!p) return DS_VIT_OK;
  cudaDeviceSynchronize();
  cudaFree(p->patch_w_pad);
  cudaFree(p->m1_perm);
  cudaFree(p->rope_cs);
  cudaFree(p->qkv_perm);
  cudaFree(p->pix_lut);
  cudaFree(p->status);
  delete p;
  return DS_VIT_OK;
}

int ds_vit_layout(int32_t gh, int32_t gw, int32_t image_token_id, int32_t base_pos, int32_t* ids,
                  int32_t* pos, uint8_t* type, int32_t* src, int64_t cap, int64_t* n_rows) {
  if (gh <= 0 || gw <= 0) return DS_VIT_EINVAL;
  const int64_t h = (gh + 2) / 3, w = (gw + 2) / 3;
  const int64_t n = 2 + h * (w + 1);
  if (n_rows) *n_rows = n;
  if (cap < n) return DS_VIT_ECAP;
  if (static_cast<int64_t>(base_pos) + n - 1 > INT32_MAX) return DS_VIT_ERANGE;
  for (int64_t r = 0; r < n; ++r) {
    uint8_t t;
    int32_t s = -1;
    if (r == 0) {
      t = DS_VIT_TOK_START;
    } else if (r == n - 1) {
      t = DS_VIT_TOK_END;
    } else {
      const int64_t q = r - 1, yy = q / (w + 1), xx = q % (w + 1);
      if (xx == w) {
        t = DS_VIT_TOK_NEWLINE;
      } else {
        t = DS_VIT_TOK_IMAGE;
        s = static_cast<int32_t>(yy * w + xx);
      }
    }
    if (ids) ids[r] = image_token_id;
    if (pos) pos[r] = static_cast<int32_t>(base_pos + r);
    if (type) type[r] = t;
    if (src) src[r] = s;
  }
  return DS_VIT_OK;
}

int ds_vit_workspace_bytes(const ds_vit_prepared* p, int n, const int32_t* H, const int32_t* W,
                           size_t* bytes) {
  if (!p || !bytes) return DS_VIT_EINVAL;
  DSV_TRY(check_images(n, H, W));
  *bytes = make_plan(n, H, W, false).total;
  return DS_VIT_OK;
}

int ds_vit_workspace_bytes_host(const ds_vit_prepared* p, int n, const int32_t* H, const int32_t* W,
                                size_t* bytes) {
  if (!p || !bytes) return DS_VIT_EINVAL;
  DSV_TRY(check_images(n, H, W));
  *bytes = make_plan(n, H, W, true).total;
  return DS_VIT_OK;
}

int ds_vit_encode_batch(const ds_vit_prepared* p, int n, const uint8_t* const* pixels,
                        const int32_t* H, const int32_t* W, void* out, int64_t* tok_offsets,
                        void* ws, size_t ws_bytes, void* stream) {
  return encode_common(p, n, pixels, H, W, out, tok_offsets, ws, ws_bytes, nullptr, nullptr, stream);
}

int ds_vit_encode(const ds_vit_prepared* p, const uint8_t* pixels, int32_t H, int32_t W, void* out,
                  void* ws, size_t ws_bytes, void* stream) {
  int64_t offs[2];
  const uint8_t* px[1] = {pixels};
  if (!pixels) return DS_VIT_EINVAL;
  return encode_common(p, 1, px, &H, &W, out, offs, ws, ws_bytes, nullptr, nullptr, stream);
}

int ds_vit_encode_debug(const ds_vit_prepared* p, int n, const uint8_t* const* pixels,
                        const int32_t* H, const int32_t* W, void* out, int64_t* tok_offsets,
                        void* ws, size_t ws_bytes, void* blocks, void* final_norm, void* stream) {
  return encode_common(p, n, pixels, H, W, out, tok_offsets, ws, ws_bytes, blocks, final_norm,
                       stream);
}

int ds_vit_encode_batch_host(const ds_vit_prepared* p, int n, const uint8_t* const* pixels,
                             const int32_t* H, const int32_t* W, void* out_host,
                             int64_t* tok_offsets, void* ws, size_t ws_bytes, void* stream) {
  if (!p || !pixels || !out_host || !tok_offsets || !ws || !aligned16(ws)) return DS_VIT_EINVAL;
  DSV_TRY(check_images(n, H, W));
  for (int i = 0; i < n; ++i)
    if (!pixels[i]) return DS_VIT_EINVAL;
  const Plan pl = make_plan(n, H, W, true);
  if (ws_bytes < pl.total) return DS_VIT_ECAP;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const uint8_t* dpix[DS_VIT_MAX_IMAGES];
  for (int i = 0; i < n; ++i) {
    dpix[i] = wsb + pl.pix_off[i];
    DSV_CUDA(cudaMemcpyAsync(wsb + pl.pix_off[i], pixels[i], static_cast<size_t>(H[i]) * W[i] * 3,
                             cudaMemcpyHostToDevice, st));
  }
  bf16* dout = reinterpret_cast<bf16*>(wsb + pl.off_out);
  DSV_TRY(run_encode(p, n, dpix, H, W, dout, tok_offsets, wsb, pl, nullptr, nullptr, st));
  DSV_CUDA(cudaMemcpyAsync(out_host, dout, static_cast<size_t>(pl.T) * 5120 * 2,
                           cudaMemcpyDeviceToHost, st));
  return DS_VIT_OK;
}

int ds_vit_graph_create(const ds_vit_prepared* p, int host, int n, const uint8_t* const* pixels,
                        const int32_t* H, const int32_t* W, void* out, int64_t* tok_offsets, void* ws,
                        size_t ws_bytes, void** graph) {
  if (!p || !graph) return DS_VIT_EINVAL;
  *graph = nullptr;
  cudaStream_t st = nullptr;
  DSV_CUDA(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    cudaStreamDestroy(st);
    return DS_VIT_ECUDA;
  }
  const int rc = host ? ds_vit_encode_batch_host(p, n, pixels, H, W, out, tok_offsets, ws, ws_bytes, st)
                      : encode_common(p, n, pixels, H, W, out, tok_offsets, ws, ws_bytes, nullptr, nullptr, st);
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(st, &g);
  cudaStreamDestroy(st);
  if (rc != DS_VIT_OK || ec != cudaSuccess || g == nullptr) {
    if (g != nullptr) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != DS_VIT_OK ? rc : DS_VIT_ECUDA;
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, g, 0);
  cudaGraphDestroy(g);
  if (ei != cudaSuccess) {
    cudaGetLastError();
    return DS_VIT_ECUDA;
  }
  *graph = exec;
  return DS_VIT_OK;
}

int ds_vit_graph_launch(void* graph, void* stream) {
  if (!graph) return DS_VIT_EINVAL;
  DSV_CUDA(cudaGraphLaunch(static_cast<cudaGraphExec_t>(graph), static_cast<cudaStream_t>(stream)));
  return DS_VIT_OK;
}

int ds_vit_graph_destroy(void* graph) {
  if (!graph) return DS_VIT_EINVAL;
  DSV_CUDA(cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(graph)));
  return DS_VIT_OK;
}

int ds_vit_overlay(void* hidden, int64_t n_hidden, int32_t width, const ds_vit_span* spans,
                   int n_spans, const void* embeds, int64_t n_embeds, const void* sentinel,
                   void* stream) {
  if (!hidden || !embeds || !sentinel || width <= 0 || width % 8 != 0 || n_hidden <= 0)
    return DS_VIT_EINVAL;
  if (!aligned16(hidden) || !aligned16(embeds) || !aligned16(sentinel)) return DS_VIT_EINVAL;
  OverlaySpans os{};
  DSV_TRY(build_spans(spans, n_spans, n_embeds, n_hidden, &os));
  return launch_overlay(static_cast<bf16*>(hidden), width, os, static_cast<const bf16*>(embeds),
                        static_cast<const bf16*>(sentinel), static_cast<cudaStream_t>(stream));
}

int ds_vit_overlay_rows(void* hidden, int64_t n_hidden, int32_t width, const int32_t* rows,
                        const uint8_t* type, const int32_t* src, int64_t n, const void* embeds,
                        int64_t n_embeds, const void* sentinel, int32_t* status, void* stream) {
  if (!hidden || !rows || !type || !src || !embeds || !sentinel || !status || width <= 0 ||
      width % 8 != 0 || n_hidden <= 0 || n_hidden > INT32_MAX || n < 0 || n > INT32_MAX ||
      n_embeds < 0 || n_embeds > INT32_MAX)
    return DS_VIT_EINVAL;
  if (!aligned16(hidden) || !aligned16(embeds) || !aligned16(sentinel) ||
      (reinterpret_cast<uintptr_t>(rows) & 3) || (reinterpret_cast<uintptr_t>(src) & 3) ||
      (reinterpret_cast<uintptr_t>(status) & 3))
    return DS_VIT_EINVAL;
  return launch_overlay_rows(static_cast<bf16*>(hidden), n_hidden, width, rows, type, src, n,
                             static_cast<const bf16*>(embeds), n_embeds, static_cast<const bf16*>(sentinel),
                             reinterpret_cast<int*>(status), static_cast<cudaStream_t>(stream));
}

int ds_vit_overlay_chunk(void* chunk, int64_t chunk_begin, int64_t chunk_rows, int32_t width,
                         const ds_vit_span* spans, int n_spans, const void* embeds,
                         int64_t n_embeds, const void* sentinel, uint8_t* row_type,
                         void* stream) {
  if (!chunk || !embeds || !sentinel || width <= 0 || width % 8 != 0 || chunk_begin < 0 ||
      chunk_rows < 1 || chunk_rows > INT32_MAX)
    return DS_VIT_EINVAL;
  if (!aligned16(chunk) || !aligned16(embeds) || !aligned16(sentinel)) return DS_VIT_EINVAL;
  OverlaySpans os{};
  DSV_TRY(build_spans(spans, n_spans, n_embeds, -1, &os));
  return launch_overlay_chunk(static_cast<bf16*>(chunk), chunk_begin, chunk_rows, width, os,
                              static_cast<const bf16*>(embeds), static_cast<const bf16*>(sentinel),
                              row_type, static_cast<cudaStream_t>(stream));
}

int ds_vit_set_kernel_timer(ds_vit_prepared* p, void* const* events, int32_t* kinds,
                            int32_t n_slots, int32_t* n_recorded) {
  if (!p) return DS_VIT_EINVAL;
  if (!events) {
    p->t_events = nullptr;
    p->t_kinds = nullptr;
    p->t_slots = 0;
    p->t_count = nullptr;
    return DS_VIT_OK;
  }
  if (!kinds || !n_recorded || n_slots < 1) return DS_VIT_EINVAL;
  for (int i = 0; i < 2 * n_slots; ++i)
    if (!events[i]) return DS_VIT_EINVAL;
  p->t_events = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
  p->t_kinds = kinds;
  p->t_slots = n_slots;
  p->t_count = n_recorded;
  *n_recorded = 0;
  return DS_VIT_OK;
}

int ds_vit_device_status(const ds_vit_prepared* p, void* stream) {
  if (!p) return DS_VIT_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  DSV_CUDA(cudaStreamSynchronize(st));
  DSV_CUDA(cudaMemcpy(&v, p->status, sizeof(int), cudaMemcpyDeviceToHost));
  DSV_CUDA(cudaMemset(p->status, 0, sizeof(int)));
  return v == 0 ? DS_VIT_OK : v;
}

int ds_vit_selftest_wait_timeout(int32_t* status, uint64_t* elapsed_ns, uint32_t limit_us, void* stream) {
  if (!status || !elapsed_ns || limit_us < 1 || limit_us > 1000000) return DS_VIT_EINVAL;
  return launch_selftest_wait(reinterpret_cast<int*>(status), reinterpret_cast<unsigned long long*>(elapsed_ns),
                              static_cast<unsigned long long>(limit_us) * 1000ull, static_cast<cudaStream_t>(stream));
}

int ds_vit_op_layernorm(const void* x, const void* g, const void* b, void* y, int64_t M, float eps,
                        void* stream) {
  if (!x || !g || !b || !y || M < 0 || !(eps > 0.f)) return DS_VIT_EINVAL;
  if (!aligned16(x) || !aligned16(g) || !aligned16(b) || !aligned16(y) || x == y) return DS_VIT_EINVAL;
  return launch_layernorm(static_cast<const bf16*>(x), static_cast<const bf16*>(g),
                          static_cast<const bf16*>(b), static_cast<bf16*>(y), M, eps,
                          static_cast<cudaStream_t>(stream));
}

int ds_vit_op_rmsnorm(const void* x, const void* g, void* y, int64_t M, float eps, void* stream) {
  if (!x || !g || !y || M < 0 || !(eps > 0.f)) return DS_VIT_EINVAL;
  if (!aligned16(x) || !aligned16(g) || !aligned16(y) || x == y) return DS_VIT_EINVAL;
  return launch_layernorm(static_cast<const bf16*>(x), static_cast<const bf16*>(g), nullptr,
                          static_cast<bf16*>(y), M, eps, static_cast<cudaStream_t>(stream), true);
}

int ds_vit_op_linear(const void* a, int64_t M, int32_t K, const void* w, int32_t N, const void* bias,
                     void* out, int32_t epilogue, const int32_t* rowpos, const float* rope_cs,
                     int32_t* status, void* stream) {
  if (!a || !w || !bias || !out || !status || M < 1 || M > INT32_MAX || K < 64 || K % 64 != 0 ||
      N < 128 || N % 128 != 0 || epilogue < 0 || epilogue > 4)
    return DS_VIT_EINVAL;
  if (epilogue == kEpiQkvRope && (N != 3072 || !rowpos || !rope_cs)) return DS_VIT_EINVAL;
  if (!aligned16(a) || !aligned16(w) || !aligned16(bias) || !aligned16(out)) return DS_VIT_EINVAL;
  CUtensorMap tA, tC;
  WeightMap tB;
  if (!make_tmap_bf16(&tA, a, M, K, 128) || !make_weight_map(&tB, w, N, K) ||
      !make_tmap_store_bf16(&tC, out, M, epilogue == kEpiSwiglu ? N / 2 : N))
    return DS_VIT_ECUDA;
  return launch_gemm(tA, tB, tC, static_cast<int>(M), N, K, static_cast<const bf16*>(bias),
                     static_cast<bf16*>(out), epilogue, rowpos, rope_cs, status,
                     static_cast<cudaStream_t>(stream));
}

int ds_vit_op_rope_table(float* rope_cs, int32_t max_pos, float theta, void* stream) {
  if (!rope_cs || max_pos < 1 || !(theta > 0.f)) return DS_VIT_EINVAL;
  return launch_rope_table(rope_cs, max_pos, theta, static_cast<cudaStream_t>(stream));
}

int ds_vit_op_attention(const void* qkv, const int32_t* seqlens, int n_images, void* out,
                        int32_t* status, void* stream) {
  if (!qkv || !seqlens || !out || !status || n_images < 1 || n_images > DS_VIT_MAX_IMAGES)
    return DS_VIT_EINVAL;
  if (!aligned16(qkv) || !aligned16(out)) return DS_VIT_EINVAL;
  AttnBatch ab{};
  ab.n_images = n_images;
  for (int i = 0; i < n_images; ++i) {
    if (seqlens[i] < 1 || seqlens[i] > DS_VIT_MAX_PATCHES) return DS_VIT_ERANGE;
    ab.cu[i + 1] = ab.cu[i] + seqlens[i];
    ab.order[i] = i;
    ab.tile_start[i + 1] = ab.tile_start[i] + (seqlens[i] + kAttnRowsPerCta - 1) / kAttnRowsPerCta;
  }
  CUtensorMap tm;
  if (!make_tmap_bf16(&tm, qkv, ab.cu[n_images], 3072, 128)) return DS_VIT_ECUDA;
  return launch_attention(tm, ab, static_cast<bf16*>(out), status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
