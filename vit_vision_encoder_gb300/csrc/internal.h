// Declarations shared by the translation units of libdsvit (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/dsvit.h"

namespace dsvit {

using bf16 = __nv_bfloat16;

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream finishes; it synchronises with
// griddepcontrol.wait (grid_dep_wait) before touching dependent data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Epilogue kinds of the tcgen05 GEMM (same values as DS_VIT_EPI_*).
enum Epilogue : int { kEpiBias = 0, kEpiBiasGelu = 1, kEpiBiasResid = 2, kEpiQkvRope = 3, kEpiSwiglu = 4,
                      // Internal: the Qwen-style tower's QKV (80-wide heads, rotation pairs 8
                      // columns apart in 16-column groups, per-row cos/sin table in rope_cs).
                      kEpiQkvRope72 = 5 };
// q and k columns of that QKV output (2 x 16 heads x 80); V follows.
constexpr int kQwenQkCols = 2560;

// cuTensorMapEncodeTiled through the runtime's driver entry point.
// Row-major bf16 matrix [rows, cols], box [box_rows, 64 cols], 128-byte swizzle,
// zero fill out of bounds.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);

// The same matrix with boxes [box_rows, 16 cols] and 32-byte swizzle (rows of
// 32 B, the layout of a 16-column tail atom).
bool make_tmap_bf16_tail16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows);

// Store map of a row-major bf16 output [rows, cols]: 32x32 boxes, 64-byte swizzle.
bool make_tmap_store_bf16(CUtensorMap* map, void* base, uint64_t rows, uint64_t cols);

int num_sms();

// The device a prepared model was built on (its weights, tensor maps and
// status word live there).
int prepared_device(const ds_vit_prepared* p);

// Lets `kernel` use `bytes` of dynamic shared memory on the current device,
// once per (kernel, device): a process that drives several GPUs sets it on
// each.  Returns the result of that first cudaFuncSetAttribute.
cudaError_t allow_smem(const void* kernel, int bytes);

// TMA maps of one weight matrix B [N, K] for both GEMM tile widths.
struct WeightMap {
  CUtensorMap bn256;   // box 256 rows
  CUtensorMap bn128;   // box 128 rows
  CUtensorMap bn64;    // box 64 rows (the last rows of a 320-row tile)
  CUtensorMap bn32;    // box 32 rows (the last rows of a 288-row tile)
};
bool make_weight_map(WeightMap* m, const void* w, uint64_t n, uint64_t k);

// out[M, N] = epi(A[M, K] B[N, K]^T + bias); tmC is the store map of `out`
// (make_tmap_store_bf16).  The tile width (gemm_bn) picks the map of B.
// Returns DS_VIT_OK or DS_VIT_ECUDA.
int launch_gemm(const CUtensorMap& tmA, const WeightMap& B, const CUtensorMap& tmC, int M, int N,
                int K, const bf16* bias, bf16* out, int epi, const int* rowpos,
                const float* rope_cs, int* status, cudaStream_t stream);

// Tile width: 128x256 tiles, or 128x128 when 128x256 tiles would leave more
// than a quarter of the SMs idle (small M).
int gemm_bn(int M, int N);

// out[M, N] = epi(A B^T + bias) in 256 x 256 tiles on 2-CTA clusters
// (tcgen05 cta_group::2; gemm_pair.cu); B through its 128-row-box map.  N a
// multiple of 256.  Returns kGemmNoPair, launching nothing, when no cluster of
// two such CTAs fits on the device.
constexpr int kGemmNoPair = 1;
int launch_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB128, const CUtensorMap& tmC, int M, int N,
                     int K, const bf16* bias, bf16* out, int epi, const int* rowpos, const float* rope_cs,
                     int* status, cudaStream_t stream);

// Query rows per attention CTA (two 128-row tiles).
constexpr int kAttnRowsPerCta = 256;

struct AttnBatch {
  int n_images;
  int cu[DS_VIT_MAX_IMAGES + 1];          // packed row offsets of the images
  int tile_start[DS_VIT_MAX_IMAGES + 1];  // CTA prefix sums (kAttnRowsPerCta rows each), launch order
  int order[DS_VIT_MAX_IMAGES];           // launch slot -> image index
};

int launch_attention(const CUtensorMap& tm_qkv, const AttnBatch& batch, bf16* out, int* status,
                     cudaStream_t stream);

// Rows of `width` values: 1024 (LayerNorm or RMS) or 1152 (LayerNorm).
int launch_layernorm(const bf16* x, const bf16* g, const bf16* b, bf16* y, int64_t M, float eps,
                     cudaStream_t stream, bool rms = false, int width = 1024);

// W'[r] = W[swap(r)], b'[r] = b[swap(r)] for the q and k rows (r < 2 hidden),
// swap exchanging head dims 16..31 and 32..47; v rows copied.  [3 hidden, K].
int launch_permute_qk_rows(const bf16* w, const bf16* b, bf16* w_perm, bf16* b_perm, int hidden, int K,
                           cudaStream_t stream);

struct ImageBatch {
  int n;
  int64_t row_off[DS_VIT_MAX_IMAGES + 1];  // patch row offsets
  int64_t tok_off[DS_VIT_MAX_IMAGES + 1];  // merged token offsets
  const uint8_t* pix[DS_VIT_MAX_IMAGES];
  int gh[DS_VIT_MAX_IMAGES];
  int gw[DS_VIT_MAX_IMAGES];
};

struct PixelNorm {
  float mean[3];
  float std[3];
};

// lut[c * 256 + v] = bf16((v/255 - mean_c)/std_c), fp32 arithmetic (3 x 256 entries).
int launch_pixel_lut(const PixelNorm& norm, bf16* lut, cudaStream_t stream);

// One thread waits on an mbarrier that never completes until limit_ns has
// passed, then records DS_VIT_ETIMEOUT in *status; *elapsed = the time waited.
int launch_selftest_wait(int* status, unsigned long long* elapsed, unsigned long long limit_ns,
                         cudaStream_t stream);

// The patch projection's K order inside the GEMM: patch row y fills columns
// y*64 .. y*64+41 in pixel order (x*3 + c), columns y*64+42 .. y*64+63 are
// zero.  The weight is permuted to match once at preparation; the product is
// the same sum as over the pages' c*196 + y*14 + x order.
constexpr int kPatchK = 14 * 64;

// Where a fused GEMM's A tile comes from.
enum ASource : int {
  kATma = 0,      // TMA from a row-major bf16 matrix
  kAPixels = 1,   // patchify + normalise (K = kPatchK, one patch row per 64 columns)
  kAMerge = 2     // 3x3 merge-gather of the final-norm output, column p*1024 + c
};

struct AGenParams {
  ImageBatch batch;
  const bf16* lut;   // kAPixels: normalised pixel values [3][256]
  const bf16* z;     // kAMerge: final-norm output [sum N, 1024]
  int* rowpos;       // kAPixels writes gy << 16 | gx of every patch row here
};

// launch_gemm with the A tile built in shared memory by producer warps
// (asrc = kAPixels: M = sum N patches, K = kPatchK; kAMerge: M = sum T tokens, K = 9216).
// kAPixels needs every image's pixel pointer 4-byte aligned.
int launch_gemm_agen(int asrc, const AGenParams& g, const WeightMap& B, const CUtensorMap& tmC,
                     int M, int N, int K, const bf16* bias, bf16* out, int epi, int* status,
                     cudaStream_t stream);

int launch_rope_table(float* table, int max_pos, float theta, cudaStream_t stream);

// W'[o, p*1024 + c] = W[o, c*9 + p]  (rows of 9216).
int launch_permute_m1(const bf16* w, bf16* w_perm, int rows, cudaStream_t stream);

// W'[o, y*64 + x*3 + c] = W[o, c*196 + y*14 + x] for x < 14, zero in columns
// y*64 + 42 .. y*64 + 63  (rows of kPatchK).
int launch_pad_patch_w(const bf16* w, bf16* w_pad, int rows, cudaStream_t stream);

struct OverlaySpans {
  int n;
  int64_t base_row[DS_VIT_MAX_IMAGES];
  int64_t embed_row[DS_VIT_MAX_IMAGES];
  int h[DS_VIT_MAX_IMAGES];   // merged grid
  int w[DS_VIT_MAX_IMAGES];
  int64_t row_start[DS_VIT_MAX_IMAGES + 1];  // prefix of span row counts
};

int launch_overlay(bf16* hidden, int width, const OverlaySpans& spans, const bf16* embeds,
                   const bf16* sentinel, cudaStream_t stream);
int launch_overlay_chunk(bf16* chunk, int64_t chunk_begin, int64_t chunk_rows, int width,
                         const OverlaySpans& spans, const bf16* embeds, const bf16* sentinel,
                         uint8_t* row_type, cudaStream_t stream);

int launch_overlay_rows(bf16* hidden, int64_t n_hidden, int width, const int32_t* rows, const uint8_t* type,
                        const int32_t* src, int64_t n, const bf16* embeds, int64_t n_embeds, const bf16* sentinel,
                        int* status, cudaStream_t stream);

}  // namespace dsvit
