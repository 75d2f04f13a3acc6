/*
 * dsvit.h — C ABI of the GB300 (sm_103a) vision-tower encode.
 *
 * The encode turns uint8 RGB pixels into language-space image tokens:
 * 14x14 patchify + CLIP normalisation + patch projection, a pre-LayerNorm ViT
 * (hidden 1024, 16 heads of 64, raw patch-grid 2D RoPE, bf16 activations at
 * every stored boundary), a final LayerNorm, the 3x3 spatial merge and the two
 * merger linears to width 5120; then the row-major image token span and the
 * overlay of the embeddings onto the prompt's hidden-state rows.
 *
 * Sources (cited by page title and section):
 *   [A] "DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision" (zLLM).
 *   [B] ds4-learning glossary, "vision" (V4.1 Flash vision paragraph, family table).
 *   [C] Lucebox "Image input" (DS4V section: failed encodes publish nothing partial).
 *
 * Conventions for every entry point:
 *   - Pointers are caller-owned.  "device" pointers are CUDA device (or managed)
 *     memory on the current device; "host" pointers are CPU memory.
 *   - bf16 tensors are row-major with the stated shapes; every device pointer
 *     must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Launching entry points are asynchronous on that stream.
 *   - Return value: DS_VIT_OK (0) or a negative DS_VIT_E* code.  All argument
 *     checks run before the first launch; on an error nothing has been written
 *     ([C], DS4V: a failed encode publishes no partial embedding matrices).
 *   - Every spin-wait inside a kernel gives up after about two seconds, records
 *     DS_VIT_ETIMEOUT in a device status word and returns; read it with
 *     ds_vit_device_status (or, for the ds_vit_op_* calls, from `status`).
 */
#ifndef DSVIT_H
#define DSVIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS_VIT_OK 0
#define DS_VIT_EINVAL (-1)   /* null pointer, bad size, unsupported config */
#define DS_VIT_ERANGE (-2)   /* an image over the patch/token limits, a row outside the buffer */
#define DS_VIT_ECAP (-3)     /* an output capacity or the workspace is too small */
#define DS_VIT_ECUDA (-4)    /* a CUDA runtime / driver call failed */
#define DS_VIT_ETIMEOUT (-5) /* a kernel's bounded wait gave up (device status word) */
#define DS_VIT_ENOMEM (-6)   /* ds_vit_prepare could not allocate its device copies */

#define DS_VIT_MAX_LAYERS 32
#define DS_VIT_MAX_IMAGES 64       /* images per batch call */
#define DS_VIT_MAX_PATCHES 9216    /* patches of one image (96 x 96 grid) */
#define DS_VIT_MAX_TOKENS 1024     /* merged tokens of one image ([A] Step 1) */

/* Row types of the image token span ([A] "Connect the complete image-to-text path first"). */
#define DS_VIT_TOK_START 0
#define DS_VIT_TOK_IMAGE 1
#define DS_VIT_TOK_NEWLINE 2
#define DS_VIT_TOK_END 3

/* Epilogues of ds_vit_op_linear. */
#define DS_VIT_EPI_BIAS 0        /* out = bf16(a w^T + bias) */
#define DS_VIT_EPI_BIAS_GELU 1   /* out = bf16(gelu_erf(a w^T + bias)) */
#define DS_VIT_EPI_BIAS_RESID 2  /* out = bf16(out + (a w^T + bias))   (in place) */
#define DS_VIT_EPI_QKV_ROPE 3    /* N = 3072: q, k rotated by 2D RoPE, then bf16 */
#define DS_VIT_EPI_SWIGLU 4      /* N = 2F accumulators (w rows: F gate, F up) -> out [M, F] =
                                    bf16(silu(gate + b_gate) * (up + b_up)) */

/* Model constants.  Only hidden 1024, heads 16, head_dim 64, mlp 4096,
 * out_dim 5120, patch 14 and merge 3 are supported; n_layers 1..32. */
typedef struct ds_vit_config {
  int32_t n_layers;
  int32_t hidden;
  int32_t heads;
  int32_t head_dim;
  int32_t mlp;
  int32_t out_dim;
  int32_t patch;
  int32_t merge;
  float rope_theta;      /* 10000 */
  float ln_eps;          /* 1e-6 */
  float mean[3];         /* pixel mean per channel (CLIP) */
  float std[3];          /* pixel std per channel (CLIP) */
  int32_t image_token_id;
  /* Block variant ([A] comparison table and Step 3 describe the released
   * tower as RMSNorm + SwiGLU with the half-vector RoPE pairing). */
  int32_t norm_kind;     /* DS_VIT_NORM_LAYER (gamma, beta) or DS_VIT_NORM_RMS (gamma; beta unused) */
  int32_t mlp_kind;      /* DS_VIT_MLP_GELU or DS_VIT_MLP_SWIGLU (fc1 [2*mlp, hidden]: gate rows, then up rows) */
  int32_t rope_pairing;  /* DS_VIT_ROPE_AXIS_HALVES or DS_VIT_ROPE_HALF_VECTOR */
} ds_vit_config;

#define DS_VIT_NORM_LAYER 0
#define DS_VIT_NORM_RMS 1
#define DS_VIT_MLP_GELU 0
#define DS_VIT_MLP_SWIGLU 1
/* per head: dims 0..31 rotated by the patch row and 32..63 by the patch column,
 * each half as a rotate-half vector with pairs (j, j+16) */
#define DS_VIT_ROPE_AXIS_HALVES 0
/* per head: angle vector [row*f0..row*f15, col*f0..col*f15], dim i paired with i+32 */
#define DS_VIT_ROPE_HALF_VECTOR 1

/* One ViT block's weights: device bf16, nn.Linear layout [out, in]. */
typedef struct ds_vit_layer_weights {
  const void *ln1_g, *ln1_b;     /* [1024] */
  const void *qkv_w, *qkv_b;     /* [3072, 1024], [3072]; rows: q (head h at h*64), k, v */
  const void *proj_w, *proj_b;   /* [1024, 1024], [1024] */
  const void *ln2_g, *ln2_b;     /* [1024] */
  const void *fc1_w, *fc1_b;     /* [4096, 1024], [4096] */
  const void *fc2_w, *fc2_b;     /* [1024, 4096], [1024] */
} ds_vit_layer_weights;

/* All weights: device bf16. */
typedef struct ds_vit_weights {
  const void *patch_w, *patch_b; /* [1024, 588], input index c*196 + y*14 + x; [1024] */
  ds_vit_layer_weights layers[DS_VIT_MAX_LAYERS];
  const void *lnm_g, *lnm_b;     /* final (merger) LayerNorm [1024] */
  const void *m1_w, *m1_b;       /* [5120, 9216], input index c*9 + dy*3 + dx; [5120] */
  const void *m2_w, *m2_b;       /* [5120, 5120], [5120] */
  const void *sentinel;          /* [3, 5120]: START, NEWLINE, END vectors */
} ds_vit_weights;

typedef struct ds_vit_prepared ds_vit_prepared;

/* One image span for ds_vit_overlay. */
typedef struct ds_vit_span {
  int64_t base_row;     /* destination row of the span's first (START) row */
  int32_t gh, gw;       /* patch grid of the image */
  int64_t embed_row;    /* row of the image's first merged token in `embeds` */
} ds_vit_span;

/* Human-readable text of a return code (static storage). */
const char* ds_vit_strerror(int code);

/*
 * ds_vit_prepare: validate `cfg`, keep the weight pointers (they must stay
 * valid until ds_vit_release), allocate the device copies the kernels need
 * (patch weight reordered to the pixel order of each patch row and padded to
 * 64 columns per patch row, K = 896, [A] Step 5; the
 * first merger weight with its input permuted from c*9+p to p*1024+c; the RoPE
 * cos/sin table; a device status word) and build the TMA descriptors.
 * Synchronises `stream` before returning.  On error *out is NULL.
 */
int ds_vit_prepare(const ds_vit_config* cfg, const ds_vit_weights* w,
                   ds_vit_prepared** out, void* stream);

/* Free what ds_vit_prepare allocated (device-synchronising).  NULL is a no-op. */
int ds_vit_release(ds_vit_prepared* p);

/*
 * Image preprocessing upstream of the encode ([A] "Step 1: Reproduce the
 * discrete image-processing rules"; [B] V4.1 paragraph: minimum pixel budget
 * 295,936, at most 1,024 image tokens, no aspect clamp; Lucebox "Image input":
 * bicubic resizing that matches Pillow byte for byte).
 *
 * ds_vit_plan_image (host only): the plan of an H x W image.  Unit u = 42
 * pixels (patch 14 x merge 3).  An image under 295,936 pixels is first
 * enlarged by s = sqrt(295936 / (H W)); the merged grid is (h, w) =
 * (ceil(sH/u), ceil(sW/u)) when h*w <= 1024, otherwise the aspect-preserving
 * floor grid under 1,024 tokens (each side >= 1).  Canvas Hc x Wc = hu x wu
 * (patch grid 3h x 3w).  The image is resized to Hr x Wr with PIL "contain"
 * rules (the side that does not fill the canvas is round(...), half to even)
 * and placed at (y0, x0) = ((Hc - Hr)/2, (Wc - Wr)/2) rounded down; the rest of
 * the canvas is RGB 127.  H, W in [1, 65535] with H*W <= 2^28, else
 * DS_VIT_EINVAL.
 */
typedef struct ds_vit_plan {
  int32_t H, W;     /* input image */
  int32_t h, w;     /* merged grid: h*w image tokens (<= DS_VIT_MAX_TOKENS) */
  int32_t Hc, Wc;   /* canvas pixels = 42h x 42w: the encode's H and W */
  int32_t Hr, Wr;   /* resized image inside the canvas */
  int32_t y0, x0;   /* top-left corner of the resized image */
} ds_vit_plan;

int ds_vit_plan_image(int32_t H, int32_t W, ds_vit_plan* out);

/* Device workspace of ds_vit_preprocess for `plan` (host only). */
int ds_vit_preprocess_workspace_bytes(const ds_vit_plan* plan, size_t* bytes);

/*
 * ds_vit_preprocess: pixels (device uint8 [H, W, 3], HWC RGB) -> canvas
 * (device uint8 [Hc, Wc, 3]), ready for ds_vit_encode(canvas, Hc, Wc).
 * Bicubic (Keys, a = -0.5, support 2 widened by the reduction factor), weights
 * in float64 normalised per output pixel and rounded to 22 fraction bits;
 * horizontal pass then vertical pass, each rounded and clamped to uint8
 * ((2^21 + sum) >> 22); a pass whose size does not change is skipped.  This
 * is the separable fixed-point scheme Pillow documents for 8-bit images;
 * agreement with Pillow itself is not tested here.  The canvas is written
 * completely.  `plan` must equal ds_vit_plan_image(H, W) (DS_VIT_EINVAL
 * otherwise); ws: device workspace, 256-byte aligned (DS_VIT_EINVAL
 * otherwise), of at least ds_vit_preprocess_workspace_bytes (DS_VIT_ECAP
 * otherwise); pixels need no alignment (a 16-byte aligned image takes the
 * faster passes).  Pixel, canvas and workspace memory stay caller-owned;
 * nothing is written on an error.
 */
int ds_vit_preprocess(const ds_vit_plan* plan, const uint8_t* pixels, void* canvas, void* ws,
                      size_t ws_bytes, void* stream);

/*
 * ds_vit_layout (host only, no GPU needed): the token span of one image with a
 * gh x gw patch grid ([A] "Connect the complete image-to-text path first";
 * [B] V4.1 paragraph).  h = ceil(gh/3), w = ceil(gw/3); n = 2 + h*(w+1) rows:
 * row 0 START; row 1 + y*(w+1) + x IMAGE with src = y*w + x; row
 * 1 + y*(w+1) + w NEWLINE; row n-1 END.  ids[r] = image_token_id for every
 * row, pos[r] = base_pos + r, src[r] = -1 for non-IMAGE rows.  Output arrays
 * (host) need `cap` entries; *n_rows receives n (also when cap is too small,
 * which returns DS_VIT_ECAP).  Any output pointer may be NULL to skip it.
 */
int ds_vit_layout(int32_t gh, int32_t gw, int32_t image_token_id, int32_t base_pos,
                  int32_t* ids, int32_t* pos, uint8_t* type, int32_t* src,
                  int64_t cap, int64_t* n_rows);

/* Workspace bytes that ds_vit_encode_batch needs for these image sizes (host
 * arrays of n entries).  Writes *bytes. */
int ds_vit_workspace_bytes(const ds_vit_prepared* p, int n, const int32_t* H,
                           const int32_t* W, size_t* bytes);

/*
 * ds_vit_encode_batch: encode n images (n <= DS_VIT_MAX_IMAGES) packed into one
 * varlen pass; attention never crosses images.
 *   pixels: host array of n device pointers, image i is uint8 [H[i], W[i], 3]
 *           (HWC, RGB), each 4-byte aligned (DS_VIT_EINVAL otherwise).
 *           H[i], W[i] (host) must be positive multiples of 14;
 *           (H/14)*(W/14) <= DS_VIT_MAX_PATCHES and the merged token count
 *           ceil(H/42)*ceil(W/42) <= DS_VIT_MAX_TOKENS.
 *   out:    device bf16 [sum T_i, 5120], image i's tokens at rows
 *           tok_offsets[i] .. tok_offsets[i+1]-1 (row-major merged order).
 *   tok_offsets: host int64 [n+1], written before the first launch.
 *   ws, ws_bytes: device workspace of at least ds_vit_workspace_bytes.
 */
int ds_vit_encode_batch(const ds_vit_prepared* p, int n, const uint8_t* const* pixels,
                        const int32_t* H, const int32_t* W, void* out, int64_t* tok_offsets,
                        void* ws, size_t ws_bytes, void* stream);

/* ds_vit_encode: one image (ds_vit_encode_batch with n = 1). */
int ds_vit_encode(const ds_vit_prepared* p, const uint8_t* pixels, int32_t H, int32_t W,
                  void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * ds_vit_encode_batch_host: as ds_vit_encode_batch, but `pixels` holds HOST
 * pointers and `out_host` is host memory.  The pixels are copied into the
 * workspace (so ws_bytes must also cover sum H*W*3 rounded up, see
 * ds_vit_workspace_bytes_host), the encode runs, and the result is copied to
 * out_host; all on `stream`.  For full overlap the host buffers should be
 * pinned.  The call returns after queueing; synchronise `stream` before reading
 * out_host.
 */
int ds_vit_workspace_bytes_host(const ds_vit_prepared* p, int n, const int32_t* H,
                                const int32_t* W, size_t* bytes);
int ds_vit_encode_batch_host(const ds_vit_prepared* p, int n, const uint8_t* const* pixels,
                             const int32_t* H, const int32_t* W, void* out_host,
                             int64_t* tok_offsets, void* ws, size_t ws_bytes, void* stream);

/*
 * ds_vit_graph_create / ds_vit_graph_launch / ds_vit_graph_destroy: one encode
 * recorded once as a CUDA graph and replayed.  The pages have no counterpart:
 * an encode is a few hundred kernel launches (seven per block), and on small
 * images the host's launch calls take about as long as the device work, so a
 * serving loop that encodes the same image sizes again records the encode
 * once and replays it.
 *   ds_vit_graph_create records ds_vit_encode_batch (host == 0) or
 *   ds_vit_encode_batch_host (host != 0; pixels and out then in page-locked
 *   host memory) with exactly these arguments on an internal stream, runs
 *   nothing, and stores an opaque executable-graph handle in *graph;
 *   tok_offsets is filled as by the recorded call.  Every replay repeats the
 *   whole encode (all its kernels and, for host == 1, both copies) on the same
 *   buffers: their contents may change between replays, their addresses and
 *   the image sizes may not, and the buffers must outlive the handle.
 *   Replays on different streams need different workspaces and outputs.  The
 *   kernel timer (ds_vit_set_kernel_timer) must be detached while recording.
 *   Errors: DS_VIT_EINVAL for a null p or graph (nothing else is touched),
 *   the recorded call's own error code (nothing is kept), DS_VIT_ECUDA when
 *   the stream, the recording or the instantiation fails.
 *   ds_vit_graph_launch queues one replay on `stream` (DS_VIT_EINVAL for a null
 *   handle, DS_VIT_ECUDA when the launch fails); ds_vit_graph_destroy frees the
 *   handle (the caller ensures no replay is still running on the device).
 */
int ds_vit_graph_create(const ds_vit_prepared* p, int host, int n, const uint8_t* const* pixels,
                        const int32_t* H, const int32_t* W, void* out, int64_t* tok_offsets, void* ws,
                        size_t ws_bytes, void** graph);
int ds_vit_graph_launch(void* graph, void* stream);
int ds_vit_graph_destroy(void* graph);

/*
 * ds_vit_encode_noalloc: ds_vit_encode for callers that cannot allocate device
 * memory when they encode (an application that owns the whole device budget
 * through its own pool, a latency-critical loop that must not pay cudaMalloc's
 * implicit synchronisation, a plugin interface that passes only inputs and
 * outputs).  The pages have no counterpart: it is a deployment variant.
 *   Same arguments and results as ds_vit_encode, without ws/ws_bytes: the
 *   scratch is a file-scope device array of DS_VIT_NOALLOC_SCRATCH_BYTES
 *   inside the library, held by every GPU that loads the library until exit.
 *   Checks, in this order, each failing before anything is written:
 *   DS_VIT_EINVAL for a null pointer, `out` not 16-byte or `pixels` not
 *   4-byte aligned, or H / W not positive multiples of 14; DS_VIT_ERANGE for
 *   an image over the ds_vit_encode limits; DS_VIT_EINVAL when the current
 *   device is not the one `p` was prepared on; DS_VIT_ERANGE for an image
 *   over DS_VIT_NOALLOC_MAX_PATCHES patches.
 *   The call allocates and frees nothing.  The array's device address belongs
 *   to the current CUDA context: the first call in each context (a device's
 *   primary context, again after cudaDeviceReset, or a context the caller
 *   created) looks it up with cudaGetSymbolAddress, with the device current;
 *   make that first call before any stream capture.
 *   All calls share the array and it keeps the last call's contents (no part
 *   needs to start at zero); calls whose kernels overlap on the GPU race.
 */
#define DS_VIT_NOALLOC_MAX_PATCHES 1024                   /* e.g. 448 x 448 pixels */
#define DS_VIT_NOALLOC_SCRATCH_BYTES (21u * 1024u * 1024u) /* 21 MiB */
int ds_vit_encode_noalloc(const ds_vit_prepared* p, const uint8_t* pixels, int32_t H, int32_t W,
                          void* out, void* stream);

/*
 * ds_vit_encode_debug: ds_vit_encode_batch that also copies named boundaries
 * ([A] Step 2: block outputs, final norm output) into caller buffers:
 *   blocks: device bf16 [n_layers + 1, sum N_i, 1024] — the patch-projection
 *           output followed by each block's output (NULL to skip);
 *   final_norm: device bf16 [sum N_i, 1024] (NULL to skip).
 */
int ds_vit_encode_debug(const ds_vit_prepared* p, int n, const uint8_t* const* pixels,
                        const int32_t* H, const int32_t* W, void* out, int64_t* tok_offsets,
                        void* ws, size_t ws_bytes, void* blocks, void* final_norm,
                        void* stream);

/*
 * ds_vit_overlay: write image spans into a prompt's hidden states
 * ([A] "Connect the complete image-to-text path first": aligner rows replace
 * IMAGE rows, learned vectors fill START / NEWLINE / END rows).  For span s
 * and its row r (layout of ds_vit_layout for gh, gw):
 *   hidden[base_row + r] = IMAGE ? embeds[embed_row + src] : sentinel[START/NEWLINE/END].
 *   hidden:   device bf16 [n_hidden, width]; width = 5120.
 *   spans:    host array of n_spans entries (n_spans <= DS_VIT_MAX_IMAGES);
 *             every span must lie inside [0, n_hidden) and its embed rows
 *             inside [0, n_embeds); spans must not overlap.
 *   embeds:   device bf16 [n_embeds, width]; sentinel: device bf16 [3, width].
 * Exact copy (bit-for-bit); rows outside the spans are not touched.
 */
int ds_vit_overlay(void* hidden, int64_t n_hidden, int32_t width, const ds_vit_span* spans,
                   int n_spans, const void* embeds, int64_t n_embeds, const void* sentinel,
                   void* stream);

/*
 * ds_vit_overlay_rows: the overlay driven by caller-given per-row arrays
 * ([A] "Connect the complete image-to-text path first": IMAGE rows take
 * aligner rows, START / NEWLINE / END rows the learned vectors; [A]'s routing
 * section: the rows travel with their type).  For entry i < n:
 *   hidden[rows[i]] = type[i] == IMAGE ? embeds[src[i]] : sentinel[START/NEWLINE/END].
 * This form places rows anywhere (a non-contiguous placeholder layout, spans
 * already interleaved with text by the caller); ds_vit_overlay is the compact
 * form for contiguous spans.
 *   hidden:  device bf16 [n_hidden, width]; width a multiple of 8.
 *   rows, src: device int32 [n]; type: device uint8 [n] (DS_VIT_TOK_*), as
 *            written by ds_vit_layout (rows = the destination rows, e.g. the
 *            layout's pos when positions equal prompt rows).  src is read only
 *            for IMAGE entries.  Rows must be distinct (two entries naming one
 *            row leave either one's value).
 *   embeds:  device bf16 [n_embeds, width]; sentinel: device bf16 [3, width].
 *   status:  device int32, 0 on entry.  The entries live on the device, so
 *            they are checked there, all of them before any row is written:
 *            a type above DS_VIT_TOK_END records DS_VIT_EINVAL, a row outside
 *            [0, n_hidden) or an IMAGE src outside [0, n_embeds) records
 *            DS_VIT_ERANGE, and then nothing is written.  Read it after the
 *            stream's work completes; a nonzero value left in it also stops
 *            later calls from writing.
 * Returns DS_VIT_EINVAL for null or misaligned pointers (rows, src, status
 * 4-byte; hidden, embeds, sentinel 16-byte) or bad sizes, before any launch.
 * Exact copy (bit-for-bit); rows not listed are not touched.
 */
int ds_vit_overlay_rows(void* hidden, int64_t n_hidden, int32_t width, const int32_t* rows,
                        const uint8_t* type, const int32_t* src, int64_t n, const void* embeds,
                        int64_t n_embeds, const void* sentinel, int32_t* status, void* stream);

/*
 * ds_vit_overlay_chunk: the overlay for chunked prefill ([A] "Connect the
 * complete image-to-text path first": an image span may cross a chunk
 * boundary, so each embedding chunk replaces only the rows of the spans that
 * intersect it; [A]'s routing section: a row-level image-rows mask).
 *   chunk:       device bf16 [chunk_rows, width], prompt rows
 *                chunk_begin .. chunk_begin + chunk_rows - 1 (chunk_rows >= 1).
 *   spans:       as ds_vit_overlay, in prompt rows (base_row >= 0); they may
 *                extend past the chunk; embed rows inside [0, n_embeds); no overlap.
 *   row_type:    device uint8 [chunk_rows] or NULL: 0 for rows outside every
 *                span, 1 + the layout type for span rows (START 1, IMAGE 2,
 *                NEWLINE 3, END 4); the image-rows mask is row_type != 0.
 * Span rows inside the chunk are written exactly as ds_vit_overlay writes
 * them; the other rows of the chunk are not touched.  Overlaying every chunk
 * of a prompt equals one ds_vit_overlay of the whole prompt.
 */
int ds_vit_overlay_chunk(void* chunk, int64_t chunk_begin, int64_t chunk_rows, int32_t width,
                         const ds_vit_span* spans, int n_spans, const void* embeds,
                         int64_t n_embeds, const void* sentinel, uint8_t* row_type,
                         void* stream);

/* Kernel kinds reported by ds_vit_set_kernel_timer. */
/* PATCH_GEMM patchifies and normalises the pixels inside its A-tile load;
 * MERGER_GEMM1 gathers the 3x3 windows inside its A-tile load. */
#define DS_VIT_KERNEL_PATCH_GEMM 0
#define DS_VIT_KERNEL_LAYERNORM 1
#define DS_VIT_KERNEL_QKV_GEMM 2
#define DS_VIT_KERNEL_ATTENTION 3
#define DS_VIT_KERNEL_PROJ_GEMM 4
#define DS_VIT_KERNEL_FC1_GEMM 5
#define DS_VIT_KERNEL_FC2_GEMM 6
#define DS_VIT_KERNEL_MERGER_GEMM1 7
#define DS_VIT_KERNEL_MERGER_GEMM2 8

/*
 * ds_vit_set_kernel_timer (profiling aid): after this call, every kernel that
 * an encode call on `p` launches is bracketed on its stream by
 * cudaEventRecord(events[2i]) and cudaEventRecord(events[2i+1]) for the i-th
 * launch of that call; kinds[i] receives its DS_VIT_KERNEL_* code and
 * *n_recorded the number of launches of the latest call (launches past n_slots
 * run untimed).  events: host array of 2*n_slots cudaEvent_t (created by the
 * caller with timing enabled); kinds: host int32 [n_slots]; n_recorded: host
 * int32.  All stay caller-owned and must outlive the attachment.
 * events = NULL detaches.  Encodes on `p` must not run concurrently while
 * attached.
 */
int ds_vit_set_kernel_timer(ds_vit_prepared* p, void* const* events, int32_t* kinds,
                            int32_t n_slots, int32_t* n_recorded);

/* ---------------------------------------------------------------------------
 * The Qwen3-VL-style tower ([A] comparison table, "Patch order reflects the
 * spatial reducer", "Qwen3-VL has two layers of positional meaning",
 * "DeepStack means that 'vision output' is plural"): 16x16x2 patches (a still
 * image fills both temporal slots) in 2x2-merge-group order, a learned 48x48
 * position table interpolated (bilinear, align corners) to the grid, n_layers
 * pre-LayerNorm blocks (hidden 1152, 16 heads of 72, 2D RoPE: dims 0..35 at
 * the patch row and 36..71 at the column, pairs (j, j+18), GELU MLP 4608), a
 * 2x2 merger (LayerNorm, 4 rows -> 4608, Linear 4608 + GELU, Linear 5120), and
 * three DeepStack mergers of the same shape on the outputs of blocks 8, 16, 24.
 * Config: hidden 1152, heads 16, head_dim 72, mlp 4608, out_dim 5120, patch
 * 16, merge 2, norm_kind LAYER, mlp_kind GELU (DS_VIT_EINVAL otherwise).
 * ------------------------------------------------------------------------- */
typedef struct ds_vit_qwen_merger {
  const void *ln_g, *ln_b;   /* [1152] */
  const void *w1, *b1;       /* [4608, 4608] (input = 4 patch rows concatenated), [4608] */
  const void *w2, *b2;       /* [5120, 4608], [5120] */
} ds_vit_qwen_merger;

typedef struct ds_vit_qwen_weights {
  const void* patch_w;       /* [1152, 1536], column ((c*2 + t)*16 + y)*16 + x */
  const void* patch_b;       /* [1152] */
  const void* pos_table;     /* [48*48, 1152], row y*48 + x */
  ds_vit_layer_weights layers[DS_VIT_MAX_LAYERS];   /* qkv [3456, 1152] (q, k, v heads of 72), */
                                                    /* proj [1152, 1152], fc1 [4608, 1152], fc2 [1152, 4608] */
  ds_vit_qwen_merger merger;        /* primary output */
  ds_vit_qwen_merger deepstack[3];  /* taps after blocks 8, 16, 24 (needed when n_layers reaches them) */
} ds_vit_qwen_weights;

typedef struct ds_vit_qwen_prepared ds_vit_qwen_prepared;

/* Device copies (W_qkv with every head padded to 80 rows, the q and k rows of
 * each head reordered so that rotation pairs share a 16-row group; the pixel
 * table; the RoPE table) and TMA descriptors.  Synchronises `stream`. */
int ds_vit_qwen_prepare(const ds_vit_config* cfg, const ds_vit_qwen_weights* w,
                        ds_vit_qwen_prepared** out, void* stream);
int ds_vit_qwen_release(ds_vit_qwen_prepared* p);

/* Workspace of one H x W encode (host only).  H, W positive multiples of 32,
 * T = (H/32)(W/32) <= DS_VIT_MAX_TOKENS, grid sides <= 2048 (else
 * DS_VIT_EINVAL / DS_VIT_ERANGE). */
int ds_vit_qwen_workspace_bytes(int32_t H, int32_t W, size_t* bytes);

/*
 * ds_vit_qwen_encode: one image, device uint8 [H, W, 3] -> out device bf16
 * [T, 5120] (merged tokens in merge-group = row-major order of the 2x2 grid)
 * and, when `deepstack` is not NULL, device bf16 [3, T, 5120] (taps 8, 16, 24;
 * taps past n_layers are not written).  blocks (NULL to skip): device bf16
 * [n_layers + 1, N, 1152], the patch embedding and each block's output, rows in
 * merge-group order.  ws: device workspace of at least
 * ds_vit_qwen_workspace_bytes.  Nothing is written on an argument error.
 */
int ds_vit_qwen_encode(const ds_vit_qwen_prepared* p, const uint8_t* pixels, int32_t H, int32_t W,
                       void* out, void* deepstack, void* ws, size_t ws_bytes, void* blocks,
                       void* stream);

/*
 * ds_vit_qwen_layout (host only): three-axis (t, h, w) M-RoPE positions of the
 * span <vision_start>, h*w <image_pad>, <vision_end> that starts at sequence
 * index seq_start, text before it holding positions equal to its indices
 * ([A] "Qwen3-VL has two layers of positional meaning").  vision_start at
 * p = seq_start on all axes; pad (y, x) at (p+1, p+1+y, p+1+x); vision_end at
 * q = p+1+max(h, w); *rope_delta = q + 1 - (seq_start + h*w + 2), the offset
 * that keeps later positions continuous.  pos: host int32 [3, h*w + 2] (axis
 * major) with cap >= 3*(h*w + 2) entries, or NULL for rope_delta only.
 */
int ds_vit_qwen_layout(int32_t h, int32_t w, int32_t seq_start, int32_t* pos, int64_t cap,
                       int32_t* rope_delta);

/* Synchronise `stream`, then read and clear p's device status word: DS_VIT_OK,
 * or DS_VIT_ETIMEOUT if a kernel's bounded wait gave up since the last read. */
int ds_vit_device_status(const ds_vit_prepared* p, void* stream);

/*
 * ds_vit_selftest_wait_timeout: the failure path of every bounded wait, on the
 * device, without a fault.  One thread waits on a shared-memory mbarrier that
 * nothing completes; after limit_us microseconds of %globaltimer it gives up,
 * sets *status (device int32, caller-owned; not cleared first) to
 * DS_VIT_ETIMEOUT as a timed-out kernel does, stores the time it waited in
 * *elapsed_ns (device uint64) and returns.  The context stays usable.
 * 1 <= limit_us <= 1000000, non-NULL pointers, else DS_VIT_EINVAL (nothing
 * launched).  Asynchronous on `stream`.
 */
int ds_vit_selftest_wait_timeout(int32_t* status, uint64_t* elapsed_ns, uint32_t limit_us, void* stream);

/* ---------------------------------------------------------------------------
 * Single-kernel entry points (the steps of the encode, for step-level parity
 * checks and profiling).  `status` is a caller-owned device int32 that kernels
 * with bounded waits set to DS_VIT_ETIMEOUT on a timeout (never cleared here).
 * ------------------------------------------------------------------------- */

/* y = bf16(LN(x) * g + b) over rows of 1024 (biased variance, fp32 statistics).
 * x, y: device bf16 [M, 1024] (may not alias); g, b: device bf16 [1024]. */
int ds_vit_op_layernorm(const void* x, const void* g, const void* b, void* y, int64_t M,
                        float eps, void* stream);

/* y = bf16(x * (1/sqrt(mean(x^2) + eps)) * g) over rows of 1024 (RMSNorm, the
 * released tower's norm per [A]'s comparison table).  As ds_vit_op_layernorm. */
int ds_vit_op_rmsnorm(const void* x, const void* g, void* y, int64_t M, float eps, void* stream);

/* out[M, N] = epilogue(a[M, K] w[N, K]^T + bias[N]) on the tcgen05 tensor cores.
 * K % 64 == 0, N % 128 == 0 (N % 256 == 0 for SWIGLU), M >= 1.  For DS_VIT_EPI_QKV_ROPE: N = 3072,
 * rowpos (device int32 [M]) holds gy << 16 | gx of each row and rope_cs is the
 * table of ds_vit_op_rope_table; otherwise both may be NULL.  For
 * DS_VIT_EPI_SWIGLU, w and bias hold N/2 gate rows then N/2 up rows and out is
 * [M, N/2]. */
int ds_vit_op_linear(const void* a, int64_t M, int32_t K, const void* w, int32_t N,
                     const void* bias, void* out, int32_t epilogue, const int32_t* rowpos,
                     const float* rope_cs, int32_t* status, void* stream);

/* rope_cs (device fp32 [max_pos, 32]): for pos < max_pos and i < 16,
 * [pos][i] = cos(pos * theta^(-i/16)), [pos][16 + i] = sin(...), evaluated in
 * double precision and rounded to fp32 ([A] Step 3). */
int ds_vit_op_rope_table(float* rope_cs, int32_t max_pos, float theta, void* stream);

/* Bidirectional attention per image over packed rows ([A] "Multimodal basics").
 * qkv: device bf16 [total, 3072] (q | k | v, head h at columns h*64 of each);
 * seqlens: host int32 [n_images]; out: device bf16 [total, 1024] =
 * bf16(softmax(q k^T / 8) v) per image and head. */
int ds_vit_op_attention(const void* qkv, const int32_t* seqlens, int n_images, void* out,
                        int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSVIT_H */
