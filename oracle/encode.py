"""CPU oracle of the vision-tower encode.  TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import or run anything in this
package.  The product path (the C-ABI library and its Python binding) never
calls it, and this package imports nothing from the product path.

What it computes follows the pages it cites, written as plain numpy:

* page A: "DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision" (zLLM);
* page B: the ds4-learning glossary entry "vision" (the DeepSeek V4.1 Flash
  vision family paragraph and the per-family table);
* the model constants (hidden 1024, 16 heads of 64, pre-LayerNorm, MLP 4096
  with erf GELU, merger LN -> Linear 9216->5120 -> GELU -> Linear 5120->5120,
  CLIP pixel statistics, theta 10000) are inputs (``cfg``), as given by the
  workload definition.

Precision: arithmetic in fp32 (numpy float32, BLAS sgemm for the matrix
products); every tensor that is stored between steps is rounded to bf16 with
round-to-nearest-even (page B's table: "intermediate results rounded to BF16").
Trigonometric and erf values are evaluated in float64 and then cast to fp32.

Function -> pin (tests/test_oracle_pins.py): round_bf16 (bit patterns of known
values), patchify (index definition, inverse, one-hot weight selectors),
normalise ([-1, 1] endpoints, closed form), rope (one-hot pairs, blocked axes,
norm, relative position, angle order fixture), layer_norm (moments, constant
row), attention (row sums, uniform case, brute force in float64, block-diagonal
packing, peaked softmax), gelu (float64 closed form, tanh gap), vit_block
(identity when the residual branches are zero), merge_unfold (integer-coded
grid, the right-edge padding fixture), layout (closed-form counts, types,
permutation) and overlay (exact copy, untouched rows).  End-to-end embedding
values have no published dump to compare with; their pins are the step pins
above.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

F32 = np.float32

# Row types of the image token span.
TOK_START, TOK_IMAGE, TOK_NEWLINE, TOK_END = 0, 1, 2, 3


# Evaluation modes.  The definition fixes every bf16 rounding point but not
# the order of the fp32 sums inside a matrix product, so several evaluations
# are equally valid; tests use the spread between them to bound how strongly
# the bf16 boundaries amplify summation-order noise over many layers.
#
# ``order`` selects how ``mm`` accumulates each dot product:
#   "f32"      fp32 matrix product (BLAS sgemm; the library's summation order);
#   "f64"      accumulated in float64 and rounded to fp32 once (correctly
#              rounded in practice);
#   "f32_rev"  fp32 product with the summation index reversed (BLAS again, so
#              its blocking falls on other terms).
# The order also governs the row statistics of the norms (mean and variance,
# or mean square): numpy's fp32 pairwise sum, a float64 sum, or the fp32 sum
# over the reversed row.
# ``p_bf16`` selects the attention reading in which the unnormalised softmax
# numerators exp(s - max) are rounded to bf16 before the product with V and
# the row sum is taken over the fp32 numerators (a tensor-core kernel feeds P
# to the PV product as bf16); the default keeps P in fp32.
# ``fn32`` evaluates GELU and SiLU in fp32 arithmetic (fp32 erf / exp and fp32
# products) instead of float64 cast to fp32: the same functions, rounded
# differently.
_MODE = {"order": "f32", "p_bf16": False, "fn32": False}


def _row_mean(x: np.ndarray) -> np.ndarray:
    """Mean over the last axis in the order of the evaluation mode, as fp32."""
    order = _MODE["order"]
    if order == "f64":
        return x.astype(np.float64).mean(axis=-1, keepdims=True).astype(F32)
    if order == "f32_rev":
        return x[..., ::-1].mean(axis=-1, dtype=F32, keepdims=True)
    return x.mean(axis=-1, dtype=F32, keepdims=True)


def mm(a, b) -> np.ndarray:
    order = _MODE["order"]
    if order == "f64":
        return (np.asarray(a, np.float64) @ np.asarray(b, np.float64)).astype(F32)
    if order == "f32_rev":
        return (np.ascontiguousarray(np.asarray(a, F32)[:, ::-1])
                @ np.ascontiguousarray(np.asarray(b, F32)[::-1]))
    return np.asarray(a, F32) @ np.asarray(b, F32)


class evaluation:
    """Context manager selecting the evaluation mode (see above)."""

    def __init__(self, order: str = "f32", p_bf16: bool = False, fn32: bool = False):
        assert order in ("f32", "f64", "f32_rev")
        self.mode = {"order": order, "p_bf16": bool(p_bf16), "fn32": bool(fn32)}

    def __enter__(self):
        self.prev = dict(_MODE)
        _MODE.update(self.mode)
        return self

    def __exit__(self, *exc):
        _MODE.update(self.prev)


def products(order: str):
    """Only the accumulation order ("f32", "f64" or "f32_rev")."""
    return evaluation(order, _MODE["p_bf16"], _MODE["fn32"])


def round_bf16(x) -> np.ndarray:
    """fp32 -> nearest bf16 value (ties to even), returned as fp32.

    Bit arithmetic on the fp32 pattern: add 0x7FFF plus the lowest kept bit,
    then clear the 16 dropped bits.  NaN passes through unchanged.
    """
    x = np.ascontiguousarray(x, dtype=F32)
    u = x.view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    r = np.where(np.isnan(x), u, r)
    return r.view(F32)


def bits_to_f32(b) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(F32)


def f32_to_bits(x) -> np.ndarray:
    """fp32 values that are already bf16 values -> their uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=F32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------- preprocessing

def patchify(pix: np.ndarray, patch: int = 14) -> np.ndarray:
    """uint8 [H, W, 3] -> uint8 [gh*gw, 3*patch*patch].

    Page A, "Step 1: Reproduce the discrete image-processing rules", item 5:
    patches are flattened in (grid_y, grid_x, channel, y, x) order, so row
    n = gy*gw + gx and column k = c*patch*patch + y*patch + x hold the pixel at
    image row gy*patch + y, column gx*patch + x, channel c.  Page A, "Step 5":
    one 14x14 RGB patch has 3*14*14 = 588 values.
    """
    H, W, C = pix.shape
    gh, gw = H // patch, W // patch
    t = pix[:gh * patch, :gw * patch].reshape(gh, patch, gw, patch, C)   # gy, y, gx, x, c
    return np.ascontiguousarray(t.transpose(0, 2, 4, 1, 3)).reshape(gh * gw, C * patch * patch)


def unpatchify(P: np.ndarray, gh: int, gw: int, patch: int = 14) -> np.ndarray:
    """Inverse of ``patchify`` (used by its pin)."""
    C = P.shape[1] // (patch * patch)
    t = P.reshape(gh, gw, C, patch, patch).transpose(0, 3, 1, 4, 2)       # gy, y, gx, x, c
    return np.ascontiguousarray(t).reshape(gh * patch, gw * patch, C)


def normalise(P: np.ndarray, mean, std, patch: int = 14) -> np.ndarray:
    """uint8 patch rows -> bf16 values r((p/255 - mean_c)/std_c), fp32 arithmetic.

    Page A, Step 1 item 6 maps [0, 255] to [-1, 1] (mean = std = 0.5); the
    workload's model uses the CLIP mean/std (page B's table pairs bicubic resize
    with CLIP normalisation).  Channel c owns columns [c*196, (c+1)*196).
    """
    pp = patch * patch
    c = np.arange(P.shape[1]) // pp
    m = np.asarray(mean, dtype=F32)[c]
    s = np.asarray(std, dtype=F32)[c]
    v = P.astype(F32) / F32(255.0)
    return round_bf16((v - m[None, :]) / s[None, :])


# ---------------------------------------------------------------- 2D RoPE

def rope_freqs(theta: float, n: int = 16) -> np.ndarray:
    """f_i = theta^(-i/n), i = 0..n-1, float64 (one 32-dim rotary half per axis)."""
    return float(theta) ** (-np.arange(n, dtype=np.float64) / n)


def rope_angles(gy: np.ndarray, gx: np.ndarray, theta: float) -> np.ndarray:
    """Angle vector of each patch, [n, 32] float64: [gy*f0..gy*f15, gx*f0..gx*f15].

    Page A, "Step 3: Height and width occupy blocks in 2D RoPE": height
    frequencies first, then width frequencies (blocked, not interleaved).
    Page B's table: positions are the raw patch grid (not the merged grid).
    """
    f = rope_freqs(theta)
    return np.concatenate([np.asarray(gy, np.float64)[:, None] * f[None, :],
                           np.asarray(gx, np.float64)[:, None] * f[None, :]], axis=1)


def rope_half_vector(v: np.ndarray, gy: np.ndarray, gx: np.ndarray, theta: float) -> np.ndarray:
    """Page A's pairing, taken literally ("Step 3": the angle vector
    [h*f0..h*fn, w*f0..w*fn] with the half-vector rotation convention): per
    head, dim i (i < 32) pairs with dim i + 32 and the pair turns by angle
    ang[i] of rope_angles:  v'[i] = v[i] cos - v[i+32] sin,
    v'[i+32] = v[i+32] cos + v[i] sin.  fp32 rotation, float64 cos/sin."""
    n = v.shape[0]
    ang = rope_angles(gy, gx, theta)                      # [n, 32]
    cos = np.cos(ang).astype(F32)[:, None, :]
    sin = np.sin(ang).astype(F32)[:, None, :]
    h = v.reshape(n, -1, 64)
    a, b = h[:, :, :32], h[:, :, 32:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=2).reshape(n, -1)


def rope(v: np.ndarray, gy: np.ndarray, gx: np.ndarray, theta: float) -> np.ndarray:
    """Rotate one projection (q or k), fp32 [n, heads*64] -> fp32 [n, heads*64].

    Per head: dims [0, 32) form a 32-dim rotary vector at position gy and dims
    [32, 64) one at position gx.  Inside each 32-dim half, the half-vector
    ("rotate half") convention pairs dim j with dim j+16 and rotates the pair by
    angle pos*f_j:  v'[j] = v[j] cos - v[j+16] sin,  v'[j+16] = v[j+16] cos + v[j] sin.
    cos/sin are evaluated in float64 and cast to fp32; the rotation is fp32.
    """
    n = v.shape[0]
    ang = rope_angles(gy, gx, theta)                      # [n, 32]
    cos = np.cos(ang).astype(F32)
    sin = np.sin(ang).astype(F32)
    h = v.reshape(n, -1, 64)
    out = np.empty_like(h)
    for half in range(2):                                  # 0: height (gy), 1: width (gx)
        c = cos[:, None, half * 16:(half + 1) * 16]
        s = sin[:, None, half * 16:(half + 1) * 16]
        a = h[:, :, half * 32: half * 32 + 16]
        b = h[:, :, half * 32 + 16: half * 32 + 32]
        out[:, :, half * 32: half * 32 + 16] = a * c - b * s
        out[:, :, half * 32 + 16: half * 32 + 32] = b * c + a * s
    return out.reshape(n, -1)


# ---------------------------------------------------------------- block pieces

def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float) -> np.ndarray:
    """(x - mu) * (1/sqrt(var + eps)) * g + b over the last axis, fp32, biased variance."""
    x = x.astype(F32)
    mu = _row_mean(x)
    d = x - mu
    var = _row_mean(d * d)
    inv = F32(1.0) / np.sqrt(var + F32(eps))
    return d * inv * g.astype(F32) + b.astype(F32)


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x * (1/sqrt(mean(x^2) + eps)) * g over the last axis, fp32 (page A's
    comparison table: the official vision tower uses RMSNorm; "Step 2" table:
    "RMSNorm semantics" at the final norm output)."""
    x = x.astype(F32)
    ms = _row_mean(x * x)
    inv = F32(1.0) / np.sqrt(ms + F32(eps))
    return x * inv * g.astype(F32)


def norm(x: np.ndarray, g, b, cfg: dict) -> np.ndarray:
    """The block / final norm of the model variant: LayerNorm (default) or RMSNorm."""
    if cfg.get("norm", "layernorm") == "rmsnorm":
        return rms_norm(x, _f(g), cfg["ln_eps"])
    return layer_norm(x, _f(g), _f(b), cfg["ln_eps"])


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z)), float64, returned as fp32 (fp32
    arithmetic under the fn32 evaluation mode)."""
    if _MODE["fn32"]:
        zf = np.asarray(z, dtype=F32)
        return zf / (F32(1.0) + np.exp(-zf))
    zz = np.asarray(z, dtype=np.float64)
    return (zz / (1.0 + np.exp(-zz))).astype(F32)


def gelu(z: np.ndarray) -> np.ndarray:
    """GELU with erf (page A, "End-to-end results and their limits": the official
    vision path uses erf, not the tanh approximation): 0.5 z (1 + erf(z/sqrt 2)),
    evaluated in float64, returned as fp32 (fp32 arithmetic under the fn32
    evaluation mode)."""
    if _MODE["fn32"]:
        zf = np.asarray(z, dtype=F32)
        e = _erf(zf * F32(1.0 / math.sqrt(2.0))).astype(F32)
        return F32(0.5) * zf * (F32(1.0) + e)
    zz = np.asarray(z, dtype=np.float64)
    return (0.5 * zz * (1.0 + _erf(zz / math.sqrt(2.0)))).astype(F32)


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax in fp32 with the row maximum subtracted first."""
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True, dtype=F32)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, heads: int,
              head_dim: int = 64) -> np.ndarray:
    """Bidirectional attention of one image: every patch attends to every patch
    of the same image, no mask (page A, "Multimodal basics": attention gives
    each patch information from the whole image).

    q: [nq, heads*64] (bf16 values), k, v: [n, heads*64].  Scale 1/sqrt(64).
    Returns r(softmax(q k^T / 8) v), [nq, heads*64].
    """
    scale = F32(1.0 / math.sqrt(head_dim))
    out = np.empty((q.shape[0], heads * head_dim), dtype=F32)
    for h in range(heads):
        sl = slice(h * head_dim, (h + 1) * head_dim)
        s = mm(q[:, sl], k[:, sl].T) * scale
        if _MODE["p_bf16"]:
            e = np.exp(s - s.max(axis=-1, keepdims=True))
            out[:, sl] = mm(round_bf16(e), v[:, sl]) / e.sum(axis=-1, keepdims=True, dtype=F32)
        else:
            p = softmax_rows(s)
            out[:, sl] = mm(p, v[:, sl])
    return round_bf16(out)


# ---------------------------------------------------------------- ViT block

def _f(w):
    return bits_to_f32(w) if np.asarray(w).dtype == np.uint16 else np.asarray(w, dtype=F32)


def qkv_project(y, L, cfg, gy, gx):
    """t = y W_qkv^T + b (fp32); q = r(rope(t_q)), k = r(rope(t_k)), v = r(t_v).
    Page A, "Step 2" table (block 0 output isolates QKV bias, attention and
    residual order); page B's table: no QK norm."""
    D = cfg["hidden"]
    t = mm(y, _f(L["qkv_w"]).T) + _f(L["qkv_b"])
    rot = rope_half_vector if cfg.get("rope_pairing", "axis_halves") == "half_vector" else rope
    q = round_bf16(rot(t[:, :D], gy, gx, cfg["rope_theta"]))
    k = round_bf16(rot(t[:, D:2 * D], gy, gx, cfg["rope_theta"]))
    v = round_bf16(t[:, 2 * D:])
    return q, k, v


def mlp_hidden(y, L, cfg):
    """The MLP's stored hidden activation.  GELU MLP (default): r(GELU(y W_1^T +
    b_1)).  SwiGLU (page A's comparison table for the official tower): W_1 and
    b_1 hold the gate rows first and the up rows second, each ``mlp`` rows;
    r(SiLU(y W_gate^T + b_gate) * (y W_up^T + b_up)), the product in fp32."""
    t = mm(y, _f(L["fc1_w"]).T) + _f(L["fc1_b"])
    if cfg.get("mlp_kind", "gelu") == "swiglu":
        F = cfg["mlp"]
        return round_bf16(silu(t[:, :F]) * t[:, F:2 * F])
    return round_bf16(gelu(t))


def block_tail(x_rows, o_rows, L, cfg):
    """x = r(x + (o W_o^T + b_o)); y = r(norm2(x)); g = mlp_hidden(y);
    x = r(x + (g W_2^T + b_2)).  Every stored activation is bf16 (page B)."""
    x = round_bf16(x_rows + (mm(o_rows, _f(L["proj_w"]).T) + _f(L["proj_b"])))
    y = round_bf16(norm(x, L["ln2_g"], L["ln2_b"], cfg))
    g = mlp_hidden(y, L, cfg)
    return round_bf16(x + (mm(g, _f(L["fc2_w"]).T) + _f(L["fc2_b"])))


def vit_block(x, L, cfg, seqlens, gy, gx, rows=None):
    """One pre-LayerNorm ViT block over the packed patches of several images.

    ``seqlens`` gives the patch count of each packed image (attention never
    crosses images).  With ``rows`` (indices into x) only those output rows are
    computed: the same definition evaluated at a subset of query rows (keys and
    values still come from every patch of the row's image).
    """
    heads = cfg["heads"]
    y = round_bf16(norm(x, L["ln1_g"], L["ln1_b"], cfg))
    q, k, v = qkv_project(y, L, cfg, gy, gx)
    starts = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    sel = np.arange(x.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.empty((sel.shape[0], x.shape[1]), dtype=F32)
    for i in range(len(seqlens)):
        a, b = starts[i], starts[i + 1]
        m = (sel >= a) & (sel < b)
        if m.any():
            o[m] = attention(q[sel[m]], k[a:b], v[a:b], heads, cfg["head_dim"])
    return block_tail(x[sel], o, L, cfg)


# ---------------------------------------------------------------- merger

def merge_unfold(z: np.ndarray, gh: int, gw: int, m: int = 3) -> np.ndarray:
    """[gh*gw, C] -> [h*w, C*m*m], h = ceil(gh/m), w = ceil(gw/m).

    Page A, "Step 4: The aligner pads a two-dimensional grid": pad the right and
    bottom edges of the 2-D grid with zeros to multiples of 3, map each
    (source_y, source_x) to its 3x3 window (y//3, x//3) and offset
    (y%3, x%3), and unfold channel-major: the 9 positions of channel 0, then the
    9 of channel 1, ...  Inside one channel the 9 window positions are taken
    row-major (dy*3 + dx).
    """
    C = z.shape[1]
    h, w = -(-gh // m), -(-gw // m)
    grid = np.zeros((h * m, w * m, C), dtype=z.dtype)
    grid[:gh, :gw] = z.reshape(gh, gw, C)
    t = grid.reshape(h, m, w, m, C).transpose(0, 2, 4, 1, 3)          # my, mx, c, dy, dx
    return np.ascontiguousarray(t).reshape(h * w, C * m * m)


def merger(A: np.ndarray, W: dict) -> np.ndarray:
    """e = r(r(GELU(A W_m1^T + b_m1)) W_m2^T + b_m2) (page A, "Multimodal basics",
    third step, and "Step 2" table: the aligner's two linear projections)."""
    u = round_bf16(gelu(mm(A, _f(W["m1_w"]).T) + _f(W["m1_b"])))
    return round_bf16(mm(u, _f(W["m2_w"]).T) + _f(W["m2_b"]))


# ---------------------------------------------------------------- encode

def grid_positions(gh: int, gw: int):
    n = np.arange(gh * gw)
    return n // gw, n % gw


def encode(images, W: dict, cfg: dict, n_layers: int | None = None, dump: dict | None = None):
    """uint8 images [H, W, 3] (H, W multiples of 14) -> ([sum T, out_dim] bf16
    values as fp32, token offsets [n+1]).

    Patchify + normalise, patch projection, ``n_layers`` ViT blocks over the
    packed images, final (merger) LayerNorm, 3x3 merge, two linears.  With
    ``dump`` the named boundaries are stored in it: "patches", "x0", "blocks"
    (list of block outputs), "final_norm", "merge_A", "out" (page A, "Step 2":
    patches, block outputs, final norm output, aligner output).
    """
    p = cfg["patch"]
    L_all = W["layers"] if n_layers is None else W["layers"][:n_layers]
    grids = [(im.shape[0] // p, im.shape[1] // p) for im in images]
    P = np.concatenate([normalise(patchify(im, p), cfg["mean"], cfg["std"], p) for im in images])
    gy = np.concatenate([grid_positions(*g)[0] for g in grids])
    gx = np.concatenate([grid_positions(*g)[1] for g in grids])
    seqlens = [gh * gw for gh, gw in grids]
    x = round_bf16(mm(P, _f(W["patch_w"]).T) + _f(W["patch_b"]))
    if dump is not None:
        dump["patches"], dump["x0"], dump["blocks"] = P, x, []
    for L in L_all:
        x = vit_block(x, L, cfg, seqlens, gy, gx)
        if dump is not None:
            dump["blocks"].append(x)
    z = round_bf16(norm(x, W["lnm_g"], W["lnm_b"], cfg))
    starts = np.concatenate([[0], np.cumsum(seqlens)])
    A = np.concatenate([merge_unfold(z[starts[i]:starts[i + 1]], *grids[i], cfg["merge"])
                        for i in range(len(images))])
    e = merger(A, W)
    offs = np.concatenate([[0], np.cumsum([-(-gh // 3) * -(-gw // 3) for gh, gw in grids])])
    if dump is not None:
        dump.update(final_norm=z, merge_A=A, out=e)
    return e, offs.astype(np.int64)


# ---------------------------------------------------------------- layout / overlay

def layout(gh: int, gw: int, image_token_id: int, base_pos: int = 0, m: int = 3):
    """Token span of one image (page A, "Connect the complete image-to-text path
    first"; page B, V4.1 paragraph: plain row-major START, per merged row
    w x IMAGE + NEWLINE, END, identity order, every row carries the image token
    id).  Returns ids, pos, type, src (src = merged-token index for IMAGE rows,
    -1 otherwise).  Positions advance one per row (page A, comparison table:
    "the serialized image grid advances through the text sequence")."""
    h, w = -(-gh // m), -(-gw // m)
    types, src = [TOK_START], [-1]
    for y in range(h):
        for x in range(w):
            types.append(TOK_IMAGE)
            src.append(y * w + x)
        types.append(TOK_NEWLINE)
        src.append(-1)
    types.append(TOK_END)
    src.append(-1)
    n = len(types)
    ids = np.full(n, image_token_id, dtype=np.int32)
    pos = (base_pos + np.arange(n)).astype(np.int32)
    return ids, pos, np.asarray(types, dtype=np.uint8), np.asarray(src, dtype=np.int32)


def overlay_chunk(chunk: np.ndarray, chunk_begin: int, spans, embeds, sentinel):
    """Overlay for chunked prefill (page A, "Connect the complete image-to-text
    path first": an image span may cross a chunk boundary, so the engine keeps
    each image's token range and, when it assembles an embedding chunk, replaces
    only the intersecting part; page A's routing section: a row-level
    image-rows mask travels with the rows).

    chunk: [R, width] bit patterns of prompt rows chunk_begin .. chunk_begin+R-1;
    spans: (base_row, gh, gw, embed_row) per image, spans in prompt rows.
    Returns the chunk with every span row inside it written as ``overlay``
    writes it, and row_type uint8 [R]: 0 for rows outside every span, 1 + the
    layout type (START 1, IMAGE 2, NEWLINE 3, END 4) for span rows."""
    out = np.array(chunk, copy=True)
    row_type = np.zeros(out.shape[0], dtype=np.uint8)
    for base, gh, gw, erow in spans:
        _, _, types, src = layout(gh, gw, 0)
        for r, (t, s) in enumerate(zip(types, src)):
            i = base + r - chunk_begin
            if 0 <= i < out.shape[0]:
                if t == TOK_IMAGE:
                    out[i] = embeds[erow + s]
                else:
                    out[i] = sentinel[{TOK_START: 0, TOK_NEWLINE: 1, TOK_END: 2}[int(t)]]
                row_type[i] = 1 + int(t)
    return out, row_type


def overlay_rows(hidden: np.ndarray, rows, types, src, embeds, sentinel) -> np.ndarray:
    """Copy of ``hidden`` with entry i written at row rows[i]: IMAGE entries take
    aligner row embeds[src[i]], START / NEWLINE / END entries the learned
    vector sentinel[0 / 1 / 2] (page A, "Connect the complete image-to-text path
    first"; the rows may lie anywhere in the prompt).  Entries are applied in
    order; bit patterns, exact copy."""
    out = np.array(hidden, copy=True)
    for r, t, s in zip(rows, types, src):
        if t == TOK_IMAGE:
            out[r] = embeds[s]
        else:
            out[r] = sentinel[{TOK_START: 0, TOK_NEWLINE: 1, TOK_END: 2}[int(t)]]
    return out


def overlay(hidden: np.ndarray, base_row: int, types, src, embeds, sentinel) -> np.ndarray:
    """Copy of ``hidden`` (bf16 bit patterns) with the span written at base_row:
    IMAGE rows take aligner rows ``embeds[src]``; START / NEWLINE / END rows take
    the learned vectors ``sentinel[0 / 1 / 2]`` (page A, "Connect the complete
    image-to-text path first").  All arrays are uint16 bit patterns; exact copy."""
    out = np.array(hidden, copy=True)
    for r, (t, s) in enumerate(zip(types, src)):
        if t == TOK_IMAGE:
            out[base_row + r] = embeds[s]
        else:
            out[base_row + r] = sentinel[{TOK_START: 0, TOK_NEWLINE: 1, TOK_END: 2}[int(t)]]
    return out
