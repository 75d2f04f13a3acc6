"""CPU oracle of the Qwen3-VL-style vision tower.  TEST INFRASTRUCTURE ONLY
(same rules as ``oracle/encode.py``).

Page A ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision"),
sections "Comparing the DeepSeek V4.1 Flash and Qwen3-VL vision towers",
"Patch order reflects the spatial reducer", "Qwen3-VL has two layers of
positional meaning" and "DeepStack means that 'vision output' is plural":
16 x 16 patches with temporal patch 2 (a still image fills both temporal
slots; 3 x 2 x 16 x 16 = 1,536 columns), 27 layers, hidden 1,152, 16 heads,
LayerNorm and GELU MLP; a learned 48 x 48 position table interpolated to the
image grid, then visual 2D RoPE; patches of one 2 x 2 merge group contiguous,
so the 2 x 2 merger is a direct merge; DeepStack takes ViT layers 8, 16 and 24
through three separate mergers: one primary embedding plus three DeepStack
tensors.  At the language boundary, visual tokens get temporal / height /
width M-RoPE positions, text tokens equal positions on all three axes, and
rope_delta keeps positions continuous after the image.

Readings (the page does not give these; each is the plainest choice and is
listed in the design notes):
* head_dim = 1152 / 16 = 72; MLP width 4 x 1152 = 4608; LayerNorm eps 1e-6.
* Patch row (c, t, y, x) -> column ((c*2 + t)*16 + y)*16 + x, pixels
  normalised with the config's per-channel mean/std.  Row order: merge group
  (gy//2, gx//2) row-major, inside a group (gy%2, gx%2) row-major.
* Position table [48, 48, 1152] sampled bilinearly at align-corners positions
  y = gy * 47 / (gh - 1), x = gx * 47 / (gw - 1) (0 for a side of 1), in fp32;
  x0 = r(r(pos) + (A W^T + b)).
* 2D RoPE per head: dims [0, 36) a rotate-half vector at the patch row, dims
  [36, 72) one at the patch column, pairs (j, j + 18), f_j = theta^(-j/18).
  q and k are stored in bf16 before and after the rotation: q = r(rot(r(t))).
* Merger (main and each DeepStack tap): LayerNorm(1152) per patch, the four
  consecutive rows of a merge group concatenated to 4608, Linear 4608 -> 4608
  + bias, GELU (erf), Linear 4608 -> 5120 + bias.  Taps: the outputs of blocks
  8, 16 and 24 (1-based).
* Span: <vision_start>, h*w <image_pad>, <vision_end> at sequence index s with
  text positions equal to the index before it.  vision_start at p = s on all
  axes; pad (y, x) at (p+1, p+1+y, p+1+x); vision_end at q = p+1+max(h, w) on
  all axes; rope_delta = (q + 1) - (s + h*w + 2).

Function -> pin (tests/test_qwen_pins.py): patchify (column formula, both
temporal slots, merge-group order and its inverse), pos_interp (grid 48 x 48
returns the table, constant table, linear table reproduced exactly), rope
(one-hot pairs, angle order, relative position), block (identity with zero
branches, float64 brute force of attention at head_dim 72), merger (one-hot
weights select the merge-group concatenation), layout (pages' three-axis rule
and rope_delta on small grids).
"""
from __future__ import annotations

import math

import numpy as np

from .encode import F32, attention, gelu, layer_norm, mm, round_bf16, _f

QWEN = dict(hidden=1152, heads=16, head_dim=72, mlp=4608, out_dim=5120, patch=16, temporal=2,
            merge=2, pos_side=48, rope_theta=10000.0, ln_eps=1e-6, taps=(8, 16, 24))


def patch_order(gh: int, gw: int):
    """(gy, gx) of each patch row in merge-group order."""
    gy, gx = [], []
    for my in range(gh // 2):
        for mx in range(gw // 2):
            for dy in range(2):
                for dx in range(2):
                    gy.append(2 * my + dy)
                    gx.append(2 * mx + dx)
    return np.asarray(gy, dtype=np.int64), np.asarray(gx, dtype=np.int64)


def patchify(img: np.ndarray, mean, std) -> np.ndarray:
    """uint8 [H, W, 3] (H, W multiples of 32) -> normalised bf16 values [N, 1536]
    (r((p/255 - mean_c)/std_c), fp32 arithmetic: the patch matrix is a stored
    tensor), rows in merge-group order, column ((c*2 + t)*16 + y)*16 + x, both
    temporal slots holding the same frame."""
    H, W = img.shape[:2]
    gh, gw = H // 16, W // 16
    gy, gx = patch_order(gh, gw)
    px = (img.astype(F32) / F32(255.0) - np.asarray(mean, F32)) / np.asarray(std, F32)   # [H, W, 3]
    out = np.empty((gh * gw, 1536), dtype=F32)
    for r, (y, x) in enumerate(zip(gy, gx)):
        p = px[16 * y:16 * y + 16, 16 * x:16 * x + 16, :].transpose(2, 0, 1)            # [c, y, x]
        out[r] = np.stack([p, p], axis=1).reshape(-1)                                    # [c, t, y, x]
    return round_bf16(out)


def pos_interp(table: np.ndarray, gh: int, gw: int) -> np.ndarray:
    """Bilinear sample of a [S, S, D] (or [S*S, D]) table at the align-corners
    positions of a gh x gw grid, fp32, [gh*gw, D] in row-major grid order."""
    t = _f(table)
    S = t.shape[0] if t.ndim == 3 else int(round(math.sqrt(t.shape[0])))
    t = t.reshape(S, S, -1)
    ys = np.zeros(gh) if gh == 1 else np.arange(gh) * (S - 1) / (gh - 1)
    xs = np.zeros(gw) if gw == 1 else np.arange(gw) * (S - 1) / (gw - 1)
    out = np.empty((gh, gw, t.shape[2]), dtype=F32)
    for i, yv in enumerate(ys):
        y0 = min(int(math.floor(yv)), S - 1)
        y1 = min(y0 + 1, S - 1)
        fy = F32(yv - y0)
        for j, xv in enumerate(xs):
            x0 = min(int(math.floor(xv)), S - 1)
            x1 = min(x0 + 1, S - 1)
            fx = F32(xv - x0)
            top = t[y0, x0] * (F32(1) - fx) + t[y0, x1] * fx
            bot = t[y1, x0] * (F32(1) - fx) + t[y1, x1] * fx
            out[i, j] = top * (F32(1) - fy) + bot * fy
    return out.reshape(gh * gw, -1)


def rope(v: np.ndarray, gy, gx, theta: float) -> np.ndarray:
    """Per head of 72: dims [0, 36) rotated at the patch row, [36, 72) at the
    patch column; inside each half pairs (j, j+18), angle pos * theta^(-j/18)."""
    n = v.shape[0]
    f = theta ** (-np.arange(18, dtype=np.float64) / 18.0)
    h = v.reshape(n, -1, 72)
    out = np.empty_like(h)
    for half, pos in enumerate((gy, gx)):
        ang = np.asarray(pos, np.float64)[:, None] * f[None, :]
        c = np.cos(ang).astype(F32)[:, None, :]
        s = np.sin(ang).astype(F32)[:, None, :]
        a = h[:, :, half * 36: half * 36 + 18]
        b = h[:, :, half * 36 + 18: half * 36 + 36]
        out[:, :, half * 36: half * 36 + 18] = a * c - b * s
        out[:, :, half * 36 + 18: half * 36 + 36] = b * c + a * s
    return out.reshape(n, -1)


def block(x, L, cfg, gy, gx):
    """One pre-LayerNorm block over the patches of one image (bf16 stored)."""
    D, heads = cfg["hidden"], cfg["heads"]
    y = round_bf16(layer_norm(x, _f(L["ln1_g"]), _f(L["ln1_b"]), cfg["ln_eps"]))
    t = round_bf16(mm(y, _f(L["qkv_w"]).T) + _f(L["qkv_b"]))
    q = round_bf16(rope(t[:, :D], gy, gx, cfg["rope_theta"]))
    k = round_bf16(rope(t[:, D:2 * D], gy, gx, cfg["rope_theta"]))
    v = t[:, 2 * D:]
    o = attention(q, k, v, heads, cfg["head_dim"])
    x = round_bf16(x + (mm(o, _f(L["proj_w"]).T) + _f(L["proj_b"])))
    y = round_bf16(layer_norm(x, _f(L["ln2_g"]), _f(L["ln2_b"]), cfg["ln_eps"]))
    g = round_bf16(gelu(mm(y, _f(L["fc1_w"]).T) + _f(L["fc1_b"])))
    return round_bf16(x + (mm(g, _f(L["fc2_w"]).T) + _f(L["fc2_b"])))


def merger(x, M, cfg) -> np.ndarray:
    """LayerNorm per patch, four consecutive rows concatenated, two linears."""
    z = round_bf16(layer_norm(x, _f(M["ln_g"]), _f(M["ln_b"]), cfg["ln_eps"]))
    A = z.reshape(-1, 4 * z.shape[1])
    u = round_bf16(gelu(mm(A, _f(M["w1"]).T) + _f(M["b1"])))
    return round_bf16(mm(u, _f(M["w2"]).T) + _f(M["b2"]))


def encode(img: np.ndarray, W: dict, cfg: dict, n_layers: int | None = None, dump: dict | None = None):
    """uint8 [H, W, 3] -> (primary [T, 5120], deepstack list of [T, 5120] for the
    taps that ``n_layers`` reaches).  With ``dump``: "x0", "blocks"."""
    H, Wd = img.shape[:2]
    gh, gw = H // 16, Wd // 16
    gy, gx = patch_order(gh, gw)
    A = patchify(img, cfg["mean"], cfg["std"])
    pos = pos_interp(W["pos_table"], gh, gw).reshape(gh, gw, -1)[gy, gx]
    x = round_bf16(round_bf16(pos) + (mm(A, _f(W["patch_w"]).T) + _f(W["patch_b"])))
    layers = W["layers"] if n_layers is None else W["layers"][:n_layers]
    deep = []
    if dump is not None:
        dump["x0"], dump["blocks"] = x, []
    for l, L in enumerate(layers):
        x = block(x, L, cfg, gy, gx)
        if dump is not None:
            dump["blocks"].append(x)
        if l + 1 in cfg["taps"]:
            deep.append(merger(x, W["deepstack"][cfg["taps"].index(l + 1)], cfg))
    return merger(x, W["merger"], cfg), deep


def layout(h: int, w: int, seq_start: int):
    """M-RoPE positions (t, h, w) of the span <vision_start>, h*w <image_pad>,
    <vision_end> starting at sequence index seq_start (text before it has
    positions equal to its index), and rope_delta.  Returns int32 [3, h*w + 2]
    and rope_delta."""
    p = seq_start
    n = h * w + 2
    pos = np.empty((3, n), dtype=np.int32)
    pos[:, 0] = p
    yy, xx = np.divmod(np.arange(h * w), w)
    pos[0, 1:-1] = p + 1
    pos[1, 1:-1] = p + 1 + yy
    pos[2, 1:-1] = p + 1 + xx
    q = p + 1 + max(h, w)
    pos[:, -1] = q
    return pos, (q + 1) - (seq_start + n)
