"""Seeded synthetic inputs for the vision-tower encode.

This module draws random numbers and stores them; it holds none of the encode's
arithmetic. Both the CUDA path and the CPU oracle take what it returns as plain
inputs: weights as bf16 bit patterns (uint16), images as uint8 HWC RGB, prompt
hidden-state buffers as bf16 bit patterns.

Recipe (all streams are numpy PCG64 seeded through ``SeedSequence``):

* weights, seed 1000: every matrix and bias ~ N(0, 0.02); LayerNorm gamma
  1 + N(0, 0.02), beta ~ N(0, 0.02); START/NEWLINE/END vectors ~ N(0, 0.02).
  Drawn in fp32 and rounded to bf16 (round to nearest even).  Layer ``l`` draws
  from the stream ``[seed, 1 + l]``, so a 2-layer model is the first two layers
  of the 32-layer one.
* images: uint8 uniform 0..255, or a smooth random gradient plus N(0, 20) noise.
* the named workloads (sizes cycle as stated): ``tiny`` 84x84, 2 layers;
  ``min`` 546x546 gradient; ``max`` 1344x1344 uniform; ``batch16`` 16 mixed
  sizes; ``aspect`` 2688x336.
"""
from __future__ import annotations

import numpy as np

# Model constants of the encode (dims, rope theta, LN eps, CLIP pixel statistics,
# the image token id).  They are part of the model definition that both sides
# receive as an input.
MODEL = dict(
    hidden=1024, heads=16, head_dim=64, mlp=4096, out_dim=5120,
    patch=14, merge=3, rope_theta=10000.0, ln_eps=1e-6,
    mean=(0.48145466, 0.4578275, 0.40821073),
    std=(0.26862954, 0.26130258, 0.27577711),
    image_token_id=129264,
)

# The tower as the pages describe the released checkpoint (page A's comparison
# table and Step 1 / Step 3): RMSNorm, SwiGLU MLP (gate and up of 4096 rows
# each), pixels mapped to [-1, 1], and page A's RoPE pairing (angle vector
# [h*f, w*f], dim i paired with dim i + 32).
MODEL_OFFICIAL = dict(MODEL, norm="rmsnorm", mlp_kind="swiglu", rope_pairing="half_vector",
                      mean=(0.5, 0.5, 0.5), std=(0.5, 0.5, 0.5))

WEIGHT_SEED = 1000

LAYER_KEYS = ("ln1_g", "ln1_b", "qkv_w", "qkv_b", "proj_w", "proj_b",
              "ln2_g", "ln2_b", "fc1_w", "fc1_b", "fc2_w", "fc2_b")


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (storage format of the draws)."""
    # uint32 arithmetic does not wrap for finite inputs (all draws are finite).
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, std=0.02, mean=0.0):
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
                        + np.float32(mean))


def make_layer(layer: int, seed: int = WEIGHT_SEED, hidden=1024, mlp=4096) -> dict:
    r = _rng(seed, 1 + layer)
    return dict(
        ln1_g=_normal(r, hidden, mean=1.0), ln1_b=_normal(r, hidden),
        qkv_w=_normal(r, (3 * hidden, hidden)), qkv_b=_normal(r, 3 * hidden),
        proj_w=_normal(r, (hidden, hidden)), proj_b=_normal(r, hidden),
        ln2_g=_normal(r, hidden, mean=1.0), ln2_b=_normal(r, hidden),
        fc1_w=_normal(r, (mlp, hidden)), fc1_b=_normal(r, mlp),
        fc2_w=_normal(r, (hidden, mlp)), fc2_b=_normal(r, hidden),
    )


def make_weights_official(n_layers: int, seed: int = WEIGHT_SEED) -> dict:
    """Weights of MODEL_OFFICIAL: the default draws, with each layer's fc1
    extended to the SwiGLU layout (rows [0, 4096) gate = the default fc1, rows
    [4096, 8192) up, drawn from stream tag 500 + layer).  Norm betas are drawn
    as usual and unused by RMSNorm."""
    w = make_weights(n_layers, seed)
    for l, L in enumerate(w["layers"]):
        r = _rng(seed, 500 + l)
        mlp, hidden = L["fc1_w"].shape
        L["fc1_w"] = np.concatenate([L["fc1_w"], _normal(r, (mlp, hidden))])
        L["fc1_b"] = np.concatenate([L["fc1_b"], _normal(r, mlp)])
    return w


# The Qwen3-VL-style tower (page A's comparison table; oracle/qwen.py lists the
# readings): hidden 1152, 16 heads of 72, MLP 4608, 27 layers, 16x16x2
# patches, 48x48 position table, 2x2 merger to 5120, DeepStack taps 8/16/24.
QWEN_MODEL = dict(hidden=1152, heads=16, head_dim=72, mlp=4608, out_dim=5120, patch=16, temporal=2,
                  merge=2, pos_side=48, rope_theta=10000.0, ln_eps=1e-6, taps=(8, 16, 24),
                  n_layers=27, mean=MODEL["mean"], std=MODEL["std"])
QWEN_SEED = 2000


def _qwen_merger(r, D=1152, out=5120):
    return dict(ln_g=_normal(r, D, mean=1.0), ln_b=_normal(r, D), w1=_normal(r, (4 * D, 4 * D)),
                b1=_normal(r, 4 * D), w2=_normal(r, (out, 4 * D)), b2=_normal(r, out))


def make_weights_qwen(n_layers: int, seed: int = QWEN_SEED) -> dict:
    """bf16 bit patterns: patch_w [1152, 1536] (column ((c*2 + t)*16 + y)*16 + x),
    pos_table [48*48, 1152] (row y*48 + x), per layer the fields of a block
    (qkv_w [3456, 1152], fc1_w [4608, 1152], ...), "merger" and three
    "deepstack" mergers (ln_g, ln_b, w1 [4608, 4608], b1, w2 [5120, 4608], b2).
    Stream tags: 0 patch/pos, 1 + l layer l, 100 merger, 101..103 DeepStack."""
    D, F = 1152, 4608
    r0 = _rng(seed, 0)
    w = dict(patch_w=_normal(r0, (D, 1536)), patch_b=_normal(r0, D), pos_table=_normal(r0, (48 * 48, D)))
    layers = []
    for l in range(n_layers):
        r = _rng(seed, 1 + l)
        layers.append(dict(
            ln1_g=_normal(r, D, mean=1.0), ln1_b=_normal(r, D),
            qkv_w=_normal(r, (3 * D, D)), qkv_b=_normal(r, 3 * D),
            proj_w=_normal(r, (D, D)), proj_b=_normal(r, D),
            ln2_g=_normal(r, D, mean=1.0), ln2_b=_normal(r, D),
            fc1_w=_normal(r, (F, D)), fc1_b=_normal(r, F),
            fc2_w=_normal(r, (D, F)), fc2_b=_normal(r, D)))
    w["layers"] = layers
    w["merger"] = _qwen_merger(_rng(seed, 100))
    w["deepstack"] = [_qwen_merger(_rng(seed, 101 + i)) for i in range(3)]
    return w


def make_weights(n_layers: int, seed: int = WEIGHT_SEED) -> dict:
    """All weights as bf16 bit patterns (uint16), nn.Linear layout [out, in].

    ``patch_w`` is [1024, 588] with input index k = c*196 + y*14 + x (the
    [1024, 3, 14, 14] convolution weight flattened); ``m1_w`` is [5120, 9216]
    with input index c*9 + dy*3 + dx; ``sentinel`` is [3, 5120] holding the
    START, NEWLINE and END vectors in that order.
    """
    h, o = MODEL["hidden"], MODEL["out_dim"]
    r0 = _rng(seed, 0)
    w = dict(patch_w=_normal(r0, (h, 3 * 14 * 14)), patch_b=_normal(r0, h))
    w["layers"] = [make_layer(l, seed) for l in range(n_layers)]
    rm = _rng(seed, 100)
    w.update(lnm_g=_normal(rm, h, mean=1.0), lnm_b=_normal(rm, h),
             m1_w=_normal(rm, (o, 9 * h)), m1_b=_normal(rm, o),
             m2_w=_normal(rm, (o, o)), m2_b=_normal(rm, o),
             sentinel=_normal(rm, (3, o)))
    return w


def uniform_image(H: int, W: int, seed: int) -> np.ndarray:
    return _rng(seed).integers(0, 256, size=(H, W, 3), dtype=np.uint8)


def gradient_image(H: int, W: int, seed: int) -> np.ndarray:
    """pix = clip(round(a_c + b_c*x + d_c*y + N(0, 20)), 0, 255) with
    a_c ~ U(64, 192) and b_c, d_c ~ U(-128/W, 128/W)."""
    r = _rng(seed)
    a = r.uniform(64, 192, size=3)
    b = r.uniform(-128 / W, 128 / W, size=3)
    d = r.uniform(-128 / W, 128 / W, size=3)
    y, x = np.mgrid[0:H, 0:W]
    img = (a[None, None, :] + b[None, None, :] * x[..., None] + d[None, None, :] * y[..., None]
           + r.normal(0.0, 20.0, size=(H, W, 3)))
    return np.clip(np.rint(img), 0, 255).astype(np.uint8)


# Inputs of the preprocessing step (plan, contain resize, gray canvas): images
# off the patch grid, as a camera or a rendered chart delivers them.
#   photo: 3024 x 4032 (H x W) gradient + noise, seed 6 -> 27 x 36 merged grid;
#   chart: 600 x 800 uniform, seed 7 -> 15 x 20 grid (resized up by 1.05).
PREPROCESS_WORKLOADS = {
    "photo": (3024, 4032, "gradient", 6),
    "chart": (600, 800, "uniform", 7),
}


def hidden_buffer(rows: int, width: int, seed: int) -> np.ndarray:
    """Prompt hidden states ~ N(0, 1) as bf16 bit patterns."""
    return to_bf16_bits(_rng(seed).standard_normal((rows, width), dtype=np.float32))


BATCH16_SIZES = ((546, 546), (1344, 672), (672, 1344), (1008, 1008), (840, 420))

# Named workloads.  ``images`` gives (H, W, kind, seed) per image.
WORKLOADS = {
    "tiny": dict(n_layers=2, images=[(84, 84, "uniform", 1)]),
    "min": dict(n_layers=32, images=[(546, 546, "gradient", 2)]),
    "max": dict(n_layers=32, images=[(1344, 1344, "uniform", 3)],
                hidden_rows=4096, hidden_seed=30, base_seed=31),
    "batch16": dict(n_layers=32,
                    images=[BATCH16_SIZES[i % 5] + ("uniform", 40 + i) for i in range(16)],
                    hidden_rows=16384, hidden_seed=56, base0=64, gap=32),
    "aspect": dict(n_layers=32, images=[(2688, 336, "uniform", 5)], repeats=8),
}


def make_image(H: int, W: int, kind: str, seed: int) -> np.ndarray:
    if kind == "uniform":
        return uniform_image(H, W, seed)
    if kind == "gradient":
        return gradient_image(H, W, seed)
    raise ValueError(kind)


def workload_images(name: str) -> list:
    return [make_image(*spec) for spec in WORKLOADS[name]["images"]]


def span_bases(name: str, span_rows: list) -> list:
    """Destination row of each image's span in the prompt buffer, given the row
    count of each span (``span_rows``, from a layout computed elsewhere).

    ``max``: one span at a seeded base ~ U[0, rows - span].  ``batch16``: spans in
    request order starting at row 64 with 32 text rows between consecutive spans.
    """
    wl = WORKLOADS[name]
    if "base_seed" in wl:
        return [int(_rng(wl["base_seed"]).integers(0, wl["hidden_rows"] - span_rows[0] + 1))]
    if "base0" in wl:
        bases, b = [], wl["base0"]
        for n in span_rows:
            bases.append(b)
            b += n + wl["gap"]
        return bases
    return [0] * len(span_rows)
