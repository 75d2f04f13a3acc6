"""CPU oracle of the image preprocessing upstream of the encode.  TEST
INFRASTRUCTURE ONLY (same rules as ``oracle/encode.py``: only the test suite,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import it).

Page A ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision", section
"Step 1: Reproduce the discrete image-processing rules") lists the chain:
plan the largest grid that fits the aspect ratio and the token budget (at most
1,024 image tokens; images under the minimum pixel budget are enlarged first),
constrain the target to the patch and merge grid, resize with PIL "contain"
semantics and bicubic filtering (the other side by *round*, not ceil), centre
on RGB 127 gray.  Page B (ds4-learning glossary "vision", V4.1 paragraph) gives
the minimum pixel budget 295,936 and no 8:1 aspect clamp; the Lucebox page
("Image input", code layout) resizes bicubically to match Pillow byte for byte.

Readings (the pages do not print the planner or the filter arithmetic):

* plan: unit u = 14 * 3 = 42 px.  If H*W < 295,936 the image is enlarged by
  s = sqrt(295,936 / (H W)).  The merged grid covers the (enlarged) image,
  (h, w) = (ceil(sH / u), ceil(sW / u)), when h w <= 1,024; otherwise it is the
  largest grid with the image's aspect ratio under the budget,
  (floor(sH r / u), floor(sW r / u)) with r = sqrt(1,024 u^2 / (s^2 H W)), each
  side at least 1 and the other then capped so that h w <= 1,024.  Canvas =
  (h u) x (w u) pixels.  The encode workloads of 546^2 and up (1344^2, the batch
  sizes, 2688x336) are their own canvases; the 84x84 test image is enlarged.
* contain: PIL's rule on the aspect ratios W/H and Wc/Hc: the wider image keeps
  the canvas width and takes height round(H / W * Wc), the taller one keeps the
  height and takes width round(W / H * Hc) (round half to even, as Python's
  ``round``); equal ratios keep the canvas size.  Placed at
  ((Wc - Wr) // 2, (Hc - Hr) // 2), gray 127 elsewhere.
* bicubic: Keys' cubic convolution kernel with a = -0.5, support 2, widened by
  the scale factor when reducing (antialiasing); per output index i the taps
  start at xmin = trunc(c - support + 0.5) (>= 0) with c = (i + 0.5) in/out and
  end before min(trunc(c + support + 0.5), in); weights filter((x - c + 0.5) /
  max(scale, 1)) summed in order and divided by their sum, then fixed point with
  22 fraction bits rounded half away from zero; each output = clamp((2^21 +
  sum pixel * weight) >> 22, 0, 255).  Horizontal pass first, then vertical;
  a pass whose size does not change is skipped.  This is the separable
  resampling Pillow documents for 8-bit images (32 - 8 - 2 = 22 bits).

Function -> pin (tests/test_preprocess_pins.py): keys (closed-form values,
partition of unity), coeffs (sum, symmetry, identity at scale 1), resample
(identity, constants, linear ramps up and down in the interior, against a
float64 two-dimensional evaluation), contain_size (round versus ceil, half to
even), plan (workload grids, minimum budget, token budget) and preprocess
(gray border, placement).
"""
from __future__ import annotations

import math

import numpy as np

UNIT = 42                  # patch 14 x merge 3
MAX_TOKENS = 1024
MIN_PIXELS = 295936
GRAY = 127
A = -0.5                   # Keys' cubic convolution parameter
SUPPORT = 2.0
PRECISION_BITS = 22        # 32 - 8 - 2


def keys(x: float) -> float:
    """Keys' cubic convolution kernel, a = -0.5, in Horner form (float64)."""
    x = abs(x)
    if x < 1.0:
        return ((A + 2.0) * x - (A + 3.0)) * x * x + 1.0
    if x < 2.0:
        return (((x - 5.0) * x + 8.0) * x - 4.0) * A
    return 0.0


def coeffs(in_size: int, out_size: int):
    """Per output index: first input tap and the fixed-point weights (int64
    array [out_size, ksize], zero past each index's taps)."""
    scale = in_size / out_size
    filterscale = max(scale, 1.0)
    support = SUPPORT * filterscale
    ksize = int(math.ceil(support)) * 2 + 1
    ss = 1.0 / filterscale
    xmin = np.zeros(out_size, dtype=np.int64)
    kk = np.zeros((out_size, ksize), dtype=np.int64)
    for i in range(out_size):
        center = (i + 0.5) * scale
        lo = int(center - support + 0.5)          # truncation toward zero
        lo = max(lo, 0)
        hi = min(int(center + support + 0.5), in_size)
        n = hi - lo
        w = [keys((x + lo - center + 0.5) * ss) for x in range(n)]
        total = 0.0
        for v in w:                                # summed in order
            total += v
        for x in range(n):
            k = w[x] / total if total != 0.0 else w[x]
            f = k * (1 << PRECISION_BITS)
            kk[i, x] = int(f + 0.5) if k >= 0 else int(f - 0.5)
        xmin[i] = lo
    return xmin, kk


def _pass(img: np.ndarray, out_size: int, axis: int) -> np.ndarray:
    """One separable pass along ``axis`` (1 = width, 0 = height) of a uint8
    [H, W, C] image."""
    in_size = img.shape[axis]
    xmin, kk = coeffs(in_size, out_size)
    src = np.moveaxis(img, axis, 0).astype(np.int64)      # [in, other, C]
    out = np.empty((out_size,) + src.shape[1:], dtype=np.uint8)
    for i in range(out_size):
        n = min(kk.shape[1], in_size - xmin[i])
        acc = np.full(src.shape[1:], 1 << (PRECISION_BITS - 1), dtype=np.int64)
        for x in range(n):
            if kk[i, x] != 0:
                acc += src[xmin[i] + x] * kk[i, x]
        out[i] = np.clip(acc >> PRECISION_BITS, 0, 255).astype(np.uint8)
    return np.moveaxis(out, 0, axis)


def resample(img: np.ndarray, out_w: int, out_h: int) -> np.ndarray:
    """Bicubic resize of a uint8 [H, W, C] image to [out_h, out_w, C]."""
    out = np.ascontiguousarray(img)
    if out_w != out.shape[1]:
        out = _pass(out, out_w, 1)
    if out_h != out.shape[0]:
        out = _pass(out, out_h, 0)
    return np.ascontiguousarray(out)


def contain_size(W: int, H: int, Wc: int, Hc: int):
    """Size of an H x W image fitted inside Wc x Hc with PIL contain rules."""
    im_ratio = W / H
    dest_ratio = Wc / Hc
    Wr, Hr = Wc, Hc
    if im_ratio != dest_ratio:
        if im_ratio > dest_ratio:
            Hr = max(1, round(H / W * Wc))
        else:
            Wr = max(1, round(W / H * Hc))
    return Wr, Hr


def plan(H: int, W: int) -> dict:
    """Grid, canvas, resized size and placement for an H x W image."""
    s = 1.0
    if H * W < MIN_PIXELS:
        s = math.sqrt(MIN_PIXELS / (H * W))
    He, We = H * s, W * s
    h, w = math.ceil(He / UNIT), math.ceil(We / UNIT)
    if h * w > MAX_TOKENS:
        r = math.sqrt(MAX_TOKENS * UNIT * UNIT / (He * We))
        h, w = max(1, math.floor(He * r / UNIT)), max(1, math.floor(We * r / UNIT))
        h = max(1, min(h, MAX_TOKENS // w))
        w = min(w, MAX_TOKENS // h)
    Hc, Wc = h * UNIT, w * UNIT
    Wr, Hr = contain_size(W, H, Wc, Hc)
    return {"h": h, "w": w, "gh": 3 * h, "gw": 3 * w, "Hc": Hc, "Wc": Wc, "Hr": Hr, "Wr": Wr,
            "y0": (Hc - Hr) // 2, "x0": (Wc - Wr) // 2}


def preprocess(img: np.ndarray) -> np.ndarray:
    """uint8 [H, W, 3] image -> uint8 [Hc, Wc, 3] canvas of its plan."""
    p = plan(img.shape[0], img.shape[1])
    canvas = np.full((p["Hc"], p["Wc"], 3), GRAY, dtype=np.uint8)
    canvas[p["y0"]:p["y0"] + p["Hr"], p["x0"]:p["x0"] + p["Wr"]] = resample(img, p["Wr"], p["Hr"])
    return canvas
