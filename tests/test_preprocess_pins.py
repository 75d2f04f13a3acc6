"""Pins of the preprocessing oracle (oracle/preprocess.py) against closed forms,
invariants and an independent float64 evaluation.  CPU only.

Page A ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision", "Step 1:
Reproduce the discrete image-processing rules"): grid planning under the token
budget, contain resizing with bicubic filtering and round (not ceil), centring
on RGB 127 gray.  Page B (ds4-learning glossary "vision", V4.1): minimum pixel
budget 295,936, at most 1,024 image tokens.
"""
import math

import numpy as np
import pytest

import oracle.preprocess as P


# ------------------------------------------------------------------ kernel


def test_keys_closed_form_values():
    """Keys' kernel with a = -0.5: (a+2)|x|^3 - (a+3)|x|^2 + 1 on [0, 1) and
    a|x|^3 - 5a|x|^2 + 8a|x| - 4a on [1, 2), expanded here term by term."""
    a = -0.5
    for x in (0.0, 0.1, 0.25, 0.5, 0.75, 0.99, 1.0, 1.25, 1.5, 1.75, 1.99, 2.0, 2.5, 7.0):
        if x < 1:
            ref = (a + 2) * x ** 3 - (a + 3) * x ** 2 + 1
        elif x < 2:
            ref = a * x ** 3 - 5 * a * x ** 2 + 8 * a * x - 4 * a
        else:
            ref = 0.0
        assert P.keys(x) == pytest.approx(ref, abs=1e-15)
        assert P.keys(-x) == P.keys(x)
    assert P.keys(0.5) == 0.5625 and P.keys(1.5) == -0.0625
    assert P.keys(1.0) == 0.0 and P.keys(2.0) == 0.0 and P.keys(0.0) == 1.0


def test_keys_partition_of_unity_and_linear_reproduction():
    """For a = -0.5 the integer shifts of the kernel sum to 1 and reproduce
    linear functions: sum_k f(t - k) = 1, sum_k k f(t - k) = t."""
    for t in np.linspace(0, 1, 37):
        ks = range(-2, 4)
        assert sum(P.keys(t - k) for k in ks) == pytest.approx(1.0, abs=1e-14)
        assert sum(k * P.keys(t - k) for k in ks) == pytest.approx(t, abs=1e-14)


# ------------------------------------------------------------------ coefficients


@pytest.mark.parametrize("n_in,n_out", [(10, 10), (64, 32), (32, 64), (1000, 333), (7, 29), (4032, 1512)])
def test_coeffs_sum_and_range(n_in, n_out):
    xmin, kk = P.coeffs(n_in, n_out)
    one = 1 << P.PRECISION_BITS
    assert kk.shape[0] == n_out
    assert np.all(np.abs(kk.sum(axis=1) - one) <= kk.shape[1])    # each weight rounded once
    assert np.all(xmin >= 0)
    nz = [np.nonzero(kk[i])[0] for i in range(n_out)]
    assert all(xmin[i] + (z.max() if len(z) else 0) < n_in for i, z in enumerate(nz))


def test_coeffs_identity_at_scale_one():
    xmin, kk = P.coeffs(17, 17)
    for i in range(17):
        row = kk[i]
        assert row[i - xmin[i]] == 1 << P.PRECISION_BITS
        assert np.count_nonzero(row) == 1


# ------------------------------------------------------------------ resample


def smooth_image(h, w, seed):
    """Low-frequency image (no bicubic overshoot past 0..255)."""
    rng = np.random.default_rng(seed)
    yy, xx = np.mgrid[0:h, 0:w]
    out = np.empty((h, w, 3), dtype=np.uint8)
    for c in range(3):
        f = 40 + 80 * (0.5 + 0.5 * np.sin(xx / (w / rng.uniform(1, 3)) + yy / (h / rng.uniform(1, 3)) + c))
        out[..., c] = np.round(f + 40 * (yy / h)).astype(np.uint8)
    return out


def test_resample_identity_and_constants():
    img = np.random.default_rng(1).integers(0, 256, (23, 31, 3), dtype=np.uint8)
    assert np.array_equal(P.resample(img, 31, 23), img)
    for v in (0, 1, 127, 254, 255):
        c = np.full((40, 50, 3), v, dtype=np.uint8)
        for (w, h) in ((17, 23), (123, 71), (50, 13), (7, 40)):
            assert np.all(P.resample(c, w, h) == v)


def test_resample_linear_ramp_up_and_down():
    """Bicubic (a = -0.5) reproduces linear functions away from the borders.
    Upsampling x2: out[i] = v((i + 0.5)/2 - 0.5); downsampling x2 with the
    widened kernel: out[i] = v(2 i + 0.5)."""
    x = np.arange(32)
    ramp = np.repeat((10 + 3 * x).astype(np.uint8)[None, :, None], 3, axis=2)
    up = P.resample(ramp, 64, 1)[0, :, 0].astype(np.float64)
    i = np.arange(64)
    ref = 10 + 3 * ((i + 0.5) / 2 - 0.5)            # fractional parts .25 / .75
    inner = slice(4, 60)
    assert np.array_equal(up[inner], np.round(ref[inner]))
    x = np.arange(64)
    ramp = np.repeat((10 + 2 * x).astype(np.uint8)[None, :, None], 3, axis=2)
    dn = P.resample(ramp, 32, 1)[0, :, 0].astype(np.int64)
    i = np.arange(32)
    inner = slice(3, 29)
    assert np.array_equal(dn[inner], (11 + 4 * i)[inner])
    # the same along the height (vertical pass)
    col = np.repeat((10 + 2 * x).astype(np.uint8)[:, None, None], 3, axis=2)
    dv = P.resample(col, 1, 32)[:, 0, 0].astype(np.int64)
    assert np.array_equal(dv[inner], (11 + 4 * i)[inner])


@pytest.mark.parametrize("shape,out", [((40, 52), (31, 17)), ((30, 30), (71, 45)), ((64, 21), (64, 9))])
def test_resample_against_float64_2d(shape, out):
    """Fixed-point separable result vs a float64 two-dimensional evaluation of
    the same normalised filter without intermediate rounding.  Bound: the
    horizontal pass rounds to uint8 (<= 1/2), which the vertical filter scales
    by its absolute row sum, and the vertical pass rounds again (<= 1/2)."""
    img = smooth_image(*shape, seed=3)
    Wo, Ho = out
    got = P.resample(img, Wo, Ho).astype(np.float64)

    def weights(n_in, n_out):
        scale = n_in / n_out
        fs = max(scale, 1.0)
        W = np.zeros((n_out, n_in))
        for i in range(n_out):
            c = (i + 0.5) * scale
            for x in range(n_in):
                d = (x - c + 0.5) / fs
                if abs(d) < 2 and x >= int(c - 2 * fs + 0.5) and x < int(c + 2 * fs + 0.5):
                    W[i, x] = P.keys(d)
            W[i] /= W[i].sum()
        return W

    Wx = weights(shape[1], Wo) if Wo != shape[1] else np.eye(Wo)
    Wy = weights(shape[0], Ho) if Ho != shape[0] else np.eye(Ho)
    ref = np.einsum("yi,ijc,xj->yxc", Wy, img.astype(np.float64), Wx)
    bound = 0.5 + (0.5 * np.abs(Wy).sum(axis=1).max() if Wo != shape[1] else 0.0) + 1e-6
    assert np.abs(got - np.clip(ref, 0, 255)).max() <= bound


# ------------------------------------------------------------------ contain and plan


def test_contain_round_not_ceil_and_half_even():
    # 1/3 of 100 = 33.3: round gives 33 where a covering ceil gives 34 (page A, Step 1).
    assert P.contain_size(300, 100, 100, 100) == (100, 33)
    assert P.contain_size(100, 300, 100, 100) == (33, 100)
    # exact halves round to even: 2.5 -> 2, 7.5 -> 8
    assert P.contain_size(4, 1, 10, 10) == (10, 2)
    assert P.contain_size(4, 3, 10, 10) == (10, 8)
    # equal aspect ratios keep the canvas size
    assert P.contain_size(544, 544, 546, 546) == (546, 546)
    assert P.contain_size(1000, 500, 84, 42) == (84, 42)


@pytest.mark.parametrize("H,W,hw", [(546, 546, (13, 13)), (1344, 1344, (32, 32)), (2688, 336, (64, 8)),
                                    (1344, 672, (32, 16)), (672, 1344, (16, 32)), (1008, 1008, (24, 24)),
                                    (840, 420, (20, 10))])
def test_plan_workloads_are_their_own_canvas(H, W, hw):
    p = P.plan(H, W)
    assert (p["h"], p["w"]) == hw
    assert (p["Hc"], p["Wc"], p["Hr"], p["Wr"], p["y0"], p["x0"]) == (H, W, H, W, 0, 0)


def test_plan_minimum_budget_and_token_budget():
    # 544^2 = 295,936 exactly: not enlarged, covered by 13 x 13 units of 42.
    p = P.plan(544, 544)
    assert (p["h"], p["w"], p["Hc"], p["Hr"]) == (13, 13, 546, 546)
    # small images are enlarged proportionally to the minimum budget first
    for H, W in ((100, 100), (84, 84), (300, 150)):
        p = P.plan(H, W)
        s = math.sqrt(P.MIN_PIXELS / (H * W))
        assert (p["h"], p["w"]) == (math.ceil(H * s / 42), math.ceil(W * s / 42))
    # over the budget: the aspect-preserving floor grid, at most 1,024 tokens
    p = P.plan(3024, 4032)
    assert (p["h"], p["w"]) == (27, 36)
    rng = np.random.default_rng(7)
    for _ in range(300):
        H, W = int(rng.integers(1, 20000)), int(rng.integers(1, 20000))
        p = P.plan(H, W)
        assert 1 <= p["h"] * p["w"] <= P.MAX_TOKENS
        assert p["Hr"] <= p["Hc"] and p["Wr"] <= p["Wc"]
        assert p["Hr"] == p["Hc"] or p["Wr"] == p["Wc"]          # contain fills one side
        s = max(1.0, math.sqrt(P.MIN_PIXELS / (H * W)))
        ceil_grid = (math.ceil(H * s / 42), math.ceil(W * s / 42))
        if ceil_grid[0] * ceil_grid[1] <= P.MAX_TOKENS:
            assert (p["h"], p["w"]) == ceil_grid


def test_preprocess_places_image_on_gray():
    img = smooth_image(100, 300, seed=5)
    p = P.plan(100, 300)
    canvas = P.preprocess(img)
    assert canvas.shape == (p["Hc"], p["Wc"], 3)
    inside = canvas[p["y0"]:p["y0"] + p["Hr"], p["x0"]:p["x0"] + p["Wr"]]
    assert np.array_equal(inside, P.resample(img, p["Wr"], p["Hr"]))
    mask = np.ones(canvas.shape[:2], dtype=bool)
    mask[p["y0"]:p["y0"] + p["Hr"], p["x0"]:p["x0"] + p["Wr"]] = False
    assert mask.any() and np.all(canvas[mask] == P.GRAY)
