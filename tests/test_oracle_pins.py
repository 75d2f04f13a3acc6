"""Pins of the CPU oracle against facts fixed outside it: values the pages print
(tests/golden/), closed forms, invariants, library routines for special cases,
and brute force in float64 on tiny inputs.  No GPU needed."""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL

GOLD = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _gold(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ bf16 rounding

def test_round_bf16_ties_to_even():
    one = 1.0
    assert O.round_bf16(np.array([one], F32))[0] == 1.0
    assert O.round_bf16(np.array([1 + 2 ** -8], F32))[0] == 1.0               # tie -> even (0)
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8], F32))[0] == 1 + 2 ** -6   # tie -> even (2)
    assert O.round_bf16(np.array([1 + 2 ** -8 + 2 ** -20], F32))[0] == 1 + 2 ** -7
    assert np.isnan(O.round_bf16(np.array([np.nan], F32))[0])
    assert O.round_bf16(np.array([3.4e38], F32))[0] == np.inf                  # past bf16 max


def test_round_bf16_matches_torch_rne():
    x = np.random.default_rng(0).standard_normal(100000).astype(F32) * 100
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(O.round_bf16(x), ref)


# ------------------------------------------------------------------ patchify / normalise

def test_patch_geometry_fixture():
    g = {k: int(v) for k, v in _gold("patch_geometry.txt")}
    assert g["patch_values"] == 3 * g["patch"] * g["patch"]
    img = WL.uniform_image(28, 42, seed=7)
    P = O.patchify(img, g["patch"])
    assert P.shape == (2 * 3, g["patch_values"])
    assert WL.MODEL["hidden"] == g["hidden"] and WL.MODEL["heads"] == g["heads"]
    assert WL.MODEL["merge"] == g["merge"] and WL.MODEL["out_dim"] == g["out_dim"]
    assert WL.MODEL["image_token_id"] == g["image_token_id"]
    # the largest workload image stays within the 1,024-token budget
    assert (1344 // 14 // 3) ** 2 == g["max_tokens"]


def test_patchify_index_definition():
    """(grid_y, grid_x, channel, y, x) order, element by element."""
    img = WL.uniform_image(42, 56, seed=3)
    P = O.patchify(img)
    gw = 56 // 14
    rng = np.random.default_rng(1)
    for _ in range(500):
        gy, gx, c, y, x = (int(rng.integers(0, 3)), int(rng.integers(0, gw)),
                           int(rng.integers(0, 3)), int(rng.integers(0, 14)), int(rng.integers(0, 14)))
        assert P[gy * gw + gx, c * 196 + y * 14 + x] == img[gy * 14 + y, gx * 14 + x, c]


def test_patchify_roundtrip():
    img = WL.uniform_image(70, 98, seed=4)
    assert np.array_equal(O.unpatchify(O.patchify(img), 5, 7), img)


def test_normalise_endpoints_half():
    """mean = std = 0.5 is the [0,255] -> [-1,1] map: 0 -> -1, 255 -> 1 exactly."""
    P = np.array([[0] * 196 + [255] * 196 + [0] * 196], dtype=np.uint8)
    v = O.normalise(P, (0.5,) * 3, (0.5,) * 3)
    assert np.all(v[0, :196] == -1.0) and np.all(v[0, 196:392] == 1.0)


def test_normalise_clip_closed_form():
    vals = np.arange(256, dtype=np.uint8)
    P = np.tile(vals, 3)[:588][None, :]
    P = np.concatenate([np.repeat(vals[None, :196], 1, 0)] * 3, axis=1)
    v = O.normalise(P, WL.MODEL["mean"], WL.MODEL["std"])
    for c in range(3):
        exact = (vals[:196].astype(np.float64) / 255 - WL.MODEL["mean"][c]) / WL.MODEL["std"][c]
        got = v[0, c * 196:(c + 1) * 196].astype(np.float64)
        assert np.all(np.abs(got - exact) <= np.abs(exact) * 2 ** -8 + 1e-7)


def test_patch_embed_one_hot_selector():
    """With W_pe rows one-hot at column k, output column j = normalised patch value k_j."""
    img = WL.uniform_image(28, 28, seed=9)
    W = WL.make_weights(0)
    ks = np.random.default_rng(2).choice(588, size=1024)
    pw = np.zeros((1024, 588), np.uint16)
    pw[np.arange(1024), ks] = 0x3F80                      # bf16 1.0
    W["patch_w"], W["patch_b"] = pw, np.zeros(1024, np.uint16)
    d = {}
    O.encode([img], W, WL.MODEL, dump=d)
    P = d["patches"]
    assert np.array_equal(d["x0"], P[:, ks])


# ------------------------------------------------------------------ RoPE

def test_rope_angle_order_fixture():
    f = O.rope_freqs(10000.0)
    h, w = 3.0, 5.0
    ang = O.rope_angles(np.array([h]), np.array([w]), 10000.0)[0]
    for slot, axis, fi in _gold("rope_angle_order.txt"):
        coord = h if axis == "h" else w
        assert abs(ang[int(slot)] - coord * f[int(fi)]) <= 1e-15 * coord * f[int(fi)]


def test_rope_frequencies_closed_form():
    f = O.rope_freqs(10000.0)
    assert f[0] == 1.0 and abs(f[8] - 0.01) < 1e-15 and abs(f[4] - 0.1) < 1e-15


def test_rope_one_hot_pairs():
    """rotate-half: e_j -> cos e_j + sin e_{j+16};  e_{j+16} -> cos e_{j+16} - sin e_j,
    height angle on dims 0..31, width angle on dims 32..63."""
    gy, gx = 7, 3
    f = O.rope_freqs(10000.0)
    for j in (0, 5, 15):
        for half, pos in ((0, gy), (1, gx)):
            a = pos * f[j]
            c, s = np.float32(math.cos(a)), np.float32(math.sin(a))
            v = np.zeros((1, 64), F32)
            v[0, half * 32 + j] = 1
            r = O.rope(v, np.array([gy]), np.array([gx]), 10000.0)[0]
            exp = np.zeros(64, F32)
            exp[half * 32 + j], exp[half * 32 + j + 16] = c, s
            assert np.array_equal(r, exp)
            v = np.zeros((1, 64), F32)
            v[0, half * 32 + j + 16] = 1
            r = O.rope(v, np.array([gy]), np.array([gx]), 10000.0)[0]
            exp = np.zeros(64, F32)
            exp[half * 32 + j + 16], exp[half * 32 + j] = c, -s
            assert np.array_equal(r, exp)


def _rope_interleaved(v, gy, gx, theta):
    """A plausible mistake (page A, Step 3): angles interleaved h, w, h, w..."""
    f = O.rope_freqs(theta)
    ang = np.empty((v.shape[0], 32))
    ang[:, 0::2] = np.asarray(gy)[:, None] * f[None, :]
    ang[:, 1::2] = np.asarray(gx)[:, None] * f[None, :]
    cos, sin = np.cos(ang).astype(F32), np.sin(ang).astype(F32)
    h = v.reshape(v.shape[0], -1, 64)
    out = np.empty_like(h)
    for half in range(2):
        c = cos[:, None, half * 16:(half + 1) * 16]
        s = sin[:, None, half * 16:(half + 1) * 16]
        a, b = h[:, :, half * 32:half * 32 + 16], h[:, :, half * 32 + 16:half * 32 + 32]
        out[:, :, half * 32:half * 32 + 16] = a * c - b * s
        out[:, :, half * 32 + 16:half * 32 + 32] = b * c + a * s
    return out.reshape(v.shape[0], -1)


def _blocked_axes_hold(fn):
    v = np.random.default_rng(5).standard_normal((1, 128)).astype(F32)
    a = fn(v, np.array([4]), np.array([2]), 10000.0)
    b = fn(v, np.array([4]), np.array([9]), 10000.0)      # only the width moved
    c = fn(v, np.array([11]), np.array([2]), 10000.0)     # only the height moved
    ah, aw = a.reshape(2, 64)[:, :32], a.reshape(2, 64)[:, 32:]
    return (np.array_equal(ah, b.reshape(2, 64)[:, :32])
            and np.array_equal(aw, c.reshape(2, 64)[:, 32:]))


def test_rope_blocked_axes_and_mutation():
    assert _blocked_axes_hold(O.rope)
    assert not _blocked_axes_hold(_rope_interleaved)


def test_rope_norm_identity_relative():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 1024)).astype(F32)
    k = rng.standard_normal((1, 1024)).astype(F32)
    z = np.array([0])
    assert np.array_equal(O.rope(q, z, z, 1e4), q)
    r = O.rope(q, np.array([191]), np.array([23]), 1e4)
    pn = lambda v: np.hypot(v.reshape(-1, 2, 2, 16)[:, :, 0], v.reshape(-1, 2, 2, 16)[:, :, 1])
    assert np.allclose(pn(r), pn(q), rtol=1e-6, atol=1e-6)
    # q.k depends only on the position difference, separately per axis
    def dot(py, px, ky, kx):
        a = O.rope(q.astype(np.float64).astype(F32), np.array([py]), np.array([px]), 1e4)
        b = O.rope(k, np.array([ky]), np.array([kx]), 1e4)
        return float((a.astype(np.float64) * b).reshape(16, 64).sum(1).sum())
    d0 = dot(0, 0, 5, 3)
    assert abs(dot(10, 7, 15, 10) - d0) < 1e-3 * (1 + abs(d0))
    assert abs(dot(100, 0, 105, 3) - d0) < 1e-3 * (1 + abs(d0))
    assert abs(dot(0, 2, 5, 4) - d0) > 1e-2                        # a different offset


def test_rope_cos_sin_float64_at_max_row():
    gy = np.arange(192)
    ang = O.rope_angles(gy, gy, 1e4)
    f = [10000.0 ** (-i / 16) for i in range(16)]
    for p in (0, 1, 95, 191):
        for i in range(16):
            assert abs(ang[p, i] - p * f[i]) <= 1e-15 * p * f[i]
            assert abs(ang[p, 16 + i] - p * f[i]) <= 1e-15 * p * f[i]


# ------------------------------------------------------------------ LayerNorm / GELU

def test_layernorm_moments_and_constant_row():
    x = np.random.default_rng(7).standard_normal((64, 1024)).astype(F32) * 3 + 1
    y = O.layer_norm(x, np.ones(1024, F32), np.zeros(1024, F32), 1e-6)
    assert np.allclose(y.mean(1), 0, atol=1e-5) and np.allclose(y.var(1), 1, atol=1e-4)
    b = np.random.default_rng(8).standard_normal(1024).astype(F32)
    g = np.random.default_rng(9).standard_normal(1024).astype(F32)
    y = O.layer_norm(np.full((2, 1024), 0.375, F32), g, b, 1e-6)
    assert np.array_equal(y, np.broadcast_to(b, (2, 1024)))


def test_gelu_closed_form_and_tanh_gap():
    z = np.linspace(-6, 6, 2001).astype(F32)
    g = O.gelu(z)
    ref = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in z.astype(np.float64)])
    assert np.allclose(g, ref, rtol=1e-6, atol=1e-7)
    tanh = 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))
    gap = np.abs(tanh - g).max()
    assert 1e-4 < gap < 3e-3                     # page A: local differences around 1e-3


# ------------------------------------------------------------------ attention

def _attn_bruteforce(q, k, v, heads, d=64):
    nq, n = q.shape[0], k.shape[0]
    out = np.zeros((nq, heads * d))
    for h in range(heads):
        for i in range(nq):
            s = [sum(float(q[i, h * d + t]) * float(k[j, h * d + t]) for t in range(d)) / 8.0
                 for j in range(n)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            tot = sum(e)
            for t in range(d):
                out[i, h * d + t] = sum(e[j] / tot * float(v[j, h * d + t]) for j in range(n))
    return out


def test_attention_bruteforce_float64():
    rng = np.random.default_rng(10)
    q, k, v = (O.round_bf16(rng.standard_normal((5, 128)).astype(F32)) for _ in range(3))
    got = O.attention(q, k, v, heads=2)
    ref = _attn_bruteforce(q, k, v, heads=2)
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-6)


def test_attention_peaked_softmax():
    """Large logits (q, k scaled x10) exercise the max subtraction."""
    rng = np.random.default_rng(11)
    q, k, v = (O.round_bf16(rng.standard_normal((6, 64)).astype(F32) * s) for s in (10, 10, 1))
    got = O.attention(q, k, v, heads=1)
    ref = _attn_bruteforce(q, k, v, heads=1)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-5)


def test_attention_bf16_numerators_reading():
    """The p_bf16 evaluation: numerators exp(s - max) rounded to bf16 before the
    product with V, row sums over the unrounded numerators.  Float64 brute force
    of that reading, and it differs from the fp32-P default by at most the bf16
    rounding of P."""
    rng = np.random.default_rng(21)
    q, k, v = (O.round_bf16(rng.standard_normal((7, 128)).astype(F32) * sc) for sc in (3, 3, 1))
    with O.evaluation("f32", p_bf16=True):
        got = O.attention(q, k, v, heads=2)
    ref, mag = np.zeros((7, 128)), np.zeros((7, 128))
    for h in range(2):
        sl = slice(64 * h, 64 * h + 64)
        s = q[:, sl].astype(np.float64) @ k[:, sl].astype(np.float64).T / 8.0
        e = np.exp(s - s.max(axis=1, keepdims=True))
        ref[:, sl] = _bf16(e) @ v[:, sl] / e.sum(axis=1, keepdims=True)
        mag[:, sl] = e @ np.abs(v[:, sl]) / e.sum(axis=1, keepdims=True)    # sum of p |v|
    # each side rounds its output to bf16 once (2^-9 relative) after fp32 sums
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-5 * mag)
    base = O.attention(q, k, v, heads=2)
    assert not np.array_equal(got, base)                  # the reading changes results
    # P's own rounding moves the output by at most 2^-9 of sum p |v| (plus 2^-9
    # of it again through the row sum), besides the two output roundings
    assert np.all(np.abs(got - base) <= 2 ** -8 * mag + 2 ** -8 * np.abs(base) + 1e-6)


def test_fp32_function_mode_and_norm_orders():
    """fn32 evaluates GELU / SiLU in fp32 arithmetic: within a few fp32 units
    of the float64 closed form (and not always equal to the float64 path);
    every norm-statistics order gives the same LayerNorm / RMSNorm within fp32
    rounding (and the float64 order differs from the default somewhere)."""
    z = np.linspace(-8, 8, 20001, dtype=F32)
    ref = 0.5 * z.astype(np.float64) * (1 + np.array([math.erf(v / math.sqrt(2)) for v in z.astype(np.float64)]))
    with O.evaluation("f32", fn32=True):
        g32 = O.gelu(z)
        s32 = O.silu(z)
    assert g32.dtype == F32 and s32.dtype == F32
    assert np.all(np.abs(g32 - ref) <= 4 * 2.0 ** -24 * (np.abs(ref) + 1.0))
    assert not np.array_equal(g32, O.gelu(z))
    sref = z.astype(np.float64) / (1 + np.exp(-z.astype(np.float64)))
    assert np.all(np.abs(s32 - sref) <= 4 * 2.0 ** -24 * (np.abs(sref) + 1.0))
    x = np.random.default_rng(25).standard_normal((64, 1024)).astype(F32) * 3 + 1
    g, b = np.full(1024, 1.0, F32), np.zeros(1024, F32)
    base, rbase = O.layer_norm(x, g, b, 1e-6), O.rms_norm(x, g, 1e-6)
    outs = []
    for order in ("f64", "f32_rev"):
        with O.evaluation(order):
            outs.append(O.layer_norm(x, g, b, 1e-6))
            rms = O.rms_norm(x, g, 1e-6)
        assert np.abs(outs[-1] - base).max() <= 1e-5 and np.abs(rms - rbase).max() <= 1e-5
    assert not np.array_equal(outs[0], base)


def test_product_orders_are_valid_evaluations():
    """Every accumulation order of ``mm`` is the same product within the fp32
    bound K * 2^-24 * (|a| |b|); the reversed order is a different evaluation."""
    rng = np.random.default_rng(22)
    a = rng.standard_normal((16, 1024)).astype(F32)
    b = rng.standard_normal((1024, 24)).astype(F32)
    exact = a.astype(np.float64) @ b.astype(np.float64)
    bound = 1024 * 2.0 ** -24 * (np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64))
    outs = {}
    for order in ("f32", "f64", "f32_rev"):
        with O.evaluation(order):
            outs[order] = O.mm(a, b)
        assert outs[order].dtype == F32
        assert np.all(np.abs(outs[order] - exact) <= bound)
    assert np.abs(outs["f64"] - exact).max() <= 2.0 ** -23 * np.abs(exact).max()
    assert not np.array_equal(outs["f32_rev"], outs["f32"])
    with O.evaluation("f64", True):
        with O.products("f32_rev"):                       # keeps the P reading
            assert O.encode.__module__ == "oracle.encode"
    assert O.mm(a, b).dtype == F32                        # modes restored on exit


def test_softmax_rows_sum_to_one():
    s = np.random.default_rng(12).standard_normal((50, 300)).astype(F32) * 20
    p = O.softmax_rows(s)
    assert np.allclose(p.sum(1), 1.0, atol=1e-6) and np.all(p >= 0)


def test_attention_uniform_when_q_zero():
    rng = np.random.default_rng(13)
    k, v = (O.round_bf16(rng.standard_normal((9, 128)).astype(F32)) for _ in range(2))
    got = O.attention(np.zeros((9, 128), F32), k, v, heads=2)
    assert np.allclose(got, O.round_bf16(v.mean(0, dtype=np.float64).astype(F32))[None, :],
                       atol=2 ** -8)


# ------------------------------------------------------------------ blocks (tiny dims)

def _small_cfg():
    return dict(WL.MODEL, hidden=128, heads=2, mlp=256)


def _small_layer(seed):
    rng = np.random.default_rng(seed)
    n = lambda *s: WL.to_bf16_bits(rng.standard_normal(s).astype(F32) * 0.2)
    return dict(ln1_g=WL.to_bf16_bits(1 + rng.standard_normal(128).astype(F32) * 0.1), ln1_b=n(128),
                qkv_w=n(384, 128), qkv_b=n(384), proj_w=n(128, 128), proj_b=n(128),
                ln2_g=WL.to_bf16_bits(1 + rng.standard_normal(128).astype(F32) * 0.1), ln2_b=n(128),
                fc1_w=n(256, 128), fc1_b=n(256), fc2_w=n(128, 256), fc2_b=n(128))


def _bf16(a):
    """Round to bf16 through torch (an independent RNE routine), back to float64."""
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _block_bruteforce(x, L, gy, gx, eps=1e-6):
    """Pre-LN block in float64 loops, each step from its definition; the stored
    activations (LN outputs, q, k, v, attention output, residual stream, MLP
    hidden) are rounded to bf16 at the same points as the definition says."""
    f = {k: O.bits_to_f32(v).astype(np.float64) for k, v in L.items()}
    n, D = x.shape

    def ln(a, g, b):
        out = np.zeros_like(a)
        for i in range(a.shape[0]):
            mu = sum(a[i]) / D
            var = sum((t - mu) ** 2 for t in a[i]) / D
            out[i] = [(a[i, j] - mu) / math.sqrt(var + eps) * g[j] + b[j] for j in range(D)]
        return out

    def lin(a, w, b):
        return np.array([[sum(a[i, t] * w[o, t] for t in range(a.shape[1])) + b[o]
                          for o in range(w.shape[0])] for i in range(a.shape[0])])

    fr = [10000.0 ** (-i / 16) for i in range(16)]

    def rot(vec, i):
        out = vec.copy()
        for hd in range(D // 64):
            for half, pos in ((0, gy[i]), (1, gx[i])):
                base = hd * 64 + half * 32
                for j in range(16):
                    c, s = math.cos(pos * fr[j]), math.sin(pos * fr[j])
                    a, b = vec[base + j], vec[base + j + 16]
                    out[base + j], out[base + j + 16] = a * c - b * s, b * c + a * s
        return out

    x = x.astype(np.float64)
    y = _bf16(ln(x, f["ln1_g"], f["ln1_b"]))
    t = lin(y, f["qkv_w"], f["qkv_b"])
    q = _bf16([rot(t[i, :D], i) for i in range(n)])
    k = _bf16([rot(t[i, D:2 * D], i) for i in range(n)])
    v = _bf16(t[:, 2 * D:])
    o = _bf16(_attn_bruteforce(q, k, v, heads=D // 64))
    x = _bf16(x + lin(o, f["proj_w"], f["proj_b"]))
    y = _bf16(ln(x, f["ln2_g"], f["ln2_b"]))
    hdn = lin(y, f["fc1_w"], f["fc1_b"])
    g = _bf16([[0.5 * a * (1 + math.erf(a / math.sqrt(2))) for a in row] for row in hdn])
    return _bf16(x + lin(g, f["fc2_w"], f["fc2_b"]))


def test_vit_block_bruteforce_tiny():
    cfg = _small_cfg()
    L = _small_layer(14)
    rng = np.random.default_rng(15)
    x = O.round_bf16(rng.standard_normal((6, 128)).astype(F32))
    gy, gx = O.grid_positions(2, 3)
    got = O.vit_block(x, L, cfg, [6], gy, gx)
    ref = _block_bruteforce(x, L, gy, gx)
    err = np.abs(got - ref) / (1 + np.abs(ref))
    assert err.max() < 2 ** -7, err.max()        # allows a rare one-ulp rounding flip
    # a transposed projection is far off
    L2 = dict(L, proj_w=np.ascontiguousarray(L["proj_w"].T))
    bad = O.vit_block(x, L2, cfg, [6], gy, gx)
    assert (np.abs(bad - ref) / (1 + np.abs(ref))).max() > 0.05


def test_vit_block_rows_subset_matches_full():
    cfg = _small_cfg()
    L = _small_layer(16)
    x = O.round_bf16(np.random.default_rng(17).standard_normal((20, 128)).astype(F32))
    gy = np.concatenate([O.grid_positions(3, 4)[0], O.grid_positions(2, 4)[0]])
    gx = np.concatenate([O.grid_positions(3, 4)[1], O.grid_positions(2, 4)[1]])
    full = O.vit_block(x, L, cfg, [12, 8], gy, gx)
    rows = [0, 5, 11, 12, 19]
    assert np.array_equal(O.vit_block(x, L, cfg, [12, 8], gy, gx, rows=rows), full[rows])


def test_varlen_packing_is_block_diagonal():
    cfg = _small_cfg()
    L = _small_layer(18)
    rng = np.random.default_rng(19)
    xa = O.round_bf16(rng.standard_normal((12, 128)).astype(F32))
    xb = O.round_bf16(rng.standard_normal((8, 128)).astype(F32))
    ga, gb = O.grid_positions(3, 4), O.grid_positions(2, 4)
    a = O.vit_block(xa, L, cfg, [12], *ga)
    b = O.vit_block(xb, L, cfg, [8], *gb)
    gy, gx = np.concatenate([ga[0], gb[0]]), np.concatenate([ga[1], gb[1]])
    ab = O.vit_block(np.concatenate([xa, xb]), L, cfg, [12, 8], gy, gx)
    assert np.array_equal(ab, np.concatenate([a, b]))


def test_zero_residual_branches_give_identity_blocks():
    W = WL.make_weights(2)
    for L in W["layers"]:
        for key in ("proj_w", "proj_b", "fc2_w", "fc2_b"):
            L[key] = np.zeros_like(L[key])
    img = WL.uniform_image(42, 42, seed=20)
    d = {}
    O.encode([img], W, WL.MODEL, dump=d)
    assert np.array_equal(d["blocks"][-1], d["x0"])
    z = O.round_bf16(O.layer_norm(d["x0"], O.bits_to_f32(W["lnm_g"]), O.bits_to_f32(W["lnm_b"]), 1e-6))
    assert np.array_equal(d["final_norm"], z)


# ------------------------------------------------------------------ merge

def test_merge_right_edge_fixture():
    C = 4
    z = np.array([[100 * (n + 1) + c for c in range(C)] for n in range(10)], F32)   # gh=2, gw=5
    A = O.merge_unfold(z, 2, 5)
    assert A.shape == (2, C * 9)
    for t, slot, srcp in _gold("aligner_right_edge.txt"):
        for c in range(C):
            want = 0 if srcp == "Z" else 100 * (int(srcp) + 1) + c
            assert A[int(t), c * 9 + int(slot)] == want
    # the page's early mistake (append zeros to the flattened tensor) fails
    flat = np.concatenate([z, np.zeros((8, C), F32)]).reshape(3, 6, C)
    wrong = flat.reshape(1, 3, 2, 3, C).transpose(0, 2, 4, 1, 3).reshape(2, C * 9)
    assert not np.array_equal(wrong, A)


def test_merge_5x5_pads_column_and_row_six():
    z = np.arange(1, 26, dtype=F32)[:, None].repeat(2, 1)
    A = O.merge_unfold(z, 5, 5)                     # -> 2x2 merged grid
    grid = np.zeros((6, 6))
    for t in range(4):
        my, mx = divmod(t, 2)
        for dy in range(3):
            for dx in range(3):
                grid[3 * my + dy, 3 * mx + dx] = A[t, 0 * 9 + dy * 3 + dx]
    assert np.all(grid[:, 5] == 0) and np.all(grid[5, :] == 0)
    assert np.array_equal(grid[:5, :5].ravel(), np.arange(1, 26))


def test_merger_one_hot_selector_recovers_unfold():
    W = WL.make_weights(0)
    rng = np.random.default_rng(21)
    cols = rng.choice(9216, size=5120)
    m1 = np.zeros((5120, 9216), np.uint16)
    m1[np.arange(5120), cols] = 0x3F80
    W.update(m1_w=m1, m1_b=np.zeros(5120, np.uint16),
             m2_w=(np.eye(5120, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16),
             m2_b=np.zeros(5120, np.uint16))
    img = WL.uniform_image(70, 56, seed=22)
    d = {}
    e, _ = O.encode([img], W, WL.MODEL, dump=d)
    assert np.array_equal(e, O.round_bf16(O.gelu(d["merge_A"][:, cols])))


# ------------------------------------------------------------------ layout / overlay

def test_layout_fixture():
    code = {"S": O.TOK_START, "I": O.TOK_IMAGE, "N": O.TOK_NEWLINE, "E": O.TOK_END}
    for row in _gold("span_layout.txt"):
        h, w, types = int(row[0]), int(row[1]), [code[c] for c in row[2:]]
        ids, pos, typ, src = O.layout(3 * h, 3 * w, 129264, base_pos=40)
        assert typ.tolist() == types
        assert np.all(ids == 129264) and pos.tolist() == list(range(40, 40 + len(types)))


@pytest.mark.parametrize("H,W,rows", [(84, 84, 8), (546, 546, 184), (1344, 1344, 1058),
                                      (2688, 336, 578), (1344, 672, 546), (840, 420, 222)])
def test_layout_counts_and_permutation(H, W, rows):
    gh, gw = H // 14, W // 14
    h, w = -(-gh // 3), -(-gw // 3)
    ids, pos, typ, src = O.layout(gh, gw, 7)
    assert len(typ) == rows == 2 + h * (w + 1)
    img = src[typ == O.TOK_IMAGE]
    assert np.array_equal(img, np.arange(h * w))                       # identity order
    assert np.all(src[typ != O.TOK_IMAGE] == -1)
    assert (typ == O.TOK_NEWLINE).sum() == h and typ[0] == O.TOK_START and typ[-1] == O.TOK_END


def test_layout_batch16_total():
    tot = sum(len(O.layout(H // 14, W // 14, 1)[0]) for H, W, _, _ in WL.WORKLOADS["batch16"]["images"])
    assert tot == 6436


def test_overlay_exact_and_untouched():
    rng = np.random.default_rng(23)
    hidden = rng.integers(0, 65535, size=(64, 32), dtype=np.uint16)
    emb = rng.integers(0, 65535, size=(6, 32), dtype=np.uint16)
    sent = rng.integers(0, 65535, size=(3, 32), dtype=np.uint16)
    ids, pos, typ, src = O.layout(6, 9, 1)                               # 2x3 merged
    out = O.overlay(hidden, 10, typ, src, emb, sent)
    n = len(typ)
    assert np.array_equal(out[:10], hidden[:10]) and np.array_equal(out[10 + n:], hidden[10 + n:])
    assert np.array_equal(out[10], sent[0]) and np.array_equal(out[10 + n - 1], sent[2])
    assert np.array_equal(out[11:14], emb[0:3]) and np.array_equal(out[14], sent[1])
    assert np.array_equal(out[15:18], emb[3:6]) and np.array_equal(out[18], sent[1])


def test_overlay_rows_contiguous_equals_span_and_scattered_rows():
    """With rows = base + r the per-row form is the span overlay; scattered
    rows (text rows interleaved) write each listed row from its own source and
    leave every other row untouched."""
    rng = np.random.default_rng(24)
    hidden = rng.integers(0, 65535, size=(64, 32), dtype=np.uint16)
    emb = rng.integers(0, 65535, size=(6, 32), dtype=np.uint16)
    sent = rng.integers(0, 65535, size=(3, 32), dtype=np.uint16)
    ids, pos, typ, src = O.layout(6, 9, 1, base_pos=10)
    assert np.array_equal(O.overlay_rows(hidden, pos, typ, src, emb, sent),
                          O.overlay(hidden, 10, typ, src, emb, sent))
    rows = np.sort(rng.choice(64, len(typ), replace=False))
    out = O.overlay_rows(hidden, rows, typ, src, emb, sent)
    for r, t, s_ in zip(rows, typ, src):
        want = emb[s_] if t == O.TOK_IMAGE else sent[{0: 0, 2: 1, 3: 2}[int(t)]]
        assert np.array_equal(out[r], want)
    rest = np.setdiff1d(np.arange(64), rows)
    assert np.array_equal(out[rest], hidden[rest])


def _two_span_prompt(rng, rows=120, width=16):
    """Prompt with two spans (2x3 and 3x2 merged grids) and text around them."""
    hidden = rng.integers(0, 65535, size=(rows, width), dtype=np.uint16)
    emb = rng.integers(0, 65535, size=(12, width), dtype=np.uint16)
    sent = rng.integers(0, 65535, size=(3, width), dtype=np.uint16)
    spans = [(7, 6, 9, 0), (50, 9, 6, 6)]          # (base_row, gh, gw, embed_row)
    return hidden, emb, sent, spans


def test_overlay_chunks_assemble_to_the_whole_prompt():
    """Page A: a span may cross a chunk boundary and each chunk replaces only
    the intersecting rows.  Any split of the prompt into chunks, overlaid
    chunk by chunk, equals the whole-prompt overlay (pinned above), and the
    row types are the layout's types on span rows, 0 elsewhere."""
    rng = np.random.default_rng(29)
    hidden, emb, sent, spans = _two_span_prompt(rng)
    whole = hidden
    want_type = np.zeros(len(hidden), dtype=np.uint8)
    for base, gh, gw, erow in spans:
        _, _, typ, src = O.layout(gh, gw, 1)
        src = np.where(src >= 0, src + erow, src)
        whole = O.overlay(whole, base, typ, src, emb, sent)
        want_type[base:base + len(typ)] = typ + 1
    for cuts in ([0, 120], [0, 9, 120], [0, 8, 13, 51, 52, 60, 119, 120], list(range(0, 121, 5)),
                 [0, 1, 2, 3, 120]):
        parts, types = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            out, rt = O.overlay_chunk(hidden[a:b], a, spans, emb, sent)
            parts.append(out)
            types.append(rt)
        assert np.array_equal(np.concatenate(parts), whole)
        assert np.array_equal(np.concatenate(types), want_type)


def test_overlay_chunk_outside_spans_is_untouched():
    rng = np.random.default_rng(31)
    hidden, emb, sent, spans = _two_span_prompt(rng)
    out, rt = O.overlay_chunk(hidden[20:50], 20, spans, emb, sent)    # between the spans
    assert np.array_equal(out, hidden[20:50]) and not rt.any()
    out, rt = O.overlay_chunk(hidden[5:8], 5, spans, emb, sent)       # one START row at 7
    assert np.array_equal(out[:2], hidden[5:7]) and np.array_equal(out[2], sent[0])
    assert list(rt) == [0, 0, 1 + O.TOK_START]


# ------------------------------------------------------------------ the official tower variant
# (page A's comparison table: RMSNorm and SwiGLU; Step 3: [h*f, w*f] angles with the
# half-vector rotation; Step 1 item 6: pixels to [-1, 1])

def test_rms_norm_closed_forms():
    g = np.full(1024, 1.0, F32)
    for c in (0.375, -2.0, 13.0):
        y = O.rms_norm(np.full((1, 1024), c, F32), g, 1e-6)
        assert np.allclose(y, np.sign(c) * abs(c) / math.sqrt(c * c + 1e-6), rtol=1e-6)
    x = np.random.default_rng(41).standard_normal((4, 1024)).astype(F32) * 3
    y = O.rms_norm(x, g, 1e-6)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-5)                 # unit mean square
    assert np.allclose(O.rms_norm(8 * x, g, 1e-6), y, rtol=1e-5, atol=1e-6)  # scale invariance
    gg = np.random.default_rng(42).standard_normal(1024).astype(F32)
    assert np.allclose(O.rms_norm(x, gg, 1e-6), y * gg, rtol=1e-6)


def test_silu_closed_forms():
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 30.0, -30.0, 1.7])
    s = O.silu(z).astype(np.float64)
    assert s[0] == 0.0
    assert s[1] == pytest.approx(0.75 * math.log(3.0), rel=1e-7)           # sigma(ln 3) = 3/4
    assert s[2] == pytest.approx(-0.25 * math.log(3.0), rel=1e-7)
    assert s[3] == pytest.approx(30.0, rel=1e-7) and abs(s[4]) < 1e-11
    w = np.linspace(-6, 6, 101)
    assert np.allclose(O.silu(w) - O.silu(-w), w, atol=1e-6)                # silu(x) - silu(-x) = x


def test_swiglu_hidden_selects_gate_and_up():
    """One-hot gate row j and up row k: hidden = r(silu(y_j) * y_k)."""
    F, D = 8, 16
    cfg = dict(WL.MODEL, mlp=F, mlp_kind="swiglu")
    rng = np.random.default_rng(43)
    y = O.round_bf16(rng.standard_normal((5, D)).astype(F32))
    w = np.zeros((2 * F, D), F32)
    pairs = [(3, 7), (0, 0), (15, 2), (9, 9), (1, 14), (4, 5), (6, 11), (12, 8)]
    for n, (j, k) in enumerate(pairs):
        w[n, j] = 1.0
        w[F + n, k] = 1.0
    L = {"fc1_w": w, "fc1_b": np.zeros(2 * F, F32)}
    h = O.mlp_hidden(y, L, cfg)
    for n, (j, k) in enumerate(pairs):
        assert np.array_equal(h[:, n], O.round_bf16(O.silu(y[:, j]) * y[:, k]))


def test_rope_half_vector_pairs_and_angle_order():
    """Dim i < 32 pairs with i + 32 and turns by the i-th angle of
    [h*f0..h*f15, w*f0..w*f15] (page A, Step 3)."""
    gy, gx = np.array([5]), np.array([11])
    ang = O.rope_angles(gy, gx, 10000.0)[0]
    for i in (0, 7, 15, 16, 23, 31):
        v = np.zeros((1, 64), F32)
        v[0, i] = 1.0
        out = O.rope_half_vector(v, gy, gx, 10000.0)[0]
        assert out[i] == pytest.approx(math.cos(ang[i]), abs=1e-6)
        assert out[i + 32] == pytest.approx(math.sin(ang[i]), abs=1e-6)
        assert np.count_nonzero(out) == 2
        pos, f = (5, i) if i < 16 else (11, i - 16)
        assert ang[i] == pytest.approx(pos * 10000.0 ** (-f / 16), rel=1e-12)


def test_rope_pairings_differ_by_a_fixed_permutation():
    """Swapping head dims 16..31 with 32..47 maps page A's pairing onto the
    axis-halves pairing exactly, so q.k is the same under both when W_q, W_k
    rows are permuted (the GPU applies the permutation to the weights)."""
    perm = np.r_[0:16, 32:48, 16:32, 48:64]
    rng = np.random.default_rng(44)
    v = rng.standard_normal((9, 128)).astype(F32)
    gy, gx = np.arange(9) % 3, np.arange(9) // 3 + 4
    full = np.concatenate([perm + 64 * h for h in range(2)])
    a = O.rope(v[:, full], gy, gx, 10000.0)
    b = O.rope_half_vector(v, gy, gx, 10000.0)[:, full]
    assert np.array_equal(a, b)


def test_official_block_identity_with_zero_branches():
    cfg = WL.MODEL_OFFICIAL
    L = WL.make_weights_official(1)["layers"][0]
    L = dict(L, proj_w=np.zeros_like(L["proj_w"]), proj_b=np.zeros_like(L["proj_b"]),
             fc2_w=np.zeros_like(L["fc2_w"]), fc2_b=np.zeros_like(L["fc2_b"]))
    x = O.round_bf16(np.random.default_rng(45).standard_normal((36, 1024)).astype(F32))
    gy, gx = O.grid_positions(6, 6)
    assert np.array_equal(O.vit_block(x, L, cfg, [36], gy, gx), x)
