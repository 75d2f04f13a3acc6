"""Pins of the Qwen3-VL-style tower oracle (oracle/qwen.py) against closed
forms, invariants, brute force and the page's rules.  CPU only.

Page A ("DeepSeek V4.1 Flash Engineering, Part 3: Integrating Vision"): the
comparison table, "Patch order reflects the spatial reducer", "Qwen3-VL has
two layers of positional meaning", "DeepStack means that 'vision output' is
plural"."""
import math

import numpy as np
import pytest

import oracle as O
import oracle.qwen as Q
import workloads as WL

F32 = np.float32


def test_patch_order_groups_are_contiguous():
    gy, gx = Q.patch_order(4, 6)
    first = list(zip(gy[:8], gx[:8]))
    assert first == [(0, 0), (0, 1), (1, 0), (1, 1), (0, 2), (0, 3), (1, 2), (1, 3)]
    assert sorted(zip(gy, gx)) == [(y, x) for y in range(4) for x in range(6)]
    for r in range(0, 24, 4):                     # each run of 4 is one 2x2 group
        assert len({(int(y) // 2, int(x) // 2) for y, x in zip(gy[r:r + 4], gx[r:r + 4])}) == 1


def test_patchify_columns_and_temporal_slots():
    H, W = 32, 64
    yy, xx = np.mgrid[0:H, 0:W]
    img = np.stack([(yy * 3 + xx) % 256, (yy + 5 * xx) % 256, (7 * yy + xx) % 256], axis=2).astype(np.uint8)
    mean, std = (0.5, 0.25, 0.125), (0.5, 0.5, 0.25)
    A = Q.patchify(img, mean, std)
    gy, gx = Q.patch_order(H // 16, W // 16)
    assert A.shape == (8, 1536)
    for r in (0, 3, 5, 7):
        for c, t, y, x in ((0, 0, 0, 0), (2, 1, 15, 15), (1, 0, 7, 3), (1, 1, 7, 3)):
            px = img[16 * gy[r] + y, 16 * gx[r] + x, c]
            ref = O.round_bf16(np.array([(F32(px) / F32(255) - F32(mean[c])) / F32(std[c])], F32))[0]
            assert A[r, ((c * 2 + t) * 16 + y) * 16 + x] == ref
    assert np.array_equal(A.reshape(8, 3, 2, 256)[:, :, 0], A.reshape(8, 3, 2, 256)[:, :, 1])


def test_pos_interp_identity_constant_and_linear():
    rng = np.random.default_rng(61)
    table = rng.standard_normal((48, 48, 8)).astype(F32)
    assert np.array_equal(Q.pos_interp(table, 48, 48), table.reshape(-1, 8))
    assert np.all(Q.pos_interp(np.full((48, 48, 4), 0.75, F32), 13, 29) == F32(0.75))
    yv, xv = np.mgrid[0:48, 0:48]
    lin = (0.5 + 0.25 * yv - 0.125 * xv).astype(F32)[..., None]
    got = Q.pos_interp(lin, 10, 7).reshape(10, 7)
    ys, xs = np.arange(10) * 47 / 9, np.arange(7) * 47 / 6
    ref = 0.5 + 0.25 * ys[:, None] - 0.125 * xs[None, :]
    assert np.allclose(got, ref, atol=1e-5)
    one = Q.pos_interp(table, 1, 1)
    assert np.array_equal(one[0], table[0, 0])


def test_rope_pairs_angles_and_relative_position():
    theta = 10000.0
    for i, axis in ((0, 0), (5, 0), (17, 0), (36, 1), (44, 1), (53, 1)):
        v = np.zeros((1, 72), F32)
        v[0, i] = 1.0
        gy, gx = np.array([9]), np.array([4])
        out = Q.rope(v, gy, gx, theta)[0]
        j = i % 36
        pos = (9, 4)[axis]
        ang = pos * theta ** (-j / 18)
        assert out[i] == pytest.approx(math.cos(ang), abs=1e-6)
        assert out[i + 18] == pytest.approx(math.sin(ang), abs=1e-6)
        assert np.count_nonzero(out) == 2
    rng = np.random.default_rng(62)
    q, k = rng.standard_normal((2, 1, 72)).astype(F32)
    d = []
    for shift in (0, 3, 11):
        qr = Q.rope(q, np.array([2 + shift]), np.array([5 + shift]), theta)
        kr = Q.rope(k, np.array([7 + shift]), np.array([1 + shift]), theta)
        d.append(float((qr * kr).sum()))
    assert np.allclose(d, d[0], atol=1e-4)
    x = rng.standard_normal((3, 144)).astype(F32)
    r = Q.rope(x, np.arange(3), np.arange(3) * 2, theta)
    assert np.allclose(np.linalg.norm(r.reshape(6, 72), axis=1), np.linalg.norm(x.reshape(6, 72), axis=1), rtol=1e-5)


def test_attention_head72_against_float64():
    rng = np.random.default_rng(63)
    n, heads = 20, 2
    q, k, v = (O.round_bf16(rng.standard_normal((n, heads * 72)).astype(F32)) for _ in range(3))
    got = O.attention(q, k, v, heads, 72)
    ref = np.empty((n, heads * 72))
    for h in range(heads):
        sl = slice(72 * h, 72 * h + 72)
        s = q[:, sl].astype(np.float64) @ k[:, sl].astype(np.float64).T / math.sqrt(72)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ref[:, sl] = (p / p.sum(axis=1, keepdims=True)) @ v[:, sl]
    assert np.abs(got - ref).max() <= 1e-2 * (1 + np.abs(ref)).max()


def test_block_identity_with_zero_branches():
    W = WL.make_weights_qwen(1)
    L = dict(W["layers"][0])
    for f in ("proj_w", "proj_b", "fc2_w", "fc2_b"):
        L[f] = np.zeros_like(L[f])
    x = O.round_bf16(np.random.default_rng(64).standard_normal((16, 1152)).astype(F32))
    gy, gx = Q.patch_order(4, 4)
    assert np.array_equal(Q.block(x, L, Q.QWEN, gy, gx), x)


def _small_qwen_layer(seed, D=144, F=288):
    rng = np.random.default_rng(seed)
    n = lambda *sh: WL.to_bf16_bits(rng.standard_normal(sh).astype(F32) * 0.1)
    g = lambda: WL.to_bf16_bits(1 + rng.standard_normal(D).astype(F32) * 0.1)
    return dict(ln1_g=g(), ln1_b=n(D), qkv_w=n(3 * D, D), qkv_b=n(3 * D), proj_w=n(D, D), proj_b=n(D),
                ln2_g=g(), ln2_b=n(D), fc1_w=n(F, D), fc1_b=n(F), fc2_w=n(D, F), fc2_b=n(D))


def _bf16(a):
    """Round to bf16 through torch (an independent RNE routine), back to float64."""
    import torch
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _qwen_block_bruteforce(x, L, gy, gx, heads=2, hd=72, theta=10000.0, eps=1e-6):
    """The Qwen-style block in float64 loops, each step from its definition,
    with the stored activations rounded to bf16 where the oracle's header puts
    them: LN outputs, the QKV projection before the rotation, q and k after it,
    the attention output, the residual stream and the MLP hidden."""
    f = {k: O.bits_to_f32(v).astype(np.float64) for k, v in L.items()}
    n, D = x.shape

    def ln(a, g, b):
        out = np.zeros_like(a)
        for i in range(n):
            mu = sum(a[i]) / D
            var = sum((t - mu) ** 2 for t in a[i]) / D
            out[i] = [(a[i, j] - mu) / math.sqrt(var + eps) * g[j] + b[j] for j in range(D)]
        return out

    def lin(a, w, b):
        return np.array([[sum(a[i, t] * w[o, t] for t in range(a.shape[1])) + b[o]
                          for o in range(w.shape[0])] for i in range(a.shape[0])])

    fr = [theta ** (-j / 18) for j in range(18)]

    def rot(vec, i):
        out = vec.copy()
        for h in range(heads):
            for half, pos in ((0, gy[i]), (1, gx[i])):
                base = h * hd + half * 36
                for j in range(18):
                    c, s = math.cos(pos * fr[j]), math.sin(pos * fr[j])
                    a, b = vec[base + j], vec[base + j + 18]
                    out[base + j], out[base + j + 18] = a * c - b * s, b * c + a * s
        return out

    x = x.astype(np.float64)
    y = _bf16(ln(x, f["ln1_g"], f["ln1_b"]))
    t = _bf16(lin(y, f["qkv_w"], f["qkv_b"]))
    q = _bf16([rot(t[i, :D], i) for i in range(n)])
    k = _bf16([rot(t[i, D:2 * D], i) for i in range(n)])
    v = t[:, 2 * D:]
    o = np.zeros((n, D))
    for h in range(heads):
        sl = slice(h * hd, (h + 1) * hd)
        for i in range(n):
            sc = [sum(q[i, sl] * k[j, sl]) / math.sqrt(hd) for j in range(n)]
            m = max(sc)
            e = [math.exp(a - m) for a in sc]
            o[i, sl] = sum(e[j] * v[j, sl] for j in range(n)) / sum(e)
    o = _bf16(o)
    x = _bf16(x + lin(o, f["proj_w"], f["proj_b"]))
    y = _bf16(ln(x, f["ln2_g"], f["ln2_b"]))
    hdn = lin(y, f["fc1_w"], f["fc1_b"])
    g = _bf16([[0.5 * a * (1 + math.erf(a / math.sqrt(2))) for a in row] for row in hdn])
    return _bf16(x + lin(g, f["fc2_w"], f["fc2_b"]))


def test_block_against_float64_bruteforce():
    """Q.block at hidden 144 (2 heads of 72) on a 2 x 4 grid in merge-group
    order, against the float64 brute force; a transposed projection, a wrong
    head split (4 heads of 36) and swapped RoPE axes are each far off."""
    cfg = dict(Q.QWEN, hidden=144, heads=2, mlp=288)
    L = _small_qwen_layer(67)
    x = O.round_bf16(np.random.default_rng(68).standard_normal((8, 144)).astype(F32))
    gy, gx = Q.patch_order(2, 4)
    ref = _qwen_block_bruteforce(x, L, gy, gx)
    err = lambda got: (np.abs(got - ref) / (1 + np.abs(ref))).max()
    assert err(Q.block(x, L, cfg, gy, gx)) < 2 ** -7           # allows a rare one-ulp rounding flip
    assert err(Q.block(x, dict(L, proj_w=np.ascontiguousarray(L["proj_w"].T)), cfg, gy, gx)) > 0.05
    assert err(Q.block(x, L, dict(cfg, heads=4, head_dim=36), gy, gx)) > 0.05
    assert err(Q.block(x, L, cfg, gx, gy)) > 0.05


def test_merger_concatenates_each_group_in_order():
    """One-hot w1 rows pick column r*1152 + c of the group concatenation: the
    c-th channel of the group's r-th patch (after the merger LayerNorm)."""
    rng = np.random.default_rng(65)
    x = O.round_bf16(rng.standard_normal((8, 1152)).astype(F32))
    M = dict(ln_g=np.ones(1152, F32), ln_b=np.zeros(1152, F32), w1=np.zeros((4608, 4608), F32),
             b1=np.zeros(4608, F32), w2=np.zeros((5120, 4608), F32), b2=np.zeros(5120, F32))
    picks = [(0, 5), (1, 0), (2, 1151), (3, 700)]
    for n, (r, c) in enumerate(picks):
        M["w1"][n, r * 1152 + c] = 1.0
        M["w2"][n, n] = 1.0
    e = Q.merger(x, M, Q.QWEN)
    z = O.round_bf16(O.layer_norm(x, M["ln_g"], M["ln_b"], 1e-6))
    for g in range(2):
        for n, (r, c) in enumerate(picks):
            assert e[g, n] == O.round_bf16(O.gelu(z[4 * g + r, c:c + 1]))[0]


def test_layout_three_axis_positions_and_rope_delta():
    pos, delta = Q.layout(2, 3, 5)
    assert pos[:, 0].tolist() == [5, 5, 5]                       # vision_start: equal axes
    assert pos[0, 1:-1].tolist() == [6] * 6                      # still image: one temporal index
    assert pos[1, 1:-1].tolist() == [6, 6, 6, 7, 7, 7]           # rows
    assert pos[2, 1:-1].tolist() == [6, 7, 8, 6, 7, 8]           # columns
    assert pos[:, -1].tolist() == [9, 9, 9]                      # vision_end after max(h, w)
    assert delta == 10 - (5 + 8)                                 # next text position = index + delta
    pos, delta = Q.layout(32, 32, 0)
    assert pos.shape == (3, 1026) and pos[:, -1].tolist() == [33] * 3 and delta == 34 - 1026


def test_small_encode_runs_and_taps():
    W = WL.make_weights_qwen(9)
    img = WL.uniform_image(64, 32, seed=66)
    cfg = dict(Q.QWEN, mean=WL.MODEL["mean"], std=WL.MODEL["std"])
    e, deep = Q.encode(img, W, cfg)
    assert e.shape == (2, 5120) and len(deep) == 1 and deep[0].shape == (2, 5120)
    assert np.all(np.isfinite(e))
