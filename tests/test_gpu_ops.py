"""Single-kernel parity on the GPU through the C ABI: LayerNorm, the tcgen05
GEMM with each fused epilogue, the RoPE table and varlen attention, each
against the CPU oracle on the same seeded inputs (several tiles plus ragged
tails)."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import assert_parity, dev, host, rand_bits, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import vit_vision_encoder_gb300
    return vit_vision_encoder_gb300


def test_layernorm(dv):
    for M in (1, 7, 300, 9216):
        x = rand_bits((M, 1024), 1, 3.0)
        g = WL.to_bf16_bits(1 + np.random.default_rng(2).standard_normal(1024).astype(np.float32) * 0.1)
        b = rand_bits(1024, 3, 0.1)
        y = dv.op_layernorm(dev(x, torch), dev(g, torch), dev(b, torch), 1e-6)
        ref = O.round_bf16(O.layer_norm(O.bits_to_f32(x), O.bits_to_f32(g), O.bits_to_f32(b), 1e-6))
        got = host(y)
        assert rel_err(got, ref).max() <= 8e-3, M
        assert (got == ref).mean() > 0.99


def test_rope_table(dv):
    t = dv.op_rope_table(192, 10000.0).cpu().numpy()
    pos = np.arange(192)
    ang = O.rope_angles(pos, pos, 10000.0)[:, :16]
    for got, ref in ((t[:, :16], np.cos(ang).astype(np.float32)),
                     (t[:, 16:], np.sin(ang).astype(np.float32))):
        ulps = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
        assert ulps.max() <= 1 and (ulps == 0).mean() > 0.999


GEMM_CASES = [
    (1, 64, 256, "bias"), (77, 640, 1024, "bias"), (300, 1024, 1024, "bias"),
    (1000, 1024, 4096, "gelu"), (513, 4096, 1024, "resid"), (169, 9216, 5120, "gelu"),
    (2000, 1024, 1024, "resid"),
    # N = 1152 (the Qwen-style tower's hidden width, a multiple of 288 but not
    # of 256): 288-wide tiles where they fit one round (two MMAs per K step, a
    # 256-row and a 32-row B box; odd chunk count in the epilogue), ragged M in
    # the second case, the tower's FC2 shape (K = 4608); 128-wide tiles where
    # they do not (5000 rows: 160 tiles of 288) and for other widths.
    (4096, 1152, 1152, "resid"), (3000, 1152, 1152, "bias"), (1700, 1152, 1152, "gelu"),
    (4096, 4608, 1152, "resid"), (5000, 1152, 1152, "resid"), (2500, 640, 1408, "gelu"),
    # K >= 2048 with enough 256 x 256 tiles: the 2-CTA-cluster kernel.  FC2-like
    # K = 4096; M = 4200, whose last tile's second 128-row half lies wholly past
    # M; the second merger linear's K = N = 5120.
    (3840, 4096, 1024, "resid"), (4200, 2048, 1024, "gelu"), (4200, 4096, 1024, "resid"),
    # The out-projection shape with a ragged last tile: residual rows by TMA,
    # 4 valid rows in the last tile's first half, none in its second.
    (4100, 1024, 1024, "resid"), (9216, 1024, 1024, "resid"),
    # The merger linears' width at about a thousand rows: 320-wide tiles in one
    # round (two MMAs per K step, a 256-row and a 64-row B box); ragged M.
    (1024, 5120, 5120, "bias"), (1100, 2048, 5120, "gelu"), (1000, 1024, 5120, "bias"),
]


@pytest.mark.parametrize("M,K,N,epi", GEMM_CASES)
def test_linear_epilogues(dv, M, K, N, epi):
    a = rand_bits((M, K), 10 + M)
    w = rand_bits((N, K), 11 + K, 1.0 / math.sqrt(K))
    b = rand_bits(N, 12, 0.5)
    af, wf, bf = O.bits_to_f32(a), O.bits_to_f32(w), O.bits_to_f32(b)
    t = af @ wf.T + bf
    code = {"bias": dv.EPI_BIAS, "gelu": dv.EPI_BIAS_GELU, "resid": dv.EPI_BIAS_RESID}[epi]
    out = None
    if epi == "resid":
        x = rand_bits((M, N), 13)
        out = dev(x, torch)
        ref = O.round_bf16(O.bits_to_f32(x) + t)
    elif epi == "gelu":
        ref = O.round_bf16(O.gelu(t))
    else:
        ref = O.round_bf16(t)
    y, st = dv.op_linear(dev(a, torch), dev(w, torch), dev(b, torch), code, out=out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = host(y)
    e = rel_err(got, ref)
    assert e.max() <= 1e-2, f"max {e.max()}"
    assert (got == ref).mean() > 0.98


def test_gelu_epilogue_every_bf16_input(dv):
    """Every bf16 value in [-10, 10] passes through the GELU epilogue unchanged
    by the product (one-hot A column times unit weights), so the output is
    bf16(GELU(x)) of the kernel's erf evaluation: it must equal the oracle's
    float64 erf rounded to bf16, up to one ulp where the exact value lies
    within the approximation error of a rounding boundary.  Below x = -8.3
    the oracle's 1 + erf cancels to 0 in float64 while the kernel keeps the
    tail (about 1e-16): those compare by absolute difference."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bits_to_f32(bits)
    keep = np.isfinite(vals) & (np.abs(vals) <= 10.0)
    bits, vals = bits[keep], vals[keep]
    M = len(bits)
    a = np.zeros((M, 64), dtype=np.uint16)
    a[:, 0] = bits
    w = np.zeros((256, 64), dtype=np.uint16)
    w[:, 0] = WL.to_bf16_bits(np.ones(256, dtype=np.float32))
    b = np.zeros(256, dtype=np.uint16)
    y, st = dv.op_linear(dev(a, torch), dev(w, torch), dev(b, torch), dv.EPI_BIAS_GELU)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = O.f32_to_bits(host(y)).astype(np.int32)
    ref = O.f32_to_bits(O.round_bf16(O.gelu(vals))).astype(np.int32)
    ulps = np.abs(got - ref[:, None])
    tiny = np.abs(host(y) - O.round_bf16(O.gelu(vals))[:, None]) <= 1e-6
    assert ulps[~tiny].max() <= 1, f"max {ulps[~tiny].max()} ulp"
    assert (ulps == 0).mean() > 0.995


@pytest.mark.parametrize("gh,gw", [(6, 6), (25, 21), (192, 2), (64, 80)])
def test_linear_qkv_rope(dv, gh, gw):
    M = gh * gw
    cfg = WL.MODEL
    y = rand_bits((M, 1024), 20)
    L = {"qkv_w": rand_bits((3072, 1024), 21, 1 / 32), "qkv_b": rand_bits(3072, 22, 0.5)}
    gy, gx = O.grid_positions(gh, gw)
    q, k, v = O.qkv_project(O.bits_to_f32(y), L, cfg, gy, gx)
    ref = np.concatenate([q, k, v], axis=1)
    rowpos = torch.from_numpy((gy.astype(np.int32) << 16) | gx.astype(np.int32)).cuda()
    cs = dv.op_rope_table(max(gh, gw), cfg["rope_theta"])
    out, st = dv.op_linear(dev(y, torch), dev(L["qkv_w"], torch), dev(L["qkv_b"], torch),
                           dv.EPI_QKV_ROPE, rowpos=rowpos, rope_cs=cs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = host(out)
    e = rel_err(got, ref)
    assert e.max() <= 1e-2, f"max {e.max()}"


@pytest.mark.parametrize("seqlens,scale", [([36], 1.0), ([525], 1.0), ([128, 300, 1, 257], 1.0),
                                           ([700], 3.0), ([1521], 1.0)])
def test_attention_varlen(dv, seqlens, scale):
    tot = sum(seqlens)
    rng = np.random.default_rng(30 + tot)
    qkv = WL.to_bf16_bits(np.concatenate([
        rng.standard_normal((tot, 2048)).astype(np.float32) * scale,
        rng.standard_normal((tot, 1024)).astype(np.float32)], axis=1))
    out, st = dv.op_attention(dev(qkv, torch), seqlens)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = host(out)
    f = O.bits_to_f32(qkv)
    ref = np.empty((tot, 1024), np.float32)
    s0 = 0
    for n in seqlens:
        ref[s0:s0 + n] = O.attention(f[s0:s0 + n, :1024], f[s0:s0 + n, 1024:2048],
                                     f[s0:s0 + n, 2048:], heads=16)
        s0 += n
    assert_parity(got, ref, what=f"attention {seqlens}")
    assert rel_err(got, ref).mean() < 2e-3
