"""The released tower's block variant on the GPU (page A's comparison table:
RMSNorm and SwiGLU; Step 3: the half-vector RoPE pairing on [h*f, w*f];
Step 1 item 6: pixels to [-1, 1]) against the oracle computing that variant
directly: the RMSNorm and SwiGLU kernels alone, then whole encodes with every
step teacher-forced and the free-running output within the oracle's own
summation-order spread; and the benchmarked 1344x1344 image at 32 layers
with sampled rows of every block teacher-forced."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import (assert_end_to_end, assert_steps_teacher_forced, dev, host, rand_bits, rel_err, sample_rows,
                      sample_tokens)

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


def test_rmsnorm(dv):
    for M in (1, 7, 300, 9216):
        x = rand_bits((M, 1024), 51, 3.0)
        g = WL.to_bf16_bits(1 + np.random.default_rng(52).standard_normal(1024).astype(np.float32) * 0.1)
        y = dv.op_rmsnorm(dev(x, torch), dev(g, torch), 1e-6)
        ref = O.round_bf16(O.rms_norm(O.bits_to_f32(x), O.bits_to_f32(g), 1e-6))
        got = host(y)
        assert rel_err(got, ref).max() <= 8e-3, M
        assert (got == ref).mean() > 0.99


@pytest.mark.parametrize("M,K,F", [(1, 64, 128), (300, 1024, 512), (1000, 1024, 4096), (2000, 256, 1024),
                                   (2000, 2048, 1024)])
def test_linear_swiglu(dv, M, K, F):
    a = rand_bits((M, K), 53 + M)
    w = rand_bits((2 * F, K), 54 + K, 1.0 / math.sqrt(K))
    b = rand_bits(2 * F, 55, 0.5)
    cfg = dict(WL.MODEL, mlp=F, mlp_kind="swiglu")
    ref = O.mlp_hidden(O.bits_to_f32(a), {"fc1_w": w, "fc1_b": b}, cfg)
    y, st = dv.op_linear(dev(a, torch), dev(w, torch), dev(b, torch), dv.EPI_SWIGLU)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and tuple(y.shape) == (M, F)
    got = host(y)
    e = rel_err(got, ref)
    assert e.max() <= 1e-2, f"max {e.max()}"
    assert (got == ref).mean() > 0.98


@pytest.fixture(scope="module")
def w2():
    return WL.make_weights_official(2)


@pytest.fixture(scope="module")
def enc2(dv, w2):
    e = dv.Encoder(dv.weights_to_device(w2), WL.MODEL_OFFICIAL)
    yield e
    e.close()


def _run(dv, enc, imgs):
    d = [torch.from_numpy(im).cuda() for im in imgs]
    r = enc.encode(d, dump=True)
    torch.cuda.synchronize()
    assert enc.status() == dv.OK
    return r


@pytest.mark.parametrize("sizes", [[(84, 84)], [(546, 546)], [(350, 294), (14, 28), (126, 1260)]])
def test_official_encode(dv, enc2, w2, sizes):
    imgs = [WL.uniform_image(h, w, seed=200 + i) for i, (h, w) in enumerate(sizes)]
    out, offs, blocks, fnorm = _run(dv, enc2, imgs)
    assert_steps_teacher_forced(imgs, w2, WL.MODEL_OFFICIAL, blocks, fnorm, out, layers=(0, 1))
    ref_offs, _ = assert_end_to_end(host(out), imgs, w2, WL.MODEL_OFFICIAL, what=f"official {sizes}")
    assert np.array_equal(offs, ref_offs)


def test_official_differs_from_default(dv, enc2, w2):
    """The variant switches really change the computation (not a silent default)."""
    img = WL.uniform_image(84, 84, seed=7)
    out, *_ = _run(dv, enc2, [img])
    ref_default, _ = O.encode([img], w2 | {"layers": [dict(L, fc1_w=L["fc1_w"][:4096], fc1_b=L["fc1_b"][:4096])
                                                      for L in w2["layers"]]}, WL.MODEL)
    assert np.abs(host(out) - ref_default).max() > 0.05


def test_official_full_size_every_block(dv):
    """The benchmarked configuration: 1344x1344 (9216 patches), 32 layers of
    the variant.  Sampled query rows of every block (each image's first and
    last row, its last query tile's first row and 96 random rows) and sampled
    merged tokens, each recomputed from the GPU's own inputs."""
    w = WL.make_weights_official(32)
    e = dv.Encoder(dv.weights_to_device(w), WL.MODEL_OFFICIAL)
    try:
        img = WL.workload_images("max")[0]
        out, offs, blocks, fnorm = _run(dv, e, [img])
    finally:
        e.close()
    assert offs[-1] == 1024
    assert_steps_teacher_forced([img], w, WL.MODEL_OFFICIAL, blocks, fnorm, out, layers=range(32),
                                rows=sample_rows([9216], 96, seed=13), toks=sample_tokens(offs, 8, seed=14))
