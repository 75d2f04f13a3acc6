"""The Qwen3-VL-style tower on the GPU (ds_vit_qwen_encode) against the
oracle (oracle/qwen.py): every step recomputed from the GPU's own input to it
(patch embedding with the interpolated position table, each block, the
primary merger, the DeepStack merger of block 8) within the encode's step
bound, and the free-running outputs within the oracle's own summation-order
spread.  Grids: 2x2 merged (one partial query tile), 7x7 (ragged tiles),
16x12; 9 blocks so that the first DeepStack tap is reached; and the
benchmarked 1024x1024 image with all 27 blocks, every step teacher-forced."""
import math

import numpy as np
import pytest

import oracle as O
import oracle.qwen as Q
import workloads as WL
from gpu_util import (SPREAD_MODES, assert_parity, assert_within_spread, bits_of, dev, host, rand_bits,
                      rel_err, spread_of)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N_LAYERS = 9


@pytest.fixture(scope="module")
def dv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import vit_vision_encoder_gb300
    return vit_vision_encoder_gb300


@pytest.fixture(scope="module")
def wq():
    return WL.make_weights_qwen(N_LAYERS)


@pytest.fixture(scope="module")
def encq(dv, wq):
    e = dv.QwenEncoder(dv.weights_to_device(wq), WL.QWEN_MODEL, n_layers=N_LAYERS)
    yield e
    e.close()


def test_linear_width_1152(dv):
    M, K, N = 777, 1152, 1152
    a = rand_bits((M, K), 71)
    w = rand_bits((N, K), 72, 1.0 / math.sqrt(K))
    b = rand_bits(N, 73, 0.5)
    x = rand_bits((M, N), 74)
    ref = O.round_bf16(O.bits_to_f32(x) + (O.bits_to_f32(a) @ O.bits_to_f32(w).T + O.bits_to_f32(b)))
    out = dev(x, torch)
    y, st = dv.op_linear(dev(a, torch), dev(w, torch), dev(b, torch), dv.EPI_BIAS_RESID, out=out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    e = rel_err(host(y), ref)
    assert e.max() <= 1e-2


@pytest.mark.parametrize("H,W", [(64, 64), (224, 224), (512, 384)])
def test_qwen_encode(dv, encq, wq, H, W):
    cfg = WL.QWEN_MODEL
    img = WL.uniform_image(H, W, seed=300 + H)
    out, deep, blocks = encq.encode(torch.from_numpy(img).cuda(), dump=True)
    torch.cuda.synchronize()
    bl = blocks.cpu()
    gh, gw = H // 16, W // 16
    gy, gx = Q.patch_order(gh, gw)
    # patch embedding: r(r(pos) + A W^T + b)
    A = Q.patchify(img, cfg["mean"], cfg["std"])
    pos = Q.pos_interp(wq["pos_table"], gh, gw).reshape(gh, gw, -1)[gy, gx]
    x0 = O.round_bf16(O.round_bf16(pos) + (O.mm(A, O.bits_to_f32(wq["patch_w"]).T) + O.bits_to_f32(wq["patch_b"])))
    assert_parity(bits_of(bl[0]), x0, what="patch embedding")
    for l in range(N_LAYERS):
        ref = Q.block(bits_of(bl[l]), wq["layers"][l], cfg, gy, gx)
        assert_parity(bits_of(bl[l + 1]), ref, what=f"block {l}")
    assert_parity(host(out), Q.merger(bits_of(bl[N_LAYERS]), wq["merger"], cfg), what="merger")
    assert_parity(host(deep[0]), Q.merger(bits_of(bl[8]), wq["deepstack"][0], cfg), what="deepstack 8")
    # free-running outputs against the oracle, within the spread of its valid evaluations
    outs = []
    for mode in SPREAD_MODES:
        with O.evaluation(*mode):
            prim, deep_ref = Q.encode(img, wq, cfg, n_layers=N_LAYERS)
        outs.append((prim, deep_ref[0]))
    assert_within_spread(host(out), outs[0][0], spread_of([o[0] for o in outs]), what="primary")
    assert_within_spread(host(deep[0]), outs[0][1], spread_of([o[1] for o in outs]), what="deepstack 8")


def test_qwen_rejects_bad_sizes(dv, encq):
    img = torch.zeros((48, 64, 3), dtype=torch.uint8, device="cuda")
    with pytest.raises(dv.DsVitError):
        encq.encode(img)


def test_qwen_full_grid_block_repeatable(dv, wq):
    """1024x1024 (4096 patches: 16 query blocks of 256 rows per head, 32 K/V
    tiles): block 0 teacher-forced against the oracle, and three encodes
    bit-identical.  The attention writes P over the scores it has read and
    issues the next scores after the PV MMA; an ordering fault there would
    show as run-to-run differences."""
    cfg = WL.QWEN_MODEL
    e = dv.QwenEncoder(dv.weights_to_device(wq), cfg, n_layers=1)
    try:
        img = WL.uniform_image(1024, 1024, seed=1024)
        dimg = torch.from_numpy(img).cuda()
        runs = []
        for _ in range(3):
            out, _, blocks = e.encode(dimg, deepstack=False, dump=True)
            torch.cuda.synchronize()
            runs.append((out.clone(), blocks.clone()))
        for out, blocks in runs[1:]:
            assert torch.equal(out, runs[0][0]) and torch.equal(blocks, runs[0][1])
        bl = runs[0][1].cpu()
        gy, gx = Q.patch_order(64, 64)
        ref = Q.block(bits_of(bl[0]), wq["layers"][0], cfg, gy, gx)
        assert_parity(bits_of(bl[1]), ref, what="block 0 at 4096 patches")
    finally:
        e.close()


def test_qwen_full_size_every_block(dv):
    """The benchmarked configuration: 1024x1024 (4096 patches), all 27 blocks
    of the tower.  Every block teacher-forced on every row, the primary merger
    and the three DeepStack mergers (taps after blocks 8, 16 and 24) from the
    GPU's own inputs."""
    cfg = WL.QWEN_MODEL
    n = cfg["n_layers"]
    w = WL.make_weights_qwen(n)
    e = dv.QwenEncoder(dv.weights_to_device(w), cfg)
    try:
        img = WL.uniform_image(1024, 1024, seed=2048)
        out, deep, blocks = e.encode(torch.from_numpy(img).cuda(), dump=True)
        torch.cuda.synchronize()
        bl = blocks.cpu()
    finally:
        e.close()
    gy, gx = Q.patch_order(64, 64)
    for l in range(n):
        ref = Q.block(bits_of(bl[l]), w["layers"][l], cfg, gy, gx)
        assert_parity(bits_of(bl[l + 1]), ref, what=f"block {l} at 4096 patches")
    assert_parity(host(out), Q.merger(bits_of(bl[n]), w["merger"], cfg), what="merger at 4096 patches")
    for k, tap in enumerate(cfg["taps"]):
        assert_parity(host(deep[k]), Q.merger(bits_of(bl[tap]), w["deepstack"][k], cfg),
                      what=f"deepstack {tap} at 4096 patches")


def test_qwen_peaked_attention(dv, wq):
    """q and k projection rows scaled x8 (logits of standard deviation ~10 in
    log2 units): the running maximum rises by more than 8 inside a row, so the
    head-72 kernel rescales O and the row sum mid-row.  512x512 image (1024
    patches, 8 K/V tiles per row); block 0 teacher-forced."""
    cfg = WL.QWEN_MODEL
    L0 = dict(wq["layers"][0])
    w = O.bits_to_f32(L0["qkv_w"]).copy()
    w[:2 * 1152] *= 8.0
    L0["qkv_w"] = WL.to_bf16_bits(w)
    wp = dict(wq)
    wp["layers"] = [L0]
    e = dv.QwenEncoder(dv.weights_to_device(wp), cfg, n_layers=1)
    try:
        img = WL.uniform_image(512, 512, seed=512)
        _, _, blocks = e.encode(torch.from_numpy(img).cuda(), deepstack=False, dump=True)
        torch.cuda.synchronize()
        bl = blocks.cpu()
        gy, gx = Q.patch_order(32, 32)
        ref = Q.block(bits_of(bl[0]), L0, cfg, gy, gx)
        assert_parity(bits_of(bl[1]), ref, what="peaked block 0")
    finally:
        e.close()


@pytest.mark.parametrize("H,W", [(32, 32), (96, 1024), (736, 416)])
def test_qwen_irregular_grids(dv, wq, H, W):
    """Grids of 2x2 (one merge group), 6x64 and 46x26 patches (ragged query
    and key tiles, N = 4, 384, 1196): the patch embedding and two blocks
    teacher-forced, and the merger of the second block's output."""
    cfg = WL.QWEN_MODEL
    e = dv.QwenEncoder(dv.weights_to_device(wq), cfg, n_layers=2)
    try:
        img = WL.uniform_image(H, W, seed=700 + H)
        out, _, blocks = e.encode(torch.from_numpy(img).cuda(), deepstack=False, dump=True)
        torch.cuda.synchronize()
        bl = blocks.cpu()
        gh, gw = H // 16, W // 16
        gy, gx = Q.patch_order(gh, gw)
        A = Q.patchify(img, cfg["mean"], cfg["std"])
        pos = Q.pos_interp(wq["pos_table"], gh, gw).reshape(gh, gw, -1)[gy, gx]
        x0 = O.round_bf16(O.round_bf16(pos) + (O.mm(A, O.bits_to_f32(wq["patch_w"]).T) +
                                              O.bits_to_f32(wq["patch_b"])))
        assert_parity(bits_of(bl[0]), x0, what="patch embedding")
        for l in range(2):
            ref = Q.block(bits_of(bl[l]), wq["layers"][l], cfg, gy, gx)
            assert_parity(bits_of(bl[l + 1]), ref, what=f"block {l}")
        assert_parity(host(out), Q.merger(bits_of(bl[2]), wq["merger"], cfg), what="merger")
    finally:
        e.close()
