"""Preprocessing on the GPU through the C ABI (ds_vit_preprocess): the canvas
must equal the oracle's byte for byte (integer work), on downscales,
enlargements, one-axis resizes, identity plans, noise that drives the bicubic
overshoot into the clamp, and extreme aspect ratios."""
import numpy as np
import pytest

import oracle.preprocess as PP
import workloads as WL

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


CASES = [
    ((1000, 333), "uniform", 1),     # tall: fills the canvas height, width by round
    ((333, 1000), "gradient", 2),    # wide
    ((100, 100), "uniform", 3),      # under the pixel budget: enlarged to 546
    ((544, 544), "gradient", 4),     # exactly the budget: 544 -> 546
    ((546, 546), "uniform", 5),      # its own canvas: copy
    ((600, 800), "uniform", 7),      # chart: up by 1.05
    ((1, 1), "uniform", 8),          # one pixel -> 546 x 546
    ((3, 700), "uniform", 9),        # one axis far below the other
    ((1344, 1000), "gradient", 10),  # height kept (1344 = 32 units), width resized
    ((20000, 100), "gradient", 11),  # 200:1, no aspect clamp
    ((4500, 6000), "uniform", 12),   # downscale by 4: 17-tap filters (generic horizontal pass)
    ((2640, 112), "gradient", 13),   # width kept, height resized from the input's 336-byte rows
    ((2136, 140), "uniform", 14),    # width kept, 420-byte rows (not 16-byte multiples)
    ((1200, 5000), "gradient", 15),  # wide downscale: 21 column blocks with a ragged last one
]


@pytest.mark.parametrize("hw,kind,seed", CASES)
def test_preprocess_matches_oracle_bytes(dv, hw, kind, seed):
    img = WL.make_image(hw[0], hw[1], kind, seed)
    canvas, plan = dv.preprocess(torch.from_numpy(img).cuda())
    torch.cuda.synchronize()
    ref = PP.preprocess(img)
    assert plan["Hc"] == ref.shape[0] and plan["Wc"] == ref.shape[1]
    got = canvas.cpu().numpy()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


@pytest.mark.parametrize("hw", [(2640, 112), (1000, 333)])
def test_preprocess_unaligned_source(dv, hw):
    """An image that starts one byte into its allocation (a view): the passes
    that read 16-byte words of the source must not be taken."""
    img = WL.make_image(hw[0], hw[1], "uniform", 16)
    flat = torch.empty(img.size + 1, dtype=torch.uint8, device="cuda")
    view = flat[1:].view(hw[0], hw[1], 3)
    view.copy_(torch.from_numpy(img).cuda())
    canvas, _ = dv.preprocess(view)
    torch.cuda.synchronize()
    assert np.array_equal(canvas.cpu().numpy(), PP.preprocess(img))


def test_preprocess_photo_full_size(dv):
    """The 3024 x 4032 photo workload, downscaled by 2.67 on both axes."""
    H, W, kind, seed = WL.PREPROCESS_WORKLOADS["photo"]
    img = WL.make_image(H, W, kind, seed)
    canvas, plan = dv.preprocess(torch.from_numpy(img).cuda())
    torch.cuda.synchronize()
    assert (plan["h"], plan["w"]) == (27, 36)
    assert np.array_equal(canvas.cpu().numpy(), PP.preprocess(img))


def test_preprocessed_canvas_encodes(dv):
    """The canvas is a valid encode input: its token count is the plan's."""
    W2 = WL.make_weights(2)
    enc = dv.Encoder(dv.weights_to_device(W2), WL.MODEL)
    try:
        img = WL.make_image(600, 800, "uniform", 7)
        canvas, plan = dv.preprocess(torch.from_numpy(img).cuda())
        out, offs = enc.encode([canvas])
        torch.cuda.synchronize()
        assert out.shape[0] == plan["h"] * plan["w"] == int(offs[-1])
        assert bool(torch.isfinite(out.float()).all())
    finally:
        enc.close()
