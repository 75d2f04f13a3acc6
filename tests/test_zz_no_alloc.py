"""ds_vit_encode_noalloc: the encode for callers that cannot allocate device
memory when they encode (their application owns the whole device budget, or
they must not pay cudaMalloc's synchronisation, or their interface passes only
inputs and outputs).  Its scratch is a fixed array inside the library.

Checked through the C ABI against ds_vit_encode (the entry point with a
caller workspace) on two calls in a row with different image sizes, so the
second call runs on scratch that still holds the first call's data; and the
size limit.  Collected last on purpose (file name)."""
import ctypes as C

import numpy as np
import pytest

import workloads as WL
from gpu_util import assert_parity, host

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


@pytest.fixture(scope="module")
def enc(dv):
    e = dv.Encoder(dv.weights_to_device(WL.make_weights(2)), WL.MODEL)
    yield e
    e.close()


def _p(t):
    return C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _with_workspace(dv, enc, img):
    H, W = img.shape[:2]
    out = torch.empty((enc.tokens([(H, W)]), 5120), dtype=torch.bfloat16, device="cuda")
    ws = enc.workspace([(H, W)])
    dv.check(dv.lib.ds_vit_encode(enc.handle, _p(img), H, W, _p(out), _p(ws), ws.numel(), _stream()),
             "ds_vit_encode")
    return out


def _no_alloc(dv, enc, img):
    H, W = img.shape[:2]
    out = torch.full((enc.tokens([(H, W)]), 5120), float("nan"), dtype=torch.bfloat16, device="cuda")
    dv.check(dv.lib.ds_vit_encode_noalloc(enc.handle, _p(img), H, W, _p(out), _stream()),
             "ds_vit_encode_noalloc")
    return out


def test_no_alloc_matches_workspace_entry_point_twice(dv, enc):
    imgs = [torch.from_numpy(WL.uniform_image(h, w, seed=500 + i)).cuda()
            for i, (h, w) in enumerate([(448, 448), (350, 294)])]   # 1024 and 525 patches
    refs = [_with_workspace(dv, enc, im) for im in imgs]
    torch.cuda.synchronize()
    for im, ref in zip(imgs, refs):                                # two calls in a row
        got = _no_alloc(dv, enc, im)
        torch.cuda.synchronize()
        assert enc.status() == dv.OK
        assert_parity(host(got), host(ref), what="no-alloc encode")
        assert torch.equal(got, ref)                               # same kernels, same inputs


def test_no_alloc_rejects_images_over_the_limit(dv, enc):
    img = torch.from_numpy(WL.uniform_image(462, 462, seed=7)).cuda()      # 33 x 33 = 1089 patches
    out = torch.full((121, 5120), 3.0, dtype=torch.bfloat16, device="cuda")
    rc = dv.lib.ds_vit_encode_noalloc(enc.handle, _p(img), 462, 462, _p(out), _stream())
    assert rc == dv.ERANGE
    assert dv.lib.ds_vit_encode_noalloc(enc.handle, _p(img), 463, 462, _p(out), _stream()) == dv.EINVAL
    # A misaligned output is reported as such even for an image over the limit:
    # the alignment checks come before the patch limit.
    odd = C.c_void_p(out.data_ptr() + 2)
    assert dv.lib.ds_vit_encode_noalloc(enc.handle, _p(img), 462, 462, odd, _stream()) == dv.EINVAL
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
