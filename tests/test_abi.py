"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, validates arguments before touching CUDA, and its host-only layout
matches the oracle exactly."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as WL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dv():
    import __graft_entry__
    __graft_entry__.build()
    import vit_vision_encoder_gb300
    return vit_vision_encoder_gb300


def _declared():
    src = open(os.path.join(ROOT, "include", "dsvit.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_vit_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(dv):
    names = _declared()
    assert len(names) >= 15
    h = C.CDLL(dv.LIB_PATH)
    for n in names:
        assert hasattr(h, n), n
    assert set(names) == set(dv.SIGNATURES)


def test_graph_calls_reject_null_handles(dv):
    """The graph entry points check their handles before any CUDA call."""
    g = C.c_void_p(123)
    assert dv.lib.ds_vit_graph_create(None, 0, 0, None, None, None, None, None, None, 0, C.byref(g)) == dv.EINVAL
    assert g.value == 123                     # untouched: rejected before anything is written
    assert dv.lib.ds_vit_graph_create(C.c_void_p(1), 0, 0, None, None, None, None, None, None, 0, None) == dv.EINVAL
    assert dv.lib.ds_vit_graph_launch(None, None) == dv.EINVAL
    assert dv.lib.ds_vit_graph_destroy(None) == dv.EINVAL


def test_strerror(dv):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert dv.lib.ds_vit_strerror(code)
    assert dv.lib.ds_vit_strerror(-99) == b"unknown error"


@pytest.mark.parametrize("H,W", [(84, 84), (546, 546), (1344, 1344), (2688, 336), (1344, 672),
                                 (672, 1344), (1008, 1008), (840, 420), (14, 14), (14, 9 * 14 * 14),
                                 (70, 28)])
def test_layout_matches_oracle(dv, H, W):
    gh, gw = H // 14, W // 14
    got = dv.layout(gh, gw, 129264, base_pos=1000)
    ref = O.layout(gh, gw, 129264, base_pos=1000)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_layout_capacity_and_args(dv):
    n = C.c_int64(0)
    ids = np.zeros(3, np.int32)
    assert dv.lib.ds_vit_layout(6, 6, 1, 0, ids.ctypes.data, None, None, None, 3, C.byref(n)) == dv.ECAP
    assert n.value == 8 and np.all(ids == 0)          # nothing written on error
    assert dv.lib.ds_vit_layout(0, 6, 1, 0, None, None, None, None, 0, C.byref(n)) == dv.EINVAL
    assert dv.lib.ds_vit_layout(6, 6, 1, 2 ** 31 - 5, None, None, None, None, 100, C.byref(n)) == dv.ERANGE


def test_null_arguments_rejected_before_cuda(dv):
    L = dv.lib
    assert L.ds_vit_prepare(None, None, None, None) == dv.EINVAL
    h = C.c_void_p()
    cfg = dv.make_config(WL.MODEL, 2)
    assert L.ds_vit_prepare(C.byref(cfg), None, C.byref(h), None) == dv.EINVAL
    bad = dv.make_config(dict(WL.MODEL, hidden=768), 2)
    w = dv.Weights()
    assert L.ds_vit_prepare(C.byref(bad), C.byref(w), C.byref(h), None) == dv.EINVAL
    assert L.ds_vit_overlay(None, 10, 5120, None, 1, None, 1, None, None) == dv.EINVAL
    sp = (dv.Span * 2)()
    sp[0].base_row, sp[0].gh, sp[0].gw, sp[0].embed_row = 10, 6, 6, 0
    sp[1].base_row, sp[1].gh, sp[1].gw, sp[1].embed_row = 12, 6, 6, 4        # overlaps span 0
    ok = C.c_void_p(256)
    assert L.ds_vit_overlay_chunk(None, 0, 4, 5120, sp, 1, ok, 4, ok, None, None) == dv.EINVAL
    assert L.ds_vit_overlay_chunk(ok, -1, 4, 5120, sp, 1, ok, 4, ok, None, None) == dv.EINVAL
    assert L.ds_vit_overlay_chunk(ok, 0, 0, 5120, sp, 1, ok, 4, ok, None, None) == dv.EINVAL
    assert L.ds_vit_overlay_chunk(ok, 0, 4, 5120, sp, 2, ok, 8, ok, None, None) == dv.EINVAL
    assert L.ds_vit_overlay_chunk(ok, 0, 4, 5120, sp, 1, ok, 3, ok, None, None) == dv.ERANGE
    assert L.ds_vit_encode(None, None, 84, 84, None, None, 0, None) == dv.EINVAL
    assert L.ds_vit_release(None) == dv.OK
    assert L.ds_vit_device_status(None, None) == dv.EINVAL
    fake = C.c_void_p(16)   # never dereferenced: the checks reject before any launch
    assert L.ds_vit_selftest_wait_timeout(None, fake, 1000, None) == dv.EINVAL
    assert L.ds_vit_selftest_wait_timeout(fake, None, 1000, None) == dv.EINVAL
    assert L.ds_vit_selftest_wait_timeout(fake, fake, 0, None) == dv.EINVAL
    assert L.ds_vit_selftest_wait_timeout(fake, fake, 1000001, None) == dv.EINVAL
    assert L.ds_vit_op_attention(None, None, 1, None, None, None) == dv.EINVAL
    assert L.ds_vit_op_linear(None, 1, 64, None, 256, None, None, 0, None, None, None, None) == dv.EINVAL


def test_plan_matches_oracle(dv):
    """The host planner of the C ABI agrees with the oracle's plan exactly
    (every field), on the workload sizes and on random sizes up to 16000."""
    import oracle.preprocess as PP
    sizes = [(546, 546), (1344, 1344), (2688, 336), (544, 544), (100, 100), (3024, 4032),
             (1080, 1920), (1000, 333), (20000, 100), (1, 1), (1, 65535), (65535, 1), (300, 100),
             (100, 300), (4, 1), (4, 3)]
    rng = np.random.default_rng(11)
    sizes += [(int(h), int(w)) for h, w in rng.integers(1, 16000, (400, 2))]   # H*W <= 2^28
    sizes += [(int(h), int(w)) for h, w in rng.integers(1, 700, (400, 2))]
    for H, W in sizes:
        got = dv.plan_image(H, W)
        ref = PP.plan(H, W)
        for k in ("h", "w", "Hc", "Wc", "Hr", "Wr", "y0", "x0"):
            assert got[k] == ref[k], (H, W, k, got, ref)


def test_qwen_layout_matches_oracle(dv):
    import oracle.qwen as Q
    for h, w, s in ((2, 3, 5), (32, 32, 0), (1, 1, 100), (5, 17, 12345), (64, 16, 7)):
        pos, delta = dv.qwen_layout(h, w, s)
        rp, rd = Q.layout(h, w, s)
        assert np.array_equal(pos, rp) and delta == rd
    b = C.c_int32(0)
    assert dv.lib.ds_vit_qwen_layout(0, 3, 0, None, 0, C.byref(b)) == dv.EINVAL
    small = np.zeros(5, np.int32)
    assert dv.lib.ds_vit_qwen_layout(2, 3, 0, small.ctypes.data, 5, C.byref(b)) == dv.ECAP
    n = C.c_size_t(0)
    assert dv.lib.ds_vit_qwen_workspace_bytes(48, 64, C.byref(n)) == dv.EINVAL        # not a multiple of 32
    assert dv.lib.ds_vit_qwen_workspace_bytes(1088, 1056, C.byref(n)) == dv.ERANGE    # 34 x 33 > 1024 tokens
    assert dv.lib.ds_vit_qwen_workspace_bytes(1024, 1024, C.byref(n)) == dv.OK and n.value > 0


def test_plan_and_preprocess_argument_checks(dv):
    L = dv.lib
    p = dv.Plan()
    for H, W in ((0, 10), (10, 0), (65536, 10), (20000, 20000)):
        assert L.ds_vit_plan_image(H, W, C.byref(p)) == dv.EINVAL
    assert L.ds_vit_plan_image(10, 10, None) == dv.EINVAL
    assert L.ds_vit_plan_image(1000, 333, C.byref(p)) == dv.OK
    b = C.c_size_t(0)
    assert L.ds_vit_preprocess_workspace_bytes(C.byref(p), C.byref(b)) == dv.OK and b.value > 0
    p.Hr += 1                                     # a plan that is not the image's plan
    assert L.ds_vit_preprocess_workspace_bytes(C.byref(p), C.byref(b)) == dv.EINVAL
    assert L.ds_vit_preprocess(C.byref(p), C.c_void_p(16), C.c_void_p(16), C.c_void_p(256), 1 << 30,
                               None) == dv.EINVAL
    p.Hr -= 1
    assert L.ds_vit_preprocess(None, None, None, None, 0, None) == dv.EINVAL
    assert L.ds_vit_preprocess(C.byref(p), C.c_void_p(16), C.c_void_p(16), C.c_void_p(256), 0,
                               None) == dv.ECAP


def test_workspace_size_validation(dv):
    # a non-multiple of 14 and an image over the 9216-patch limit are refused
    L = dv.lib
    b = C.c_size_t(0)
    fake = C.c_void_p(1)
    H = (C.c_int32 * 1)(85)
    W = (C.c_int32 * 1)(84)
    assert L.ds_vit_workspace_bytes(fake, 1, H, W, C.byref(b)) == dv.EINVAL
    H[0], W[0] = 1358, 1344        # 97 x 96 patches
    assert L.ds_vit_workspace_bytes(fake, 1, H, W, C.byref(b)) == dv.ERANGE
    H[0], W[0] = 1344, 1344
    assert L.ds_vit_workspace_bytes(fake, 1, H, W, C.byref(b)) == dv.OK
    assert b.value >= 9216 * (1024 * 3 + 3072 + 4096) * 2


def test_no_alloc_scratch_covers_every_grid_up_to_the_limit(dv):
    """Every grid of at most NOALLOC_MAX_PATCHES patches fits the static scratch."""
    L = dv.lib
    b = C.c_size_t(0)
    fake = C.c_void_p(1)
    worst = 0
    for gh in range(1, dv.NOALLOC_MAX_PATCHES + 1):
        for gw in (dv.NOALLOC_MAX_PATCHES // gh,):
            H = (C.c_int32 * 1)(14 * gh)
            W = (C.c_int32 * 1)(14 * gw)
            assert L.ds_vit_workspace_bytes(fake, 1, H, W, C.byref(b)) == dv.OK
            worst = max(worst, b.value)
    assert worst <= dv.NOALLOC_SCRATCH_BYTES
