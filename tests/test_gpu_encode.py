"""End-to-end encode parity on the GPU through the C ABI, against the CPU
oracle on the same seeded inputs.

Two criteria (the reasons are stated in gpu_util.py):
* every step (patch projection, each ViT block, final norm, merger) is
  recomputed by the oracle from the GPU's own input to that step and must
  meet |gpu - oracle| <= 2e-2 (1 + |oracle|) per element, row cosine >= 0.999;
* free-running embeddings must meet row cosine >= 0.999 and an elementwise
  bound given by the spread between valid evaluations of the oracle.

Workloads: the tiny 84x84 image (2 layers), ragged grids and varlen batches
(2 layers), and at full depth (32 layers) the 546x546 image, the 1344x1344 and
2688x336 images (every block on sampled rows, and free running) and the
16-image varlen batch (every block on sampled rows of every image).  Also error paths, the device
status word, the host-buffer entry point and the overlay."""
import numpy as np
import pytest

import oracle as O
import workloads as WL
from gpu_util import (assert_end_to_end, assert_steps_teacher_forced, dev, host, sample_rows, sample_tokens,
                      stored_spread)

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
def w2():
    return WL.make_weights(2)


@pytest.fixture(scope="module")
def enc2(dv, w2):
    e = dv.Encoder(dv.weights_to_device(w2), WL.MODEL)
    yield e
    e.close()


def _run(dv, enc, imgs, dump=False):
    d = [torch.from_numpy(im).cuda() for im in imgs]
    r = enc.encode(d, dump=dump)
    torch.cuda.synchronize()
    assert enc.status() == dv.OK
    return r


def test_tiny_workload(dv, enc2, w2):
    img = WL.workload_images("tiny")[0]
    out, offs, blocks, fnorm = _run(dv, enc2, [img], dump=True)
    assert out.shape == (4, 5120)
    assert_steps_teacher_forced([img], w2, WL.MODEL, blocks, fnorm, out, layers=(0, 1))
    ref_offs, _ = assert_end_to_end(host(out), [img], w2, WL.MODEL, what="tiny")
    assert np.array_equal(offs, ref_offs)


@pytest.mark.parametrize("sizes", [[(350, 294)], [(84, 84), (350, 294), (14, 28)],
                                   [(126, 1260), (42, 14)], [(14, 14)]])
def test_ragged_and_batch(dv, enc2, w2, sizes):
    imgs = [WL.uniform_image(h, w, seed=100 + i) for i, (h, w) in enumerate(sizes)]
    out, offs, blocks, fnorm = _run(dv, enc2, imgs, dump=True)
    assert_steps_teacher_forced(imgs, w2, WL.MODEL, blocks, fnorm, out, layers=(0, 1))
    ref_offs, _ = assert_end_to_end(host(out), imgs, w2, WL.MODEL, what=str(sizes))
    assert np.array_equal(offs, ref_offs)


def test_batch_equals_single(dv, enc2):
    imgs = [WL.uniform_image(h, w, seed=200 + i) for i, (h, w) in enumerate([(84, 126), (210, 168)])]
    both, offs = _run(dv, enc2, imgs)
    one, _ = _run(dv, enc2, imgs[:1])
    two, _ = _run(dv, enc2, imgs[1:])
    assert torch.equal(both[offs[0]:offs[1]], one) and torch.equal(both[offs[1]:offs[2]], two)


def test_repeat_is_deterministic(dv, enc2):
    img = [WL.uniform_image(350, 294, seed=9)]
    a, _ = _run(dv, enc2, img)
    a = a.clone()
    b, _ = _run(dv, enc2, img)
    assert torch.equal(a, b)


def test_two_streams_match_one(dv, enc2, w2):
    """Two prepared handles encoding concurrently on two streams (each with
    its own workspace and output, as the throughput measurement runs) give
    the one-stream embeddings bit for bit: nothing is shared between handles."""
    imgs = [WL.uniform_image(h, w, seed=400 + i) for i, (h, w) in enumerate([(350, 294), (210, 1008)])]
    d = [torch.from_numpy(im).cuda() for im in imgs]
    ref, offs = _run(dv, enc2, imgs)
    ref = ref.clone()
    enc_b = dv.Encoder(dv.weights_to_device(w2), WL.MODEL)
    try:
        encs = (enc2, enc_b)
        outs = [torch.zeros_like(ref) for _ in range(4)]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        cur = torch.cuda.current_stream()
        for st in streams:
            st.wait_stream(cur)
        for i in range(4):
            with torch.cuda.stream(streams[i % 2]):
                encs[i % 2].encode(d, out=outs[i])
        for st in streams:
            cur.wait_stream(st)
        torch.cuda.synchronize()
        assert enc2.status() == dv.OK and enc_b.status() == dv.OK
        for o in outs:
            assert torch.equal(o, ref)
    finally:
        enc_b.close()


def test_host_buffers_match_device(dv, enc2):
    imgs = [WL.uniform_image(h, w, seed=300 + i) for i, (h, w) in enumerate([(84, 84), (168, 98)])]
    dev_out, offs = _run(dv, enc2, imgs)
    hin = [torch.from_numpy(im).pin_memory() for im in imgs]
    hout = torch.empty((int(offs[-1]), 5120), dtype=torch.bfloat16).pin_memory()
    offs2 = enc2.encode_host(hin, hout)
    torch.cuda.synchronize()
    assert np.array_equal(offs, offs2) and torch.equal(hout, dev_out.cpu())


def test_graph_replays_the_encode(dv, enc2):
    """An encode recorded as a graph (ds_vit_graph_create) and replayed gives
    the direct encode's embeddings bit for bit, and recomputes them: after new
    pixels are written into the same buffers, a replay matches a direct encode
    of the new images.  Replays alternate between two graphs on two streams."""
    sizes = [(350, 294), (84, 84)]
    first = [torch.from_numpy(WL.uniform_image(h, w, seed=500 + i)).cuda() for i, (h, w) in enumerate(sizes)]
    second = [torch.from_numpy(WL.uniform_image(h, w, seed=600 + i)).cuda() for i, (h, w) in enumerate(sizes)]
    ref1, offs = enc2.encode(first)
    ref1 = ref1.clone()
    ref2, _ = enc2.encode(second)
    ref2 = ref2.clone()
    torch.cuda.synchronize()
    bufs = [[im.clone() for im in first] for _ in range(2)]
    graphs = []
    try:
        for b in bufs:
            g, out, goffs = enc2.graph(b)
            assert np.array_equal(goffs, offs)
            graphs.append((g, out))
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        cur = torch.cuda.current_stream()
        for st in streams:
            st.wait_stream(cur)
        for i in range(4):
            graphs[i % 2][0].launch(streams[i % 2])
        for st in streams:
            cur.wait_stream(st)
        torch.cuda.synchronize()
        for _, out in graphs:
            assert torch.equal(out, ref1)
        for b in bufs:                       # same buffers, new contents
            for dst, src in zip(b, second):
                dst.copy_(src)
        for g, _ in graphs:
            g.launch()
        torch.cuda.synchronize()
        assert enc2.status() == dv.OK
        for _, out in graphs:
            assert torch.equal(out, ref2)
    finally:
        for g, _ in graphs:
            g.close()


def test_graph_create_failure_keeps_nothing(dv, enc2):
    """A recording whose encode rejects its arguments returns that error,
    stores no handle and leaves no capture open: a direct encode right after
    works and matches a fresh one."""
    import ctypes as C
    img = torch.from_numpy(WL.uniform_image(84, 84, seed=11)).cuda()
    out = torch.zeros((4, 5120), dtype=torch.bfloat16, device="cuda")
    ws = enc2.workspace([(84, 84)])
    px = (C.c_void_p * 1)(img.data_ptr())
    offs = (C.c_int64 * 2)()
    h = C.c_void_p(7)
    bad_h, bad_w = (C.c_int32 * 1)(85), (C.c_int32 * 1)(84)
    rc = dv.lib.ds_vit_graph_create(enc2.handle, 0, 1, px, bad_h, bad_w, C.c_void_p(out.data_ptr()), offs,
                                    C.c_void_p(ws.data_ptr()), ws.numel(), C.byref(h))
    assert rc == dv.EINVAL and not h.value
    small = (C.c_int32 * 1)(84)
    rc = dv.lib.ds_vit_graph_create(enc2.handle, 0, 1, px, small, small, C.c_void_p(out.data_ptr()), offs,
                                    C.c_void_p(ws.data_ptr()), 1024, C.byref(h))
    assert rc == dv.ECAP and not h.value
    a, _ = _run(dv, enc2, [WL.uniform_image(84, 84, seed=11)])
    b, _ = enc2.encode([img])
    torch.cuda.synchronize()
    assert torch.equal(a, b) and bool((out == 0).all())


def test_graph_host_buffers(dv, enc2):
    """The host-buffer encode recorded as a graph: both copies and the encode
    in every replay, page-locked buffers."""
    imgs = [WL.uniform_image(h, w, seed=700 + i) for i, (h, w) in enumerate([(168, 98), (84, 84)])]
    dev_out, offs = _run(dv, enc2, imgs)
    hin = [torch.from_numpy(im).pin_memory() for im in imgs]
    hout = torch.zeros((int(offs[-1]), 5120), dtype=torch.bfloat16).pin_memory()
    g, goffs = enc2.graph_host(hin, hout)
    try:
        g.launch()
        torch.cuda.synchronize()
        assert np.array_equal(goffs, offs) and torch.equal(hout, dev_out.cpu())
        new = [WL.uniform_image(h, w, seed=800 + i) for i, (h, w) in enumerate([(168, 98), (84, 84)])]
        new_out, _ = _run(dv, enc2, new)
        for dst, src in zip(hin, new):
            dst.copy_(torch.from_numpy(src))
        g.launch()
        torch.cuda.synchronize()
        assert torch.equal(hout, new_out.cpu())
    finally:
        g.close()


def test_errors_write_nothing(dv, enc2):
    import ctypes as C
    img = torch.from_numpy(WL.uniform_image(84, 84, seed=5)).cuda()
    out = torch.full((4, 5120), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = enc2.workspace([(84, 84)])
    L = dv.lib
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: C.c_void_p(t.data_ptr())
    assert L.ds_vit_encode(enc2.handle, P(img), 85, 84, P(out), P(ws), ws.numel(), st) == dv.EINVAL
    assert L.ds_vit_encode(enc2.handle, P(img), 84, 84, P(out), P(ws), 1024, st) == dv.ECAP
    assert L.ds_vit_encode(enc2.handle, P(img), 14 * 200, 14 * 200, P(out), P(ws), ws.numel(),
                           st) == dv.ERANGE
    # Pixels must start on a 4-byte boundary (rejected before any launch).
    padded = torch.zeros(84 * 84 * 3 + 4, dtype=torch.uint8, device="cuda")
    assert L.ds_vit_encode(enc2.handle, C.c_void_p(padded.data_ptr() + 2), 84, 84, P(out), P(ws),
                           ws.numel(), st) == dv.EINVAL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


# ------------------------------------------------------------------ full depth

@pytest.fixture(scope="module")
def w32():
    return WL.make_weights(32)


@pytest.fixture(scope="module")
def enc32(dv, w32):
    e = dv.Encoder(dv.weights_to_device(w32), WL.MODEL)
    yield e
    e.close()


def test_min_image_full_depth(dv, enc32, w32):
    """546x546 gradient image, 32 layers: every block teacher-forced, and the
    free-running output within the stored spread of the oracle's valid
    evaluations."""
    img = WL.workload_images("min")[0]
    out, offs, blocks, fnorm = _run(dv, enc32, [img], dump=True)
    assert_steps_teacher_forced([img], w32, WL.MODEL, blocks, fnorm, out, layers=range(32))
    assert_end_to_end(host(out), [img], w32, WL.MODEL, what="546x546 full depth",
                      env=stored_spread("min"))


@pytest.fixture(scope="module")
def max_run(dv, enc32):
    """The 1344x1344 image through ds_vit_encode (plain) and through the debug
    entry point (block dumps); both outputs must be bit-identical."""
    img = WL.workload_images("max")[0]
    H, W = img.shape[:2]
    d = torch.from_numpy(img).cuda()
    plain = torch.empty((1024, 5120), dtype=torch.bfloat16, device="cuda")
    ws = enc32.workspace([(H, W)])
    import ctypes as C
    P = lambda t: C.c_void_p(t.data_ptr())
    dv.check(dv.lib.ds_vit_encode(enc32.handle, P(d), H, W, P(plain), P(ws), ws.numel(),
                                  C.c_void_p(torch.cuda.current_stream().cuda_stream)), "ds_vit_encode")
    out, offs, blocks, fnorm = _run(dv, enc32, [img], dump=True)
    assert torch.equal(plain, out)
    return img, out, offs, blocks, fnorm


def test_max_image_all_blocks(dv, max_run, w32):
    """1344x1344, 9216 patches, 32 layers: sampled query rows of every block
    and sampled merged tokens, each recomputed from the GPU's own inputs."""
    img, out, offs, blocks, fnorm = max_run
    assert offs[-1] == 1024
    rows = sample_rows([9216], 96, seed=7)
    assert_steps_teacher_forced([img], w32, WL.MODEL, blocks, fnorm, out, layers=range(32),
                                rows=rows, toks=sample_tokens(offs, 8, seed=8))


def test_max_image_free_running(dv, max_run, w32):
    """The 1024-token image's embeddings (ds_vit_encode) against the oracle's
    whole encode: row cosine >= 0.999 and the elementwise error within the
    stored spread of the oracle's valid evaluations."""
    img, out, offs, _, _ = max_run
    ref_offs, stats = assert_end_to_end(host(out), [img], w32, WL.MODEL, what="1344x1344 free running",
                                        env=stored_spread("max"))
    assert np.array_equal(offs, ref_offs)


def test_aspect_image_all_blocks_and_free_running(dv, enc32, w32):
    """2688x336 (192 x 24 grid, row positions up to 191): sampled rows of every
    block, including the last grid rows, teacher-forced; then the free-running
    output against the oracle within the stored spread."""
    img = WL.workload_images("aspect")[0]
    out, offs, blocks, fnorm = _run(dv, enc32, [img], dump=True)
    assert offs[-1] == 512
    rows = np.union1d(sample_rows([4608], 24, seed=9), [23, 24, 4584, 4600])
    assert_steps_teacher_forced([img], w32, WL.MODEL, blocks, fnorm, out, layers=range(32),
                                rows=rows, toks=sample_tokens(offs, 6, seed=10))
    del blocks, fnorm
    assert_end_to_end(host(out), [img], w32, WL.MODEL, what="2688x336 free running",
                      env=stored_spread("aspect"))


def test_batch16_full_size(dv, enc32, w32):
    """The 16-image varlen batch (sizes cycling 546^2, 1344x672, 672x1344,
    1008^2, 840x420; 54,684 patches, up to 5,184 per image), 32 layers, through
    ds_vit_encode_batch: token offsets exact; every block teacher-forced on
    sampled rows of every image (first and last row, a row of the last query
    tile, random rows), with keys and values from that image only; the merger
    on sampled tokens of every image.  The debug entry point that dumps the
    blocks gives bit-identical embeddings."""
    imgs = WL.workload_images("batch16")
    d = [torch.from_numpy(im).cuda() for im in imgs]
    plain, offs_plain = _run(dv, enc32, imgs)
    plain = plain.clone()
    out, offs, blocks, fnorm = _run(dv, enc32, imgs, dump=True)
    assert torch.equal(plain, out) and np.array_equal(offs_plain, offs)
    seqlens = [(im.shape[0] // 14) * (im.shape[1] // 14) for im in imgs]
    assert sum(seqlens) == 54684 and max(seqlens) == 5184
    ntok = [O.merge_unfold(np.zeros((n, 1), np.float32), im.shape[0] // 14, im.shape[1] // 14).shape[0]
            for n, im in zip(seqlens, imgs)]
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(ntok)]))
    assert offs[-1] == 6076
    del d
    assert_steps_teacher_forced(imgs, w32, WL.MODEL, blocks, fnorm, out, layers=range(32),
                                rows=sample_rows(seqlens, 4, seed=11), toks=sample_tokens(offs, 1, seed=12))


# ------------------------------------------------------------------ overlay

def test_overlay_max_workload_exact(dv, w32):
    """Overlay of one 1,058-row span into a 4096 x 5120 prompt at the seeded base."""
    ids, pos, typ, src = O.layout(96, 96, WL.MODEL["image_token_id"])
    base = WL.span_bases("max", [len(ids)])[0]
    hidden = WL.hidden_buffer(4096, 5120, WL.WORKLOADS["max"]["hidden_seed"])
    emb = WL.hidden_buffer(1024, 5120, 77)
    ref = O.overlay(hidden, base, typ, src, emb, w32["sentinel"])
    h = dev(hidden, torch)
    dv.overlay(h, [(base, 96, 96, 0)], dev(emb, torch), dev(w32["sentinel"], torch))
    torch.cuda.synchronize()
    assert np.array_equal(h.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_overlay_batch16_exact(dv, w32):
    sizes = [(H, W) for H, W, _, _ in WL.WORKLOADS["batch16"]["images"]]
    lays = [O.layout(H // 14, W // 14, 1) for H, W in sizes]
    bases = WL.span_bases("batch16", [len(l[0]) for l in lays])
    ntok = [int((l[2] == O.TOK_IMAGE).sum()) for l in lays]
    eoff = np.concatenate([[0], np.cumsum(ntok)])
    hidden = WL.hidden_buffer(16384, 5120, WL.WORKLOADS["batch16"]["hidden_seed"])
    emb = WL.hidden_buffer(int(eoff[-1]), 5120, 78)
    ref = hidden.copy()
    for i, (ids, pos, typ, src) in enumerate(lays):
        ref = O.overlay(ref, bases[i], typ, src, emb[eoff[i]:eoff[i + 1]], w32["sentinel"])
    h = dev(hidden, torch)
    spans = [(bases[i], H // 14, W // 14, int(eoff[i])) for i, (H, W) in enumerate(sizes)]
    dv.overlay(h, spans, dev(emb, torch), dev(w32["sentinel"], torch))
    torch.cuda.synchronize()
    assert np.array_equal(h.view(torch.int16).cpu().numpy().view(np.uint16), ref)


def test_overlay_chunks_batch16_exact(dv, w32):
    """Chunked prefill over the 16-span prompt: chunks of 2048 rows and a
    ragged split (spans cross chunk boundaries) against the oracle, chunk by
    chunk, with the row-type mask; the chunks reassemble to the whole overlay."""
    sizes = [(H, W) for H, W, _, _ in WL.WORKLOADS["batch16"]["images"]]
    lays = [O.layout(H // 14, W // 14, 1) for H, W in sizes]
    bases = WL.span_bases("batch16", [len(l[0]) for l in lays])
    ntok = [int((l[2] == O.TOK_IMAGE).sum()) for l in lays]
    eoff = np.concatenate([[0], np.cumsum(ntok)])
    hidden = WL.hidden_buffer(16384, 5120, WL.WORKLOADS["batch16"]["hidden_seed"])
    emb = WL.hidden_buffer(int(eoff[-1]), 5120, 78)
    spans = [(bases[i], H // 14, W // 14, int(eoff[i])) for i, (H, W) in enumerate(sizes)]
    d_emb, d_sent = dev(emb, torch), dev(w32["sentinel"], torch)
    whole = dev(hidden, torch)
    dv.overlay(whole, spans, d_emb, d_sent)
    for cuts in (list(range(0, 16385, 2048)), [0, 65, 700, 701, 3000, 6979, 6980, 16384]):
        parts = []
        for a, b in zip(cuts[:-1], cuts[1:]):
            ch = dev(hidden[a:b], torch)
            rt = torch.full((b - a,), 255, dtype=torch.uint8, device="cuda")
            dv.overlay_chunk(ch, a, spans, d_emb, d_sent, row_type=rt)
            torch.cuda.synchronize()
            ref, ref_rt = O.overlay_chunk(hidden[a:b], a, spans, emb, w32["sentinel"])
            assert np.array_equal(ch.view(torch.int16).cpu().numpy().view(np.uint16), ref), (a, b)
            assert np.array_equal(rt.cpu().numpy(), ref_rt), (a, b)
            parts.append(ch)
        assert torch.equal(torch.cat(parts).view(torch.int16), whole.view(torch.int16))


def test_overlay_rows_exact(dv, w32):
    """Per-row overlay (rows / type / src arrays on the device) of the 16-image
    batch's spans: at the spans' own rows it equals the span overlay bit for
    bit, and with the rows scattered over the prompt (text interleaved) it
    equals the oracle; the entries are checked on the device and an invalid one
    (a row past the buffer, or an unknown type) writes nothing."""
    sizes = [(H, W) for H, W, _, _ in WL.WORKLOADS["batch16"]["images"]]
    lays = [O.layout(H // 14, W // 14, 1) for H, W in sizes]
    bases = WL.span_bases("batch16", [len(l[0]) for l in lays])
    ntok = [int((l[2] == O.TOK_IMAGE).sum()) for l in lays]
    eoff = np.concatenate([[0], np.cumsum(ntok)])
    hidden = WL.hidden_buffer(16384, 5120, WL.WORKLOADS["batch16"]["hidden_seed"])
    emb = WL.hidden_buffer(int(eoff[-1]), 5120, 78)
    typ = np.concatenate([l[2] for l in lays])
    src = np.concatenate([np.where(l[3] >= 0, l[3] + eoff[i], -1) for i, l in enumerate(lays)]).astype(np.int32)
    rows = np.concatenate([bases[i] + np.arange(len(l[0])) for i, l in enumerate(lays)]).astype(np.int32)
    d_emb, d_sent = dev(emb, torch), dev(w32["sentinel"], torch)
    I = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    spans = [(bases[i], H // 14, W // 14, int(eoff[i])) for i, (H, W) in enumerate(sizes)]
    a, b = dev(hidden, torch), dev(hidden, torch)
    dv.overlay(a, spans, d_emb, d_sent)
    st = dv.overlay_rows(b, I(rows), I(typ), I(src), d_emb, d_sent)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert np.array_equal(bits(b), O.overlay_rows(hidden, rows, typ, src, emb, w32["sentinel"]))
    scattered = np.sort(np.random.default_rng(79).choice(16384, len(rows), replace=False)).astype(np.int32)
    c = dev(hidden, torch)
    st = dv.overlay_rows(c, I(scattered), I(typ), I(src), d_emb, d_sent)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bits(c), O.overlay_rows(hidden, scattered, typ, src, emb, w32["sentinel"]))
    for bad_rows, bad_typ, code in ((np.where(np.arange(len(rows)) == 5000, 16384, rows), typ, dv.ERANGE),
                                    (rows, np.where(np.arange(len(typ)) == 17, 9, typ).astype(np.uint8),
                                     dv.EINVAL)):
        e = dev(hidden, torch)
        st = dv.overlay_rows(e, I(bad_rows.astype(np.int32)), I(bad_typ), I(src), d_emb, d_sent)
        torch.cuda.synchronize()
        assert int(st.item()) == code
        assert np.array_equal(bits(e), hidden)


def test_overlay_rejects_out_of_range(dv, w32):
    h = torch.zeros((100, 5120), dtype=torch.bfloat16, device="cuda")
    emb = torch.zeros((4, 5120), dtype=torch.bfloat16, device="cuda")
    s = dev(w32["sentinel"], torch)
    with pytest.raises(dv.DsVitError):
        dv.overlay(h, [(95, 6, 6, 0)], emb, s)          # 8 rows from 95 leave the buffer
    with pytest.raises(dv.DsVitError):
        dv.overlay(h, [(0, 6, 6, 1)], emb, s)           # embed rows 1..4 leave embeds
    with pytest.raises(dv.DsVitError):
        dv.overlay(h, [(0, 6, 6, 0), (5, 6, 6, 0)], emb, s)   # overlapping spans
    torch.cuda.synchronize()
    assert bool((h == 0).all())


def test_seeded_size_sweep(dv, enc2, w2):
    """A seeded batch of irregular grids (ragged query and key tiles, grids that
    are not multiples of 3, extreme aspects), at most ~4000 patches in all:
    every step teacher-forced, the free-running output within the oracle's
    spread, and the token offsets exact."""
    rng = np.random.default_rng(4242)
    sizes = [(1, 1), (3, 37)]
    while sum(gh * gw for gh, gw in sizes) < 3000:
        sizes.append((int(rng.integers(1, 41)), int(rng.integers(1, 41))))
    imgs = [WL.uniform_image(14 * gh, 14 * gw, seed=500 + i) for i, (gh, gw) in enumerate(sizes)]
    out, offs, blocks, fnorm = _run(dv, enc2, imgs, dump=True)
    assert_steps_teacher_forced(imgs, w2, WL.MODEL, blocks, fnorm, out, layers=(0, 1))
    ref_offs, _ = assert_end_to_end(host(out), imgs, w2, WL.MODEL, what=f"sweep {sizes}")
    assert np.array_equal(offs, ref_offs)
