"""Helpers shared by the GPU tests (conversion and tolerance checks only)."""
import numpy as np

import oracle as O
import workloads as WL

# Per-element bound and per-row cosine of the embeddings, applied to every
# step of the encode recomputed by the oracle from the GPU's own input to that
# step (patch projection, each block, final norm, merger).
REL_TOL = 2e-2
COS_MIN = 0.999
# Free-running end-to-end comparisons: the bf16 rounding at every boundary
# amplifies any fp32 summation-order difference, so the elementwise bound is
# a multiple of the definition's own noise floor (the oracle with BLAS sgemm
# products against the oracle with float64-accumulated products).
FLOOR_FACTOR = 2.5


def dev(bits, torch):
    """bf16 bit patterns (numpy uint16) -> CUDA bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host(t):
    """CUDA bf16 tensor -> fp32 numpy."""
    return t.float().cpu().numpy()


def rand_bits(shape, seed, scale=1.0):
    return WL.to_bf16_bits(np.random.default_rng(seed).standard_normal(shape).astype(np.float32) * scale)


def rel_err(got, ref):
    return np.abs(got.astype(np.float64) - ref) / (1.0 + np.abs(ref.astype(np.float64)))


def row_cos(got, ref):
    g, r = got.astype(np.float64), ref.astype(np.float64)
    return (g * r).sum(-1) / (np.linalg.norm(g, axis=-1) * np.linalg.norm(r, axis=-1) + 1e-30)


def assert_parity(got, ref, rel=REL_TOL, cos=COS_MIN, what=""):
    e = rel_err(got, ref)
    c = row_cos(got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1]))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert e.max() <= rel, f"{what}: max rel err {e.max():.4g} (mean {e.mean():.3g}) > {rel}"
    assert c.min() >= cos, f"{what}: min row cosine {c.min():.6f} < {cos}"


def assert_end_to_end(got, imgs, W, cfg, n_layers=None, what=""):
    """Free-running embeddings vs the oracle: per-row cosine >= COS_MIN and an
    elementwise bound of FLOOR_FACTOR x the oracle's own summation-order spread
    (never tighter than REL_TOL)."""
    ref, offs = O.encode(imgs, W, cfg, n_layers=n_layers)
    with O.products("f64"):
        alt, _ = O.encode(imgs, W, cfg, n_layers=n_layers)
    floor = rel_err(alt, ref)
    e = rel_err(got, ref)
    c = row_cos(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert c.min() >= COS_MIN, f"{what}: min row cosine {c.min():.6f}"
    lim_max = max(REL_TOL, FLOOR_FACTOR * floor.max())
    lim_mean = max(REL_TOL / 10, FLOOR_FACTOR * floor.mean())
    assert e.max() <= lim_max, f"{what}: max rel err {e.max():.4g} > {lim_max:.4g} (floor {floor.max():.4g})"
    assert e.mean() <= lim_mean, f"{what}: mean rel err {e.mean():.4g} > {lim_mean:.4g}"
    return offs, dict(max=float(e.max()), mean=float(e.mean()), floor_max=float(floor.max()),
                      floor_mean=float(floor.mean()), cos=float(c.min()))


def bits_of(t):
    """CPU bf16 tensor -> fp32 numpy (exact)."""
    import torch
    return O.bits_to_f32(t.view(torch.int16).numpy().view(np.uint16))


def assert_steps_teacher_forced(imgs, W, cfg, blocks, fnorm, out, layers, rows=None, toks=None):
    """Each step recomputed by the oracle from the GPU's own input to it."""
    grids = [(im.shape[0] // 14, im.shape[1] // 14) for im in imgs]
    seqlens = [gh * gw for gh, gw in grids]
    gy = np.concatenate([O.grid_positions(*g)[0] for g in grids])
    gx = np.concatenate([O.grid_positions(*g)[1] for g in grids])
    bl = blocks.cpu()
    sel = np.arange(sum(seqlens)) if rows is None else np.asarray(rows)
    P = np.concatenate([O.normalise(O.patchify(im), cfg["mean"], cfg["std"]) for im in imgs])
    x0 = O.round_bf16(O.mm(P[sel], O.bits_to_f32(W["patch_w"]).T) + O.bits_to_f32(W["patch_b"]))
    assert_parity(bits_of(bl[0])[sel], x0, what="patch projection")
    for l in layers:
        xin, xout = bits_of(bl[l]), bits_of(bl[l + 1])
        ref = O.vit_block(xin, W["layers"][l], cfg, seqlens, gy, gx, rows=rows)
        assert_parity(xout[sel], ref, what=f"block {l}")
    L = len(bl) - 1
    z = O.round_bf16(O.norm(bits_of(bl[L])[sel], W["lnm_g"], W["lnm_b"], cfg))
    zg = fnorm.float().cpu().numpy()
    assert_parity(zg[sel], z, what="final norm")
    starts = np.concatenate([[0], np.cumsum(seqlens)])
    A = np.concatenate([O.merge_unfold(zg[starts[i]:starts[i + 1]], *grids[i])
                        for i in range(len(imgs))])
    t = np.arange(A.shape[0]) if toks is None else np.asarray(toks)
    assert_parity(out.float().cpu().numpy()[t], O.merger(A[t], W), what="merger")
