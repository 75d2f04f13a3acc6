"""The disk cache of oracle encodes used by the GPU tests: a cached result is
the oracle's own output, the key changes with every input that determines it,
and an unreadable entry is recomputed."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_util as G  # noqa: E402
import oracle as O  # noqa: E402
import workloads as WL  # noqa: E402


def test_cached_encode_equals_oracle(tmp_path, monkeypatch):
    monkeypatch.setenv("DSVIT_ORACLE_CACHE", str(tmp_path))
    W = WL.make_weights(2)
    imgs = [WL.uniform_image(84, 84, seed=1)]
    ref, offs = O.encode(imgs, W, WL.MODEL)
    e1, o1 = G.oracle_encode_cached(imgs, W, WL.MODEL)
    assert len(list(tmp_path.iterdir())) == 1
    e2, o2 = G.oracle_encode_cached(imgs, W, WL.MODEL)      # from disk
    for e, o in ((e1, o1), (e2, o2)):
        assert np.array_equal(e, ref) and np.array_equal(o, offs)


def test_key_follows_inputs(tmp_path):
    W = WL.make_weights(2)
    img = WL.uniform_image(84, 84, seed=1)
    k = G._oracle_cache_key([img], W, WL.MODEL, None)
    other = img.copy()
    other[0, 0, 0] ^= 1
    W2 = WL.make_weights(2)
    W2["layers"][1]["fc2_b"] = W2["layers"][1]["fc2_b"].copy()
    W2["layers"][1]["fc2_b"][0] ^= 1
    assert G._oracle_cache_key([other], W, WL.MODEL, None) != k
    assert G._oracle_cache_key([img], W2, WL.MODEL, None) != k
    assert G._oracle_cache_key([img], W, WL.MODEL, 1) != k
    assert G._oracle_cache_key([img], W, dict(WL.MODEL, ln_eps=1e-5), None) != k
    assert G._oracle_cache_key([img], W, WL.MODEL, None) == k


def test_unreadable_entry_is_recomputed(tmp_path, monkeypatch):
    monkeypatch.setenv("DSVIT_ORACLE_CACHE", str(tmp_path))
    W = WL.make_weights(2)
    imgs = [WL.uniform_image(84, 84, seed=2)]
    path = tmp_path / (G._oracle_cache_key(imgs, W, WL.MODEL, None) + ".npz")
    path.write_bytes(b"not an npz")
    e, offs = G.oracle_encode_cached(imgs, W, WL.MODEL)
    ref, roffs = O.encode(imgs, W, WL.MODEL)
    assert np.array_equal(e, ref) and np.array_equal(offs, roffs)
