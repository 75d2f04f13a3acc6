"""The two bounds the planar resize passes rely on, checked against the
oracle's filter coefficients (oracle/preprocess.py: coeffs) over many sizes.

* Nonzero taps: every output index's taps lie in [lo, hi) with
  hi - lo <= floor(4 max(scale, 1)) + 1 (both ends are truncations of
  c -+ support + 1/2 and support = 2 max(scale, 1)); the passes read
  4 ceil(that / 4) taps per output (weight groups of four for dp4a), so no
  nonzero weight is dropped.
* Staging start: the horizontal pass stages its input span from
  max(0, floor(e) - 1), with e the exact rational value of c - support + 1/2
  for the block's first output ((2x - 3) W + Wr) / (2 Wr) when W > Wr, else
  ((2x + 1) W - 3 Wr) / (2 Wr)); that start must be at most the first tap
  the float64 table computes and at most 2 below it (the span has room for 2).
"""
import math

import numpy as np
import pytest

import oracle.preprocess as PP


def _sizes(n, seed):
    rng = np.random.default_rng(seed)
    pairs = [(4032, 1512), (3024, 1134), (800, 840), (600, 630), (1, 546), (3, 700), (20000, 16800),
             (6000, 1512), (112, 112), (1000, 333), (333, 1000)]
    pairs += [(int(a), int(b)) for a, b in zip(rng.integers(1, 9000, n), rng.integers(1, 4000, n))]
    return pairs


def _nonzero_bound(n_in, n_out):
    s = n_in / n_out
    return int(math.floor(4.0 * (s if s > 1.0 else 1.0) + 1e-6)) + 1


@pytest.mark.parametrize("n_in,n_out", _sizes(150, 1))
def test_nonzero_taps_within_bound(n_in, n_out):
    xmin, kk = PP.coeffs(n_in, n_out)
    nz = kk != 0
    last = np.where(nz.any(axis=1), nz.shape[1] - np.argmax(nz[:, ::-1], axis=1), 0)
    assert last.max() <= _nonzero_bound(n_in, n_out)
    # and the span itself: hi - lo from the same truncations
    s = n_in / n_out
    sup = 2.0 * max(s, 1.0)
    for i in range(0, n_out, max(1, n_out // 64)):
        c = (i + 0.5) * s
        lo = max(int(c - sup + 0.5), 0)
        hi = min(int(c + sup + 0.5), n_in)
        assert hi - lo <= _nonzero_bound(n_in, n_out)


@pytest.mark.parametrize("W,Wr", _sizes(150, 2))
def test_staging_start(W, Wr):
    xmin, _ = PP.coeffs(W, Wr)
    for xb in range(0, Wr, 128):
        num = (2 * xb - 3) * W + Wr if W > Wr else (2 * xb + 1) * W - 3 * Wr
        start = max(num // (2 * Wr) - 1, 0)
        assert start <= int(xmin[xb]) <= start + 2, (W, Wr, xb)
