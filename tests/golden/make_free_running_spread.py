"""Writes free_running_spread.json: the spread envelope of the oracle's valid
evaluations on the full-depth (32-layer) workloads, which the free-running
GPU tests use as their elementwise bound.

Runs only the oracle (and the seeded input generators): for each workload the
whole encode in every mode of ``gpu_util.SPREAD_MODES`` (accumulation order
of products and norm statistics: fp32 BLAS, float64, fp32 reversed; fp32 or
bf16 softmax numerators; GELU in float64 or fp32 arithmetic), then the
envelope of the pairwise relative errors (``gpu_util.spread_of``).  Several minutes per workload on a few cores; the
1344 x 1344 image takes the longest.

    python tests/golden/make_free_running_spread.py [min] [aspect] [max]
"""
from __future__ import annotations

import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))                 # tests/ (gpu_util)
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))  # repo root (oracle, workloads)

import oracle as O  # noqa: E402
import workloads as WL  # noqa: E402
from gpu_util import SPREAD_FILE, SPREAD_MODES, SPREAD_Z, spread_of  # noqa: E402

NAMES = ("min", "aspect", "max")


def envelope(name: str) -> dict:
    wl = WL.WORKLOADS[name]
    imgs = WL.workload_images(name)
    if name == "aspect":
        imgs = imgs[:1]                  # one image; the workload repeats it on one stream
    W = WL.make_weights(wl["n_layers"])
    outs, secs = [], []
    for mode in SPREAD_MODES:
        t = time.time()
        with O.evaluation(*mode):
            outs.append(O.encode(imgs, W, WL.MODEL)[0])
        secs.append(round(time.time() - t, 1))
        print(f"{name}: {mode} {secs[-1]} s", flush=True)
    env = spread_of(outs)
    env.update(images=[list(im.shape[:2]) for im in imgs], layers=wl["n_layers"],
               modes=[list(m) for m in SPREAD_MODES], seconds=secs)
    return env


def main(argv):
    names = [a for a in argv if a in NAMES] or list(NAMES)
    d = {"z": SPREAD_Z, "workloads": {}}
    if os.path.exists(SPREAD_FILE):
        with open(SPREAD_FILE) as f:
            d = json.load(f)
    d["z"] = SPREAD_Z
    d["written_by"] = "tests/golden/make_free_running_spread.py (oracle only)"
    for name in names:
        d["workloads"][name] = envelope(name)
        with open(SPREAD_FILE, "w") as f:
            json.dump(d, f, indent=1)
            f.write("\n")
        print(name, {k: d["workloads"][name][k] for k in ("max", "mean")}, flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
