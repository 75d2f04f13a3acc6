#!/usr/bin/env python
"""Benchmark: merged visual tokens/s of the vision-tower encode on the
1024-token image (1344x1344 uint8 RGB, 9216 patches, 32 layers, 1024 merged
tokens at width 5120), plus the token layout and the overlay of the span into
a 4096 x 5120 prompt buffer.  One step = one pass of that whole path.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --profile encode|attention|overlay|gemm-qkv|gemm-fc1|gemm-fc2|gemm-proj   (for ncu)

N > 1 runs under torchrun: every rank encodes its own copy of the workload
(replicas, no data-path collective); the timed region is bracketed by barriers
and the slowest rank's time is reported.  Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import ctypes as C
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "merged visual tokens/sec (ViT+merger, 1024-token image); % of BF16 TC peak"
WORKLOAD = "max"
IMG_H = IMG_W = 1344
GH = GW = 96
N_PATCH = GH * GW
N_TOK = 1024
N_LAYERS = 32
# Algorithmic FLOPs of one encode: unpadded K (588), full bidirectional attention.
KIND_FLOP = {"patch_gemm": 2 * N_PATCH * 1024 * 588, "qkv_gemm": 2 * N_PATCH * 1024 * 3072,
             "attention": 4 * N_PATCH * N_PATCH * 64 * 16, "proj_gemm": 2 * N_PATCH * 1024 * 1024,
             "fc1_gemm": 2 * N_PATCH * 1024 * 4096, "fc2_gemm": 2 * N_PATCH * 4096 * 1024,
             "merger_gemm1": 2 * N_TOK * 5120 * 9216, "merger_gemm2": 2 * N_TOK * 5120 * 5120}
ENCODE_FLOP = (KIND_FLOP["patch_gemm"] + KIND_FLOP["merger_gemm1"] + KIND_FLOP["merger_gemm2"]
               + N_LAYERS * sum(KIND_FLOP[k] for k in ("qkv_gemm", "attention", "proj_gemm",
                                                        "fc1_gemm", "fc2_gemm")))
KIND_NAMES = ["patch_gemm", "layernorm", "qkv_gemm", "attention", "proj_gemm",
              "fc1_gemm", "fc2_gemm", "merger_gemm1", "merger_gemm2"]
LAUNCHES_PER_ENCODE = 1 + N_LAYERS * 7 + 1 + 2


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def tensor_peak(pk, clk):
    """The measured bf16 peak that applies to a kernel timed at the sampled SM
    clock: the burst figure (cuBLAS timed alone, at the maximum SM clock) when
    the median SM clock under load is within 5% of the maximum, else the
    sustained one (a seconds-long loop under the power cap, at a lower clock).
    Returns (peak TFLOP/s, label)."""
    if clk and clk.get("sm_mhz") and clk.get("sm_max_mhz") and clk["sm_mhz"] < 0.95 * clk["sm_max_mhz"]:
        return pk["bf16_sus"], f"{pk['source']} bf16 dense, sustained (median SM clock {clk['sm_mhz']:.0f} MHz)"
    mhz = f"{clk['sm_mhz']:.0f} MHz" if clk and clk.get("sm_mhz") else "not sampled"
    return pk["bf16"], f"{pk['source']} bf16 dense, burst (median SM clock {mhz}, at its maximum)"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def aggregate(elapsed_s: float, units_per_rank: int, world: int):
    """(slowest rank's seconds, whole-job units/s).  Needs an initialised
    process group when world > 1."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64)
    if world > 1:
        if dist.get_backend() == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    tmax = float(t.item())
    return tmax, units_per_rank * world / tmax


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self):
        self.proc, self.lines = None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [[c.strip() for c in l.split(",")] for l in self.lines if l]
        rows = [r for r in rows if len(r) >= 9]
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis and vis.split(",")[0].isdigit():
            mine = [r for r in rows if r[0] == vis.split(",")[int(os.environ.get("LOCAL_RANK", 0))]]
            rows = mine or rows
        num = lambda s: float(s) if s.replace(".", "", 1).isdigit() else None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        if not sm or not mx:
            return None
        reasons = sorted({self.NAMES[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows)}


def kernel_source_hash(name: str) -> str:
    p = os.path.join(ROOT, "vit_vision_encoder_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def measured_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, or None
    when the attention source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_sha256_16") != kernel_source_hash("attention.cu"):
        return None
    return d.get("dram_bytes_per_launch")


def _threads():
    return int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count())))


def _oracle_block_timing(imgs, n_layers, cfg, W):
    """Oracle time of one encode of ``imgs``: patch projection, block 0 over
    all packed patches (measured), final LN + merger (measured); the whole
    encode derived as embed + n_layers x block + merger.  Returns
    (embed_s, block_s, merger_s, tokens)."""
    import numpy as np

    import oracle as O
    grids = [(im.shape[0] // 14, im.shape[1] // 14) for im in imgs]
    t0 = time.perf_counter()
    P = np.concatenate([O.normalise(O.patchify(im), cfg["mean"], cfg["std"]) for im in imgs])
    x = O.round_bf16(O.mm(P, O.bits_to_f32(W["patch_w"]).T) + O.bits_to_f32(W["patch_b"]))
    t1 = time.perf_counter()
    gy = np.concatenate([O.grid_positions(*g)[0] for g in grids])
    gx = np.concatenate([O.grid_positions(*g)[1] for g in grids])
    seqlens = [gh * gw for gh, gw in grids]
    x = O.vit_block(x, W["layers"][0], cfg, seqlens, gy, gx)
    t2 = time.perf_counter()
    z = O.round_bf16(O.norm(x, W["lnm_g"], W["lnm_b"], cfg))
    starts = np.concatenate([[0], np.cumsum(seqlens)])
    A = np.concatenate([O.merge_unfold(z[starts[i]:starts[i + 1]], *grids[i]) for i in range(len(imgs))])
    O.merger(A, W)
    t3 = time.perf_counter()
    return t1 - t0, t2 - t1, t3 - t2, A.shape[0]


def cpu_baseline():
    """The oracle as it stands, on a bounded sample of the same workload: the
    1344x1344 image through patch projection, one ViT block over all 9216
    patches, the final LN and the merger (measured).  The full-encode time is
    derived as embed + 32 x block + merger."""
    import workloads as WL
    W = WL.make_weights(1)
    img = WL.workload_images(WORKLOAD)[0]
    emb, blk, mrg, T = _oracle_block_timing([img], N_LAYERS, WL.MODEL, W)
    full = emb + N_LAYERS * blk + mrg
    return dict(value=T / full, unit="tokens/s", cores=_threads(), kind="oracle", derived=True,
                measured={"embed_s": round(emb, 3), "block_s": round(blk, 3), "merger_s": round(mrg, 3)},
                sample=f"1344x1344 image: patch projection, 1 of the 32 ViT blocks over all 9216 patches, "
                       f"final LN + merger, measured; full encode derived as embed + 32 x block + merger "
                       f"= {full:.1f} s (block {blk:.2f} s)")


def oracle_timings():
    """The oracle on every synthetic workload, on the host cores: the tiny
    image and the 546x546 image as whole encodes (measured); the 2688x336 image
    and the first five images of the 16-image batch (one cycle of its sizes, a
    declared subset) as patch projection + one block + merger, measured, with
    the whole encode derived as embed + 32 x block + merger."""
    import oracle as O
    import workloads as WL
    cfg = WL.MODEL
    res = {}
    for name in ("tiny", "min"):
        wl = WL.WORKLOADS[name]
        imgs = WL.workload_images(name)
        W = WL.make_weights(wl["n_layers"])
        t0 = time.perf_counter()
        e, _ = O.encode(imgs, W, cfg)
        sec = time.perf_counter() - t0
        res[name] = {"oracle_s": round(sec, 3), "oracle_tokens_per_s": round(e.shape[0] / sec, 3),
                     "oracle_images_per_s": round(len(imgs) / sec, 4), "cores": _threads(), "derived": False,
                     "sample": "whole encode"}
    W1 = WL.make_weights(1)
    for name, imgs, label in (("aspect", WL.workload_images("aspect")[:1], "one 2688x336 image"),
                              ("batch16", WL.workload_images("batch16")[:5],
                               "subset: the first 5 of the 16 images (one cycle of the sizes)")):
        emb, blk, mrg, T = _oracle_block_timing(imgs, N_LAYERS, cfg, W1)
        full = emb + N_LAYERS * blk + mrg
        res[name] = {"oracle_s": round(full, 2), "oracle_tokens_per_s": round(T / full, 3),
                     "oracle_images_per_s": round(len(imgs) / full, 5), "cores": _threads(), "derived": True,
                     "measured": {"embed_s": round(emb, 3), "block_s": round(blk, 3), "merger_s": round(mrg, 3)},
                     "sample": f"{label}: patch projection, 1 of the 32 blocks, final LN + merger measured; "
                               f"whole encode derived as embed + 32 x block + merger"}
    return res


def run_reference(args):
    """The oracle, timed on the host cores on this workload: each step is one of
    the 32 ViT blocks over all 9216 patches; the full encode is estimated as
    embed + 32 x mean block + merger."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle as O
    import workloads as WL
    img = WL.workload_images(WORKLOAD)[0]
    cfg = WL.MODEL
    W = WL.make_weights(N_LAYERS)
    gy, gx = O.grid_positions(GH, GW)
    t0 = time.perf_counter()
    P = O.normalise(O.patchify(img), cfg["mean"], cfg["std"])
    x = O.round_bf16(O.mm(P, O.bits_to_f32(W["patch_w"]).T) + O.bits_to_f32(W["patch_b"]))
    t_embed = time.perf_counter() - t0
    t0 = time.perf_counter()
    z = O.round_bf16(O.layer_norm(x, O.bits_to_f32(W["lnm_g"]), O.bits_to_f32(W["lnm_b"]), cfg["ln_eps"]))
    O.merger(O.merge_unfold(z, GH, GW), W)
    t_merge = time.perf_counter() - t0
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        x = O.vit_block(x, W["layers"][s % N_LAYERS], cfg, [N_PATCH], gy, gx)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    block = statistics.mean(times)
    full = t_embed + N_LAYERS * block + t_merge
    value = N_TOK / full
    sample = (f"each step: one of the 32 ViT blocks of the oracle over all 9216 patches of the 1344x1344 "
              f"image (measured, {block:.2f} s mean); the value is derived for the whole encode as embed "
              f"({t_embed:.2f} s) + 32 x mean block + final LN and merger ({t_merge:.2f} s) = {full:.1f} s")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": block * 1e3,
        "step": "one ViT block of the oracle (measured); value derived for the whole encode",
        "derived_encode_s": full, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "1344x1344 uint8 uniform (seed 3), 9216 patches, 32 layers, 1024 tokens; "
                               "CPU oracle (numpy fp32 with bf16 rounding)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _threads(), "kind": "oracle",
                         "derived": True, "sample": sample,
                         "measured": {"embed_s": round(t_embed, 3), "block_s": round(block, 3),
                                      "merger_s": round(t_merge, 3)}},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def encode_flop(sizes, n_layers: int, swiglu: bool = False) -> int:
    """Algorithmic FLOPs of one encode of these images (unpadded K, full
    bidirectional attention per image; SwiGLU doubles the up-projection)."""
    tot = 0
    fc1 = 8192 if swiglu else 4096
    for H, W in sizes:
        gh, gw = H // 14, W // 14
        n, t = gh * gw, ((gh + 2) // 3) * ((gw + 2) // 3)
        tot += 2 * n * 1024 * 588 + 2 * t * 5120 * 9216 + 2 * t * 5120 * 5120
        tot += n_layers * (2 * n * 1024 * (3072 + 1024 + fc1 + 4096) + 4 * n * n * 64 * 16)
    return tot


def qwen_workload(pk, reps: int = 5, H: int = 1024, W: int = 1024):
    """The Qwen3-VL-style tower (27 blocks, hidden 1152, 16 heads of 72, 2x2
    merger, three DeepStack mergers) on a 1024x1024 image (4096 patches, 1024
    tokens): CUDA events around ds_vit_qwen_encode with all four outputs.
    Algorithmic FLOPs count the real head width (72), not the padding."""
    import torch

    import workloads as WL
    import vit_vision_encoder_gb300 as dv
    cfg = WL.QWEN_MODEL
    Wq = WL.make_weights_qwen(cfg["n_layers"])
    enc = dv.QwenEncoder(dv.weights_to_device(Wq), cfg)
    img = torch.from_numpy(WL.uniform_image(H, W, seed=8)).cuda()
    T, N = (H // 32) * (W // 32), (H // 16) * (W // 16)
    out = torch.empty((T, 5120), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        enc.encode(img, out=out)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for r in range(reps):
        enc.encode(img, out=out)
        ev[r + 1].record()
    torch.cuda.synchronize()
    sec = statistics.mean(ev[r].elapsed_time(ev[r + 1]) / 1e3 for r in range(reps))
    L = cfg["n_layers"]
    fl = 2 * N * 1152 * 1536 + L * (2 * N * 1152 * (3456 + 1152 + 4608 + 4608) + 4 * N * N * 72 * 16)
    fl += 4 * (2 * T * 4608 * 4608 + 2 * T * 5120 * 4608)
    enc.close()
    return {"tower": "Qwen3-VL-style: 16x16x2 patches, 27 blocks of 1152 (16 heads of 72), 2x2 merger + 3 DeepStack",
            "image": [H, W], "patches": N, "tokens": T, "ms_per_encode": round(sec * 1e3, 4),
            "tokens_per_s": round(T / sec, 1), "tflops": round(fl / sec / 1e12, 1),
            "frac_of_peak": round(fl / sec / 1e12 / pk["tc"], 3),
            "note": "heads padded to 80 in the QKV projection and attention tiles; FLOPs counted at 72"}


def official_workload(pk, reps: int = 5):
    """The released tower's block variant (RMSNorm, SwiGLU, half-vector RoPE
    pairing, [-1, 1] pixels) on the 1344x1344 image at full depth: its own
    weights (fc1 doubled for gate and up), CUDA events around the encode."""
    import torch

    import workloads as WL
    import vit_vision_encoder_gb300 as dv
    W = WL.make_weights_official(N_LAYERS)
    enc = dv.Encoder(dv.weights_to_device(W), WL.MODEL_OFFICIAL)
    img = torch.from_numpy(WL.workload_images(WORKLOAD)[0]).cuda()
    out = torch.empty((N_TOK, 5120), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        enc.encode([img], out=out)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for r in range(reps):
        enc.encode([img], out=out)
        ev[r + 1].record()
    torch.cuda.synchronize()
    sec = statistics.mean(ev[r].elapsed_time(ev[r + 1]) / 1e3 for r in range(reps))
    fl = encode_flop([(int(img.shape[0]), int(img.shape[1]))], N_LAYERS, swiglu=True)
    if enc.status() != dv.OK:
        raise RuntimeError("device status after the official variant")
    enc.close()
    return {"variant": "RMSNorm, SwiGLU (4096 gate + 4096 up), half-vector RoPE pairing, [-1, 1] pixels",
            "image": [int(img.shape[0]), int(img.shape[1])], "layers": N_LAYERS, "tokens": N_TOK,
            "ms_per_encode": round(sec * 1e3, 4), "tokens_per_s": round(N_TOK / sec, 1),
            "tflops": round(fl / sec / 1e12, 1), "frac_of_peak": round(fl / sec / 1e12 / pk["tc"], 3)}


def other_workloads(dw, cfg, pk, reps: int = 5):
    """images/s, merged tokens/s and the fraction of the bf16 peak on the other
    synthetic workloads (CUDA events around the encode only): one stream, and
    (except the aspect-ratio workload, whose protocol is one stream) two
    encodes in flight on two streams, issued eagerly and replayed from CUDA
    graphs recorded once per stream."""
    import torch

    import workloads as WL
    import vit_vision_encoder_gb300 as dv
    res = {}
    for name in ("tiny", "min", "batch16", "aspect"):
        wl = WL.WORKLOADS[name]
        enc = dv.Encoder(dw, cfg, n_layers=wl["n_layers"])
        imgs = [torch.from_numpy(im).cuda() for im in WL.workload_images(name)]
        sizes = [(int(im.shape[0]), int(im.shape[1])) for im in imgs]
        T = enc.tokens(sizes)
        out = torch.empty((T, 5120), dtype=torch.bfloat16, device="cuda")
        runs = wl.get("repeats", reps)
        for _ in range(2):
            enc.encode(imgs, out=out)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(runs + 1)]
        ev[0].record()
        for r in range(runs):
            enc.encode(imgs, out=out)
            ev[r + 1].record()
        torch.cuda.synchronize()
        per = [ev[r].elapsed_time(ev[r + 1]) / 1e3 for r in range(runs)]
        # the 8-run protocol of the aspect-ratio workload reports runs 2..8
        sec = statistics.mean(per[1:] if name == "aspect" else per)
        fl = encode_flop(sizes, wl["n_layers"])
        res[name] = {"images": len(imgs), "layers": wl["n_layers"], "tokens": T,
                     "ms_per_encode": round(sec * 1e3, 4), "images_per_s": round(len(imgs) / sec, 2),
                     "tokens_per_s": round(T / sec, 1), "tflops": round(fl / sec / 1e12, 1),
                     "frac_of_peak": round(fl / sec / 1e12 / pk["tc"], 3)}
        if name != "aspect":
            # The same encodes alternating between two streams (own workspace
            # and output each), as the headline step runs; the aspect-ratio
            # workload's protocol is one stream.
            enc_b = dv.Encoder(dw, cfg, n_layers=wl["n_layers"])
            encs, outs = (enc, enc_b), (out, torch.empty_like(out))
            streams = [torch.cuda.Stream(), torch.cuda.Stream()]

            def two(n):
                cur = torch.cuda.current_stream()
                for st in streams:
                    st.wait_stream(cur)
                for i in range(n):
                    with torch.cuda.stream(streams[i % 2]):
                        encs[i % 2].encode(imgs, out=outs[i % 2])
                for st in streams:
                    cur.wait_stream(st)

            two(2)
            torch.cuda.synchronize()
            n2 = 2 * runs
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            two(n2)
            e1.record()
            torch.cuda.synchronize()
            sec2 = e0.elapsed_time(e1) / 1e3 / n2
            res[name]["two_streams"] = {"ms_per_encode": round(sec2 * 1e3, 4), "tokens_per_s": round(T / sec2, 1),
                                        "frac_of_peak": round(fl / sec2 / 1e12 / pk["tc"], 3)}
            # The same, each stream's encode recorded once as a CUDA graph and
            # replayed (its own input copy, workspace and output).
            imgs_b = [im.clone() for im in imgs]
            graphs = [encs[0].graph(imgs, out=outs[0])[0], encs[1].graph(imgs_b, out=outs[1])[0]]

            def two_graph(n):
                cur = torch.cuda.current_stream()
                for st in streams:
                    st.wait_stream(cur)
                for i in range(n):
                    graphs[i % 2].launch(streams[i % 2])
                for st in streams:
                    cur.wait_stream(st)

            two_graph(2)
            torch.cuda.synchronize()
            e0.record()
            two_graph(n2)
            e1.record()
            torch.cuda.synchronize()
            sec3 = e0.elapsed_time(e1) / 1e3 / n2
            res[name]["two_streams_graph"] = {"ms_per_encode": round(sec3 * 1e3, 4),
                                              "tokens_per_s": round(T / sec3, 1),
                                              "frac_of_peak": round(fl / sec3 / 1e12 / pk["tc"], 3)}
            for g in graphs:
                g.close()
            if enc_b.status() != dv.OK:
                raise RuntimeError(f"device status after {name} (second stream)")
            enc_b.close()
        if enc.status() != dv.OK:
            raise RuntimeError(f"device status after {name}")
        enc.close()
    return res


def preprocess_workloads(pk, reps: int = 20):
    """The preprocessing step (plan, contain resize, gray canvas) on images off
    the patch grid: CUDA-event time per image (median of `reps`, after warm-up)
    of the call captured in a CUDA graph (the device's time: tables, both
    passes) and issued eagerly (host planning included), and the algorithmic
    bytes (input read once, intermediate written and read once when the width
    changes, canvas written once) against the measured HBM copy bandwidth."""
    import torch

    import workloads as WL
    import vit_vision_encoder_gb300 as dv

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        per = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(per)

    res = {}
    for name, (H, W, kind, seed) in WL.PREPROCESS_WORKLOADS.items():
        img = torch.from_numpy(WL.make_image(H, W, kind, seed)).cuda()
        canvas, plan = dv.preprocess(img)
        run = lambda: dv.preprocess(img, canvas=canvas)
        eager = timed(run)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        sec = timed(g.replay)
        nbytes = H * W * 3 + plan["Hc"] * plan["Wc"] * 3
        if plan["Wr"] != W:
            nbytes += 2 * H * plan["Wr"] * 3
        res[name] = {"input": [H, W], "grid": [plan["h"], plan["w"]], "canvas": [plan["Hc"], plan["Wc"]],
                     "resized": [plan["Hr"], plan["Wr"]], "ms": round(sec * 1e3, 4),
                     "algorithmic_bytes": nbytes, "gb_per_s": round(nbytes / sec / 1e9, 1),
                     "frac_of_hbm": round(nbytes / sec / 1e9 / pk["hbm"], 3),
                     "timing": "CUDA graph of the call (coefficient tables included)",
                     "eager_ms": round(eager * 1e3, 4),
                     "eager_frac_of_hbm": round(nbytes / eager / 1e9 / pk["hbm"], 3)}
    return res


def overlay_chunk_timing(pk, chunk_rows: int = 2048, reps: int = 20):
    """Chunked-prefill overlay of the 16-image batch prompt (16384 x 5120, 16
    spans, 6436 span rows) in chunks of `chunk_rows`, with the row-type mask:
    CUDA-event time for all chunks (median of `reps`) and algorithmic bytes
    (each span row read once and written once, one mask byte per prompt row)."""
    import numpy as np
    import torch

    import oracle as O
    import workloads as WL
    import vit_vision_encoder_gb300 as dv
    sizes = [(H, W) for H, W, _, _ in WL.WORKLOADS["batch16"]["images"]]
    rows = [len(O.layout(H // 14, W // 14, 1)[0]) for H, W in sizes]
    ntok = [((H // 14 + 2) // 3) * ((W // 14 + 2) // 3) for H, W in sizes]
    bases = WL.span_bases("batch16", rows)
    eoff = np.concatenate([[0], np.cumsum(ntok)])
    spans = [(bases[i], H // 14, W // 14, int(eoff[i])) for i, (H, W) in enumerate(sizes)]
    hidden = torch.randn((16384, 5120), device="cuda").to(torch.bfloat16)
    emb = torch.randn((int(eoff[-1]), 5120), device="cuda").to(torch.bfloat16)
    sent = torch.randn((3, 5120), device="cuda").to(torch.bfloat16)
    mask = torch.empty(16384, dtype=torch.uint8, device="cuda")
    chunks = [(a, min(a + chunk_rows, 16384)) for a in range(0, 16384, chunk_rows)]

    def run():
        for a, b in chunks:
            dv.overlay_chunk(hidden[a:b], a, spans, emb, sent, row_type=mask[a:b])

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        per = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(per)

    eager = timed(run)
    # The same calls captured once in a CUDA graph and replayed (how a prefill
    # loop that owns a graph would issue them): the launches no longer wait on
    # the host.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    sec = timed(g.replay)
    nbytes = sum(rows) * 5120 * 2 * 2 + 16384
    return {"prompt_rows": 16384, "span_rows": sum(rows), "chunk_rows": chunk_rows, "chunks": len(chunks),
            "ms": round(sec * 1e3, 4), "algorithmic_bytes": nbytes, "gb_per_s": round(nbytes / sec / 1e9, 1),
            "frac_of_hbm": round(nbytes / sec / 1e9 / pk["hbm"], 3), "timing": "CUDA graph of the chunk calls",
            "eager_ms": round(eager * 1e3, 4),
            "eager_frac_of_hbm": round(nbytes / eager / 1e9 / pk["hbm"], 3)}


def run_profile_case(case: str):
    """A bounded case for ncu (run it with --profile-from-start off): warm-up
    launches, then exactly the launches of interest between
    cudaProfilerStart/Stop."""
    import numpy as np
    import torch

    import workloads as WL
    import vit_vision_encoder_gb300 as dv
    torch.cuda.set_device(0)
    rng = np.random.default_rng(0)
    if case in ("encode", "min-encode"):
        # The 1344x1344 image, or the 546x546 one (1521 patches, 169 tokens).
        W = WL.make_weights(N_LAYERS)
        enc = dv.Encoder(dv.weights_to_device(W), WL.MODEL)
        name = WORKLOAD if case == "encode" else "min"
        img = torch.from_numpy(WL.workload_images(name)[0]).cuda()
        T = enc.tokens([(int(img.shape[0]), int(img.shape[1]))])
        out = torch.empty((T, 5120), dtype=torch.bfloat16, device="cuda")
        run = lambda: enc.encode([img], out=out)
    elif case == "overlay":
        # One 1,058-row span into the 4096 x 5120 prompt at the seeded base.
        hidden = torch.from_numpy(WL.hidden_buffer(4096, 5120, WL.WORKLOADS[WORKLOAD]["hidden_seed"])
                                  .view(np.int16)).cuda().view(torch.bfloat16)
        emb = torch.randn((N_TOK, 5120), device="cuda").to(torch.bfloat16)
        sent = torch.randn((3, 5120), device="cuda").to(torch.bfloat16)
        n_rows = len(dv.layout(GH, GW, WL.MODEL["image_token_id"])[0])
        base = WL.span_bases(WORKLOAD, [n_rows])[0]
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

        def run():
            flush.zero_()                   # evict L2 so the counters see DRAM traffic
            dv.overlay(hidden, [(base, GH, GW, 0)], emb, sent)
    elif case == "attention":
        qkv = torch.from_numpy(WL.to_bf16_bits(rng.standard_normal((N_PATCH, 3072), dtype=np.float32))
                               .view(np.int16)).cuda().view(torch.bfloat16)
        o = torch.empty((N_PATCH, 1024), dtype=torch.bfloat16, device="cuda")
        run = lambda: dv.op_attention(qkv, [N_PATCH], out=o)
    elif case in ("qwen-encode", "qwen-attention"):
        cfg = WL.QWEN_MODEL
        n_layers = cfg["n_layers"] if case == "qwen-encode" else 1
        Wq = WL.make_weights_qwen(n_layers)
        enc = dv.QwenEncoder(dv.weights_to_device(Wq), cfg)
        img = torch.from_numpy(WL.uniform_image(1024, 1024, seed=8)).cuda()
        out = torch.empty((1024, 5120), dtype=torch.bfloat16, device="cuda")
        run = lambda: enc.encode(img, out=out)
    elif case == "preprocess":
        # The 3024 x 4032 photo: tables, horizontal and vertical passes.
        H, W, kind, seed = WL.PREPROCESS_WORKLOADS["photo"]
        img = torch.from_numpy(WL.make_image(H, W, kind, seed)).cuda()
        canvas, _ = dv.preprocess(img)
        run = lambda: dv.preprocess(img, canvas=canvas)
    elif case.startswith("gemm-"):
        K, N, epi = {"gemm-qkv": (1024, 3072, dv.EPI_BIAS), "gemm-fc1": (1024, 4096, dv.EPI_BIAS_GELU),
                     "gemm-fc2": (4096, 1024, dv.EPI_BIAS_RESID),
                     "gemm-proj": (1024, 1024, dv.EPI_BIAS_RESID)}[case]
        a = torch.randn((N_PATCH, K), device="cuda").to(torch.bfloat16)
        w = (torch.randn((N, K), device="cuda") * 0.02).to(torch.bfloat16)
        b = torch.zeros(N, device="cuda").to(torch.bfloat16)
        o = torch.zeros((N_PATCH, N), device="cuda").to(torch.bfloat16)
        run = lambda: dv.op_linear(a, w, b, epi, out=o)
    else:
        raise SystemExit(f"unknown profile case {case}")
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    run()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    print(f"profile case {case} done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-workloads", action="store_true",
                    help="do not time the other synthetic workloads")
    ap.add_argument("--profile", default=None,
                    help="run one bounded case for ncu instead of the benchmark")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.profile:
        return run_profile_case(args.profile)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    import workloads as WL
    import vit_vision_encoder_gb300 as dv

    cfg = WL.MODEL
    W = WL.make_weights(N_LAYERS)
    dw = dv.weights_to_device(W)
    enc = dv.Encoder(dw, cfg)
    img_np = WL.workload_images(WORKLOAD)[0]
    img = torch.from_numpy(img_np).cuda()
    out = torch.empty((N_TOK, 5120), dtype=torch.bfloat16, device="cuda")
    hidden = torch.from_numpy(WL.hidden_buffer(4096, 5120, WL.WORKLOADS[WORKLOAD]["hidden_seed"])
                              .view(np.int16)).cuda().view(torch.bfloat16)
    sentinel = dw["sentinel"]
    n_rows = len(dv.layout(GH, GW, cfg["image_token_id"])[0])
    base = WL.span_bases(WORKLOAD, [n_rows])[0]

    def step():
        enc.encode([img], out=out)
        dv.layout(GH, GW, cfg["image_token_id"], base)
        dv.overlay(hidden, [(base, GH, GW, 0)], out, sentinel)

    # Throughput steps alternate between two streams, each with its own encoder
    # workspace, output and prompt buffer, so one encode's sparse start and end
    # (patch projection, merger, overlay) overlap the other's kernels, as a
    # server would run consecutive requests.
    enc_b = dv.Encoder(dw, cfg)
    encs = (enc, enc_b)
    outs = (out, torch.empty_like(out))
    hiddens = (hidden, hidden.clone())
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def steps2(n):
        cur = torch.cuda.current_stream()
        for st in streams:
            st.wait_stream(cur)
        for i in range(n):
            with torch.cuda.stream(streams[i % 2]):
                encs[i % 2].encode([img], out=outs[i % 2])
                dv.layout(GH, GW, cfg["image_token_id"], base)
                dv.overlay(hiddens[i % 2], [(base, GH, GW, 0)], outs[i % 2], sentinel)
        for st in streams:
            cur.wait_stream(st)

    # The same steps with each stream's encode recorded once as a CUDA graph
    # (ds_vit_graph_create) on its own input, workspace and output, and
    # replayed: every replay runs every kernel of the encode; only the host's
    # launch calls are saved.  The overlay is launched directly each step.
    imgs_g = (img, img.clone())
    graphs = [encs[i].graph([imgs_g[i]], out=outs[i])[0] for i in range(2)]

    def steps2_graph(n):
        cur = torch.cuda.current_stream()
        for st in streams:
            st.wait_stream(cur)
        for i in range(n):
            with torch.cuda.stream(streams[i % 2]):
                graphs[i % 2].launch(streams[i % 2])
                dv.layout(GH, GW, cfg["image_token_id"], base)
                dv.overlay(hiddens[i % 2], [(base, GH, GW, 0)], outs[i % 2], sentinel)
        for st in streams:
            cur.wait_stream(st)

    for _ in range(args.warmup):
        step()
    steps2(2)
    steps2_graph(max(args.warmup, 2))
    torch.cuda.synchronize()

    # CUDA events around every kernel launch of every timed step.
    per = LAUNCHES_PER_ENCODE
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * per * args.steps)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    ev_arr = (C.c_void_p * len(evs))(*[e.cuda_event for e in evs])
    kinds = (C.c_int32 * (per * args.steps))()
    counts = (C.c_int32 * args.steps)()

    # Timed region 1 (the value): K steps, nothing else on the stream.
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    steps2_graph(args.steps)
    t1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed = t0.elapsed_time(t1) / 1e3
    clk = clocks.stop()

    # The same K steps issued eagerly (every kernel launched from the host).
    torch.cuda.synchronize()
    t0.record()
    steps2(args.steps)
    t1.record()
    torch.cuda.synchronize()
    eager_elapsed = t0.elapsed_time(t1) / 1e3

    # Timed region 2 (per-kernel times, the roofline): the same K steps with CUDA
    # events recorded around every kernel launch on the encode's stream.
    torch.cuda.synchronize()
    for s in range(args.steps):
        ev_ptr = C.cast(C.byref(ev_arr, s * 2 * per * C.sizeof(C.c_void_p)), C.POINTER(C.c_void_p))
        kind_ptr = C.cast(C.byref(kinds, s * per * 4), C.POINTER(C.c_int32))
        cnt_ptr = C.cast(C.byref(counts, s * 4), C.POINTER(C.c_int32))
        dv.check(dv.lib.ds_vit_set_kernel_timer(enc.handle, ev_ptr, kind_ptr, per, cnt_ptr),
                 "ds_vit_set_kernel_timer")
        step()
    torch.cuda.synchronize()
    enc.detach_timer()
    for e in encs:
        if e.status() != dv.OK:
            raise RuntimeError(f"device status {e.status()}")

    per_kind = {}
    n_launch = 0
    for s in range(args.steps):
        for i in range(counts[s]):
            k = KIND_NAMES[kinds[s * per + i]]
            ms = evs[2 * (s * per + i)].elapsed_time(evs[2 * (s * per + i) + 1])
            d = per_kind.setdefault(k, [0.0, 0])
            d[0] += ms
            d[1] += 1
            n_launch += 1
    n_launch += args.steps          # one overlay launch per step
    n_launch //= args.steps         # launches per timed step (both regions run the same steps)
    gpu_launches = n_launch * args.steps

    tmax, value = aggregate(elapsed, N_TOK * args.steps, world)
    eager_tmax, eager_value = aggregate(eager_elapsed, N_TOK * args.steps, world)

    # End to end through the host-buffer entry point: pinned pixels in, pinned
    # embeddings out, both copies inside the timed region.  Steps alternate
    # between two streams, each with its own encoder workspace and host
    # buffers, so one step's copies overlap the other's kernels (as a server
    # would run consecutive requests).
    hins = [torch.from_numpy(img_np).pin_memory() for _ in range(2)]
    houts = [torch.empty((N_TOK, 5120), dtype=torch.bfloat16).pin_memory() for _ in range(2)]

    # Each stream's host-buffer encode recorded once as a CUDA graph
    # (ds_vit_graph_create with host = 1): every replay copies the pixels in,
    # encodes and copies the embeddings out.
    hgraphs = [encs[i].graph_host([hins[i]], houts[i])[0] for i in range(2)]

    def e2e_steps(n):
        cur = torch.cuda.current_stream()
        for st in streams:
            st.wait_stream(cur)
        for i in range(n):
            with torch.cuda.stream(streams[i % 2]):
                hgraphs[i % 2].launch(streams[i % 2])
            dv.layout(GH, GW, cfg["image_token_id"], base)
        for st in streams:
            cur.wait_stream(st)

    def e2e_steps_eager(n):
        cur = torch.cuda.current_stream()
        for st in streams:
            st.wait_stream(cur)
        for i in range(n):
            with torch.cuda.stream(streams[i % 2]):
                encs[i % 2].encode_host([hins[i % 2]], houts[i % 2])
            dv.layout(GH, GW, cfg["image_token_id"], base)
        for st in streams:
            cur.wait_stream(st)

    e2e_steps(max(args.warmup, 2))
    e2e_steps_eager(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(args.steps)
    e1.record()
    torch.cuda.synchronize()
    e2e_sec = e0.elapsed_time(e1) / 1e3
    # The same K host-buffer steps issued eagerly (ds_vit_encode_batch_host per step).
    e0.record()
    e2e_steps_eager(args.steps)
    e1.record()
    torch.cuda.synchronize()
    e2e_eager_sec = e0.elapsed_time(e1) / 1e3
    for e in encs:
        if e.status() != dv.OK:
            raise RuntimeError(f"device status {e.status()}")
    for g in graphs + hgraphs:
        g.close()
    enc_b.close()
    _, e2e_value = aggregate(e2e_sec, N_TOK * args.steps, world)
    _, e2e_eager_value = aggregate(e2e_eager_sec, N_TOK * args.steps, world)

    pk = peaks()
    pk["tc"], pk["tc_label"] = tensor_peak(pk, clk)
    attn_ms, attn_n = per_kind["attention"]
    attn_tflops = KIND_FLOP["attention"] / (attn_ms / attn_n / 1e3) / 1e12
    kernels = {}
    for k, (ms, n) in per_kind.items():
        d = {"launches_per_step": n / args.steps, "ms_per_step": round(ms / args.steps, 4)}
        if k in KIND_FLOP:
            d["tflops"] = round(KIND_FLOP[k] * n / (ms / 1e3) / 1e12, 1)
            d["frac_of_peak"] = round(d["tflops"] / pk["tc"], 3)
        kernels[k] = d
    ms_step = tmax / args.steps * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "1344x1344 uint8 uniform (seed 3) -> 96x96 = 9216 patches, 32-layer ViT "
                               "(hidden 1024, 16x64 heads, MLP 4096), 3x3 merge -> 1024 tokens x 5120, "
                               "layout (1058 rows) + overlay into a 4096x5120 prompt buffer",
                   "images_per_step": 1, "parallelism": f"replicas x{world}",
                   "streams": "steps alternate between two streams (own workspace, output and prompt "
                              "buffer each), so consecutive encodes overlap; per-kernel times and the "
                              "roofline come from a single-stream pass",
                   "launch": "each stream's encode recorded once as a CUDA graph (ds_vit_graph_create) "
                             "and replayed every step (all kernels run each replay); the overlay is "
                             "launched directly; the same steps issued eagerly are under 'eager'",
                   "l2": "no flush: per-step working set above L2 (0.95 GB of weights streamed per "
                         "step, 189 MB of activations; L2 129 MB)",
                   "weights": "random N(0,0.02), seed 1000"},
        "images_per_s": value / N_TOK,
        "encode_tflops": ENCODE_FLOP / (ms_step / 1e3) / 1e12,
        "encode_tc_peak_frac": ENCODE_FLOP / (ms_step / 1e3) / 1e12 / pk["tc"],
        "roofline": {"bound": "tensor", "kernel": "attention", "achieved": attn_tflops,
                     "peak": pk["tc"], "unit": "TFLOP/s", "frac": attn_tflops / pk["tc"],
                     "peak_kind": pk["tc_label"],
                     "frac_of_burst": attn_tflops / pk["bf16"], "frac_of_sustained": attn_tflops / pk["bf16_sus"],
                     "flop_per_launch": KIND_FLOP["attention"], "traffic": measured_traffic()},
        "kernels": kernels,
        "eager": {"value": eager_value, "ms_per_step": eager_tmax / args.steps * 1e3,
                  "launch": "every kernel launched from the host (ds_vit_encode_batch per step)"},
        "gpu_launches": gpu_launches,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": IMG_H * IMG_W * 3,
                "d2h_bytes_per_step": N_TOK * 5120 * 2,
                "api": "ds_vit_encode_batch_host (pinned pixels in, pinned embeddings out) recorded once per "
                       "stream as a CUDA graph (ds_vit_graph_create, host = 1; both copies and the encode in "
                       "every replay) + ds_vit_layout; steps alternate between two streams, each with its "
                       "own workspace",
                "eager_value": e2e_eager_value,
                "eager_api": "ds_vit_encode_batch_host called every step (same buffers, streams and copies)"},
        "clocks": clk,
    }
    if not args.skip_workloads:
        line["workloads"] = other_workloads(dw, cfg, pk)
        line["preprocess"] = preprocess_workloads(pk)
        line["overlay_chunks"] = overlay_chunk_timing(pk)
        line["official_variant"] = official_workload(pk)
        line["qwen_tower"] = qwen_workload(pk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
        if "workloads" in line:
            for name, d in oracle_timings().items():
                line["workloads"][name]["oracle"] = d
    if rank == 0:
        print(json.dumps(line), flush=True)
    enc.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
