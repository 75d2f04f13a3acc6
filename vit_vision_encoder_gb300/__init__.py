"""Python binding of libdsvit (the GB300 vision-tower encode), via ctypes.

Argument marshalling only: every step of the encode runs in the library's
CUDA kernels.  PyTorch supplies device memory (tensors) and the current
stream.  Importing this package loads ``libdsvit.so`` and raises if it is
missing (build it with ``__graft_entry__.build()``); there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsvit.so")

OK, EINVAL, ERANGE, ECAP, ECUDA, ETIMEOUT, ENOMEM = 0, -1, -2, -3, -4, -5, -6
TOK_START, TOK_IMAGE, TOK_NEWLINE, TOK_END = 0, 1, 2, 3
EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESID, EPI_QKV_ROPE, EPI_SWIGLU = 0, 1, 2, 3, 4
MAX_LAYERS, MAX_IMAGES, MAX_PATCHES, MAX_TOKENS = 32, 64, 9216, 1024
NOALLOC_MAX_PATCHES, NOALLOC_SCRATCH_BYTES = 1024, 21 * 1024 * 1024


class DsVitError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib.ds_vit_strerror(code).decode()} ({code})")


class Config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("heads", C.c_int32),
                ("head_dim", C.c_int32), ("mlp", C.c_int32), ("out_dim", C.c_int32),
                ("patch", C.c_int32), ("merge", C.c_int32), ("rope_theta", C.c_float),
                ("ln_eps", C.c_float), ("mean", C.c_float * 3), ("std", C.c_float * 3),
                ("image_token_id", C.c_int32), ("norm_kind", C.c_int32), ("mlp_kind", C.c_int32),
                ("rope_pairing", C.c_int32)]


LAYER_FIELDS = ("ln1_g", "ln1_b", "qkv_w", "qkv_b", "proj_w", "proj_b",
                "ln2_g", "ln2_b", "fc1_w", "fc1_b", "fc2_w", "fc2_b")


class LayerWeights(C.Structure):
    _fields_ = [(f, C.c_void_p) for f in LAYER_FIELDS]


class Weights(C.Structure):
    _fields_ = ([("patch_w", C.c_void_p), ("patch_b", C.c_void_p),
                 ("layers", LayerWeights * MAX_LAYERS)]
                + [(f, C.c_void_p) for f in ("lnm_g", "lnm_b", "m1_w", "m1_b", "m2_w", "m2_b",
                                              "sentinel")])


class Span(C.Structure):
    _fields_ = [("base_row", C.c_int64), ("gh", C.c_int32), ("gw", C.c_int32),
                ("embed_row", C.c_int64)]


MERGER_FIELDS = ("ln_g", "ln_b", "w1", "b1", "w2", "b2")


class QwenMerger(C.Structure):
    _fields_ = [(f, C.c_void_p) for f in MERGER_FIELDS]


class QwenWeights(C.Structure):
    _fields_ = ([("patch_w", C.c_void_p), ("patch_b", C.c_void_p), ("pos_table", C.c_void_p),
                 ("layers", LayerWeights * MAX_LAYERS), ("merger", QwenMerger),
                 ("deepstack", QwenMerger * 3)])


class Plan(C.Structure):
    _fields_ = [(f, C.c_int32) for f in ("H", "W", "h", "w", "Hc", "Wc", "Hr", "Wr", "y0", "x0")]


# Every symbol include/dsvit.h declares: name -> (restype, argtypes).
_VP, _I32, _I64, _SZ, _F = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float
_P_I32, _P_I64 = C.POINTER(C.c_int32), C.POINTER(C.c_int64)
SIGNATURES = {
    "ds_vit_strerror": (C.c_char_p, [C.c_int]),
    "ds_vit_prepare": (C.c_int, [C.POINTER(Config), C.POINTER(Weights), C.POINTER(_VP), _VP]),
    "ds_vit_release": (C.c_int, [_VP]),
    "ds_vit_layout": (C.c_int, [_I32, _I32, _I32, _I32, _VP, _VP, _VP, _VP, _I64, _P_I64]),
    "ds_vit_workspace_bytes": (C.c_int, [_VP, C.c_int, _P_I32, _P_I32, C.POINTER(_SZ)]),
    "ds_vit_workspace_bytes_host": (C.c_int, [_VP, C.c_int, _P_I32, _P_I32, C.POINTER(_SZ)]),
    "ds_vit_encode_batch": (C.c_int, [_VP, C.c_int, C.POINTER(_VP), _P_I32, _P_I32, _VP, _P_I64,
                                      _VP, _SZ, _VP]),
    "ds_vit_encode": (C.c_int, [_VP, _VP, _I32, _I32, _VP, _VP, _SZ, _VP]),
    "ds_vit_encode_noalloc": (C.c_int, [_VP, _VP, _I32, _I32, _VP, _VP]),
    "ds_vit_encode_batch_host": (C.c_int, [_VP, C.c_int, C.POINTER(_VP), _P_I32, _P_I32, _VP,
                                           _P_I64, _VP, _SZ, _VP]),
    "ds_vit_encode_debug": (C.c_int, [_VP, C.c_int, C.POINTER(_VP), _P_I32, _P_I32, _VP, _P_I64,
                                      _VP, _SZ, _VP, _VP, _VP]),
    "ds_vit_graph_create": (C.c_int, [_VP, C.c_int, C.c_int, C.POINTER(_VP), _P_I32, _P_I32, _VP, _P_I64,
                                      _VP, _SZ, C.POINTER(_VP)]),
    "ds_vit_graph_launch": (C.c_int, [_VP, _VP]),
    "ds_vit_graph_destroy": (C.c_int, [_VP]),
    "ds_vit_overlay": (C.c_int, [_VP, _I64, _I32, C.POINTER(Span), C.c_int, _VP, _I64, _VP, _VP]),
    "ds_vit_overlay_rows": (C.c_int, [_VP, _I64, _I32, _VP, _VP, _VP, _I64, _VP, _I64, _VP, _VP, _VP]),
    "ds_vit_overlay_chunk": (C.c_int, [_VP, _I64, _I64, _I32, C.POINTER(Span), C.c_int, _VP, _I64, _VP,
                                       _VP, _VP]),
    "ds_vit_device_status": (C.c_int, [_VP, _VP]),
    "ds_vit_selftest_wait_timeout": (C.c_int, [_VP, _VP, C.c_uint32, _VP]),
    "ds_vit_set_kernel_timer": (C.c_int, [_VP, C.POINTER(_VP), _P_I32, _I32, _P_I32]),
    "ds_vit_op_layernorm": (C.c_int, [_VP, _VP, _VP, _VP, _I64, _F, _VP]),
    "ds_vit_op_rmsnorm": (C.c_int, [_VP, _VP, _VP, _I64, _F, _VP]),
    "ds_vit_op_linear": (C.c_int, [_VP, _I64, _I32, _VP, _I32, _VP, _VP, _I32, _VP, _VP, _VP, _VP]),
    "ds_vit_op_rope_table": (C.c_int, [_VP, _I32, _F, _VP]),
    "ds_vit_op_attention": (C.c_int, [_VP, _P_I32, C.c_int, _VP, _VP, _VP]),
    "ds_vit_plan_image": (C.c_int, [_I32, _I32, C.POINTER(Plan)]),
    "ds_vit_qwen_prepare": (C.c_int, [C.POINTER(Config), C.POINTER(QwenWeights), C.POINTER(_VP), _VP]),
    "ds_vit_qwen_release": (C.c_int, [_VP]),
    "ds_vit_qwen_workspace_bytes": (C.c_int, [_I32, _I32, C.POINTER(_SZ)]),
    "ds_vit_qwen_encode": (C.c_int, [_VP, _VP, _I32, _I32, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "ds_vit_qwen_layout": (C.c_int, [_I32, _I32, _I32, _VP, _I64, _P_I32]),
    "ds_vit_preprocess_workspace_bytes": (C.c_int, [C.POINTER(Plan), C.POINTER(_SZ)]),
    "ds_vit_preprocess": (C.c_int, [C.POINTER(Plan), _VP, _VP, _VP, _SZ, _VP]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    h = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(h, name)
        fn.restype, fn.argtypes = res, args
    return h


lib = _load()


def check(rc: int, where: str) -> None:
    if rc != OK:
        raise DsVitError(rc, where)


def _i32(vals):
    return (C.c_int32 * len(vals))(*[int(v) for v in vals])


# ---------------------------------------------------------------- host-only

def layout(gh: int, gw: int, image_token_id: int, base_pos: int = 0):
    """Token span of one image: (ids, pos, type, src) numpy arrays (host call)."""
    n = C.c_int64(0)
    lib.ds_vit_layout(gh, gw, image_token_id, base_pos, None, None, None, None, 0, C.byref(n))
    ids = np.empty(n.value, np.int32)
    pos = np.empty(n.value, np.int32)
    typ = np.empty(n.value, np.uint8)
    src = np.empty(n.value, np.int32)
    check(lib.ds_vit_layout(gh, gw, image_token_id, base_pos, ids.ctypes.data, pos.ctypes.data,
                            typ.ctypes.data, src.ctypes.data, n.value, C.byref(n)), "ds_vit_layout")
    return ids, pos, typ, src


def make_config(model: dict, n_layers: int) -> Config:
    c = Config()
    c.n_layers = n_layers
    for k in ("hidden", "heads", "head_dim", "mlp", "out_dim", "patch", "merge", "image_token_id"):
        setattr(c, k, int(model[k]))
    c.rope_theta = float(model["rope_theta"])
    c.ln_eps = float(model["ln_eps"])
    c.mean = (C.c_float * 3)(*model["mean"])
    c.std = (C.c_float * 3)(*model["std"])
    c.norm_kind = {"layernorm": 0, "rmsnorm": 1}[model.get("norm", "layernorm")]
    c.mlp_kind = {"gelu": 0, "swiglu": 1}[model.get("mlp_kind", "gelu")]
    c.rope_pairing = {"axis_halves": 0, "half_vector": 1}[model.get("rope_pairing", "axis_halves")]
    return c


# ---------------------------------------------------------------- torch side

def _torch():
    import torch
    return torch


def _stream():
    return C.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def weights_to_device(w: dict, device="cuda") -> dict:
    """bf16 bit-pattern numpy arrays -> device bf16 tensors (same nesting)."""
    torch = _torch()

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    out = {k: up(v) for k, v in w.items() if k not in ("layers", "merger", "deepstack")}
    out["layers"] = [{k: up(v) for k, v in L.items()} for L in w["layers"]]
    if "merger" in w:
        out["merger"] = {k: up(v) for k, v in w["merger"].items()}
    if "deepstack" in w:
        out["deepstack"] = [{k: up(v) for k, v in M.items()} for M in w["deepstack"]]
    return out


class Encoder:
    """A prepared model (ds_vit_prepare) plus a cached workspace."""

    def __init__(self, dev_weights: dict, model: dict, n_layers: int | None = None):
        n_layers = len(dev_weights["layers"]) if n_layers is None else n_layers
        self.n_layers = n_layers
        self._keep = dev_weights
        self.cfg = make_config(model, n_layers)
        w = Weights()
        for k in ("patch_w", "patch_b", "lnm_g", "lnm_b", "m1_w", "m1_b", "m2_w", "m2_b",
                  "sentinel"):
            setattr(w, k, dev_weights[k].data_ptr())
        for l in range(n_layers):
            for k in LAYER_FIELDS:
                setattr(w.layers[l], k, dev_weights["layers"][l][k].data_ptr())
        self._w = w
        h = C.c_void_p()
        check(lib.ds_vit_prepare(C.byref(self.cfg), C.byref(w), C.byref(h), _stream()),
              "ds_vit_prepare")
        self.handle = h
        self._ws = None
        self._host_ws = None

    def close(self):
        if self.handle:
            lib.ds_vit_release(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, sizes, host=False) -> int:
        H, W = _i32([s[0] for s in sizes]), _i32([s[1] for s in sizes])
        b = C.c_size_t(0)
        fn = lib.ds_vit_workspace_bytes_host if host else lib.ds_vit_workspace_bytes
        check(fn(self.handle, len(sizes), H, W, C.byref(b)), "ds_vit_workspace_bytes")
        return b.value

    def workspace(self, sizes, host=False):
        torch = _torch()
        need = self.workspace_bytes(sizes, host)
        attr = "_host_ws" if host else "_ws"
        ws = getattr(self, attr)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            setattr(self, attr, ws)
        return ws

    @staticmethod
    def tokens(sizes) -> int:
        return sum(-(-(h // 14) // 3) * -(-(w // 14) // 3) for h, w in sizes)

    def encode(self, images, out=None, dump=False):
        """images: list of uint8 CUDA tensors [H, W, 3].  Returns (out [sum T, 5120]
        bf16, tok_offsets int64 numpy [n+1]) and, with dump=True, also
        (blocks [n_layers+1, sum N, 1024], final_norm [sum N, 1024])."""
        torch = _torch()
        sizes = [(int(im.shape[0]), int(im.shape[1])) for im in images]
        n = len(images)
        if out is None:
            out = torch.empty((self.tokens(sizes), 5120), dtype=torch.bfloat16, device="cuda")
        ws = self.workspace(sizes)
        H, W = _i32([s[0] for s in sizes]), _i32([s[1] for s in sizes])
        px = (C.c_void_p * n)(*[im.data_ptr() for im in images])
        offs = (C.c_int64 * (n + 1))()
        if not dump:
            check(lib.ds_vit_encode_batch(self.handle, n, px, H, W, _ptr(out), offs, _ptr(ws),
                                          ws.numel(), _stream()), "ds_vit_encode_batch")
            return out, np.array(offs[:], dtype=np.int64)
        N = sum((h // 14) * (w // 14) for h, w in sizes)
        blocks = torch.empty((self.n_layers + 1, N, 1024), dtype=torch.bfloat16, device="cuda")
        fn = torch.empty((N, 1024), dtype=torch.bfloat16, device="cuda")
        check(lib.ds_vit_encode_debug(self.handle, n, px, H, W, _ptr(out), offs, _ptr(ws),
                                      ws.numel(), _ptr(blocks), _ptr(fn), _stream()),
              "ds_vit_encode_debug")
        return out, np.array(offs[:], dtype=np.int64), blocks, fn

    def encode_host(self, images_host, out_host):
        """images_host: list of (pinned) uint8 CPU tensors; out_host: CPU bf16 tensor
        [sum T, 5120].  Copies in, encodes, copies out on the current stream."""
        sizes = [(int(im.shape[0]), int(im.shape[1])) for im in images_host]
        n = len(sizes)
        ws = self.workspace(sizes, host=True)
        H, W = _i32([s[0] for s in sizes]), _i32([s[1] for s in sizes])
        px = (C.c_void_p * n)(*[im.data_ptr() for im in images_host])
        offs = (C.c_int64 * (n + 1))()
        check(lib.ds_vit_encode_batch_host(self.handle, n, px, H, W, _ptr(out_host), offs,
                                           _ptr(ws), ws.numel(), _stream()),
              "ds_vit_encode_batch_host")
        return np.array(offs[:], dtype=np.int64)

    def graph(self, images, out=None):
        """Record one encode of `images` (uint8 CUDA tensors) into `out` as a
        CUDA graph (ds_vit_graph_create); returns (EncodeGraph, out,
        tok_offsets).  Each launch() repeats the whole encode on these
        buffers, whose contents may change between launches."""
        torch = _torch()
        sizes = [(int(im.shape[0]), int(im.shape[1])) for im in images]
        if out is None:
            out = torch.empty((self.tokens(sizes), 5120), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(self.workspace_bytes(sizes), 16), dtype=torch.uint8, device="cuda")
        return self._record(0, images, sizes, out, ws), out, self._last_offsets

    def graph_host(self, images_host, out_host):
        """As graph(), recording ds_vit_encode_batch_host: page-locked CPU
        images in, page-locked CPU output out, both copies in every launch."""
        torch = _torch()
        sizes = [(int(im.shape[0]), int(im.shape[1])) for im in images_host]
        ws = torch.empty(max(self.workspace_bytes(sizes, host=True), 16), dtype=torch.uint8, device="cuda")
        return self._record(1, images_host, sizes, out_host, ws), self._last_offsets

    def _record(self, host, images, sizes, out, ws):
        n = len(sizes)
        H, W = _i32([s[0] for s in sizes]), _i32([s[1] for s in sizes])
        px = (C.c_void_p * n)(*[im.data_ptr() for im in images])
        offs = (C.c_int64 * (n + 1))()
        h = C.c_void_p()
        check(lib.ds_vit_graph_create(self.handle, host, n, px, H, W, _ptr(out), offs, _ptr(ws), ws.numel(),
                                      C.byref(h)), "ds_vit_graph_create")
        self._last_offsets = np.array(offs[:], dtype=np.int64)
        return EncodeGraph(h, (images, out, ws, self))

    def attach_timer(self, n_slots: int = 512):
        """Bracket every kernel of later encode calls with CUDA events; returns
        a callable giving [(kind, ms), ...] for the latest call (after a sync)."""
        torch = _torch()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_slots)]
        for e in evs:
            e.record()                      # materialise the underlying cudaEvent_t
        torch.cuda.synchronize()
        arr = (C.c_void_p * (2 * n_slots))(*[e.cuda_event for e in evs])
        kinds = (C.c_int32 * n_slots)()
        count = C.c_int32(0)
        check(lib.ds_vit_set_kernel_timer(self.handle, arr, kinds, n_slots, C.byref(count)),
              "ds_vit_set_kernel_timer")
        self._timer = (evs, arr, kinds, count)

        def read():
            n = count.value
            return [(int(kinds[i]), evs[2 * i].elapsed_time(evs[2 * i + 1])) for i in range(n)]
        return read

    def detach_timer(self):
        lib.ds_vit_set_kernel_timer(self.handle, None, None, 0, None)
        self._timer = None

    def status(self) -> int:
        return lib.ds_vit_device_status(self.handle, _stream())


class EncodeGraph:
    """An executable graph of one recorded encode; holds its buffers."""

    def __init__(self, handle, keep):
        self.handle, self._keep = handle, keep

    def launch(self, stream=None):
        torch = _torch()
        st = C.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)
        check(lib.ds_vit_graph_launch(self.handle, st), "ds_vit_graph_launch")

    def close(self):
        if self.handle:
            lib.ds_vit_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class QwenEncoder:
    """The Qwen3-VL-style tower (ds_vit_qwen_prepare) plus a cached workspace."""

    def __init__(self, dev_weights: dict, model: dict, n_layers: int | None = None):
        n_layers = len(dev_weights["layers"]) if n_layers is None else n_layers
        self.n_layers = n_layers
        self._keep = dev_weights
        c = Config()
        c.n_layers = n_layers
        for k in ("hidden", "heads", "head_dim", "mlp", "out_dim", "patch", "merge"):
            setattr(c, k, int(model[k]))
        c.rope_theta, c.ln_eps = float(model["rope_theta"]), float(model["ln_eps"])
        c.mean = (C.c_float * 3)(*model["mean"])
        c.std = (C.c_float * 3)(*model["std"])
        self.cfg = c
        w = QwenWeights()
        for k in ("patch_w", "patch_b", "pos_table"):
            setattr(w, k, dev_weights[k].data_ptr())
        for l in range(n_layers):
            for k in LAYER_FIELDS:
                setattr(w.layers[l], k, dev_weights["layers"][l][k].data_ptr())
        for k in MERGER_FIELDS:
            setattr(w.merger, k, dev_weights["merger"][k].data_ptr())
        for t, M in enumerate(dev_weights.get("deepstack", [])):
            for k in MERGER_FIELDS:
                setattr(w.deepstack[t], k, M[k].data_ptr())
        self._w = w
        h = C.c_void_p()
        check(lib.ds_vit_qwen_prepare(C.byref(c), C.byref(w), C.byref(h), _stream()), "ds_vit_qwen_prepare")
        self.handle = h
        self._ws = None

    def close(self):
        if self.handle:
            lib.ds_vit_qwen_release(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def encode(self, img, out=None, deepstack=True, dump=False):
        """uint8 CUDA tensor [H, W, 3] -> (out [T, 5120], deepstack [3, T, 5120] or
        None, blocks [n_layers + 1, N, 1152] or None)."""
        torch = _torch()
        H, W = int(img.shape[0]), int(img.shape[1])
        nb = C.c_size_t()
        check(lib.ds_vit_qwen_workspace_bytes(H, W, C.byref(nb)), "ds_vit_qwen_workspace_bytes")
        if self._ws is None or self._ws.numel() < nb.value:
            self._ws = torch.empty(int(nb.value), dtype=torch.uint8, device="cuda")
        T, N = (H // 32) * (W // 32), (H // 16) * (W // 16)
        if out is None:
            out = torch.empty((T, 5120), dtype=torch.bfloat16, device="cuda")
        ds = torch.empty((3, T, 5120), dtype=torch.bfloat16, device="cuda") if deepstack else None
        bl = torch.empty((self.n_layers + 1, N, 1152), dtype=torch.bfloat16, device="cuda") if dump else None
        check(lib.ds_vit_qwen_encode(self.handle, _ptr(img), H, W, _ptr(out), _ptr(ds), _ptr(self._ws),
                                     self._ws.numel(), _ptr(bl), _stream()), "ds_vit_qwen_encode")
        return out, ds, bl


def qwen_layout(h: int, w: int, seq_start: int):
    """Three-axis M-RoPE positions [3, h*w + 2] of a Qwen image span and rope_delta."""
    n = h * w + 2
    pos = np.zeros((3, n), dtype=np.int32)
    delta = C.c_int32()
    check(lib.ds_vit_qwen_layout(h, w, seq_start, pos.ctypes.data, pos.size, C.byref(delta)),
          "ds_vit_qwen_layout")
    return pos, int(delta.value)


def plan_image(H: int, W: int) -> dict:
    """Preprocessing plan of an H x W image (host call): grid, canvas, resized
    size and placement (include/dsvit.h, ds_vit_plan_image)."""
    p = Plan()
    check(lib.ds_vit_plan_image(int(H), int(W), C.byref(p)), "ds_vit_plan_image")
    return {f: int(getattr(p, f)) for f, _ in Plan._fields_}


def preprocess(img, canvas=None):
    """uint8 CUDA tensor [H, W, 3] -> (canvas uint8 CUDA tensor [Hc, Wc, 3], plan
    dict): contain-resize with bicubic filtering onto the RGB 127 canvas."""
    torch = _torch()
    H, W = int(img.shape[0]), int(img.shape[1])
    p = Plan()
    check(lib.ds_vit_plan_image(H, W, C.byref(p)), "ds_vit_plan_image")
    nbytes = C.c_size_t()
    check(lib.ds_vit_preprocess_workspace_bytes(C.byref(p), C.byref(nbytes)),
          "ds_vit_preprocess_workspace_bytes")
    ws = torch.empty(max(int(nbytes.value), 256), dtype=torch.uint8, device="cuda")
    if canvas is None:
        canvas = torch.empty((p.Hc, p.Wc, 3), dtype=torch.uint8, device="cuda")
    check(lib.ds_vit_preprocess(C.byref(p), _ptr(img), _ptr(canvas), _ptr(ws), ws.numel(), _stream()),
          "ds_vit_preprocess")
    return canvas, {f: int(getattr(p, f)) for f, _ in Plan._fields_}


def overlay(hidden, spans, embeds, sentinel):
    """spans: list of (base_row, gh, gw, embed_row).  In place on ``hidden``."""
    arr = (Span * len(spans))()
    for i, (b, gh, gw, e) in enumerate(spans):
        arr[i].base_row, arr[i].gh, arr[i].gw, arr[i].embed_row = b, gh, gw, e
    check(lib.ds_vit_overlay(_ptr(hidden), hidden.shape[0], hidden.shape[1], arr, len(spans),
                             _ptr(embeds), embeds.shape[0], _ptr(sentinel), _stream()),
          "ds_vit_overlay")


def overlay_rows(hidden, rows, types, src, embeds, sentinel, status=None):
    """Per-row overlay (ds_vit_overlay_rows), in place on ``hidden``: rows and
    src int32 CUDA tensors [n], types a uint8 CUDA tensor [n].  Entries are
    checked on the device; ``status`` (an int32 CUDA tensor [1], zeroed here
    when not given) receives the first error code.  Returns ``status``."""
    torch = _torch()
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
    check(lib.ds_vit_overlay_rows(_ptr(hidden), hidden.shape[0], hidden.shape[1], _ptr(rows), _ptr(types),
                                  _ptr(src), rows.shape[0], _ptr(embeds), embeds.shape[0], _ptr(sentinel),
                                  _ptr(status), _stream()),
          "ds_vit_overlay_rows")
    return status


def overlay_chunk(chunk, chunk_begin, spans, embeds, sentinel, row_type=None):
    """Chunked prefill: ``chunk`` holds prompt rows chunk_begin.. (in place);
    spans as ``overlay``.  row_type (uint8 CUDA tensor [rows], optional)
    receives 0 for text rows and 1 + the layout type for span rows."""
    arr = (Span * len(spans))()
    for i, (b, gh, gw, e) in enumerate(spans):
        arr[i].base_row, arr[i].gh, arr[i].gw, arr[i].embed_row = b, gh, gw, e
    check(lib.ds_vit_overlay_chunk(_ptr(chunk), int(chunk_begin), chunk.shape[0], chunk.shape[1], arr,
                                   len(spans), _ptr(embeds), embeds.shape[0], _ptr(sentinel),
                                   _ptr(row_type), _stream()),
          "ds_vit_overlay_chunk")
    return row_type


# ---------------------------------------------------------------- single kernels

def selftest_wait_timeout(limit_us: int):
    """Run the device bounded-wait self-test (ds_vit_selftest_wait_timeout);
    returns (status code written by the kernel, nanoseconds it waited)."""
    torch = _torch()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    check(lib.ds_vit_selftest_wait_timeout(_ptr(st), _ptr(el), int(limit_us), _stream()),
          "ds_vit_selftest_wait_timeout")
    torch.cuda.synchronize()
    return int(st.item()), int(el.item())


def op_layernorm(x, g, b, eps=1e-6, out=None):
    torch = _torch()
    y = torch.empty_like(x) if out is None else out
    check(lib.ds_vit_op_layernorm(_ptr(x), _ptr(g), _ptr(b), _ptr(y), x.shape[0], eps, _stream()),
          "ds_vit_op_layernorm")
    return y


def op_rmsnorm(x, g, eps=1e-6, out=None):
    torch = _torch()
    y = torch.empty_like(x) if out is None else out
    check(lib.ds_vit_op_rmsnorm(_ptr(x), _ptr(g), _ptr(y), x.shape[0], eps, _stream()), "ds_vit_op_rmsnorm")
    return y


def op_rope_table(max_pos, theta=10000.0):
    torch = _torch()
    t = torch.empty((max_pos, 32), dtype=torch.float32, device="cuda")
    check(lib.ds_vit_op_rope_table(_ptr(t), max_pos, theta, _stream()), "ds_vit_op_rope_table")
    return t


def op_linear(a, w, bias, epilogue=EPI_BIAS, out=None, rowpos=None, rope_cs=None, status=None):
    torch = _torch()
    M, K = a.shape
    N = w.shape[0]
    if out is None:
        n_out = N // 2 if epilogue == EPI_SWIGLU else N
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    check(lib.ds_vit_op_linear(_ptr(a), M, K, _ptr(w), N, _ptr(bias), _ptr(out), epilogue,
                               _ptr(rowpos), _ptr(rope_cs), _ptr(st), _stream()),
          "ds_vit_op_linear")
    return out, st


def op_attention(qkv, seqlens, out=None, status=None):
    torch = _torch()
    if out is None:
        out = torch.empty((qkv.shape[0], 1024), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    sl = _i32(seqlens)
    check(lib.ds_vit_op_attention(_ptr(qkv), sl, len(seqlens), _ptr(out), _ptr(st), _stream()),
          "ds_vit_op_attention")
    return out, st
