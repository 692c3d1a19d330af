"""Thin Python binding of include/moe_decode.h (ctypes; argument marshalling only).

Every step of the block runs in libmoe_decode.so.  PyTorch supplies device memory and streams.
If the library is missing this module raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import numpy as np
import torch

from . import synth
from .workloads import Shape

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_decode.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_OOM, MOE_ERR_BAD_ID = (
    0, -1, -2, -3, -4, -5)
DTYPE_BF16, DTYPE_F32 = 0, 1
PART_GATE_UP, PART_DOWN = 1, 2
KERNELS_FUSED, KERNELS_SEPARATE, KERNELS_COLUMNS, KERNELS_COLUMNS_AHEAD, KERNELS_POOL = 0, 1, 2, 3, 4
KERNELS_MMA = 5
NOALLOC_MAX_ACT_FLOATS = 65536
_STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA",
           -4: "MOE_ERR_OOM", -5: "MOE_ERR_BAD_ID", -6: "MOE_ERR_TIMEOUT",
           -7: "MOE_ERR_PLAN"}

EXPORTS = ["moe_decode_create", "moe_decode_forward", "moe_decode_get_error", "moe_decode_destroy",
           "moe_decode_routes",
           "moe_decode_forward_noalloc",
           "moe_gemv_bf16",
           "moe_stack_create", "moe_stack_create_chained", "moe_stack_step",
           "moe_stack_step_parts", "moe_stack_step_host",
           "moe_stack_get_error",
           "moe_stack_destroy", "moe_pack_codes", "moe_unpack_codes", "moe_unpack_codes_device",
           "moe_synth_codes", "moe_synth_scales", "moe_synth_biases", "moe_route_invert_device",
           "moe_debug_wait_timeout", "moe_router_topk", "moe_debug_col_pieces",
           "moe_debug_col_plan"]


class MoeError(RuntimeError):
    def __init__(self, fn, rc):
        super().__init__(f"{fn} returned {_STATUS.get(rc, rc)}")
        self.rc = rc


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "din", "dff", "n_experts", "top_k", "max_tokens", "bits_gate", "bits_up", "bits_down",
        "n_shared", "dff_shared", "bits_shared", "shared_gate", "resid_dtype", "out_dtype",
        "kernel_mode")]


class Proj(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("gate", Proj), ("up", Proj), ("down", Proj), ("sh_gate", Proj), ("sh_up", Proj),
                ("sh_down", Proj), ("gate_vec", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None
_timeline = False


def use_timeline_build() -> None:
    """Load libmoe_decode_timeline.so (the column-split kernel records per-CTA, per-layer time
    stamps, read by MoeStack.timeline) instead of the product library.  Call before lib()."""
    global LIB_PATH, _timeline
    with _lock:
        if _lib is not None:
            raise RuntimeError("the library is already loaded")
        LIB_PATH = os.path.join(_HERE, "libmoe_decode_timeline.so")
        _timeline = True


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() or "
                                   "python -m quantized_moe_expert_dequant_gb300.build")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
            sig = {
                "moe_decode_create": [ctypes.POINTER(Config), ctypes.POINTER(LayerWeights),
                                      ctypes.POINTER(vp)],
                "moe_decode_forward": [vp, vp, i32, vp, vp, vp, vp, vp],
                "moe_decode_get_error": [vp, ctypes.POINTER(i32)],
                "moe_decode_routes": [vp, vp, vp, vp],
                "moe_decode_destroy": [vp],
                "moe_decode_forward_noalloc": [ctypes.POINTER(Config), ctypes.POINTER(LayerWeights),
                                               vp, i32, vp, vp, vp, vp, vp, vp],
                "moe_stack_create": [ctypes.POINTER(Config), i32, ctypes.POINTER(LayerWeights),
                                     ctypes.POINTER(vp)],
                "moe_gemv_bf16": [vp, vp, ctypes.c_int64, vp, i32, i32, i32, i32, vp],
                "moe_stack_create_chained": [ctypes.POINTER(Config), i32,
                                             ctypes.POINTER(LayerWeights), vp, ctypes.c_float,
                                             ctypes.POINTER(vp)],
                "moe_stack_step": [vp, vp, i32, vp, vp, vp, vp, vp],
                "moe_stack_step_parts": [vp, i32, vp, i32, vp, vp, vp, vp, vp],
                "moe_stack_step_host": [vp, vp, i32, vp, vp, vp, vp, vp],
                "moe_stack_get_error": [vp, ctypes.POINTER(i32)],
                "moe_stack_destroy": [vp],
                "moe_pack_codes": [vp, i64, i64, i32, vp],
                "moe_unpack_codes": [vp, i64, i64, i32, vp],
                "moe_unpack_codes_device": [vp, i64, i64, i32, vp, vp],
                "moe_synth_codes": [vp, u64, i32, i32, i64, vp],
                "moe_synth_scales": [vp, u64, i32, i32, i64, vp],
                "moe_synth_biases": [vp, vp, u64, i32, i32, i64, i32, vp],
                "moe_route_invert_device": [vp, i32, i32, i32, vp, vp],
                "moe_debug_wait_timeout": [i32, vp, vp, vp],
                "moe_router_topk": [vp, i32, i32, i32, vp, vp, vp],
                "moe_debug_col_pieces": [i32, i32, i32, i32, i32, i32, i32, i32, vp, i32],
                "moe_debug_col_plan": [ctypes.POINTER(Config), i32, i32, vp, vp],
            }
            if _timeline:
                sig["moe_stack_timeline"] = [vp, vp, i64, ctypes.POINTER(i32)]
            for name, args in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = None if name.endswith("_destroy") else ctypes.c_int
            _lib = L
    return _lib


def check(fn: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def config(shape: Shape, max_tokens: int = 1, resid_dtype: int = DTYPE_BF16,
           out_dtype: int = DTYPE_F32, kernel_mode: int = KERNELS_FUSED) -> Config:
    return Config(shape.din, shape.dff, shape.n_experts, shape.top_k, max_tokens, shape.bits_gate,
                  shape.bits_up, shape.bits_down, shape.n_shared, shape.dff_shared,
                  shape.bits_shared, shape.shared_gate, resid_dtype, out_dtype, kernel_mode)


# ---------------------------------------------------------------- device weights

@dataclasses.dataclass
class DeviceProj:
    codes: torch.Tensor   # uint8 [E, rows, rowbytes]
    scales: torch.Tensor  # fp16 [E, rows, cols/64]
    biases: torch.Tensor  # fp16 [E, rows, cols/64]

    def struct(self) -> Proj:
        return Proj(self.codes.data_ptr(), self.scales.data_ptr(), self.biases.data_ptr())

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.codes, self.scales, self.biases))


@dataclasses.dataclass
class DeviceLayer:
    shape: Shape
    gate: DeviceProj | None
    up: DeviceProj | None
    down: DeviceProj | None
    sh_gate: DeviceProj | None = None
    sh_up: DeviceProj | None = None
    sh_down: DeviceProj | None = None
    gate_vec: torch.Tensor | None = None   # bf16 [din]

    def struct(self) -> LayerWeights:
        z = Proj(None, None, None)
        f = lambda p: p.struct() if p is not None else z
        return LayerWeights(f(self.gate), f(self.up), f(self.down), f(self.sh_gate),
                            f(self.sh_up), f(self.sh_down), _p(self.gate_vec))


def _empty_proj(n, rows, cols, bits, device) -> DeviceProj:
    return DeviceProj(torch.empty((n, rows, cols * bits // 8), dtype=torch.uint8, device=device),
                      torch.empty((n, rows, cols // 64), dtype=torch.float16, device=device),
                      torch.empty((n, rows, cols // 64), dtype=torch.float16, device=device))


def synth_proj_device(seed, layer, proj, n, rows, cols, bits, device="cuda", stream=None):
    """All n experts of one projection drawn in HBM by the device generator."""
    p = _empty_proj(n, rows, cols, bits, device)
    L, st = lib(), _stream(stream)
    words = rows * cols * bits // 8 // 8
    groups = rows * (cols // 64)
    check("moe_synth_codes", L.moe_synth_codes(
        p.codes.data_ptr(), synth.tensor_key(seed, layer, proj, synth.CODES), 0, n, words, st))
    check("moe_synth_scales", L.moe_synth_scales(
        p.scales.data_ptr(), synth.tensor_key(seed, layer, proj, synth.SCALES), 0, n, groups, st))
    check("moe_synth_biases", L.moe_synth_biases(
        p.biases.data_ptr(), p.scales.data_ptr(), synth.tensor_key(seed, layer, proj, synth.BIASES),
        0, n, groups, bits, st))
    return p


def synth_layer_device(shape: Shape, layer: int, device="cuda", stream=None) -> DeviceLayer:
    s, E = shape.seed, shape.n_experts
    mk = lambda proj, n, r, c, b: synth_proj_device(s, layer, proj, n, r, c, b, device, stream)
    dl = DeviceLayer(shape, None, None, None)
    if shape.top_k > 0:
        dl.gate = mk(synth.GATE, E, shape.dff, shape.din, shape.bits_gate)
        dl.up = mk(synth.UP, E, shape.dff, shape.din, shape.bits_up)
        dl.down = mk(synth.DOWN, E, shape.din, shape.dff, shape.bits_down)
    if shape.n_shared:
        n, d, b = shape.n_shared, shape.dff_shared, shape.bits_shared
        dl.sh_gate = mk(synth.SH_GATE, n, d, shape.din, b)
        dl.sh_up = mk(synth.SH_UP, n, d, shape.din, b)
        dl.sh_down = mk(synth.SH_DOWN, n, shape.din, d, b)
        if shape.shared_gate:
            dl.gate_vec = torch.from_numpy(
                synth.gate_vector(s, layer, shape.din).view(np.int16)).view(torch.bfloat16).to(device)
    return dl


def proj_from_host(codes, scales, biases, device="cuda") -> DeviceProj:
    """Stacked host arrays (uint8 codes, uint16 fp16 bits) copied to the device."""
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(device)
    return DeviceProj(t(codes, torch.uint8), t(scales.view(np.int16), torch.float16),
                      t(biases.view(np.int16), torch.float16))


# ---------------------------------------------------------------- the block

class MoeDecode:
    """One prepared layer: moe_decode_create once, moe_decode_forward per token batch."""

    def __init__(self, layer: DeviceLayer, max_tokens: int = 1, resid_dtype=DTYPE_BF16,
                 out_dtype=DTYPE_F32, kernel_mode: int = KERNELS_FUSED):
        self.layer = layer
        self.cfg = config(layer.shape, max_tokens, resid_dtype, out_dtype, kernel_mode)
        self._w = layer.struct()
        h = ctypes.c_void_p()
        check("moe_decode_create", lib().moe_decode_create(ctypes.byref(self.cfg),
                                                           ctypes.byref(self._w), ctypes.byref(h)))
        self.handle = h

    def forward(self, x: torch.Tensor, ids: torch.Tensor | None, scores: torch.Tensor | None,
                resid: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """x bf16 [m, din]; ids int32 [m, K]; scores fp32 [m, K]; resid [m, din]; out [m, din]."""
        m = x.shape[0] if x.dim() == 2 else 1
        if out is None:
            dt = torch.float32 if self.cfg.out_dtype == DTYPE_F32 else torch.bfloat16
            out = torch.empty((m, self.cfg.din), dtype=dt, device=x.device)
        check("moe_decode_forward", lib().moe_decode_forward(
            self.handle, _p(x), m, _p(ids), _p(scores), _p(resid), _p(out), _stream(stream)))
        return out

    def routes(self, m: int, slots: bool = False, stream=None):
        """The ids the last forward's kernels read, int32 [m, top_k], and (pool mode, slots=True)
        each slot's and shared expert's down output before its coefficient, fp32
        [m, top_k + n_shared, din]; device tensors (moe_decode_routes)."""
        sh = self.layer.shape
        ids = torch.empty((m, max(sh.top_k, 1)), dtype=torch.int32, device="cuda")
        y = (torch.empty((m, sh.top_k + sh.n_shared, sh.din), dtype=torch.float32, device="cuda")
             if slots else None)
        check("moe_decode_routes", lib().moe_decode_routes(self.handle, _p(ids), _p(y),
                                                           _stream(stream)))
        return (ids[:, :sh.top_k], y) if slots else ids[:, :sh.top_k]

    def get_error(self) -> int:
        v = ctypes.c_int32()
        check("moe_decode_get_error", lib().moe_decode_get_error(self.handle, ctypes.byref(v)))
        return v.value

    def close(self):
        if self.handle:
            lib().moe_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward_noalloc(layer: "DeviceLayer", x: torch.Tensor, ids: torch.Tensor | None,
                    scores: torch.Tensor | None, resid: torch.Tensor, out: torch.Tensor,
                    device_error: torch.Tensor | None = None, max_tokens: int | None = None,
                    resid_dtype=DTYPE_BF16, out_dtype=DTYPE_F32, stream=None) -> torch.Tensor:
    """moe_decode_forward_noalloc: one layer without a handle, activations in the library's
    fixed scratch array (two-kernel mode).  `out` must be given; `device_error` is an int32
    device tensor of one element that must start at 0."""
    m = x.shape[0] if x.dim() == 2 else 1
    cfg = config(layer.shape, max_tokens or m, resid_dtype, out_dtype, KERNELS_SEPARATE)
    w = layer.struct()
    check("moe_decode_forward_noalloc", lib().moe_decode_forward_noalloc(
        ctypes.byref(cfg), ctypes.byref(w), _p(x), m, _p(ids), _p(scores), _p(resid), _p(out),
        _p(device_error), _stream(stream)))
    return out


class MoeStack:
    """A stack of layers replayed as one CUDA graph per decode step.

    norm_weight (bf16 [L - 1, din] on the device) folds the next layer's RMSNorm in
    (moe_stack_create_chained): layer l >= 1 then reads RMSNorm(out of layer l - 1) instead of x,
    and step() reads x as [m, din]."""

    def __init__(self, layers: list[DeviceLayer], max_tokens: int = 1, resid_dtype=DTYPE_BF16,
                 kernel_mode: int = KERNELS_FUSED, norm_weight=None, eps: float = 1e-6):
        self.layers = layers
        self.cfg = config(layers[0].shape, max_tokens, resid_dtype, DTYPE_F32, kernel_mode)
        arr = (LayerWeights * len(layers))()
        for i, l in enumerate(layers):
            arr[i] = l.struct()
        self._w = arr
        self._norm = norm_weight
        h = ctypes.c_void_p()
        if norm_weight is None:
            check("moe_stack_create", lib().moe_stack_create(ctypes.byref(self.cfg), len(layers),
                                                             arr, ctypes.byref(h)))
        else:
            check("moe_stack_create_chained", lib().moe_stack_create_chained(
                ctypes.byref(self.cfg), len(layers), arr, _p(norm_weight), eps, ctypes.byref(h)))
        self.handle = h

    def step(self, x, ids, scores, resid0, out, stream=None):
        """x bf16 [L, m, din]; ids int32 [L, m, K]; scores fp32 [L, m, K]; resid0 [m, din];
        out fp32 [m, din]; all on the device."""
        m = resid0.shape[0]
        check("moe_stack_step", lib().moe_stack_step(self.handle, _p(x), m, _p(ids), _p(scores),
                                                     _p(resid0), _p(out), _stream(stream)))
        return out

    def step_parts(self, parts, x, ids, scores, resid0, out, stream=None):
        """Only kernel A (parts=1) or only kernel B (parts=2) of every layer: a timing aid."""
        m = resid0.shape[0]
        check("moe_stack_step_parts", lib().moe_stack_step_parts(
            self.handle, parts, _p(x), m, _p(ids), _p(scores), _p(resid0), _p(out),
            _stream(stream)))
        return out

    def step_host(self, x, ids, scores, resid0, out, stream=None):
        """The same step from host (ideally pinned) tensors; returns after out is on the host."""
        m = resid0.shape[0]
        check("moe_stack_step_host", lib().moe_stack_step_host(
            self.handle, _p(x), m, _p(ids), _p(scores), _p(resid0), _p(out), _stream(stream)))
        return out

    def get_error(self) -> int:
        v = ctypes.c_int32()
        check("moe_stack_get_error", lib().moe_stack_get_error(self.handle, ctypes.byref(v)))
        return v.value

    def timeline(self) -> np.ndarray:
        """Timeline build only: the column-split kernel's stamps of the last step,
        uint64 [grid, L, points] (see moe_timeline.cuh)."""
        P = 64  # kTlPoints
        buf = np.zeros(512 * len(self.layers) * P, np.uint64)
        g = ctypes.c_int32()
        check("moe_stack_timeline", lib().moe_stack_timeline(
            self.handle, buf.ctypes.data, buf.nbytes, ctypes.byref(g)))
        return buf[:g.value * len(self.layers) * P].reshape(g.value, len(self.layers), P)

    def close(self):
        if self.handle:
            lib().moe_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- packing

def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    rows, cols = codes.shape
    out = np.empty((rows, cols * bits // 8), dtype=np.uint8)
    check("moe_pack_codes", lib().moe_pack_codes(codes.ctypes.data, rows, cols, bits,
                                                 out.ctypes.data))
    return out


def unpack_codes(packed: np.ndarray, cols: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    rows = packed.shape[0]
    out = np.empty((rows, cols), dtype=np.uint8)
    check("moe_unpack_codes", lib().moe_unpack_codes(packed.ctypes.data, rows, cols, bits,
                                                     out.ctypes.data))
    return out


def unpack_codes_device(packed: torch.Tensor, cols: int, bits: int, stream=None) -> torch.Tensor:
    rows = packed.shape[0]
    out = torch.empty((rows, cols), dtype=torch.uint8, device=packed.device)
    check("moe_unpack_codes_device", lib().moe_unpack_codes_device(
        packed.data_ptr(), rows, cols, bits, out.data_ptr(), _stream(stream)))
    return out


def route_invert_device(ids: torch.Tensor, n_experts: int, stream=None):
    """The kernels' route inversion of ids int32 [m, k] (device): (uniq, offs, pairs) as numpy."""
    m, k = ids.shape
    out = torch.full((2 + 3 * m * k,), -7, dtype=torch.int32, device=ids.device)
    check("moe_route_invert_device", lib().moe_route_invert_device(
        _p(ids.contiguous()), m, k, n_experts, _p(out), _stream(stream)))
    o = out.cpu().numpy()
    u = int(o[0])
    uniq = o[1:1 + u]
    offs = o[1 + u:2 + 2 * u]
    pairs = o[2 + 2 * u:2 + 2 * u + int(offs[-1])]
    return uniq.copy(), offs.copy(), pairs.copy()


def debug_wait_timeout(kind: int, device_error: torch.Tensor, stream=None) -> None:
    """Runs the kernels' bounded wait on a condition nothing satisfies (kind 0: grid-barrier
    count, 1: mbarrier stage); the time-out bit lands in device_error (int32 [1], device)."""
    scratch = torch.zeros(1, dtype=torch.int32, device=device_error.device)
    check("moe_debug_wait_timeout", lib().moe_debug_wait_timeout(kind, _p(scratch), _p(device_error),
                                                                 _stream(stream)))


def router_topk(logits: torch.Tensor, top_k: int, stream=None):
    """moe_router_topk on fp32 logits [m, E] (device): (ids int32 [m, top_k], scores fp32)."""
    m, E = logits.shape
    ids = torch.empty((m, top_k), dtype=torch.int32, device=logits.device)
    scores = torch.empty((m, top_k), dtype=torch.float32, device=logits.device)
    check("moe_router_topk", lib().moe_router_topk(_p(logits.contiguous()), m, E, top_k, _p(ids),
                                                   _p(scores), _stream(stream)))
    return ids, scores


def col_pieces(top_k: int, dff: int, n_shared: int, dff_shared: int, bits_down: int,
               bits_shared: int, u0: int, u1: int, max_pieces: int = 64):
    """The column split's pieces of the activation columns [u0, u1) (host only):
    [(seg, j0, j1, a0, blk0, nb, pb, grp), ...]."""
    import numpy as np
    out = np.zeros(8 * max_pieces, dtype=np.int32)
    rc = lib().moe_debug_col_pieces(top_k, dff, n_shared, dff_shared, bits_down, bits_shared, u0,
                                    u1, out.ctypes.data, max_pieces)
    check("moe_debug_col_pieces", min(rc, 0))
    return [tuple(int(v) for v in out[8 * q:8 + 8 * q]) for q in range(rc)]


def col_plan(shape, grid: int, ring_bytes: int) -> dict:
    """The column split's launch plan for a workload shape (host only); "bounds": the CTAs'
    column ranges, CTA c owning [bounds[c], bounds[c + 1])."""
    import numpy as np
    cfg = config(shape, 1, DTYPE_BF16, DTYPE_F32, KERNELS_COLUMNS)
    out = np.zeros(10, dtype=np.int32)
    bounds = np.zeros(grid + 1, dtype=np.int32)
    check("moe_debug_col_plan", lib().moe_debug_col_plan(ctypes.byref(cfg), grid, ring_bytes,
                                                         out.ctypes.data, bounds.ctypes.data))
    keys = ("stages", "stage_bytes", "nbs", "ro", "cb_r", "cb_s", "rows_a_r", "rows_a_s", "pack",
            "prefetch")
    plan = dict(zip(keys, (int(v) for v in out)))
    plan["bounds"] = [int(v) for v in bounds]
    return plan


# ---------------------------------------------------------------- dense bf16 decode GEMV

def gemv_bf16(W, x, y=None, shared_x: bool = True, stream=None):
    """y [n_mats, m, n_out] fp32 = x W^T for every matrix of W (bf16 [n_mats, n_out, n_in] on
    the device).  x is bf16 [m, n_in] (shared_x) or [n_mats, m, n_in]."""
    import torch
    n_mats, n_out, n_in = W.shape
    m = x.shape[-2]
    if y is None:
        y = torch.empty((n_mats, m, n_out), dtype=torch.float32, device=W.device)
    x_stride = 0 if shared_x else m * n_in
    check("moe_gemv_bf16", lib().moe_gemv_bf16(_p(W), _p(x), x_stride, _p(y), n_mats, m, n_out,
                                               n_in, _stream(stream)))
    return y
