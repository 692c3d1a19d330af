"""fp64 CPU oracle of the single-token decode MoE expert block (ctypes wrapper).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It imports nothing from the
``quantized_moe_expert_dequant_gb300`` package and the package never imports it.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64, one thread).  This wrapper only
compiles it with gcc, marshals numpy arrays into its structs and gathers the slots' experts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so beside it (gcc, -O2, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class Proj(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p), ("rows", ctypes.c_int32),
                ("cols", ctypes.c_int32), ("bits", ctypes.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("MOE_ORACLE_LIB")  # a mutant build, for the oracle's own tests
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            L.oracle_f16.restype = ctypes.c_double
            L.oracle_f16.argtypes = [ctypes.c_uint16]
            L.oracle_bf16.restype = ctypes.c_double
            L.oracle_bf16.argtypes = [ctypes.c_uint16]
            L.oracle_code.restype = ctypes.c_uint32
            L.oracle_code.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64]
            L.oracle_weight.restype = ctypes.c_double
            L.oracle_weight.argtypes = [ctypes.POINTER(Proj), ctypes.c_int64, ctypes.c_int64]
            L.oracle_silu.restype = ctypes.c_double
            L.oracle_silu.argtypes = [ctypes.c_double]
            L.oracle_sigmoid.restype = ctypes.c_double
            L.oracle_sigmoid.argtypes = [ctypes.c_double]
            L.oracle_matvec.restype = None
            L.oracle_matvec.argtypes = [ctypes.POINTER(Proj), ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int32]
            L.oracle_expert_act.restype = None
            L.oracle_expert_act.argtypes = [ctypes.POINTER(Proj), ctypes.POINTER(Proj),
                                            ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_shared_scalar.restype = ctypes.c_double
            L.oracle_shared_scalar.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
            L.oracle_moe_token.restype = ctypes.c_int
            L.oracle_moe_token.argtypes = (
                [ctypes.c_int32] * 3 + [ctypes.POINTER(Proj)] * 3 + [ctypes.c_void_p]
                + [ctypes.c_int32] * 2 + [ctypes.POINTER(Proj)] * 3
                + [ctypes.c_void_p] * 3 + [ctypes.c_int32] + [ctypes.c_void_p] * 2
                + [ctypes.c_int32])
            L.oracle_route_invert.restype = ctypes.c_int32
            L.oracle_route_invert.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p]
            L.oracle_router.restype = None
            L.oracle_router.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_gemv_bf16.restype = None
            L.oracle_gemv_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
            L.oracle_round_bf16.restype = ctypes.c_uint16
            L.oracle_round_bf16.argtypes = [ctypes.c_double]
            L.oracle_rmsnorm_bf16.restype = None
            L.oracle_rmsnorm_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_float, ctypes.c_void_p]
            _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data if a is not None else None


class Packed:
    """One expert's projection in the canonical packed layout (host numpy arrays).

    codes  uint8  [rows, cols*bits/8]   little-endian, LSB-first bit stream per row
    scales uint16 [rows, cols/64]       fp16 bit patterns
    biases uint16 [rows, cols/64]       fp16 bit patterns
    """

    def __init__(self, codes, scales, biases, bits):
        self.codes = np.ascontiguousarray(codes, dtype=np.uint8)
        self.scales = np.ascontiguousarray(scales, dtype=np.uint16)
        self.biases = np.ascontiguousarray(biases, dtype=np.uint16)
        self.bits = int(bits)
        self.rows = int(self.scales.shape[0])
        self.cols = int(self.scales.shape[1]) * 64
        assert self.codes.shape == (self.rows, self.cols * self.bits // 8), self.codes.shape
        assert self.biases.shape == self.scales.shape

    def struct(self) -> Proj:
        return Proj(_ptr(self.codes), _ptr(self.scales), _ptr(self.biases),
                    self.rows, self.cols, self.bits)


def _array(projs):
    arr = (Proj * max(1, len(projs)))()
    for i, p in enumerate(projs):
        arr[i] = p.struct()
    return arr


def f16(h: int) -> float:
    return lib().oracle_f16(int(h))


def bf16(b: int) -> float:
    return lib().oracle_bf16(int(b))


def code(row: np.ndarray, bits: int, c: int) -> int:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    return int(lib().oracle_code(_ptr(row), bits, c))


def unpack_row(row: np.ndarray, bits: int, n: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    L = lib()
    return np.array([L.oracle_code(_ptr(row), bits, c) for c in range(n)], dtype=np.uint32)


def weight(p: Packed, r: int, c: int) -> float:
    s = p.struct()
    return lib().oracle_weight(ctypes.byref(s), r, c)


def silu(z: float) -> float:
    return lib().oracle_silu(float(z))


def sigmoid(z: float) -> float:
    return lib().oracle_sigmoid(float(z))


def matvec(p: Packed, v: np.ndarray, rows=None) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    assert v.shape == (p.cols,)
    s = p.struct()
    if rows is None:
        y = np.empty(p.rows, dtype=np.float64)
        lib().oracle_matvec(ctypes.byref(s), _ptr(v), _ptr(y), None, 0)
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        y = np.empty(len(rows), dtype=np.float64)
        lib().oracle_matvec(ctypes.byref(s), _ptr(v), _ptr(y), _ptr(rows), len(rows))
    return y


def expert_act(gate: Packed, up: Packed, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    act = np.empty(gate.rows, dtype=np.float64)
    g, u = gate.struct(), up.struct()
    lib().oracle_expert_act(ctypes.byref(g), ctypes.byref(u), _ptr(x), _ptr(act))
    return act


def shared_scalar(x: np.ndarray, gate_vec_bf16: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(gate_vec_bf16, dtype=np.uint16)
    return lib().oracle_shared_scalar(_ptr(x), _ptr(g), len(x))


def moe_token(x_bf16, resid, scores, gate, up, down, sh_gate=(), sh_up=(), sh_down=(),
              gate_vec_bf16=None, rows=None) -> np.ndarray:
    """Block output for one token, fp64.

    x_bf16        uint16 [din]           bf16 bit patterns
    resid         uint16 (bf16 bits) or float32 [din]
    scores        float32 [K]
    gate/up/down  K Packed projections: the experts the K slots name, in slot order
    sh_*          Packed projections of the shared experts (may be empty)
    gate_vec_bf16 uint16 [din] or None (shared scalar 1)
    rows          output rows to compute (None: all)
    """
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    din = len(x_bf16)
    K = len(gate)
    assert len(up) == K and len(down) == K
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    assert scores.shape == (K,)
    if resid.dtype == np.uint16:
        resid_kind = 0
    elif resid.dtype == np.float32:
        resid_kind = 1
    else:
        raise TypeError("resid must be bf16 bits (uint16) or float32")
    resid = np.ascontiguousarray(resid)
    dff = gate[0].rows if K else (up[0].rows if up else 0)
    n_sh = len(sh_gate)
    dff_sh = sh_gate[0].rows if n_sh else 0
    g_arr, u_arr, d_arr = _array(gate), _array(up), _array(down)
    sg, su, sd = _array(sh_gate), _array(sh_up), _array(sh_down)
    gv = None if gate_vec_bf16 is None else np.ascontiguousarray(gate_vec_bf16, dtype=np.uint16)
    if rows is None:
        out = np.empty(din, dtype=np.float64)
        rows_p, n_rows = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        out = np.empty(len(rows), dtype=np.float64)
        rows_p, n_rows = _ptr(rows), len(rows)
    rc = lib().oracle_moe_token(din, dff, K, g_arr, u_arr, d_arr, _ptr(scores), n_sh, dff_sh,
                                sg, su, sd, _ptr(gv), _ptr(x_bf16), _ptr(resid), resid_kind,
                                _ptr(out), rows_p, n_rows)
    if rc != 0:
        raise ValueError("oracle_moe_token: shape mismatch")
    return out


def route_invert(ids: np.ndarray, n_experts: int):
    """(uniq, offs, pairs) of ids [m, k]: the distinct valid experts ascending, and per expert the
    pairs p = token * k + slot that name it, ascending (see oracle_route_invert)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    m, k = ids.shape
    n = m * k
    uniq = np.empty(max(n, 1), np.int32)
    offs = np.empty(max(n, 1) + 1, np.int32)
    pairs = np.empty(max(n, 1), np.int32)
    u = lib().oracle_route_invert(_ptr(ids), m, k, n_experts, _ptr(uniq), _ptr(offs), _ptr(pairs))
    return uniq[:u].copy(), offs[:u + 1].copy(), pairs[:offs[u]].copy()


def router(logits: np.ndarray, k: int):
    """(ids int32 [k], scores float32 [k]) of one token's fp32 logits [E] (see oracle_router)."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    ids = np.empty(k, np.int32)
    scores = np.empty(k, np.float32)
    lib().oracle_router(_ptr(logits), len(logits), k, _ptr(ids), _ptr(scores))
    return ids, scores



def round_bf16(y: float) -> int:
    """bf16 bit pattern nearest to y, ties to even (see oracle_round_bf16)."""
    return int(lib().oracle_round_bf16(float(y)))


def rmsnorm_bf16(v: np.ndarray, gamma_bf16: np.ndarray, eps: float) -> np.ndarray:
    """bf16 bits [n] of the next layer's input from a layer's fp32 output v (see
    oracle_rmsnorm_bf16)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16)
    assert g.shape == v.shape
    x = np.empty(len(v), np.uint16)
    lib().oracle_rmsnorm_bf16(_ptr(v), len(v), _ptr(g), float(eps), _ptr(x))
    return x


def gemv_bf16(W_bf16: np.ndarray, x_bf16: np.ndarray) -> np.ndarray:
    """y [m, n_out] (fp64) = x [m, n_in] times W [n_out, n_in] transposed, both bf16 bit patterns
    (see oracle_gemv_bf16)."""
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n_out, n_in = W.shape
    m = x.shape[0]
    assert x.shape == (m, n_in)
    y = np.empty((m, n_out), np.float64)
    lib().oracle_gemv_bf16(_ptr(W), _ptr(x), m, n_out, n_in, _ptr(y))
    return y
