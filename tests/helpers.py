"""Test helpers that are independent of both the oracle and the CUDA path.

``pack_bigint`` / ``unpack_bigint`` restate the canonical packed layout through Python's
arbitrary-precision integers (code c occupies bits [c*b, c*b+b) of one little-endian integer per
row), a different mechanism from the oracle's bit reader and from the kernels' word masks.
``dense_*`` build full fp64 matrices with numpy so a block output can be brute-forced on tiny
shapes with library matmuls.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import synth


def pack_bigint(codes, bits) -> np.ndarray:
    codes = [int(q) for q in codes]
    assert all(0 <= q < (1 << bits) for q in codes)
    v = 0
    for c, q in enumerate(codes):
        v |= q << (c * bits)
    return np.frombuffer(v.to_bytes(len(codes) * bits // 8, "little"), dtype=np.uint8).copy()


def unpack_bigint(row_bytes, bits, n) -> np.ndarray:
    v = int.from_bytes(np.asarray(row_bytes, dtype=np.uint8).tobytes(), "little")
    mask = (1 << bits) - 1
    return np.array([(v >> (c * bits)) & mask for c in range(n)], dtype=np.int64)


def packed_from_codes(Q, scales_f16_bits, biases_f16_bits, bits) -> O.Packed:
    Q = np.asarray(Q)
    codes = np.stack([pack_bigint(r, bits) for r in Q])
    return O.Packed(codes, scales_f16_bits, biases_f16_bits, bits)


def dense(p: O.Packed) -> np.ndarray:
    """Full fp64 weight matrix of a packed projection, through numpy's fp16 conversion."""
    Q = np.stack([unpack_bigint(p.codes[r], p.bits, p.cols) for r in range(p.rows)]).astype(np.float64)
    s = p.scales.view(np.float16).astype(np.float64)
    b = p.biases.view(np.float16).astype(np.float64)
    return Q * np.repeat(s, 64, axis=1) + np.repeat(b, 64, axis=1)


def bf16_to_f64(b) -> np.ndarray:
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def dense_expert_act(gate: O.Packed, up: O.Packed, x64) -> np.ndarray:
    g = dense(gate) @ x64
    u = dense(up) @ x64
    return g * expit(g) * u


def dense_block(x_bf16, resid64, scores, gate, up, down, sh_gate=(), sh_up=(), sh_down=(),
                gate_vec=None) -> np.ndarray:
    x = bf16_to_f64(x_bf16)
    routed = np.zeros(len(x))
    for k in range(len(gate)):
        routed += float(scores[k]) * (dense(down[k]) @ dense_expert_act(gate[k], up[k], x))
    shared = np.zeros(len(x))
    for s in range(len(sh_gate)):
        shared += dense(sh_down[s]) @ dense_expert_act(sh_gate[s], sh_up[s], x)
    scalar = 1.0 if gate_vec is None else float(expit(x @ bf16_to_f64(gate_vec)))
    return resid64 + (routed + scalar * shared)


def synth_packed(seed, layer, proj, expert, rows, cols, bits) -> O.Packed:
    c, s, b = synth.expert_proj(seed, layer, proj, expert, rows, cols, bits)
    return O.Packed(c, s, b, bits)


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
