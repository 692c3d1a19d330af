"""Seeded synthetic inputs for the decode MoE expert block (host side, numpy).

This module draws inputs only; it holds none of the block's arithmetic.  Both the CUDA path and
the CPU oracle consume what it draws, and the device generator in ``csrc/synth.cu`` implements the
same counter-based definitions so that multi-GB weight stacks can be drawn in HBM and still be
recomputed here, bit for bit, for any single expert.

Definitions (all integer arithmetic is modulo 2^64):

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; constants as published by Vigna).
* ``key(*parts)`` chains ``k <- mix64(k + G*(p+1))`` over the parts, G = 0x9E3779B97F4A7C15.
* Element i of expert e of a tensor with key t is ``h(t, e, i) = mix64(t + G*(((e << 40) | i) + 1))``.

Weight tensors (canonical packed layout, one expert = ``[rows, cols]`` codes at ``bits``):

* code bytes: the expert's code stream, read as little-endian uint64 words, has word i equal to
  ``h(t_codes, e, i)``.  Random bits make every b-bit code uniform on [0, 2^b - 1].
* scale i (fp16): ``u = h >> 40``; ``s = fp16_rn(fp32(u * 2^-24) * 0.015f + 0.005f)`` with every
  fp32 operation rounded to nearest, no fused multiply-add.  s is about U(0.005, 0.02).
* bias i (fp16): ``u = h(t_bias, e, i) >> 40``; ``c = 2^(bits-1) + (u * 2^-24 - 0.5)`` (fp32);
  ``bias = fp16_rn(-(fp32(scale) * c))``: about ``-2^(bits-1) * scale``, centring the codes.

Activations and router outputs:

* normals: Box-Muller on two 53-bit uniforms per value, in fp64, then rounded to fp32 and to
  bf16 (round to nearest even) for x, resid and the shared gate vector g.
* ids: K distinct experts of E by a partial Fisher-Yates shuffle driven by ``mix64``.
* scores: softmax, in fp64, of K standard-normal logits, rounded to fp32.
* RMSNorm weight of a chained stack (one row per layer after the first): ``1 + 0.2 * normal``
  in fp64, rounded to fp32 and to bf16.
* Dense projection (bf16 GEMV workload): weights ``0.02 * normal`` and inputs ``normal``, rounded
  to fp32 and to bf16.
"""
from __future__ import annotations

import numpy as np

G = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1

# tensor roles in the key chain
GATE, UP, DOWN, SH_GATE, SH_UP, SH_DOWN = 0, 1, 2, 3, 4, 5
CODES, SCALES, BIASES = 0, 1, 2
ROLE_X, ROLE_RESID, ROLE_GVEC, ROLE_IDS, ROLE_LOGITS, ROLE_NORM = 10, 11, 12, 13, 14, 15
ROLE_DENSE_W, ROLE_DENSE_X = 16, 17

_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def mix64_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    z = (z ^ (z >> np.uint64(30))) * _C1
    z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def key(*parts: int) -> int:
    k = 0
    for p in parts:
        k = mix64_int(k + G * (int(p) + 1))
    return k


def tensor_key(seed: int, layer: int, proj: int, comp: int) -> int:
    return key(seed, layer, proj, comp)


def hashes(tkey: int, expert: int, n: int, start: int = 0) -> np.ndarray:
    """h(tkey, expert, i) for i in [start, start + n) as uint64."""
    idx = (np.uint64(expert) << np.uint64(40)) | np.arange(start, start + n, dtype=np.uint64)
    return mix64(np.uint64(tkey) + np.uint64(G) * (idx + np.uint64(1)))


# ---------------------------------------------------------------- weights (canonical layout)

def row_bytes(cols: int, bits: int) -> int:
    return cols * bits // 8


def code_bytes(seed, layer, proj, expert, rows, cols, bits) -> np.ndarray:
    """uint8 [rows, cols*bits/8]: one expert's packed codes."""
    nbytes = rows * row_bytes(cols, bits)
    assert nbytes % 8 == 0
    words = hashes(tensor_key(seed, layer, proj, CODES), expert, nbytes // 8)
    return words.astype("<u8").view(np.uint8).reshape(rows, row_bytes(cols, bits))


def scale_bits(seed, layer, proj, expert, rows, cols) -> np.ndarray:
    """uint16 [rows, cols/64]: fp16 scales, about U(0.005, 0.02)."""
    n = rows * (cols // 64)
    u = (hashes(tensor_key(seed, layer, proj, SCALES), expert, n) >> np.uint64(40))
    v = u.astype(np.float32) * np.float32(2.0 ** -24)          # exact
    v = v * np.float32(0.015)
    v = v + np.float32(0.005)
    return v.astype(np.float16).view(np.uint16).reshape(rows, cols // 64)


def bias_bits(seed, layer, proj, expert, scales_fp16_bits, bits) -> np.ndarray:
    """uint16 like scales: fp16 biases about -2^(bits-1) * scale."""
    s = np.asarray(scales_fp16_bits, dtype=np.uint16)
    u = (hashes(tensor_key(seed, layer, proj, BIASES), expert, s.size) >> np.uint64(40))
    t = u.astype(np.float32) * np.float32(2.0 ** -24) - np.float32(0.5)  # exact
    c = np.float32(2 ** (bits - 1)) + t
    m = s.reshape(-1).view(np.float16).astype(np.float32) * c
    return (-m).astype(np.float16).view(np.uint16).reshape(s.shape)


def expert_proj(seed, layer, proj, expert, rows, cols, bits):
    """(codes uint8, scales uint16, biases uint16) of one expert's projection."""
    codes = code_bytes(seed, layer, proj, expert, rows, cols, bits)
    sc = scale_bits(seed, layer, proj, expert, rows, cols)
    bi = bias_bits(seed, layer, proj, expert, sc, bits)
    return codes, sc, bi


def stacked_proj(seed, layer, proj, n_experts, rows, cols, bits):
    """All experts of one projection, stacked: codes [E, rows, rb], scales/biases [E, rows, G]."""
    parts = [expert_proj(seed, layer, proj, e, rows, cols, bits) for e in range(n_experts)]
    return tuple(np.stack([p[i] for p in parts]) for i in range(3))


# ---------------------------------------------------------------- activations, router outputs

def normals_f64(k: int, n: int) -> np.ndarray:
    h1 = hashes(k, 0, n, 0)
    h2 = hashes(k, 1, n, 0)
    u1 = (h1 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16, nearest even (finite inputs)."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(k: int, n: int, std: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits((normals_f64(k, n) * std).astype(np.float32))


def activations(seed, layer, token, din):
    """x bf16 [din] of one token of one layer."""
    return normal_bf16(key(seed, layer, ROLE_X, token), din)


def residual(seed, layer, token, din):
    return normal_bf16(key(seed, layer, ROLE_RESID, token), din)


def gate_vector(seed, layer, din, std=0.02):
    return normal_bf16(key(seed, layer, ROLE_GVEC), din, std)


def norm_weight(seed, layer, din):
    """bf16 [din]: the RMSNorm weight that turns layer ``layer - 1``'s output into layer
    ``layer``'s input in a chained stack."""
    return f32_to_bf16_bits((1.0 + 0.2 * normals_f64(key(seed, layer, ROLE_NORM), din))
                            .astype(np.float32))


def topk_ids(seed, layer, token, n_experts, top_k, step=0) -> np.ndarray:
    """K distinct expert ids, in draw order."""
    assert top_k <= n_experts
    k = key(seed, layer, ROLE_IDS, token, step)
    perm = list(range(n_experts))
    for j in range(top_k):
        r = mix64_int(k + G * (j + 1))
        t = j + r % (n_experts - j)
        perm[j], perm[t] = perm[t], perm[j]
    return np.array(perm[:top_k], dtype=np.int32)


def scores(seed, layer, token, top_k, step=0) -> np.ndarray:
    if top_k == 0:
        return np.zeros(0, dtype=np.float32)
    logits = normals_f64(key(seed, layer, ROLE_LOGITS, token, step), top_k)
    e = np.exp(logits - logits.max())
    return (e / e.sum()).astype(np.float32)


def dense_weight(seed, n_out, n_in, matrix=0):
    """bf16 [n_out, n_in] weights of one dense projection."""
    k = key(seed, matrix, ROLE_DENSE_W)
    return normal_bf16(k, n_out * n_in, 0.02).reshape(n_out, n_in)


def dense_input(seed, m, n_in, matrix=0):
    """bf16 [m, n_in] rows (tokens) multiplied by a dense projection."""
    k = key(seed, matrix, ROLE_DENSE_X)
    return normal_bf16(k, m * n_in).reshape(m, n_in)
