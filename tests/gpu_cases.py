"""Shared builders for the GPU tests: seeded problems, the oracle's expectation, and the parity bar.

Parity bar (fp32-accumulated output): max|gpu - oracle| <= 1e-3 * rms(oracle) + 1e-6 and relative
L2 error <= 1e-4.  A bf16 output must be the bf16 rounding of a value that meets that bar: every
element within one bf16 ulp of the oracle rounded to bf16, or within the fp32 bar's absolute
allowance of the oracle plus half a bf16 ulp of the element (near zero one bf16 ulp is finer than
the fp32 sums' own rounding, so the first test alone would hold a bf16 output to more than the
fp32 one).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300 import synth
from quantized_moe_expert_dequant_gb300.workloads import Shape
from tests.oracle_jobs import OracleLayer, oracle_tokens  # noqa: F401  (re-exported)

ATOL_RMS, ATOL_ABS, REL_L2 = 1e-3, 1e-6, 1e-4


def dev(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if dtype in (torch.bfloat16, torch.float16):
        return torch.from_numpy(a.view(np.int16)).view(dtype).cuda()
    return torch.from_numpy(a).cuda()


def host_layer_device(shape: Shape, layer: int = 0) -> Bn.DeviceLayer:
    """Every expert drawn on the host and copied: independent of the device generator."""
    s, E = shape.seed, shape.n_experts
    mk = lambda proj, n, r, c, b: Bn.proj_from_host(*synth.stacked_proj(s, layer, proj, n, r, c, b))
    d = Bn.DeviceLayer(shape, None, None, None)
    if shape.top_k > 0:
        d.gate = mk(synth.GATE, E, shape.dff, shape.din, shape.bits_gate)
        d.up = mk(synth.UP, E, shape.dff, shape.din, shape.bits_up)
        d.down = mk(synth.DOWN, E, shape.din, shape.dff, shape.bits_down)
    if shape.n_shared:
        n, w, b = shape.n_shared, shape.dff_shared, shape.bits_shared
        d.sh_gate = mk(synth.SH_GATE, n, w, shape.din, b)
        d.sh_up = mk(synth.SH_UP, n, w, shape.din, b)
        d.sh_down = mk(synth.SH_DOWN, n, shape.din, w, b)
        if shape.shared_gate:
            d.gate_vec = dev(synth.gate_vector(s, layer, shape.din), torch.bfloat16)
    return d


def token_inputs(shape: Shape, layer: int = 0, m: int = 1, step: int = 0):
    """x, resid (bf16 bits) [m, din]; ids int32 and scores fp32 [m, K]."""
    s = shape.seed
    x = np.stack([synth.activations(s, layer, t + 1000 * step, shape.din) for t in range(m)])
    r = np.stack([synth.residual(s, layer, t + 1000 * step, shape.din) for t in range(m)])
    ids = np.stack([synth.topk_ids(s, layer, t, shape.n_experts, shape.top_k, step)
                    for t in range(m)]).astype(np.int32).reshape(m, shape.top_k)
    sc = np.stack([synth.scores(s, layer, t, shape.top_k, step)
                   for t in range(m)]).astype(np.float32).reshape(m, shape.top_k)
    return x, r, ids, sc


def parity(gpu, ref) -> tuple[float, float, float]:
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    err = float(np.abs(gpu - ref).max())
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    return err, rms, rel


def assert_parity(gpu, ref, what=""):
    err, rms, rel = parity(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu, dtype=np.float64))), f"{what}: non-finite output"
    assert err <= ATOL_RMS * rms + ATOL_ABS, f"{what}: max err {err:.3e} vs rms {rms:.3e}"
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e}"


def assert_parity_bf16(gpu_bf16: torch.Tensor, ref: np.ndarray, what=""):
    g = gpu_bf16.float().cpu().numpy().astype(np.float64).reshape(-1)
    r = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    _, e = np.frexp(r)
    ulp = np.ldexp(1.0, e - 8)  # |r| in [2^(e-1), 2^e): bf16 spacing 2^(e-8)
    _, eg = np.frexp(g)
    half_g = np.ldexp(1.0, eg - 9)
    ref64 = np.asarray(ref, dtype=np.float64).reshape(-1)
    allow = ATOL_RMS * float(np.sqrt(np.mean(ref64 ** 2))) + ATOL_ABS
    ok = (np.abs(g - r) <= ulp) | (np.abs(g - ref64) <= allow + half_g)
    bad = np.nonzero(~ok)[0]
    assert bad.size == 0, (f"{what}: bf16 output off at {bad[:4].tolist()}: "
                           f"{g[bad[:4]].tolist()} vs {ref64[bad[:4]].tolist()}")


def oracle_stack(shape: Shape, x, ids, sc, resid0, m: int = 1, rows=None, norm=None,
                 eps: float = 0.0, layers: int | None = None):
    """The oracle's own chain through the first `layers` layers of a stack: [layers][m][rows].

    Every layer's residual is the oracle's previous output rounded to fp32 (the stack keeps layer
    outputs in fp32).  x is [L][m][din] (bf16 bits); with norm (bf16 [L - 1][din]) only x[0] is
    read and layer l >= 1 takes RMSNorm(previous output) with row l - 1, which needs every row of
    that output (rows must then be None).  No value comes from the GPU."""
    L = shape.layers if layers is None else layers
    assert norm is None or rows is None
    oras = [OracleLayer(shape, l) for l in range(L)]
    out = []
    for l in range(L):
        per = []
        for t in range(m):
            if l == 0:
                xt, resid = x[0][t], resid0[t]
            else:
                prev = out[l - 1][t].astype(np.float32)
                xt = x[l][t] if norm is None else O.rmsnorm_bf16(prev, norm[l - 1], eps)
                resid = prev
                if rows is not None:   # only the sampled rows of the previous output exist
                    full = np.zeros(shape.din, np.float32)
                    full[rows] = prev
                    resid = full
            per.append(oras[l].token(xt, resid, ids[l][t], sc[l][t], rows=rows))
        out.append(np.stack(per))
    return out
