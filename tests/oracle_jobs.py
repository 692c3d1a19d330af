"""The oracle's view of a synthetic layer, and its per-token results computed in worker processes.

Only numpy, the oracle and the seeded generators are imported here, so that spawned workers start
without CUDA.  The workers are started with the spawn method (never forked from a process that may
already hold a CUDA context).
"""
from __future__ import annotations

import multiprocessing
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import synth
from quantized_moe_expert_dequant_gb300.workloads import Shape


class OracleLayer:
    """The oracle's view of one synthetic layer: experts regenerated on the host on demand."""

    def __init__(self, shape: Shape, layer: int = 0):
        self.shape, self.layer = shape, layer
        self._cache = {}

    def packed(self, proj, e, rows, cols, bits):
        key = (proj, e)
        if key not in self._cache:
            c, s, b = synth.expert_proj(self.shape.seed, self.layer, proj, e, rows, cols, bits)
            self._cache[key] = O.Packed(c, s, b, bits)
        return self._cache[key]

    def token(self, x_bits, resid, ids, scores, rows=None):
        sh = self.shape
        valid = [(int(e), float(w)) for e, w in zip(ids, scores) if 0 <= int(e) < sh.n_experts]
        g = [self.packed(synth.GATE, e, sh.dff, sh.din, sh.bits_gate) for e, _ in valid]
        u = [self.packed(synth.UP, e, sh.dff, sh.din, sh.bits_up) for e, _ in valid]
        d = [self.packed(synth.DOWN, e, sh.din, sh.dff, sh.bits_down) for e, _ in valid]
        n, w, b = sh.n_shared, sh.dff_shared, sh.bits_shared
        sg = [self.packed(synth.SH_GATE, i, w, sh.din, b) for i in range(n)]
        su = [self.packed(synth.SH_UP, i, w, sh.din, b) for i in range(n)]
        sd = [self.packed(synth.SH_DOWN, i, sh.din, w, b) for i in range(n)]
        gv = synth.gate_vector(sh.seed, self.layer, sh.din) if (n and sh.shared_gate) else None
        sc = np.array([w_ for _, w_ in valid], dtype=np.float32)
        return O.moe_token(x_bits, resid, sc, g, u, d, sg, su, sd, gate_vec_bf16=gv, rows=rows)



def _tokens_job(shape: Shape, layer: int, x, r, ids, sc, rows):
    ora = OracleLayer(shape, layer)
    return [ora.token(x[t], r[t], ids[t], sc[t], rows=rows) for t in range(len(x))]


def oracle_tokens(shape: Shape, layer: int, x, r, ids, sc, rows=None, workers: int | None = None):
    """The oracle's output of every token of a batch ([m] arrays, fp64), the tokens shared out over
    `workers` spawned processes (default: the host's cores, at most 16, at most one per token)."""
    m = len(x)
    n = min(m, workers or min(16, os.cpu_count() or 1))
    if n <= 1:
        return _tokens_job(shape, layer, x, r, ids, sc, rows)
    parts = [c for c in np.array_split(np.arange(m), n) if len(c)]
    ctx = multiprocessing.get_context("spawn")
    with ProcessPoolExecutor(max_workers=len(parts), mp_context=ctx) as ex:
        futs = [ex.submit(_tokens_job, shape, layer, x[c], r[c], ids[c], sc[c], rows)
                for c in parts]
        out = []
        for f in futs:
            out.extend(f.result())
    return out
