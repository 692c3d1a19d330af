"""Writes tests/golden/oracle_tiny_block.json from the oracle alone.

The pages print no worked numeric example of the block (no input with its output values), so no
fixture here can quote them.  This fixture is a regression record instead: the oracle's fp64
output on one tiny seeded case, written by this script, which calls only oracle/ and the input
generators.  Re-run it only when a change to the oracle's arithmetic is justified by the pages.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import oracle as O  # noqa: E402
from quantized_moe_expert_dequant_gb300 import synth  # noqa: E402

CASE = dict(seed=0x601D, din=128, dff=64, n_experts=4, top_k=2, bits=[4, 4, 6], n_shared=1,
            dff_shared=128, bits_shared=8, shared_gate=1)


def compute(case):
    s, din, dff = case["seed"], case["din"], case["dff"]
    bg, bu, bd = case["bits"]
    ids = synth.topk_ids(s, 0, 0, case["n_experts"], case["top_k"])
    sc = synth.scores(s, 0, 0, case["top_k"])
    pk = lambda proj, e, r, c, b: O.Packed(*synth.expert_proj(s, 0, proj, e, r, c, b), b)
    gate = [pk(synth.GATE, e, dff, din, bg) for e in ids]
    up = [pk(synth.UP, e, dff, din, bu) for e in ids]
    down = [pk(synth.DOWN, e, din, dff, bd) for e in ids]
    dsh, bsh = case["dff_shared"], case["bits_shared"]
    shg = [pk(synth.SH_GATE, i, dsh, din, bsh) for i in range(case["n_shared"])]
    shu = [pk(synth.SH_UP, i, dsh, din, bsh) for i in range(case["n_shared"])]
    shd = [pk(synth.SH_DOWN, i, din, dsh, bsh) for i in range(case["n_shared"])]
    gv = synth.gate_vector(s, 0, din) if case["shared_gate"] else None
    out = O.moe_token(synth.activations(s, 0, 0, din), synth.residual(s, 0, 0, din), sc,
                      gate, up, down, shg, shu, shd, gate_vec_bf16=gv)
    return ids, sc, out


if __name__ == "__main__":
    ids, sc, out = compute(CASE)
    rec = dict(case=CASE, ids=ids.tolist(), scores=[float(v) for v in sc],
               out_hex=[float(v).hex() for v in out],
               note="oracle fp64 output; regression record, not a value printed by the pages")
    with open(os.path.join(HERE, "oracle_tiny_block.json"), "w") as f:
        json.dump(rec, f, indent=1)
    print("wrote", len(out), "values")
