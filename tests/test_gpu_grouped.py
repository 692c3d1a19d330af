"""Batches of tokens grouped by expert (each selected expert streamed once per layer), through the
C ABI: every token must meet the oracle's parity bar, computed token by token on the host."""
import numpy as np
import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300.workloads import ALL, Shape
from tests import gpu_cases as C

pytestmark = pytest.mark.gpu


def forward(layer, x, r, ids, sc, m, mode=Bn.KERNELS_FUSED):
    blk = Bn.MoeDecode(layer, max_tokens=m, kernel_mode=mode)
    out = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                      C.dev(r, torch.bfloat16))
    torch.cuda.synchronize()
    err = blk.get_error()
    blk.close()
    return out, err


def check_tokens(shape, layer_idx, out, x, r, ids, sc, rows=None, tokens=None):
    ora = C.OracleLayer(shape, layer_idx)
    tokens = range(len(x)) if tokens is None else tokens
    for t in tokens:
        ref = ora.token(x[t], r[t], ids[t], sc[t], rows=rows)
        got = out[t].cpu().numpy() if rows is None else out[t].cpu().numpy()[rows]
        C.assert_parity(got, ref, f"{shape.name}: token {t}")


SMALL = {
    "gated shared 256x128 E8 K2 4/4/6, m=5": (Shape("g1", 256, 128, 8, 2, 4, 4, 6, n_shared=1,
                                                    dff_shared=128, bits_shared=8, shared_gate=1,
                                                    seed=41), 5),
    "8-bit 512x192 E16 K4, m=8": (Shape("g2", 512, 192, 16, 4, 8, 8, 8, seed=42), 8),
    "two shared 384x256 E12 K3 8/8/4, m=11": (Shape("g3", 384, 256, 12, 3, 8, 8, 4, n_shared=2,
                                                    dff_shared=192, bits_shared=6, seed=43), 11),
    "every expert E5 K5 6/6/8, m=3": (Shape("g4", 128, 192, 5, 5, 6, 6, 8, seed=44), 3),
    "shared only 6-bit, m=4": (Shape("g5", 256, 64, 1, 0, 4, 4, 4, n_shared=2, dff_shared=128,
                                     bits_shared=6, shared_gate=1, seed=45), 4),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_batches_every_row(name):
    shape, m = SMALL[name]
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape, m=m)
    out, err = forward(layer, x, r, ids, sc, m)
    assert err == 0
    check_tokens(shape, 0, out, x, r, ids, sc)


FULL = [("qwen3_stack_8bit", 8), ("dots_stack_mixed", 8), ("dots_stack_mixed", 32),
        ("e512_stack", 16)]


@pytest.mark.parametrize("name,m", FULL)
def test_full_size_layer_batches(name, m):
    shape = ALL[name].with_(layers=1)
    layer = Bn.synth_layer_device(shape, 0)
    x, r, ids, sc = C.token_inputs(shape, m=m, step=2)
    out, err = forward(layer, x, r, ids, sc, m)
    assert err == 0
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, shape.din - 1], rng.choice(shape.din, 40, replace=False)]))
    check_tokens(shape, 0, out, x, r, ids, sc, rows=rows, tokens=[0, m // 2, m - 1])
    del layer
    torch.cuda.empty_cache()


def test_all_tokens_pick_the_same_experts_and_bad_ids():
    shape = Shape("g6", 256, 128, 6, 3, 4, 4, 4, n_shared=1, dff_shared=64, bits_shared=4,
                  shared_gate=1, seed=46)
    layer = C.host_layer_device(shape)
    m = 6
    x, r, ids, sc = C.token_inputs(shape, m=m)
    same = np.tile(ids[:1], (m, 1))
    out, err = forward(layer, x, r, same, sc, m)
    assert err == 0
    check_tokens(shape, 0, out, x, r, same, sc)
    bad = ids.copy()
    bad[1, 0] = -4
    bad[4, 2] = shape.n_experts
    out, err = forward(layer, x, r, bad, sc, m)
    assert err == Bn.MOE_ERR_BAD_ID
    check_tokens(shape, 0, out, x, r, bad, sc)   # the oracle drops the invalid slots


def test_grouped_stack_equals_grouped_layers_and_repeats_exactly():
    shape = Shape("g7", 384, 192, 10, 3, 8, 8, 6, n_shared=1, dff_shared=128, bits_shared=4,
                  shared_gate=1, layers=3, seed=47)
    layers = [C.host_layer_device(shape, l) for l in range(shape.layers)]
    m = 4
    per = [C.token_inputs(shape, layer=l, m=m) for l in range(shape.layers)]
    x = np.stack([p[0] for p in per])
    ids = np.stack([p[2] for p in per])
    sc = np.stack([p[3] for p in per])
    r0 = per[0][1]
    stack = Bn.MoeStack(layers, max_tokens=m)
    outs = []
    for _ in range(2):
        o = torch.empty((m, shape.din), dtype=torch.float32, device="cuda")
        stack.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                   C.dev(r0, torch.bfloat16), o)
        torch.cuda.synchronize()
        assert stack.get_error() == 0
        outs.append(o)
    stack.close()
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    ref = C.oracle_stack(shape, x, ids, sc, r0, m=m)
    prev = C.dev(r0, torch.bfloat16)
    for l, ld in enumerate(layers):
        blk = Bn.MoeDecode(ld, max_tokens=m, resid_dtype=Bn.DTYPE_BF16 if l == 0 else Bn.DTYPE_F32)
        o = blk.forward(C.dev(x[l], torch.bfloat16), C.dev(ids[l], torch.int32),
                        C.dev(sc[l], torch.float32), prev)
        torch.cuda.synchronize()
        assert blk.get_error() == 0
        blk.close()
        for t in range(m):
            C.assert_parity(o[t].cpu().numpy(), ref[l][t], f"layer {l} token {t}")
        prev = o
    assert torch.equal(outs[0].view(torch.int32), prev.view(torch.int32))
