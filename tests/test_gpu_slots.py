"""The route each kernel took, exported by the kernels themselves (moe_decode_routes).

Every kernel mode writes the expert ids its producer read; they must be the input ids, in slot
order, bit for bit (including duplicate and out-of-range ids).  In the pool mode (the page's
pool-and-tail form of "Red Lite dev39 -- fused expert tail", Change, kept apart) the per-slot down
outputs W_down[id] . act (before the score) and the shared experts' (before the scalar) are
exported too, and every one of them must match the oracle's own per-expert MLP element by element
at the parity bar: a slot that read the wrong expert, a swapped slot order or a dropped shared
expert fails there, not only in the summed output.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300 import synth
from quantized_moe_expert_dequant_gb300.workloads import (QWEN3_30B_A3B_4BIT_LAYER,
                                                          QWEN15_MOE_A27B_LAYER, Shape)
from tests import gpu_cases as C

pytestmark = pytest.mark.gpu

SMALL = Shape("slots", 256, 128, 12, 4, 8, 8, 4, n_shared=1, dff_shared=192, bits_shared=8,
              shared_gate=1, seed=81)
DOTS_LIKE = Shape("dots-like layer, 4/4/6, two shared", 4096, 1408, 128, 6, 4, 4, 6, n_shared=2,
                  dff_shared=1408, bits_shared=4, seed=82)


def run(layer, mode, m, x, r, ids, sc, slots=False):
    blk = Bn.MoeDecode(layer, max_tokens=m, kernel_mode=mode)
    out = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                      C.dev(r, torch.bfloat16))
    torch.cuda.synchronize()
    routes = blk.routes(m, slots=slots)
    torch.cuda.synchronize()
    err = blk.get_error()
    blk.close()
    return out, routes, err


def odd_ids(shape, ids):
    """A duplicate of slot 0 in the last slot and an id past the experts in slot 1 of token 0."""
    ids = ids.copy()
    ids[0, -1] = ids[0, 0]
    ids[0, 1] = shape.n_experts + 3
    return ids


@pytest.mark.parametrize("mode,m", [(Bn.KERNELS_FUSED, 1), (Bn.KERNELS_FUSED, 3),
                                    (Bn.KERNELS_SEPARATE, 2), (Bn.KERNELS_COLUMNS, 1),
                                    (Bn.KERNELS_POOL, 1), (Bn.KERNELS_POOL, 3)])
def test_the_kernels_read_the_input_ids_in_slot_order(mode, m):
    shape = SMALL if mode != Bn.KERNELS_COLUMNS else SMALL.with_(bits_down=8)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape, m=m)
    ids = odd_ids(shape, ids)
    out, used, err = run(layer, mode, m, x, r, ids, sc)
    assert err == Bn.MOE_ERR_BAD_ID
    assert np.array_equal(used.cpu().numpy(), ids)
    for t in range(m):
        C.assert_parity(out[t].cpu().numpy(), C.OracleLayer(shape).token(x[t], r[t], ids[t], sc[t]),
                        f"token {t}")


def oracle_slots(shape, x_bits, ids):
    """Per routed slot W_down[id] . act_slot and per shared expert the same, fp64 [K + n_sh, din]
    (None for a slot whose id is out of range)."""
    ol = C.OracleLayer(shape)
    xd = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    out = []
    for e in ids:
        e = int(e)
        if not 0 <= e < shape.n_experts:
            out.append(None)
            continue
        act = O.expert_act(ol.packed(synth.GATE, e, shape.dff, shape.din, shape.bits_gate),
                           ol.packed(synth.UP, e, shape.dff, shape.din, shape.bits_up), xd)
        out.append(O.matvec(ol.packed(synth.DOWN, e, shape.din, shape.dff, shape.bits_down), act))
    w, b = shape.dff_shared, shape.bits_shared
    for i in range(shape.n_shared):
        act = O.expert_act(ol.packed(synth.SH_GATE, i, w, shape.din, b),
                           ol.packed(synth.SH_UP, i, w, shape.din, b), xd)
        out.append(O.matvec(ol.packed(synth.SH_DOWN, i, shape.din, w, b), act))
    return out


@pytest.mark.parametrize("shape,m", [(SMALL, 1), (SMALL, 3), (QWEN3_30B_A3B_4BIT_LAYER, 2),
                                     (QWEN15_MOE_A27B_LAYER, 1), (DOTS_LIKE, 1)],
                         ids=["small m1", "small m3", "qwen3 layer m2", "qwen1.5 layer m1",
                              "dots-like layer m1"])
def test_pool_exports_every_slot_output_matching_the_oracle(shape, m):
    layer = (C.host_layer_device(shape) if shape.n_experts * shape.expert_bytes() < 1 << 30
             else Bn.synth_layer_device(shape, 0))
    x, r, ids, sc = C.token_inputs(shape, m=m)
    if m > 1:
        ids[1, 0] = ids[0, 0]     # two tokens name one expert: streamed once, two outputs
    out, (used, y), err = run(layer, Bn.KERNELS_POOL, m, x, r, ids, sc, slots=True)
    assert err == 0
    assert np.array_equal(used.cpu().numpy(), ids)
    y = y.cpu().numpy()
    for t in range(m):
        ref = oracle_slots(shape, x[t], ids[t])
        for k, yk in enumerate(ref):
            C.assert_parity(y[t, k], yk, f"token {t} slot {k} (expert "
                            f"{ids[t, k] if k < shape.top_k else 'shared'})")
        C.assert_parity(out[t].cpu().numpy(), C.OracleLayer(shape).token(x[t], r[t], ids[t], sc[t]),
                        f"token {t} output")


def test_pool_tail_is_the_pages_weighted_sum_of_the_exported_outputs():
    """out = resid + (sum_k score_k y_k + s * sum y_shared), from the exported y, in fp64."""
    shape = SMALL
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape, m=2)
    out, (used, y), err = run(layer, Bn.KERNELS_POOL, 2, x, r, ids, sc, slots=True)
    y = y.cpu().numpy().astype(np.float64)
    gv = synth.bf16_bits_to_f32(synth.gate_vector(shape.seed, 0, shape.din)).astype(np.float64)
    for t in range(2):
        s = 1.0 / (1.0 + np.exp(-np.dot(synth.bf16_bits_to_f32(x[t]).astype(np.float64), gv)))
        want = (synth.bf16_bits_to_f32(r[t]).astype(np.float64)
                + (sc[t].astype(np.float64) @ y[t, :shape.top_k] + s * y[t, shape.top_k:].sum(0)))
        C.assert_parity(out[t].cpu().numpy(), want, f"token {t}")


def test_routes_arguments():
    layer = C.host_layer_device(SMALL)
    blk = Bn.MoeDecode(layer, kernel_mode=Bn.KERNELS_FUSED)
    with pytest.raises(Bn.MoeError) as e:
        blk.routes(1)                                   # no forward yet
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG
    x, r, ids, sc = C.token_inputs(SMALL)
    blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                C.dev(r, torch.bfloat16))
    with pytest.raises(Bn.MoeError) as e:
        blk.routes(1, slots=True)                       # slot outputs: pool mode only
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    blk.close()
