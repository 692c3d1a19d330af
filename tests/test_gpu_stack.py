"""GPU parity of the layer-stack driver (one CUDA graph per decode step) through the C ABI.

The graph replay must equal the same layers run one forward at a time, byte for byte.  Small
stacks match the oracle's own chain (its outputs feed its next layer) at every layer and row; the
full-size stacks, run in the configuration the benchmark times, are checked on sampled rows of
sampled layers through each layer's block term (out_l - out_{l-1}), which the oracle computes from
the seeded inputs alone.
"""
import numpy as np
import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300 import synth
from quantized_moe_expert_dequant_gb300.workloads import ALL, Shape
from tests import gpu_cases as C

pytestmark = pytest.mark.gpu


def stack_inputs(shape, m=1, step=0):
    per = [C.token_inputs(shape, layer=l, m=m, step=step) for l in range(shape.layers)]
    x = np.stack([p[0] for p in per])                  # [L, m, din] bf16 bits
    ids = np.stack([p[2] for p in per])                # [L, m, K]
    sc = np.stack([p[3] for p in per])
    resid0 = per[0][1]                                 # [m, din] bf16 bits
    return x, ids, sc, resid0


def run_chain(layers, x, ids, sc, resid0, m, mode=Bn.KERNELS_FUSED):
    """The same layers, one moe_decode_forward each (same kernel mode); every layer's output."""
    outs = []
    prev = C.dev(resid0, torch.bfloat16)
    for l, ld in enumerate(layers):
        blk = Bn.MoeDecode(ld, max_tokens=m,
                           resid_dtype=Bn.DTYPE_BF16 if l == 0 else Bn.DTYPE_F32, kernel_mode=mode)
        o = blk.forward(C.dev(x[l], torch.bfloat16), C.dev(ids[l], torch.int32),
                        C.dev(sc[l], torch.float32), prev)
        torch.cuda.synchronize()
        assert blk.get_error() == 0
        blk.close()
        outs.append(o)
        prev = o
    return outs


def check_layers(shape, x, ids, sc, resid0, outs, rows, tokens=(0,)):
    """Every layer's output against the oracle's own chain (rows: the rows the oracle computes)."""
    ref = C.oracle_stack(shape, x, ids, sc, resid0, m=max(tokens) + 1, rows=rows)
    for l in range(shape.layers):
        for t in tokens:
            got = outs[l][t].cpu().numpy()[rows]
            C.assert_parity(got, ref[l][t], f"{shape.name}: layer {l} token {t}")


def check_contributions(shape, x, ids, sc, resid0, outs, layers_to_check, rows, tokens=(0,)):
    """Layers of a full-size stack, on sampled rows, through a property that holds at any size:
    a layer adds its block term to its residual, so out_l - out_{l-1} is the oracle's block output
    with a zero residual on the same seeded inputs (layer 0: out_0 - resid0).  The fp32 sum in the
    tail rounds once, far below the parity bar."""
    zero = np.zeros(shape.din, np.float32)
    for l in layers_to_check:
        ora = C.OracleLayer(shape, l)
        for t in tokens:
            got = outs[l][t].cpu().numpy().astype(np.float64)
            prev = (synth.bf16_bits_to_f32(resid0[t]) if l == 0
                    else outs[l - 1][t].cpu().numpy()).astype(np.float64)
            ref = ora.token(x[l][t], zero, ids[l][t], sc[l][t], rows=rows)
            C.assert_parity((got - prev)[rows], ref,
                            f"{shape.name}: layer {l} token {t} block term")


def test_small_stack_graph_equals_chain_and_oracle():
    shape = Shape("small stack", 256, 128, 8, 2, 4, 4, 6, n_shared=1, dff_shared=128,
                  bits_shared=8, shared_gate=1, layers=4, seed=31)
    layers = [C.host_layer_device(shape, l) for l in range(shape.layers)]
    x, ids, sc, resid0 = stack_inputs(shape)
    stack = Bn.MoeStack(layers, max_tokens=1)
    out = torch.empty((1, shape.din), dtype=torch.float32, device="cuda")
    stack.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
               C.dev(resid0, torch.bfloat16), out)
    torch.cuda.synchronize()
    assert stack.get_error() == 0
    outs = run_chain(layers, x, ids, sc, resid0, 1)
    assert torch.equal(out.view(torch.int32), outs[-1].view(torch.int32))
    check_layers(shape, x, ids, sc, resid0, outs, np.arange(shape.din))
    # the graph is cached per pointer set: a second step with the same buffers replays it
    out2 = torch.empty_like(out)
    xd, idd, scd, rd = (C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                        C.dev(sc, torch.float32), C.dev(resid0, torch.bfloat16))
    stack.step(xd, idd, scd, rd, out2)
    stack.step(xd, idd, scd, rd, out2)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int32), out.view(torch.int32))
    # host buffers in, host result out
    outh = torch.empty((1, shape.din), dtype=torch.float32).pin_memory()
    pin = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if dt == torch.bfloat16
                                         else np.ascontiguousarray(a)).view(dt).pin_memory()
    stack.step_host(pin(x, torch.bfloat16), pin(ids, torch.int32), pin(sc, torch.float32),
                    pin(resid0, torch.bfloat16), outh)
    assert torch.equal(outh.view(torch.int32), out.cpu().view(torch.int32))
    stack.close()


@pytest.mark.parametrize("mode", [Bn.KERNELS_FUSED, Bn.KERNELS_SEPARATE])
def test_small_stack_several_tokens(mode):
    shape = Shape("small stack m3", 384, 192, 10, 3, 6, 6, 4, layers=3, seed=32)
    layers = [C.host_layer_device(shape, l) for l in range(shape.layers)]
    m = 3
    x, ids, sc, resid0 = stack_inputs(shape, m=m)
    stack = Bn.MoeStack(layers, max_tokens=m, kernel_mode=mode)
    out = torch.empty((m, shape.din), dtype=torch.float32, device="cuda")
    stack.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
               C.dev(resid0, torch.bfloat16), out)
    torch.cuda.synchronize()
    outs = run_chain(layers, x, ids, sc, resid0, m, mode)
    assert torch.equal(out.view(torch.int32), outs[-1].view(torch.int32))
    check_layers(shape, x, ids, sc, resid0, outs, np.arange(shape.din), tokens=range(m))
    stack.close()


@pytest.mark.parametrize("name", ["qwen3_stack_8bit", "e512_stack", "dots_stack_mixed"])
def test_full_size_stack(name):
    shape = ALL[name]
    free, _ = torch.cuda.mem_get_info()
    need = shape.layer_weight_bytes() * shape.layers
    assert free > need * 1.05, f"needs {need / 1e9:.1f} GB of device memory"
    try:
        layers = [Bn.synth_layer_device(shape, l) for l in range(shape.layers)]
        x, ids, sc, resid0 = stack_inputs(shape)
        stack = Bn.MoeStack(layers, max_tokens=1)
        out = torch.empty((1, shape.din), dtype=torch.float32, device="cuda")
        stack.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                   C.dev(resid0, torch.bfloat16), out)
        torch.cuda.synchronize()
        assert stack.get_error() == 0
        stack.close()
        outs = run_chain(layers, x, ids, sc, resid0, 1)
        assert torch.equal(out.view(torch.int32), outs[-1].view(torch.int32))
        rng = np.random.default_rng(7)
        rows = np.unique(np.concatenate([[0, shape.din - 1],
                                         rng.choice(shape.din, 62, replace=False)]))
        L = shape.layers
        check_contributions(shape, x, ids, sc, resid0, outs, [0, 1, L // 2, L - 1], rows)
    finally:
        layers = None
        torch.cuda.empty_cache()
