"""The tensor-core batch mode (MOE_KERNELS_MMA) through the C ABI: every row of every token against
the oracle at the parity bar, on small shapes of every code width and on full-size layers at
8 and 32 tokens; the route it read (ids bit for bit, invalid and repeated ids); the stack; limits.
"""
import numpy as np
import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300.workloads import ALL, Shape
from tests import gpu_cases as C
from tests.test_gpu_stack import check_contributions, run_chain, stack_inputs

pytestmark = pytest.mark.gpu


def forward(layer, x, r, ids, sc, m, resid_dtype=Bn.DTYPE_BF16, out_dtype=Bn.DTYPE_F32):
    blk = Bn.MoeDecode(layer, max_tokens=m, kernel_mode=Bn.KERNELS_MMA, resid_dtype=resid_dtype,
                       out_dtype=out_dtype)
    rt = C.dev(r, torch.bfloat16) if resid_dtype == Bn.DTYPE_BF16 else C.dev(r, torch.float32)
    out = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                      rt)
    torch.cuda.synchronize()
    used = blk.routes(m)
    torch.cuda.synchronize()
    err = blk.get_error()
    blk.close()
    return out, used.cpu().numpy(), err


def check_all(shape, out, x, r, ids, sc):
    refs = C.oracle_tokens(shape, 0, x, r, ids, sc)
    for t, ref in enumerate(refs):
        C.assert_parity(out[t].cpu().numpy(), ref, f"{shape.name}: token {t}")


SMALL = {
    "gated shared 256x128 E8 K2 4/4/6, m=5": (Shape("m1", 256, 128, 8, 2, 4, 4, 6, n_shared=1,
                                                    dff_shared=128, bits_shared=8, shared_gate=1,
                                                    seed=61), 5),
    "8-bit 512x192 E16 K4, m=8": (Shape("m2", 512, 192, 16, 4, 8, 8, 8, seed=62), 8),
    "two shared 384x256 E12 K3 8/8/4, m=11": (Shape("m3", 384, 256, 12, 3, 8, 8, 4, n_shared=2,
                                                    dff_shared=192, bits_shared=6, seed=63), 11),
    "every expert E5 K5 6/6/8, m=3": (Shape("m4", 128, 192, 5, 5, 6, 6, 8, seed=64), 3),
    "shared only 6-bit, m=4": (Shape("m5", 256, 64, 1, 0, 4, 4, 4, n_shared=2, dff_shared=128,
                                     bits_shared=6, shared_gate=1, seed=65), 4),
    "one token 6/6/6, m=1": (Shape("m6", 320, 192, 9, 3, 6, 6, 6, seed=66), 1),
    "17 tokens past two pair tiles, m=17": (Shape("m7", 192, 128, 4, 2, 4, 4, 4, n_shared=1,
                                                  dff_shared=64, bits_shared=4, seed=67), 17),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_batches_every_row(name):
    shape, m = SMALL[name]
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape, m=m)
    out, used, err = forward(layer, x, r, ids, sc, m)
    assert err == 0
    assert np.array_equal(used, ids)
    check_all(shape, out, x, r, ids, sc)


def test_fp32_residual_and_bf16_output():
    shape, m = SMALL["two shared 384x256 E12 K3 8/8/4, m=11"]
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape, m=m)
    r32 = np.random.default_rng(5).standard_normal((m, shape.din)).astype(np.float32)
    out, _, err = forward(layer, x, r32, ids, sc, m, resid_dtype=Bn.DTYPE_F32,
                          out_dtype=Bn.DTYPE_BF16)
    assert err == 0
    ora = C.OracleLayer(shape)
    for t in range(m):
        C.assert_parity_bf16(out[t], ora.token(x[t], r32[t], ids[t], sc[t]), f"token {t}")


FULL = [("dots_stack_mixed", 8), ("dots_stack_mixed", 32), ("qwen3_stack_8bit", 32),
        ("qwen3_layer_4bit", 8), ("qwen15_layer_shared", 8), ("e512_stack", 16)]


@pytest.mark.parametrize("name,m", FULL)
def test_full_size_layer_every_row(name, m):
    """A full-size layer: every output row of every token against the oracle."""
    shape = ALL[name].with_(layers=1)
    layer = Bn.synth_layer_device(shape, 0)
    x, r, ids, sc = C.token_inputs(shape, m=m, step=3)
    out, used, err = forward(layer, x, r, ids, sc, m)
    assert err == 0
    assert np.array_equal(used, ids)
    del layer
    torch.cuda.empty_cache()
    check_all(shape, out, x, r, ids, sc)


def test_repeated_and_invalid_ids():
    shape = Shape("m8", 256, 128, 6, 3, 8, 8, 4, n_shared=1, dff_shared=64, bits_shared=4,
                  shared_gate=1, seed=68)
    layer = C.host_layer_device(shape)
    m = 6
    x, r, ids, sc = C.token_inputs(shape, m=m)
    same = np.tile(ids[:1], (m, 1))          # every token names the same experts
    out, used, err = forward(layer, x, r, same, sc, m)
    assert err == 0 and np.array_equal(used, same)
    check_all(shape, out, x, r, same, sc)
    bad = ids.copy()
    bad[1, 0] = -4
    bad[4, 2] = shape.n_experts
    bad[2, 2] = bad[2, 0]                    # one token names one expert twice
    out, used, err = forward(layer, x, r, bad, sc, m)
    assert err == Bn.MOE_ERR_BAD_ID
    assert np.array_equal(used, bad)
    check_all(shape, out, x, r, bad, sc)     # the oracle drops the invalid slots


def test_agrees_with_the_grouped_kernel_within_the_bar():
    shape = ALL["dots_stack_mixed"].with_(layers=1)
    layer = Bn.synth_layer_device(shape, 0)
    m = 8
    x, r, ids, sc = C.token_inputs(shape, m=m, step=4)
    a, _, ea = forward(layer, x, r, ids, sc, m)
    blk = Bn.MoeDecode(layer, max_tokens=m, kernel_mode=Bn.KERNELS_FUSED)
    b = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                    C.dev(r, torch.bfloat16))
    torch.cuda.synchronize()
    assert ea == 0 and blk.get_error() == 0
    blk.close()
    for t in range(m):
        C.assert_parity(a[t].cpu().numpy(), b[t].cpu().numpy().astype(np.float64), f"token {t}")


def test_stack_equals_its_layers_and_repeats_exactly():
    shape = Shape("m9", 384, 192, 10, 3, 8, 8, 6, n_shared=1, dff_shared=128, bits_shared=4,
                  shared_gate=1, layers=3, seed=69)
    layers = [C.host_layer_device(shape, l) for l in range(shape.layers)]
    m = 5
    per = [C.token_inputs(shape, layer=l, m=m) for l in range(shape.layers)]
    x = np.stack([p[0] for p in per])
    ids = np.stack([p[2] for p in per])
    sc = np.stack([p[3] for p in per])
    r0 = per[0][1]
    stack = Bn.MoeStack(layers, max_tokens=m, kernel_mode=Bn.KERNELS_MMA)
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
        blk = Bn.MoeDecode(ld, max_tokens=m, kernel_mode=Bn.KERNELS_MMA,
                           resid_dtype=Bn.DTYPE_BF16 if l == 0 else Bn.DTYPE_F32)
        o = blk.forward(C.dev(x[l], torch.bfloat16), C.dev(ids[l], torch.int32),
                        C.dev(sc[l], torch.float32), prev)
        torch.cuda.synchronize()
        assert blk.get_error() == 0
        blk.close()
        for t in range(m):
            C.assert_parity(o[t].cpu().numpy(), ref[l][t], f"layer {l} token {t}")
        prev = o
    assert torch.equal(outs[0].view(torch.int32), prev.view(torch.int32))


def test_limits():
    shape = SMALL["8-bit 512x192 E16 K4, m=8"][0]
    layer = C.host_layer_device(shape)
    with pytest.raises(Bn.MoeError) as e:        # more than 64 tokens
        Bn.MoeDecode(layer, max_tokens=65, kernel_mode=Bn.KERNELS_MMA)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    wide = shape.with_(top_k=8, n_experts=16)    # 40 x 8 = 320 slots > 256
    with pytest.raises(Bn.MoeError) as e:
        Bn.MoeDecode(C.host_layer_device(wide), max_tokens=40, kernel_mode=Bn.KERNELS_MMA)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    norm = torch.ones((1, shape.din), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Bn.MoeError) as e:        # the chained stack reads RMSNorm of the output
        Bn.MoeStack([layer, layer], max_tokens=2, kernel_mode=Bn.KERNELS_MMA, norm_weight=norm)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,m", [("qwen3_stack_8bit", 8), ("dots_stack_mixed", 32)])
def test_full_size_stack(name, m):
    """The full stack in the bench's launch configuration (one graph per step, five launches per
    layer): byte-identical to the same layers run one forward each, and each checked layer's block
    term out_l - out_{l-1} against the oracle on sampled rows of three tokens."""
    shape = ALL[name]
    free, _ = torch.cuda.mem_get_info()
    need = shape.layer_weight_bytes() * shape.layers * 2.1   # plus the tile-group copies
    assert free > need, f"needs {need / 1e9:.1f} GB of device memory"
    try:
        layers = [Bn.synth_layer_device(shape, l) for l in range(shape.layers)]
        x, ids, sc, resid0 = stack_inputs(shape, m=m, step=5)
        stack = Bn.MoeStack(layers, max_tokens=m, kernel_mode=Bn.KERNELS_MMA)
        out = torch.empty((m, shape.din), dtype=torch.float32, device="cuda")
        stack.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                   C.dev(resid0, torch.bfloat16), out)
        torch.cuda.synchronize()
        assert stack.get_error() == 0
        stack.close()
        outs = run_chain(layers, x, ids, sc, resid0, m, mode=Bn.KERNELS_MMA)
        assert torch.equal(out.view(torch.int32), outs[-1].view(torch.int32))
        rng = np.random.default_rng(11)
        rows = np.unique(np.concatenate([[0, shape.din - 1],
                                         rng.choice(shape.din, 62, replace=False)]))
        L = shape.layers
        check_contributions(shape, x, ids, sc, resid0, outs, [0, 1, L // 2, L - 1], rows,
                            tokens=(0, m // 2, m - 1))
    finally:
        layers = None
        torch.cuda.empty_cache()
