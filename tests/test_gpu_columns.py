"""GPU parity of the column-split kernel mode (MOE_KERNELS_COLUMNS) through the C ABI.

In this mode every CTA carries a range of activation columns through gate/up, SwiGLU and the
matching columns of a column-block-major copy of the down projections, and the row owners sum the
per-CTA partial outputs in a fixed order: one device-wide barrier per layer.  Its sums associate
differently from the row-split modes, so it is held to the oracle's parity bar (not to the other
modes bit for bit), to itself (stack graph == chain of single-layer forwards, byte for byte; the
ids-ahead variant == the strict one, byte for byte) and to repeatability.
"""
import numpy as np
import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300.workloads import (ALL, QWEN3_30B_A3B_4BIT_LAYER,
                                                          QWEN15_MOE_A27B_LAYER, Shape)
from tests import gpu_cases as C
from tests.test_gpu_stack import check_contributions, check_layers, stack_inputs

pytestmark = pytest.mark.gpu
COLS = Bn.KERNELS_COLUMNS


def run_layer(layer, x, r, ids, sc, resid_dtype=Bn.DTYPE_BF16, out_dtype=Bn.DTYPE_F32,
              resid_dev=None, out=None):
    blk = Bn.MoeDecode(layer, max_tokens=1, resid_dtype=resid_dtype, out_dtype=out_dtype,
                       kernel_mode=COLS)
    rd = C.dev(r, torch.bfloat16) if resid_dev is None else resid_dev
    o = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                    rd, out=out)
    torch.cuda.synchronize()
    err = blk.get_error()
    blk.close()
    return o, err


def run_chain(layers, x, ids, sc, resid0):
    outs, prev = [], C.dev(resid0, torch.bfloat16)
    for l, ld in enumerate(layers):
        blk = Bn.MoeDecode(ld, max_tokens=1, resid_dtype=Bn.DTYPE_BF16 if l == 0 else Bn.DTYPE_F32,
                           kernel_mode=COLS)
        o = blk.forward(C.dev(x[l], torch.bfloat16), C.dev(ids[l], torch.int32),
                        C.dev(sc[l], torch.float32), prev)
        torch.cuda.synchronize()
        assert blk.get_error() == 0
        blk.close()
        outs.append(o)
        prev = o
    return outs


LAYERS = {
    # 8-bit down, a gated 4-bit shared expert
    "256x128 E8 K2 8/8/8 + gated shared 4-bit": Shape("c1", 256, 128, 8, 2, 8, 8, 8, n_shared=1,
                                                      dff_shared=128, bits_shared=4,
                                                      shared_gate=1, seed=41),
    # 4-bit down under 4-bit gate/up, ragged widths (din not a multiple of 1024: idle lanes)
    "384x192 E10 K3 4/4/4": Shape("c2", 384, 192, 10, 3, 4, 4, 4, seed=42),
    # 6-bit gate/up (stored as bytes in the records), 4-bit down
    "384x192 E10 K3 6/6/4": Shape("c2b", 384, 192, 10, 3, 6, 6, 4, seed=55),
    # fewer columns than CTAs: most CTAs own nothing and contribute zero partials
    "64x64 E4 K2 8/8/4": Shape("c3", 64, 64, 4, 2, 8, 8, 4, seed=43),
    # din > 2048: two row quads per thread; two ungated 8-bit shared experts
    "4096x128 E6 K3 4/4/8 two shared": Shape("c4", 4096, 128, 6, 3, 4, 4, 8, n_shared=2,
                                             dff_shared=192, bits_shared=8, seed=44),
    # shared experts only
    "256 shared only 8-bit": Shape("c5", 256, 64, 1, 0, 8, 8, 8, n_shared=2, dff_shared=128,
                                   bits_shared=8, shared_gate=1, seed=45),
    # 6-bit down codes (widened to bytes in the column-block copy), 8-bit shared expert
    "512x192 E6 K2 8/8/6 + shared 6-bit": Shape("c8", 512, 192, 6, 2, 8, 8, 6, n_shared=1,
                                               dff_shared=128, bits_shared=6, seed=53),
    "qwen3-30b-a3b layer (full size)": QWEN3_30B_A3B_4BIT_LAYER,
    "qwen1.5-moe-a2.7b layer (full size)": QWEN15_MOE_A27B_LAYER,
    # dots.llm1-like layer: din 4096, 4-bit gate/up, 6-bit down, two ungated 4-bit shared experts
    "dots-like layer 4/4/6 (full size)": Shape("dots-like layer", 4096, 1408, 128, 6, 4, 4, 6,
                                                n_shared=2, dff_shared=1408, bits_shared=4,
                                                seed=54),
}


@pytest.mark.parametrize("name", list(LAYERS))
def test_columns_layer_matches_oracle_on_every_row(name):
    shape = LAYERS[name]
    layer = (C.host_layer_device(shape) if shape.layer_weight_bytes() < 1 << 30
             else Bn.synth_layer_device(shape, 0))
    x, r, ids, sc = C.token_inputs(shape)
    out, err = run_layer(layer, x, r, ids, sc)
    assert err == 0
    ref = C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0])
    C.assert_parity(out.cpu().numpy(), ref, name)
    again, _ = run_layer(layer, x, r, ids, sc)
    assert torch.equal(out.view(torch.int32), again.view(torch.int32))


def test_columns_bad_ids_set_the_error_word_and_contribute_nothing():
    shape = Shape("cbad", 256, 128, 6, 3, 8, 8, 8, seed=46)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    ids = ids.copy()
    ids[0, 0] = -1
    ids[0, 2] = shape.n_experts
    out, err = run_layer(layer, x, r, ids, sc)
    assert err == Bn.MOE_ERR_BAD_ID
    C.assert_parity(out.cpu().numpy(), C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0]),
                    "bad ids")


def test_columns_fp32_resid_aliasing_out_and_bf16_out():
    shape = Shape("cdt", 512, 256, 8, 4, 4, 4, 8, n_shared=1, dff_shared=64, bits_shared=4,
                  shared_gate=1, seed=47)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    r32 = np.random.default_rng(6).standard_normal((1, shape.din)).astype(np.float32) * 3
    buf = C.dev(r32, torch.float32)
    out, _ = run_layer(layer, x, r, ids, sc, resid_dtype=Bn.DTYPE_F32, resid_dev=buf, out=buf)
    C.assert_parity(out.cpu().numpy(), C.OracleLayer(shape).token(x[0], r32[0], ids[0], sc[0]),
                    "fp32 resid, out aliasing resid")
    out16, _ = run_layer(layer, x, r, ids, sc, out_dtype=Bn.DTYPE_BF16)
    assert out16.dtype == torch.bfloat16
    C.assert_parity_bf16(out16, C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0]), "bf16")


@pytest.mark.parametrize("shape", [
    Shape("cs1", 256, 128, 8, 2, 8, 8, 8, n_shared=1, dff_shared=128, bits_shared=4,
          shared_gate=1, layers=4, seed=48),
    Shape("cs2", 384, 192, 10, 3, 4, 4, 4, layers=3, seed=49),
])
def test_columns_small_stack_equals_chain_and_oracle(shape):
    layers = [C.host_layer_device(shape, l) for l in range(shape.layers)]
    x, ids, sc, resid0 = stack_inputs(shape)
    stack = Bn.MoeStack(layers, max_tokens=1, kernel_mode=COLS)
    out = torch.empty((1, shape.din), dtype=torch.float32, device="cuda")
    args = (C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
            C.dev(resid0, torch.bfloat16))
    stack.step(*args, out)
    torch.cuda.synchronize()
    assert stack.get_error() == 0
    out2 = torch.empty_like(out)
    stack.step(*args, out2)   # a second replay of the same graph
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
    outs = run_chain(layers, x, ids, sc, resid0)
    assert torch.equal(out.view(torch.int32), outs[-1].view(torch.int32))
    check_layers(shape, x, ids, sc, resid0, outs, np.arange(shape.din))
    stack.close()
    # ids known ahead: the same arithmetic, the weight stream running on across layers
    ahead = Bn.MoeStack(layers, max_tokens=1, kernel_mode=Bn.KERNELS_COLUMNS_AHEAD)
    out3 = torch.empty_like(out)
    ahead.step(*args, out3)
    torch.cuda.synchronize()
    assert ahead.get_error() == 0
    assert torch.equal(out.view(torch.int32), out3.view(torch.int32))
    ahead.close()


@pytest.mark.parametrize("name", ["qwen3_stack_8bit", "e512_stack", "dots_stack_mixed"])
def test_columns_full_size_stack(name):
    shape = ALL[name]
    free, _ = torch.cuda.mem_get_info()
    need = shape.layer_weight_bytes() * shape.layers * 1.4   # plus the down copies
    assert free > need, f"needs {need / 1e9:.1f} GB of device memory"
    try:
        layers = [Bn.synth_layer_device(shape, l) for l in range(shape.layers)]
        x, ids, sc, resid0 = stack_inputs(shape)
        stack = Bn.MoeStack(layers, max_tokens=1, kernel_mode=COLS)
        out = torch.empty((1, shape.din), dtype=torch.float32, device="cuda")
        stack.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                   C.dev(resid0, torch.bfloat16), out)
        torch.cuda.synchronize()
        assert stack.get_error() == 0
        stack.close()
        ahead = Bn.MoeStack(layers, max_tokens=1, kernel_mode=Bn.KERNELS_COLUMNS_AHEAD)
        out_ahead = torch.empty_like(out)
        ahead.step(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                   C.dev(resid0, torch.bfloat16), out_ahead)
        torch.cuda.synchronize()
        assert ahead.get_error() == 0
        ahead.close()
        assert torch.equal(out.view(torch.int32), out_ahead.view(torch.int32))
        outs = run_chain(layers, x, ids, sc, resid0)
        assert torch.equal(out.view(torch.int32), outs[-1].view(torch.int32))
        rng = np.random.default_rng(8)
        rows = np.unique(np.concatenate([[0, shape.din - 1],
                                         rng.choice(shape.din, 62, replace=False)]))
        L = shape.layers
        check_contributions(shape, x, ids, sc, resid0, outs, [0, 1, L // 2, L - 1], rows)
    finally:
        layers = None
        torch.cuda.empty_cache()


def test_columns_mode_rejects_what_it_does_not_run():
    wide = C.host_layer_device(Shape("c6w", 8192, 64, 2, 1, 4, 4, 8, seed=52))
    with pytest.raises(Bn.MoeError) as e:
        Bn.MoeDecode(wide, kernel_mode=COLS)           # din above 4096
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    ok = C.host_layer_device(Shape("c7", 128, 64, 4, 2, 4, 4, 8, layers=2, seed=51))
    with pytest.raises(Bn.MoeError) as e:
        Bn.MoeDecode(ok, max_tokens=2, kernel_mode=COLS)   # batches
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    norm = torch.ones((1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Bn.MoeError) as e:
        Bn.MoeStack([ok, ok], kernel_mode=COLS, norm_weight=norm)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
