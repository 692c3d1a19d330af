"""GPU parity of one layer of the decode MoE block against the fp64 oracle, through the C ABI.

Integer work (unpacked codes, the device weight generator) must match bit for bit; the fp32
output must meet the parity bar of tests/gpu_cases.py on every row.
"""
import numpy as np
import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300 import synth
from quantized_moe_expert_dequant_gb300.workloads import (QWEN3_30B_A3B_4BIT_LAYER,
                                                          QWEN15_MOE_A27B_LAYER, Shape)
from tests import gpu_cases as C
from tests import helpers as H

pytestmark = pytest.mark.gpu


def test_library_is_the_in_tree_build():
    import os
    assert os.path.dirname(Bn.LIB_PATH).endswith("quantized_moe_expert_dequant_gb300")
    Bn.lib()
    maps = open("/proc/self/maps").read()
    assert Bn.LIB_PATH in maps


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_device_unpack_is_bit_exact(bits):
    rng = np.random.default_rng(100 + bits)
    rows, cols = 7, 448
    packed = rng.integers(0, 256, size=(rows, cols * bits // 8), dtype=np.uint8)
    got = Bn.unpack_codes_device(C.dev(packed, torch.uint8), cols, bits).cpu().numpy()
    assert np.array_equal(got, Bn.unpack_codes(packed, cols, bits))
    for r in (0, rows - 1):
        assert np.array_equal(got[r], H.unpack_bigint(packed[r], bits, cols))


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_device_generator_matches_host_bit_for_bit(bits):
    rows, cols, n = 64, 384, 3
    p = Bn.synth_proj_device(0xABC, 2, synth.DOWN, n, rows, cols, bits)
    torch.cuda.synchronize()
    c, s, b = synth.stacked_proj(0xABC, 2, synth.DOWN, n, rows, cols, bits)
    assert np.array_equal(p.codes.cpu().numpy(), c)
    assert np.array_equal(p.scales.cpu().view(torch.int16).numpy().view(np.uint16), s)
    assert np.array_equal(p.biases.cpu().view(torch.int16).numpy().view(np.uint16), b)


def run_layer(shape, layer_dev, x, r, ids, sc, m=1, resid_dtype=Bn.DTYPE_BF16,
              out_dtype=Bn.DTYPE_F32, resid_values=None):
    blk = Bn.MoeDecode(layer_dev, max_tokens=m, resid_dtype=resid_dtype, out_dtype=out_dtype)
    rd = (C.dev(r, torch.bfloat16) if resid_dtype == Bn.DTYPE_BF16
          else C.dev(resid_values.astype(np.float32), torch.float32))
    out = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                      C.dev(sc, torch.float32), rd)
    torch.cuda.synchronize()
    err = blk.get_error()
    blk.close()
    return out, err


SHAPES = {
    "tiny 64x64 E4 K2 4-bit": Shape("tiny", 64, 64, 4, 2, 4, 4, 4, seed=11),
    "ragged 192x320 E6 K3 6/6/8 gated shared": Shape("ragged", 192, 320, 6, 3, 6, 6, 8, n_shared=1,
                                                     dff_shared=192, bits_shared=4, shared_gate=1,
                                                     seed=12),
    "8-bit 2048x768 E16 K8": Shape("8bit", 2048, 768, 16, 8, 8, 8, 8, seed=13),
    "4096x1408 E12 K6 4/4/6 two shared": Shape("mixed", 4096, 1408, 12, 6, 4, 4, 6, n_shared=2,
                                                dff_shared=1408, bits_shared=4, seed=14),
    "every expert selected E5 K5 8/8/4": Shape("kE", 128, 192, 5, 5, 8, 8, 4, seed=15),
    "shared experts only 6-bit": Shape("shonly", 256, 64, 1, 0, 4, 4, 4, n_shared=3,
                                       dff_shared=128, bits_shared=6, shared_gate=1, seed=16),
    "512x512 E512 K10 gated shared": Shape("e512", 512, 512, 512, 10, 4, 4, 4, n_shared=1,
                                           dff_shared=512, bits_shared=4, shared_gate=1, seed=17),
    "qwen3-30b-a3b layer (full size)": QWEN3_30B_A3B_4BIT_LAYER,
    "qwen1.5-moe-a2.7b layer (full size)": QWEN15_MOE_A27B_LAYER,
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_layer_matches_oracle_on_every_row(name):
    shape = SHAPES[name]
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    out, err = run_layer(shape, layer, x, r, ids, sc)
    assert err == 0
    ref = C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0])
    C.assert_parity(out.cpu().numpy(), ref, name)


def test_each_slot_reads_the_expert_its_id_names():
    shape = Shape("onehot", 256, 128, 8, 4, 4, 4, 6, seed=21)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    ora = C.OracleLayer(shape)
    zero = np.zeros_like(r)
    for k in range(shape.top_k):
        onehot = np.zeros_like(sc)
        onehot[0, k] = 1.0
        out, _ = run_layer(shape, layer, x, zero, ids, onehot)
        ref = ora.token(x[0], zero[0], ids[0][k:k + 1], np.ones(1, np.float32))
        C.assert_parity(out.cpu().numpy(), ref, f"slot {k} -> expert {ids[0][k]}")
        other = ora.token(x[0], zero[0], ids[0][(k + 1) % shape.top_k:][:1], np.ones(1, np.float32))
        assert C.parity(out.cpu().numpy(), other)[2] > 1e-2


def test_out_of_range_ids_set_the_error_word_and_contribute_nothing():
    shape = Shape("badid", 128, 64, 4, 3, 4, 4, 4, seed=22)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    ids = ids.copy()
    ids[0, 0] = -1
    ids[0, 2] = shape.n_experts
    out, err = run_layer(shape, layer, x, r, ids, sc)
    assert err == Bn.MOE_ERR_BAD_ID
    ref = C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0])   # drops the invalid slots
    C.assert_parity(out.cpu().numpy(), ref, "bad ids")


def test_duplicate_ids_are_separate_slots():
    shape = Shape("dup", 128, 128, 4, 3, 6, 6, 4, seed=23)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    ids = np.array([[1, 1, 3]], dtype=np.int32)
    out, err = run_layer(shape, layer, x, r, ids, sc)
    assert err == 0
    ref = C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0])
    C.assert_parity(out.cpu().numpy(), ref, "duplicate ids")


def test_repeat_runs_are_byte_identical():
    shape = QWEN15_MOE_A27B_LAYER
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    a, _ = run_layer(shape, layer, x, r, ids, sc)
    b, _ = run_layer(shape, layer, x, r, ids, sc)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_fp32_resid_and_bf16_out():
    shape = Shape("dtypes", 256, 128, 6, 2, 4, 4, 8, n_shared=1, dff_shared=64, bits_shared=8,
                  shared_gate=1, seed=24)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    r32 = np.random.default_rng(5).standard_normal((1, shape.din)).astype(np.float32) * 3
    out, _ = run_layer(shape, layer, x, r, ids, sc, resid_dtype=Bn.DTYPE_F32, resid_values=r32)
    ref = C.OracleLayer(shape).token(x[0], r32[0], ids[0], sc[0])
    C.assert_parity(out.cpu().numpy(), ref, "fp32 resid")
    out16, _ = run_layer(shape, layer, x, r, ids, sc, out_dtype=Bn.DTYPE_BF16)
    assert out16.dtype == torch.bfloat16
    ref16 = C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0])
    C.assert_parity_bf16(out16, ref16, "bf16 out")


def test_several_tokens_with_their_own_ids():
    shape = Shape("multi", 512, 256, 16, 4, 4, 4, 6, n_shared=1, dff_shared=128, bits_shared=4,
                  seed=25)
    layer = C.host_layer_device(shape)
    m = 5
    x, r, ids, sc = C.token_inputs(shape, m=m)
    out, err = run_layer(shape, layer, x, r, ids, sc, m=m)
    assert err == 0
    ora = C.OracleLayer(shape)
    for t in range(m):
        C.assert_parity(out[t].cpu().numpy(), ora.token(x[t], r[t], ids[t], sc[t]), f"token {t}")


def test_forward_rejects_bad_arguments():
    shape = Shape("args", 128, 64, 4, 2, 4, 4, 4, seed=26)
    layer = C.host_layer_device(shape)
    blk = Bn.MoeDecode(layer, max_tokens=2)
    x, r, ids, sc = C.token_inputs(shape, m=3)
    with pytest.raises(Bn.MoeError) as e:
        blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                    C.dev(r, torch.bfloat16))
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG
    xd = C.dev(x[:1], torch.bfloat16)
    with pytest.raises(Bn.MoeError):
        blk.forward(xd, C.dev(ids[:1], torch.int32), C.dev(sc[:1], torch.float32),
                    C.dev(r[:1], torch.bfloat16), out=xd)   # out may not alias x
    blk.close()


@pytest.mark.parametrize("name", ["ragged 192x320 E6 K3 6/6/8 gated shared",
                                  "4096x1408 E12 K6 4/4/6 two shared",
                                  "qwen3-30b-a3b layer (full size)"])
def test_separate_kernels_match_fused_kernel_bit_for_bit(name):
    shape = SHAPES[name]
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    outs = []
    for mode in (Bn.KERNELS_FUSED, Bn.KERNELS_SEPARATE):
        blk = Bn.MoeDecode(layer, kernel_mode=mode)
        o = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                        C.dev(sc, torch.float32), C.dev(r, torch.bfloat16))
        torch.cuda.synchronize()
        assert blk.get_error() == 0
        blk.close()
        outs.append(o)
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    C.assert_parity(outs[1].cpu().numpy(), C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0]))
