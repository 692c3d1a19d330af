"""moe_decode_forward_noalloc against moe_decode_forward, through the C ABI.

The handle-free call keeps the activations in the library's fixed scratch array.  Two consecutive
calls on different tokens must each equal the handle's forward byte for byte (the second call
reuses scratch the first one wrote), the call must not change the device's free memory, and it
must work when captured in a CUDA graph after a first call outside capture.  This file is collected
last so it also runs after every other GPU test has used the device.
"""
import ctypes

import numpy as np
import pytest
import torch

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300.workloads import QWEN15_MOE_A27B_LAYER, Shape
from tests import gpu_cases as C

pytestmark = pytest.mark.gpu

SHAPES = {
    "ragged 192x320 E6 K3 6/6/8 gated shared": Shape("ragged", 192, 320, 6, 3, 6, 6, 8, n_shared=1,
                                                     dff_shared=192, bits_shared=4, shared_gate=1,
                                                     seed=12),
    "qwen1.5-moe-a2.7b layer (full size)": QWEN15_MOE_A27B_LAYER,
}


def handle_forward(layer, x, r, ids, sc, m):
    blk = Bn.MoeDecode(layer, max_tokens=m, kernel_mode=Bn.KERNELS_SEPARATE)
    out = blk.forward(C.dev(x, torch.bfloat16), C.dev(ids, torch.int32), C.dev(sc, torch.float32),
                      C.dev(r, torch.bfloat16))
    torch.cuda.synchronize()
    assert blk.get_error() == 0
    blk.close()
    return out


@pytest.mark.parametrize("name", list(SHAPES))
def test_two_consecutive_calls_equal_the_handle_forward(name):
    shape = SHAPES[name]
    layer = C.host_layer_device(shape)
    m = 2
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in (0, 1):
        x, r, ids, sc = C.token_inputs(shape, m=m, step=step)
        ref = handle_forward(layer, x, r, ids, sc, m)
        out = torch.full((m, shape.din), float("nan"), dtype=torch.float32, device="cuda")
        Bn.forward_noalloc(layer, C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                           C.dev(sc, torch.float32), C.dev(r, torch.bfloat16), out,
                           device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"call {step}"
    ora = C.OracleLayer(shape)
    for t in range(m):
        C.assert_parity(out[t].cpu().numpy(), ora.token(x[t], r[t], ids[t], sc[t]), f"token {t}")


def test_calls_allocate_nothing_and_can_be_captured():
    shape = SHAPES["ragged 192x320 E6 K3 6/6/8 gated shared"]
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape, step=3)
    xd, idd, scd, rd = (C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                        C.dev(sc, torch.float32), C.dev(r, torch.bfloat16))
    ref = handle_forward(layer, x, r, ids, sc, 1)
    out = torch.empty((1, shape.din), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Bn.forward_noalloc(layer, xd, idd, scd, rd, out, device_error=err)   # first call: setup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        Bn.forward_noalloc(layer, xd, idd, scd, rd, out, device_error=err)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    out2 = torch.zeros_like(out)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Bn.forward_noalloc(layer, xd, idd, scd, rd, out2, device_error=err, stream=s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out2.view(torch.int32), ref.view(torch.int32))


def test_bad_ids_reach_the_callers_error_word():
    shape = Shape("badid", 128, 64, 4, 3, 4, 4, 4, seed=22)
    layer = C.host_layer_device(shape)
    x, r, ids, sc = C.token_inputs(shape)
    ids = ids.copy()
    ids[0, 1] = shape.n_experts + 3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, shape.din), dtype=torch.float32, device="cuda")
    Bn.forward_noalloc(layer, C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                       C.dev(sc, torch.float32), C.dev(r, torch.bfloat16), out, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    C.assert_parity(out[0].cpu().numpy(), C.OracleLayer(shape).token(x[0], r[0], ids[0], sc[0]))
    # NULL error word: the call still runs and drops the slot
    out2 = torch.empty_like(out)
    Bn.forward_noalloc(layer, C.dev(x, torch.bfloat16), C.dev(ids, torch.int32),
                       C.dev(sc, torch.float32), C.dev(r, torch.bfloat16), out2)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int32), out.view(torch.int32))


def test_oversized_and_fused_configs_are_rejected():
    L = Bn.lib()
    big = Shape("big", 2048, 2048, 64, 40, 4, 4, 4, seed=1)       # 40 * 2048 > 65536 activations
    assert big.top_k * big.dff > Bn.NOALLOC_MAX_ACT_FLOATS
    w = Bn.LayerWeights()
    for shape, mode in ((big, Bn.KERNELS_SEPARATE),
                        (Shape("ok", 128, 64, 4, 2, 4, 4, 4, seed=2), Bn.KERNELS_FUSED)):
        cfg = Bn.config(shape, 1, Bn.DTYPE_BF16, Bn.DTYPE_F32, mode)
        rc = L.moe_decode_forward_noalloc(ctypes.byref(cfg), ctypes.byref(w), None, 1, None, None,
                                          None, None, None, None)
        assert rc == Bn.MOE_ERR_UNSUPPORTED
