"""The C ABI on the host (no GPU): every declared symbol is exported, host packing round-trips
against the oracle's reader, and invalid arguments are rejected before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import binding as Bn
from tests import helpers as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return Bn.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_decode.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|void)\s+(moe_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(Bn.EXPORTS) == set(names)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_host_pack_matches_bigint_and_oracle(L, bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(5, 192)).astype(np.uint8)
    packed = Bn.pack_codes(codes, bits)
    for r in range(5):
        assert np.array_equal(packed[r], H.pack_bigint(codes[r], bits))
        assert np.array_equal(O.unpack_row(packed[r], bits, 192), codes[r])
    assert np.array_equal(Bn.unpack_codes(packed, 192, bits), codes)


def test_host_pack_rejects_bad_input(L):
    with pytest.raises(Bn.MoeError) as e:
        Bn.pack_codes(np.full((1, 64), 16, np.uint8), 4)
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG
    with pytest.raises(Bn.MoeError) as e:
        Bn.pack_codes(np.zeros((1, 64), np.uint8), 5)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    with pytest.raises(Bn.MoeError) as e:
        Bn.pack_codes(np.zeros((1, 65), np.uint8), 4)
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG


def _cfg(**kw):
    base = dict(din=256, dff=128, n_experts=8, top_k=2, max_tokens=1, bits_gate=4, bits_up=4,
                bits_down=4, n_shared=0, dff_shared=0, bits_shared=4, shared_gate=0,
                resid_dtype=0, out_dtype=1, kernel_mode=0)
    base.update(kw)
    return Bn.Config(**base)


def _weights(n_proj=6, gate_vec=True, misalign=False):
    # fake, never-dereferenced addresses: validation only looks at null-ness and alignment
    a = 0x10000 + (8 if misalign else 0)
    p = Bn.Proj(a, 0x20000, 0x30000)
    return Bn.LayerWeights(p, p, p, p, p, p, 0x40000 if gate_vec else None)


@pytest.mark.parametrize("kw,rc", [
    (dict(din=100), Bn.MOE_ERR_INVALID_ARG),
    (dict(dff=0), Bn.MOE_ERR_INVALID_ARG),
    (dict(top_k=9), Bn.MOE_ERR_INVALID_ARG),
    (dict(top_k=-1), Bn.MOE_ERR_INVALID_ARG),
    (dict(top_k=0, n_shared=0), Bn.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=0), Bn.MOE_ERR_INVALID_ARG),
    (dict(bits_down=5), Bn.MOE_ERR_UNSUPPORTED),
    (dict(bits_gate=8), Bn.MOE_ERR_UNSUPPORTED),
    (dict(n_shared=5, dff_shared=64), Bn.MOE_ERR_INVALID_ARG),
    (dict(n_shared=1, dff_shared=100), Bn.MOE_ERR_INVALID_ARG),
    (dict(n_shared=1, dff_shared=64, bits_shared=3), Bn.MOE_ERR_UNSUPPORTED),
    (dict(shared_gate=2), Bn.MOE_ERR_INVALID_ARG),
    (dict(resid_dtype=7), Bn.MOE_ERR_INVALID_ARG),
    (dict(out_dtype=-1), Bn.MOE_ERR_INVALID_ARG),
    (dict(kernel_mode=6), Bn.MOE_ERR_INVALID_ARG),
])
def test_create_rejects_invalid_config(L, kw, rc):
    h = ctypes.c_void_p()
    w = _weights()
    assert L.moe_decode_create(ctypes.byref(_cfg(**kw)), ctypes.byref(w), ctypes.byref(h)) == rc
    assert not h.value


def test_create_rejects_bad_weight_pointers(L):
    h = ctypes.c_void_p()
    c = _cfg()
    w = _weights(misalign=True)
    assert L.moe_decode_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == Bn.MOE_ERR_INVALID_ARG
    w = _weights()
    w.down = Bn.Proj(None, None, None)
    assert L.moe_decode_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == Bn.MOE_ERR_INVALID_ARG
    c = _cfg(n_shared=1, dff_shared=64, shared_gate=1)
    w = _weights(gate_vec=False)
    assert L.moe_decode_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_decode_create(None, ctypes.byref(w), ctypes.byref(h)) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_decode_create(ctypes.byref(c), ctypes.byref(w), None) == Bn.MOE_ERR_INVALID_ARG


def test_calls_on_null_handles_are_rejected(L):
    assert L.moe_decode_forward(None, 1, 1, 1, 1, 1, 1, None) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_stack_step(None, 1, 1, 1, 1, 1, 1, None) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_stack_step_host(None, 1, 1, 1, 1, 1, 1, None) == Bn.MOE_ERR_INVALID_ARG
    v = ctypes.c_int32()
    assert L.moe_decode_get_error(None, ctypes.byref(v)) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_stack_get_error(None, ctypes.byref(v)) == Bn.MOE_ERR_INVALID_ARG
    L.moe_decode_destroy(None)
    L.moe_stack_destroy(None)
    c = _cfg()
    h = ctypes.c_void_p()
    assert L.moe_stack_create(ctypes.byref(c), 0, None, ctypes.byref(h)) == Bn.MOE_ERR_INVALID_ARG
    c = _cfg(out_dtype=0)
    w = _weights()
    assert L.moe_stack_create(ctypes.byref(c), 1, ctypes.byref(w), ctypes.byref(h)) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_unpack_codes_device(None, 1, 64, 4, None, None) == Bn.MOE_ERR_INVALID_ARG
    assert L.moe_synth_codes(None, 0, 0, 1, 1, None) == Bn.MOE_ERR_INVALID_ARG
