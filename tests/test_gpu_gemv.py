"""GPU parity of the dense bf16 decode GEMV (moe_gemv_bf16) against the oracle.

"Measure attention projections instead of serving them, and record the amortisation trap"
measures the q/k/v/o projections of a decode token at 1, 8 and 32 rows.  Every output of every
matrix must meet the block's parity bar against the fp64 oracle; both kernels (CUDA cores up to
4 rows, tensor-core tiles from 5) are covered, with ragged row counts and column counts that are
not multiples of the kernels' chunk widths, shared and per-matrix inputs, and the full-size
projections at 1, 8 and 32 rows.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300 import synth
from quantized_moe_expert_dequant_gb300.workloads import GEMV
from tests import gpu_cases as C

pytestmark = pytest.mark.gpu


def run(Ws, xs, shared):
    Wd = C.dev(np.stack(Ws), torch.bfloat16)
    xd = C.dev(xs[0] if shared else np.stack(xs), torch.bfloat16)
    y = Bn.gemv_bf16(Wd, xd, shared_x=shared)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(Ws, xs, y, shared, what):
    for r, W in enumerate(Ws):
        ref = O.gemv_bf16(W, xs[0] if shared else xs[r])
        for t in range(ref.shape[0]):
            C.assert_parity(y[r][t], ref[t], f"{what}: matrix {r} row {t}")


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 9, 16, 17, 24, 25, 32])
@pytest.mark.parametrize("n_out,n_in", [(17, 40), (64, 256), (33, 72)])
def test_small_shapes_every_output(m, n_out, n_in):
    seed = 1000 * m + n_out + n_in
    Ws = [synth.dense_weight(seed, n_out, n_in, r) for r in range(3)]
    for shared in (True, False):
        xs = [synth.dense_input(seed, m, n_in, r) for r in range(3)]
        y = run(Ws, xs, shared)
        check(Ws, xs, y, shared, f"m {m} {n_out}x{n_in} shared {shared}")


@pytest.mark.parametrize("name", sorted(GEMV))
@pytest.mark.parametrize("m", [1, 8, 32])
def test_full_size_projections(name, m):
    g = GEMV[name]
    W = synth.dense_weight(g.seed, g.n_out, g.n_in)
    x = synth.dense_input(g.seed, m, g.n_in)
    y = run([W], [x], True)
    check([W], [x], y, True, g.name)


def test_repeat_calls_give_identical_bytes():
    g = GEMV["qwen3_8b_kv"]
    Wd = C.dev(synth.dense_weight(g.seed, g.n_out, g.n_in)[None], torch.bfloat16)
    for m in (1, 8, 32):
        xd = C.dev(synth.dense_input(g.seed, m, g.n_in), torch.bfloat16)
        a = Bn.gemv_bf16(Wd, xd)
        b = Bn.gemv_bf16(Wd, xd)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_bad_arguments_are_rejected():
    L = Bn.lib()
    W = torch.zeros((2, 16, 64), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((40, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((2, 40, 16), dtype=torch.float32, device="cuda")
    ok = (W.data_ptr(), x.data_ptr(), 0, y.data_ptr(), 2, 1, 16, 64)
    assert L.moe_gemv_bf16(*ok, None) == Bn.MOE_OK
    torch.cuda.synchronize()
    bad = [
        (W.data_ptr(), x.data_ptr(), 0, y.data_ptr(), 2, 0, 16, 64),       # m = 0
        (W.data_ptr(), x.data_ptr(), 0, y.data_ptr(), 2, 33, 16, 64),      # m > 32
        (W.data_ptr(), x.data_ptr(), 0, y.data_ptr(), 2, 1, 16, 60),       # n_in % 8
        (W.data_ptr() + 2, x.data_ptr(), 0, y.data_ptr(), 2, 1, 16, 64),   # W misaligned
        (W.data_ptr(), x.data_ptr() + 8, 0, y.data_ptr(), 2, 1, 16, 64),   # x misaligned
        (W.data_ptr(), x.data_ptr(), 4, y.data_ptr(), 2, 1, 16, 64),       # x_stride % 8
        (W.data_ptr(), x.data_ptr(), 0, y.data_ptr(), 0, 1, 16, 64),       # no matrix
        (None, x.data_ptr(), 0, y.data_ptr(), 2, 1, 16, 64),               # null
    ]
    for args in bad:
        assert L.moe_gemv_bf16(*args, None) == Bn.MOE_ERR_INVALID_ARG, args
