"""The device router against the oracle's: pool ids bit for bit (the selection compares the same
fp32 logits), weights within fp32 rounding of the fp64 softmax."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import binding as Bn

pytestmark = pytest.mark.gpu


def check(logits, k):
    ids, sc = Bn.router_topk(torch.from_numpy(logits).cuda(), k)
    ids, sc = ids.cpu().numpy(), sc.cpu().numpy()
    # fp32 softmax: k exponentials (a few ulp each), k-1 additions and one division
    rtol = (k + 4) * 2.0 ** -23
    for t in range(len(logits)):
        oi, os_ = O.router(logits[t], k)
        assert np.array_equal(ids[t], oi), f"token {t}: {ids[t].tolist()} != {oi.tolist()}"
        np.testing.assert_allclose(sc[t], os_, rtol=rtol, atol=0, err_msg=f"token {t}")


@pytest.mark.parametrize("E,k", [(128, 8), (60, 4), (512, 10), (128, 6), (1024, 64), (33, 33),
                                 (1, 1), (1000, 40)])
def test_router_matches_oracle(E, k):
    logits = np.random.default_rng(E * 100 + k).standard_normal((37, E)).astype(np.float32)
    check(logits, k)


def test_router_ties_go_to_the_lower_id():
    rng = np.random.default_rng(5)
    logits = rng.integers(-3, 4, size=(64, 128)).astype(np.float32)   # many equal logits
    check(logits, 8)
    check(np.zeros((4, 96), np.float32), 10)                          # all equal


def test_router_rejects_bad_sizes():
    x = torch.zeros((2, 2048), dtype=torch.float32, device="cuda")
    with pytest.raises(Bn.MoeError):
        Bn.router_topk(x, 8)          # more experts than the register layout holds
    with pytest.raises(Bn.MoeError):
        Bn.router_topk(x[:, :16], 17)  # more slots than experts
