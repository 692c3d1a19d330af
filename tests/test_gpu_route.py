"""The kernels' route inversion (grouping a batch of tokens' slots by expert) against the oracle's,
bit for bit: distinct experts ascending and each expert's (token, slot) pairs ascending."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import binding as Bn

pytestmark = pytest.mark.gpu


def check(ids, E):
    got = Bn.route_invert_device(torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(), E)
    want = O.route_invert(ids, E)
    for g, w, name in zip(got, want, ("uniq", "offs", "pairs")):
        assert np.array_equal(g, w), f"{name}: {g.tolist()} != {w.tolist()}"


@pytest.mark.parametrize("m,k,E,seed", [(1, 8, 128, 1), (8, 6, 128, 2), (32, 6, 128, 3),
                                        (32, 8, 128, 4), (25, 10, 512, 5), (64, 4, 1024, 6),
                                        (3, 2, 2, 7), (256, 1, 1000, 8)])
def test_distinct_ids_per_token(m, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(m)]).astype(np.int32)
    check(ids, E)


def test_duplicates_and_invalid_ids():
    rng = np.random.default_rng(11)
    ids = rng.integers(-3, 40, size=(16, 16)).astype(np.int32)   # repeats and ids out of range
    check(ids, 37)
    check(np.full((8, 8), 5, np.int32), 6)                       # one expert for every pair
    check(np.full((2, 3), -1, np.int32), 4)                      # nothing valid


def test_limits_are_rejected():
    ids = torch.zeros((33, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(Bn.MoeError):
        Bn.route_invert_device(ids, 128)                         # 264 pairs
    with pytest.raises(Bn.MoeError):
        Bn.route_invert_device(ids[:2], 2048)                    # too many experts for the bitmap
