"""The oracle still reproduces its stored regression record (CPU only)."""
import json
import os

import numpy as np

from tests.golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_stored_record():
    rec = json.load(open(os.path.join(HERE, "oracle_tiny_block.json")))
    ids, sc, out = make_golden.compute(rec["case"])
    assert ids.tolist() == rec["ids"]
    assert [float(v) for v in sc] == rec["scores"]
    stored = np.array([float.fromhex(h) for h in rec["out_hex"]])
    assert np.allclose(out, stored, rtol=1e-14, atol=1e-14)
