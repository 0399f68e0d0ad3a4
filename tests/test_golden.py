"""The oracle reproduces its stored tiny-case record on this host (cross-host regression)."""
import json
import os

import numpy as np

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_golden(oracle_mod):
    with open(os.path.join(HERE, "oracle_tiny.json")) as f:
        d = json.load(f)
    a = {k: np.array(v) for k, v in d.items() if isinstance(v, list)}
    o, fin = oracle_mod.forward(a["q"], a["k"], a["v"], a["g"], a["beta"],
                                init_state=a["init_state"], scale=d["scale"])
    np.testing.assert_allclose(o, a["o"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin, a["final_state"], rtol=1e-13, atol=1e-15)
    M, D = oracle_mod.package(a["k"], a["v"], a["g"], a["beta"], d["seg_offsets"])
    np.testing.assert_allclose(M, a["M"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(D, a["D"], rtol=1e-13, atol=1e-15)
