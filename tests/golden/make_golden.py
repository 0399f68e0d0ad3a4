"""Writes tests/golden/oracle_tiny.json: a tiny case and the oracle's answer to it.

The pages print no worked example of the recurrence, so this fixture is a regression record
of the oracle itself (written by calling only ``oracle``), used to check that the oracle
gives the same numbers on every host that runs the tests (x86_64 here, aarch64 next to the
GPU). Its correctness rests on the pins in tests/test_oracle_pins.py.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(20261202)
    T, H, dk, dv = 6, 1, 3, 2
    q = rng.standard_normal((T, H, dk)).round(3)
    k = rng.standard_normal((T, H, dk)).round(3)
    v = rng.standard_normal((T, H, dv)).round(3)
    g = -rng.uniform(0, 1, (T, H, dk)).round(3)
    beta = rng.uniform(0, 1, (T, H)).round(3)
    S0 = rng.standard_normal((1, H, dk, dv)).round(3)
    o, fin = oracle.forward(q, k, v, g, beta, init_state=S0, scale=0.5)
    M, D = oracle.package(k, v, g, beta, [0, 2, 6])
    out = {"source": "oracle (tests/golden/make_golden.py); pins in tests/test_oracle_pins.py",
           "scale": 0.5, "q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "g": g.tolist(),
           "beta": beta.tolist(), "init_state": S0.tolist(), "o": o.tolist(),
           "final_state": fin.tolist(), "seg_offsets": [0, 2, 6], "M": M.tolist(),
           "D": D.tolist()}
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
