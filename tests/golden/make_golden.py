"""Writes oracle_fixtures.json: regression values computed by the CPU oracle
alone (no GPU code is imported).  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from normalized_cross_correlation_gb300 import inputs  # noqa: E402

MOD = 2**61 - 1


def case(w, label, random_args=None, n=24, seed=0):
    S, Q = oracle.sat(w.image)
    rng = np.random.default_rng(seed)
    xs = [c[1] for c in w.crops] + [0, w.Ox - 1] + list(rng.integers(0, w.Ox, n))
    ys = [c[2] for c in w.crops] + [0, w.Oy - 1] + list(rng.integers(0, w.Oy, n))
    r, a, b, c = oracle.correlate_at(w.image, w.templates, xs, ys, with_sums=True)
    out = {"workload": label, "xs": [int(v) for v in xs], "ys": [int(v) for v in ys],
           "S_corner": int(S[-1, -1]), "Q_corner": int(Q[-1, -1]),
           "S_mod": int(S.sum() % MOD), "Q_mod": int(Q.sum() % MOD),
           "sumI": a.tolist(), "sumI2": b.tolist(), "sumIT": c.tolist(),
           "r": r.tolist()}
    if random_args is not None:
        out["random_args"] = list(random_args)
    return out


def main():
    cases = [case(inputs.tiny_ncc(), "tiny_ncc_256_t16")]
    args = (13, 203, 171, 11, 7, 3, 2)
    cases.append(case(inputs.random_case(*args), "random", random_args=args))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_fixtures.json")
    with open(path, "w") as f:
        json.dump({"writer": "tests/golden/make_golden.py (oracle only)", "cases": cases}, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
