"""Writes tests/golden/oracle_small.json: a small TTT-Linear and TTT-MLP case run
through the fp64 oracle only.  It is a regression fixture for the oracle (it flags
any later change of the oracle's arithmetic), not an independent pin.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def main():
    r = np.random.default_rng(20240601)
    B, H, T, d, m = 1, 2, 11, 4, 8
    q, k, v = (np.round(r.standard_normal((B, H, T, d)), 3) for _ in range(3))
    eta = np.round(r.uniform(0.1, 0.9, (B, H, T)), 3)
    W0 = np.round(r.standard_normal((H, d, d)) * 0.3, 3)
    W1 = np.round(r.standard_normal((H, d, m)) * 0.3, 3)
    c1 = np.round(r.standard_normal((H, m)) * 0.1, 3)
    W2 = np.round(r.standard_normal((H, m, d)) * 0.3, 3)
    c2 = np.round(r.standard_normal((H, d)) * 0.1, 3)
    cases = []
    for b, causal in [(1, True), (4, True), (4, False), (11, False)]:
        z, Wf = oracle.linear(q, k, v, W0, b=b, causal=causal, eta=eta)
        zm, W1o, c1o, W2o, c2o = oracle.mlp(q, k, v, W1, c1, W2, c2, b=b, causal=causal, eta=eta)
        cases.append({"b": b, "causal": causal, "linear_z": z.tolist(), "linear_W": Wf.tolist(),
                      "mlp_z": zm.tolist(), "mlp_W1": W1o.tolist(), "mlp_c1": c1o.tolist(),
                      "mlp_W2": W2o.tolist(), "mlp_c2": c2o.tolist()})
    out = {"about": "oracle regression fixture written by tests/golden/make_golden.py",
           "q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "eta": eta.tolist(),
           "W0": W0.tolist(), "W1": W1.tolist(), "c1": c1.tolist(), "W2": W2.tolist(),
           "c2": c2.tolist(), "cases": cases}
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=None, separators=(",", ":"))


if __name__ == "__main__":
    main()
