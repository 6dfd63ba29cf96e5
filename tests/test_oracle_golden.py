"""Oracle against the hand-worked d = 2 example and its own regression fixture."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", range(3))
def test_hand_worked_d2(case):
    g = _load("linear_hand_d2.json")
    c = g["cases"][case]
    a = lambda x: np.array(x, dtype=np.float64)[None, None]
    z, Wf = oracle.linear(a(g["q"]), a(g["k"]), a(g["v"]), np.array(g["W0"], float)[None],
                          b=c["b"], causal=c["causal"], eta_scalar=g["eta"])
    np.testing.assert_array_equal(z[0, 0], np.array(c["z"], float))
    np.testing.assert_array_equal(Wf[0, 0], np.array(c["W_final"], float))


def test_regression_fixture():
    g = _load("oracle_small.json")
    A = {k: np.array(v, dtype=np.float64) for k, v in g.items() if k not in ("about", "cases")}
    for c in g["cases"]:
        z, Wf = oracle.linear(A["q"], A["k"], A["v"], A["W0"], b=c["b"], causal=c["causal"],
                              eta=A["eta"])
        np.testing.assert_allclose(z, c["linear_z"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(Wf, c["linear_W"], rtol=0, atol=1e-12)
        out = oracle.mlp(A["q"], A["k"], A["v"], A["W1"], A["c1"], A["W2"], A["c2"], b=c["b"],
                         causal=c["causal"], eta=A["eta"])
        for got, key in zip(out, ["mlp_z", "mlp_W1", "mlp_c1", "mlp_W2", "mlp_c2"]):
            np.testing.assert_allclose(got, c[key], rtol=0, atol=1e-12)
