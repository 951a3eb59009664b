"""Stored oracle values (tests/golden/, written by make_golden.py from the
oracle alone) must be reproduced; the symmetric two-component case is also
checked against its hand-derived closed form."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name + ".json")) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["logistic_pair", "random_small"])
def test_oracle_reproduces_golden(name):
    c = _load(name)
    args = [np.array(c[k]) for k in ("Q", "K", "V", "mu", "sigma2", "log_pi")]
    assert np.allclose(oracle.responsibilities(args[0], *args[3:]), c["gamma_Q"], rtol=0, atol=1e-14)
    assert np.allclose(oracle.forward_bidir(*args, c["eps"]), c["O_bidir"], rtol=0, atol=1e-13)
    assert np.allclose(oracle.forward_causal(*args, c["eps"]), c["O_causal"], rtol=0, atol=1e-13)


def test_logistic_pair_closed_form():
    """mu = (-1, 1), v = 1, equal priors: gamma_1(x) = 1 / (1 + e^{2x}).
    Bidirectional O_i = sum_j a_ij V_j / (sum_j a_ij + eps) with
    a_ij = g(q_i) g(k_j) + (1 - g(q_i)) (1 - g(k_j)); causal sums j <= i."""
    c = _load("logistic_pair")
    g = lambda x: 1.0 / (1.0 + math.exp(2.0 * x))  # noqa: E731
    q = [r[0] for r in c["Q"]]
    k = [r[0] for r in c["K"]]
    V = np.array(c["V"])
    eps = c["eps"]
    N = len(q)
    a = np.array([[g(q[i]) * g(k[j]) + (1 - g(q[i])) * (1 - g(k[j])) for j in range(N)]
                  for i in range(N)])
    Ob = (a @ V) / (a.sum(1, keepdims=True) + eps)
    L = np.tril(a)
    Oc = (L @ V) / (L.sum(1, keepdims=True) + eps)
    assert np.max(np.abs(np.array(c["O_bidir"]) - Ob)) < 1e-13
    assert np.max(np.abs(np.array(c["O_causal"]) - Oc)) < 1e-13
    assert np.max(np.abs(np.array(c["gamma_Q"])[:, 0] - [g(x) for x in q])) < 1e-14
