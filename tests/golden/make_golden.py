"""Writes the stored oracle values under tests/golden/.

Calls only the fp64 oracle (``oracle/``).  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def case_logistic_pair():
    # d_r = 1, K = 2 symmetric components: a case with a hand-derivable
    # posterior gamma_1(x) = 1 / (1 + exp(2 m x / v)).
    x = [-1.5, -0.5, 0.5, 1.5]
    return {
        "name": "logistic_pair",
        "cite": "GMA paper (arXiv 2606.18283): Eqs. (3), (5)-(7), (8b); closed form by Bayes' rule",
        "Q": [[v] for v in x], "K": [[v] for v in reversed(x)],
        "V": [[1.0, -1.0], [2.0, 0.5], [3.0, 0.0], [4.0, 2.0]],
        "mu": [[-1.0], [1.0]], "sigma2": [[1.0], [1.0]],
        "log_pi": [math.log(0.5), math.log(0.5)], "eps": 1e-6,
    }


def case_random_small():
    rng = np.random.default_rng(20260101)
    N, d_r, d_v, K = 16, 4, 3, 5
    s2 = np.log1p(np.exp(rng.normal(scale=math.sqrt(0.5), size=(K, d_r)))) + 1e-3
    a = rng.normal(size=K)
    return {
        "name": "random_small",
        "cite": "GMA paper (arXiv 2606.18283): Eqs. (3), (5)-(7), (8b)",
        "Q": rng.normal(size=(N, d_r)).tolist(), "K": rng.normal(size=(N, d_r)).tolist(),
        "V": rng.normal(size=(N, d_v)).tolist(), "mu": rng.normal(size=(K, d_r)).tolist(),
        "sigma2": s2.tolist(), "log_pi": (a - np.log(np.exp(a).sum())).tolist(), "eps": 1e-6,
    }


def main():
    for case in (case_logistic_pair(), case_random_small()):
        args = [np.array(case[k]) for k in ("Q", "K", "V", "mu", "sigma2", "log_pi")]
        case["gamma_Q"] = oracle.responsibilities(args[0], *args[3:]).tolist()
        case["O_bidir"] = oracle.forward_bidir(*args, case["eps"]).tolist()
        case["O_causal"] = oracle.forward_causal(*args, case["eps"]).tolist()
        with open(os.path.join(HERE, case["name"] + ".json"), "w") as f:
            json.dump(case, f, indent=1)


if __name__ == "__main__":
    main()
