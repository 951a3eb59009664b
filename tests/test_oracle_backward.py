"""Pins of the oracle's gradients (oracle.backward_bidir / backward_causal).

The gradients follow "Gaussian Mixture Attention: Linear-Time Sequence Mixing
via Probabilistic Latent Routing", gradient section: Eq. (18) for the
gradient entering a score and the chain rule for everything that enters the
score.  They are pinned to things other than their own formulas:

* central finite differences of the (already pinned) forward oracle, for every
  input and parameter element of small cases;
* invariances of the score: a shift of log pi, a joint translation of the
  routing vectors and the means, and the joint scaling (x, mu, sigma2) ->
  (c x, c mu, c^2 sigma2) change no responsibility, so the gradients are
  orthogonal to those directions;
* K = 1 (responsibilities identically 1): no routing gradient at all, and the
  bidirectional dV is the closed form sum_i dO_i / (N + eps).

Each planted mistake in the backward (``GMA_ORACLE_MUTANT`` 7, 8) must fail a
pin.
"""
import numpy as np
import pytest

import oracle


def _case(seed, B=1, H=2, N=9, d_r=3, d_v=4, K=3):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, H, N, d_r))
    Kx = rng.standard_normal((B, H, N, d_r))
    V = rng.standard_normal((B, H, N, d_v))
    mu = rng.standard_normal((H, K, d_r))
    s2 = np.log1p(np.exp(rng.standard_normal((H, K, d_r)) * np.sqrt(0.5))) + 0.2
    lp = rng.standard_normal((H, K))
    lp = lp - np.log(np.exp(lp).sum(-1, keepdims=True))
    W = rng.standard_normal((B, H, N, d_v))
    return dict(Q=Q, K=Kx, V=V, mu=mu, sigma2=s2, log_pi=lp, W=W, eps=1e-3)


def _loss(c, causal, **over):
    a = dict(c, **over)
    fwd = oracle.forward_causal if causal else oracle.forward_bidir
    O = fwd(a["Q"], a["K"], a["V"], a["mu"], a["sigma2"], a["log_pi"], a["eps"])
    return float((O * a["W"]).sum())


def _grads(c, causal):
    bwd = oracle.backward_causal if causal else oracle.backward_bidir
    return bwd(c["Q"], c["K"], c["V"], c["mu"], c["sigma2"], c["log_pi"], c["eps"], c["W"])


NAMES = {"Q": "dQ", "K": "dK", "V": "dV", "mu": "dmu", "sigma2": "dsigma2", "log_pi": "dlog_pi"}


def _check_fd(causal, seed=0):
    c = _case(seed)
    g = _grads(c, causal)
    for name, gname in NAMES.items():
        x = c[name]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            h = 1e-6 * max(1.0, abs(x[idx]))
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            fd[idx] = (_loss(c, causal, **{name: xp}) - _loss(c, causal, **{name: xm})) / (2 * h)
        scale = max(1.0, np.abs(fd).max())
        err = np.abs(g[gname] - fd).max() / scale
        assert err < 1e-6, f"{gname}: max |grad - central difference| / scale = {err:.2e}"


def _check_invariances(causal, seed=1):
    c = _case(seed, B=2)
    g = _grads(c, causal)
    # log pi shift
    assert np.abs(g["dlog_pi"].sum(-1)).max() < 1e-10
    # joint translation of x (queries and keys of every batch row of the head) and mu
    tr = g["dQ"].sum(axis=(0, 2)) + g["dK"].sum(axis=(0, 2)) + g["dmu"].sum(axis=1)
    assert np.abs(tr).max() < 1e-10 * max(1.0, np.abs(g["dQ"]).max())
    # joint scaling (x, mu, sigma2) -> (c x, c mu, c^2 sigma2), derivative at c = 1
    sc = ((c["Q"] * g["dQ"]).sum(axis=(0, 2, 3)) + (c["K"] * g["dK"]).sum(axis=(0, 2, 3))
          + (c["mu"] * g["dmu"]).sum(axis=(1, 2)) + (2 * c["sigma2"] * g["dsigma2"]).sum(axis=(1, 2)))
    assert np.abs(sc).max() < 1e-9 * max(1.0, np.abs(g["dQ"]).max())


def _check_k1(causal, seed=2):
    c = _case(seed, K=1)
    g = _grads(c, causal)
    for gname in ("dQ", "dK", "dmu", "dsigma2", "dlog_pi"):
        assert np.abs(g[gname]).max() < 1e-12, gname
    N = c["Q"].shape[2]
    if causal:
        # O_i = sum_{j<=i} V_j / (i + 1 + eps): dV_j = sum_{i>=j} W_i / (i + 1 + eps)
        w = c["W"] / (np.arange(N) + 1 + c["eps"])[None, None, :, None]
        want = np.flip(np.cumsum(np.flip(w, 2), 2), 2)
    else:
        want = np.broadcast_to(c["W"].sum(2, keepdims=True) / (N + c["eps"]), c["W"].shape)
    assert np.abs(g["dV"] - want).max() < 1e-12


PINS = [
    lambda: _check_fd(False), lambda: _check_fd(True),
    lambda: _check_invariances(False), lambda: _check_invariances(True),
    lambda: _check_k1(False), lambda: _check_k1(True),
]


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_matches_central_differences(causal):
    _check_fd(causal)


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_invariances(causal):
    _check_invariances(causal)


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_backward_k1_closed_form(causal):
    _check_k1(causal)


@pytest.mark.parametrize("mutant,what", [(7, "score gradient not mean-centred"),
                                         (8, "causal key gradient from prefix sums")])
def test_backward_pins_catch_planted_mistake(mutant, what):
    caught = 0
    with oracle.use_mutant(mutant):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught += 1
    assert caught, f"no pin caught mutant {mutant} ({what})"
