"""Pins for the fp64 oracle: checks against what the GMA paper and plain
mathematics fix, independent of the oracle's own formulas.

Each ``pin_*`` function raises AssertionError on a violation.  They are run
against the oracle in ``test_oracle.py`` and against deliberately broken
builds of it in ``test_oracle_mutants.py`` (where at least one must fail).

Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
Probabilistic Latent Routing" (arXiv 2606.18283), cited [GMA, ...].
"""
from __future__ import annotations

import math

import numpy as np

import oracle


def _rng(seed=0):
    return np.random.default_rng(seed)


def random_head(rng, N, d_r, d_v, K, mu_std=1.0):
    Q = rng.normal(size=(N, d_r))
    Kx = rng.normal(size=(N, d_r))
    V = rng.normal(size=(N, d_v))
    mu = rng.normal(scale=mu_std, size=(K, d_r))
    sigma2 = np.log1p(np.exp(rng.normal(scale=math.sqrt(0.5), size=(K, d_r)))) + 1e-3
    a = rng.normal(size=K)
    log_pi = a - np.log(np.exp(a - a.max()).sum()) - a.max()
    return Q, Kx, V, mu, sigma2, log_pi


# ---------------------------------------------------------------- responsibilities

def pin_simplex_rows():
    """Rows of Gamma are probability distributions ([GMA, below Eq. 3])."""
    rng = _rng(1)
    for (N, d_r, K) in [(37, 5, 7), (16, 1, 1), (9, 16, 32)]:
        X, _, _, mu, s2, lp = random_head(rng, N, d_r, 1, K)
        G = oracle.responsibilities(X, mu, s2, lp)
        assert G.shape == (N, K)
        assert np.all(G >= 0)
        assert np.max(np.abs(G.sum(-1) - 1.0)) < 1e-13


def pin_identical_components_give_prior():
    """All components equal => the posterior equals the prior pi for every x."""
    rng = _rng(2)
    K, d_r = 6, 4
    mu = np.tile(rng.normal(size=(1, d_r)), (K, 1))
    s2 = np.tile(rng.uniform(0.3, 2.0, size=(1, d_r)), (K, 1))
    pi = rng.dirichlet(np.ones(K))
    X = rng.normal(size=(11, d_r)) * 3
    G = oracle.responsibilities(X, mu, s2, np.log(pi))
    assert np.max(np.abs(G - pi[None])) < 1e-13


def pin_single_component_is_one():
    """K = 1 => gamma == 1 for every row."""
    rng = _rng(3)
    X, _, _, mu, s2, lp = random_head(rng, 13, 3, 1, 1)
    G = oracle.responsibilities(X, mu, s2, lp)
    assert np.max(np.abs(G - 1.0)) < 1e-15


def pin_two_symmetric_components_logistic():
    """d_r = 1, K = 2, mu = (-m, +m), equal variance v, equal priors.

    Bayes' rule with two equal-variance Gaussians gives
    p(z = 1 | x) = 1 / (1 + exp(2 m x / v)) (the logistic of the linear
    discriminant), derived by hand, not from the oracle's score formula.
    """
    for m, v in [(1.0, 1.0), (0.7, 0.5), (2.0, 3.0)]:
        x = np.linspace(-3, 3, 25)[:, None]
        mu = np.array([[-m], [m]])
        s2 = np.array([[v], [v]])
        G = oracle.responsibilities(x, mu, s2, np.log([0.5, 0.5]))
        expect = 1.0 / (1.0 + np.exp(2 * m * x[:, 0] / v))
        assert np.max(np.abs(G[:, 0] - expect)) < 1e-13


def pin_matches_scipy_textbook_posterior():
    """Gamma_ik = pi_k prod_j Normal(x_j; mu_kj, sigma2_kj) / evidence, with the
    normal log-pdf from scipy.stats and the normalisation from scipy.special."""
    from scipy.special import softmax
    from scipy.stats import norm
    rng = _rng(4)
    for (N, d_r, K) in [(20, 3, 5), (8, 16, 8)]:
        X, _, _, mu, s2, lp = random_head(rng, N, d_r, 1, K)
        logp = norm.logpdf(X[:, None, :], loc=mu[None], scale=np.sqrt(s2)[None]).sum(-1) + lp
        expect = softmax(logp, axis=-1)
        G = oracle.responsibilities(X, mu, s2, lp)
        assert np.max(np.abs(G - expect)) < 1e-12


def pin_matches_sklearn_gmm_predict_proba():
    """scikit-learn's diagonal-covariance GaussianMixture with the same
    weights, means and precisions yields the same posterior (host only)."""
    try:
        from sklearn.mixture import GaussianMixture
    except ImportError:  # the GPU machine has no scikit-learn; scipy pin still runs
        return
    rng = _rng(5)
    N, d_r, K = 30, 4, 5
    X, _, _, mu, s2, lp = random_head(rng, N, d_r, 1, K)
    pi = np.exp(lp)
    pi /= pi.sum()
    gm = GaussianMixture(n_components=K, covariance_type="diag")
    gm.weights_ = pi
    gm.means_ = mu
    gm.covariances_ = s2
    gm.precisions_cholesky_ = 1.0 / np.sqrt(s2)
    expect = gm.predict_proba(X)
    G = oracle.responsibilities(X, mu, s2, np.log(pi))
    assert np.max(np.abs(G - expect)) < 1e-10


def pin_responsibility_invariances():
    """Gamma is unchanged by x -> c x + t with mu -> c mu + t, sigma2 -> c^2 sigma2,
    by adding a constant to log pi, and permutes with the components."""
    rng = _rng(6)
    X, _, _, mu, s2, lp = random_head(rng, 17, 5, 1, 6)
    G = oracle.responsibilities(X, mu, s2, lp)
    c, t = 1.7, rng.normal(size=5)
    G2 = oracle.responsibilities(c * X + t, c * mu + t, c * c * s2, lp)
    assert np.max(np.abs(G - G2)) < 1e-12
    G3 = oracle.responsibilities(X, mu, s2, lp + 3.25)
    assert np.max(np.abs(G - G3)) < 1e-13
    perm = rng.permutation(6)
    G4 = oracle.responsibilities(X, mu[perm], s2[perm], lp[perm])
    assert np.max(np.abs(G[:, perm] - G4)) < 1e-13


# ---------------------------------------------------------------- forward

def pin_bidir_equals_materialised_affinity():
    """Eq. (7) O = Gamma^Q Vt / (Gamma^Q Z + eps) equals the row-normalised
    materialised affinity applied to V ([GMA, Eqs. 9-11, footnote 4])."""
    rng = _rng(7)
    for (N, d_r, d_v, K, eps) in [(33, 4, 3, 5, 1e-6), (64, 8, 8, 16, 1e-2), (1, 2, 2, 3, 1e-6)]:
        Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
        O = oracle.forward_bidir(Q, Kx, V, mu, s2, lp, eps)
        A = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, eps, causal=False)
        assert np.max(np.abs(O - A)) <= 1e-12 * max(1.0, np.abs(A).max())


def pin_causal_equals_masked_affinity():
    """Causal O equals the brute force with the inclusive lower-triangular
    mask j <= i ([GMA, causal variant, Eq. 8b])."""
    rng = _rng(8)
    for (N, d_r, d_v, K, eps) in [(41, 4, 3, 5, 1e-6), (64, 8, 8, 16, 1e-2)]:
        Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
        O = oracle.forward_causal(Q, Kx, V, mu, s2, lp, eps)
        A = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, eps, causal=True)
        assert np.max(np.abs(O - A)) <= 1e-12 * max(1.0, np.abs(A).max())


def pin_affinity_properties():
    """The un-normalised affinity <gQ_i, gK_j> is an inner product of two
    probability vectors, so 0 <= A_ij <= 1; its rank is at most K; with the
    same rows on both sides it is symmetric positive semi-definite
    ([GMA, affinity section: non-negative, rank at most K])."""
    rng = _rng(9)
    N, d_r, K = 40, 3, 4
    Q, Kx, _, mu, s2, lp = random_head(rng, N, d_r, 1, K)
    A = oracle.affinity(Q, Kx, mu, s2, lp)
    assert np.all(A >= 0) and np.all(A <= 1.0 + 1e-15)
    assert np.linalg.matrix_rank(A, tol=1e-10) <= K
    S = oracle.affinity(Q, Q, mu, s2, lp)
    assert np.max(np.abs(S - S.T)) < 1e-15
    assert np.linalg.eigvalsh(S).min() > -1e-12


def pin_single_component_is_mean():
    """K = 1: bidirectional O_i = sum_j V_j / (N + eps); causal O_i =
    sum_{j<=i} V_j / (i + 1 + eps) (0-indexed)."""
    rng = _rng(10)
    N, d_r, d_v, eps = 29, 3, 4, 1e-3
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, 1)
    Ob = oracle.forward_bidir(Q, Kx, V, mu, s2, lp, eps)
    assert np.max(np.abs(Ob - V.sum(0) / (N + eps))) < 1e-13
    Oc = oracle.forward_causal(Q, Kx, V, mu, s2, lp, eps)
    expect = np.cumsum(V, 0) / (np.arange(1, N + 1)[:, None] + eps)
    assert np.max(np.abs(Oc - expect)) < 1e-13


def pin_identical_components_closed_form():
    """All components equal => gamma = pi for every row, so
    Gamma^Q (Gamma^K)^T has every entry p = sum_k pi_k^2 and
    O_i = p sum_j V_j / (N p + eps) (causal: over j <= i, with (i+1) p)."""
    rng = _rng(11)
    N, d_r, d_v, K, eps = 23, 3, 2, 5, 1e-2
    mu = np.tile(rng.normal(size=(1, d_r)), (K, 1))
    s2 = np.tile(rng.uniform(0.5, 2, size=(1, d_r)), (K, 1))
    pi = rng.dirichlet(np.ones(K))
    Q, Kx, V = rng.normal(size=(N, d_r)), rng.normal(size=(N, d_r)), rng.normal(size=(N, d_v))
    p = float((pi ** 2).sum())
    Ob = oracle.forward_bidir(Q, Kx, V, mu, s2, np.log(pi), eps)
    assert np.max(np.abs(Ob - p * V.sum(0) / (N * p + eps))) < 1e-13
    Oc = oracle.forward_causal(Q, Kx, V, mu, s2, np.log(pi), eps)
    expect = p * np.cumsum(V, 0) / (np.arange(1, N + 1)[:, None] * p + eps)
    assert np.max(np.abs(Oc - expect)) < 1e-13


def pin_causal_first_and_last_rows():
    """O_0 reads only key 0: O_0 = (gQ_0 . gK_0) V_0 / (gQ_0 . gK_0 + eps);
    the last causal row sees every key, so it equals the last bidirectional row."""
    rng = _rng(12)
    N, d_r, d_v, K, eps = 31, 4, 3, 6, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    Oc = oracle.forward_causal(Q, Kx, V, mu, s2, lp, eps)
    Ob = oracle.forward_bidir(Q, Kx, V, mu, s2, lp, eps)
    assert np.max(np.abs(Oc[-1] - Ob[-1])) < 1e-13
    from scipy.special import softmax
    from scipy.stats import norm
    def gam(x):
        return softmax(norm.logpdf(x[None, :], loc=mu, scale=np.sqrt(s2)).sum(-1) + lp)
    a = float(gam(Q[0]) @ gam(Kx[0]))
    assert np.max(np.abs(Oc[0] - a * V[0] / (a + eps))) < 1e-13


def pin_causal_prefix_consistency():
    """Causal O restricted to the first N' rows equals causal O computed on
    the first N' tokens alone (output i depends only on j <= i)."""
    rng = _rng(13)
    N, d_r, d_v, K, eps = 50, 3, 4, 5, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    O = oracle.forward_causal(Q, Kx, V, mu, s2, lp, eps)
    for n in (1, 7, 33):
        On = oracle.forward_causal(Q[:n], Kx[:n], V[:n], mu, s2, lp, eps)
        assert np.max(np.abs(O[:n] - On)) < 1e-13


def pin_bidir_symmetries():
    """Bidirectional O is invariant to a joint permutation of the (K_X, V_X)
    rows, permutes with the Q_X rows and is linear in V_X."""
    rng = _rng(14)
    N, d_r, d_v, K, eps = 27, 3, 4, 5, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    O = oracle.forward_bidir(Q, Kx, V, mu, s2, lp, eps)
    p = rng.permutation(N)
    assert np.max(np.abs(O - oracle.forward_bidir(Q, Kx[p], V[p], mu, s2, lp, eps))) < 1e-13
    assert np.max(np.abs(O[p] - oracle.forward_bidir(Q[p], Kx, V, mu, s2, lp, eps))) < 1e-13
    V2 = rng.normal(size=V.shape)
    O2 = oracle.forward_bidir(Q, Kx, V2, mu, s2, lp, eps)
    O3 = oracle.forward_bidir(Q, Kx, 2.0 * V - 0.5 * V2, mu, s2, lp, eps)
    assert np.max(np.abs(O3 - (2.0 * O - 0.5 * O2))) < 1e-12


def pin_rows_agree_with_full():
    """The selected-row routines give the same rows as the full forward."""
    rng = _rng(15)
    N, d_r, d_v, K, eps = 45, 4, 3, 6, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    rows = np.array([0, 1, 17, 44])
    Ob = oracle.forward_bidir(Q, Kx, V, mu, s2, lp, eps)
    Oc = oracle.forward_causal(Q, Kx, V, mu, s2, lp, eps)
    assert np.max(np.abs(oracle.bidir_rows(Q, Kx, V, mu, s2, lp, eps, rows) - Ob[rows])) < 1e-13
    assert np.max(np.abs(oracle.causal_rows(Q, Kx, V, mu, s2, lp, eps, rows) - Oc[rows])) < 1e-13


def pin_batched_heads_use_their_own_parameters():
    """[B, H, N, d] inputs take parameters per head h (same for every batch b)."""
    rng = _rng(16)
    B, H, N, d_r, d_v, K, eps = 2, 3, 9, 3, 2, 4, 1e-6
    Q = rng.normal(size=(B, H, N, d_r)); Kx = rng.normal(size=(B, H, N, d_r))
    V = rng.normal(size=(B, H, N, d_v))
    mu = rng.normal(size=(H, K, d_r)); s2 = rng.uniform(0.2, 2, size=(H, K, d_r))
    lp = np.log(rng.dirichlet(np.ones(K), size=H))
    O = oracle.forward_bidir(Q, Kx, V, mu, s2, lp, eps)
    for b in range(B):
        for h in range(H):
            Oh = oracle.forward_bidir(Q[b, h], Kx[b, h], V[b, h], mu[h], s2[h], lp[h], eps)
            assert np.max(np.abs(O[b, h] - Oh)) == 0.0


# ---------------------------------------------------------------- decode step and latent memory

def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def pin_decode_equals_masked_affinity():
    """Position-by-position decoding from an empty memory reproduces the
    causal output computed through the materialised, masked affinity
    ([GMA, causal variant, Eq. 8b]: each step adds its own key, then reads)."""
    rng = _rng(21)
    for (N, d_r, d_v, K) in [(23, 3, 4, 5), (9, 16, 2, 1), (12, 2, 3, 8)]:
        Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
        O, _, _ = oracle.decode(Q[None, None], Kx[None, None], V[None, None], mu, s2, lp, 1e-6)
        ref = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, 1e-6, causal=True)
        assert _rel(O[0, 0], ref) < 1e-12


def pin_decode_single_component_running_mean():
    """K = 1: every gamma is 1, so o_t = sum_{j<=t} V_j / (t + 1 + eps)."""
    rng = _rng(22)
    N, d_r, d_v, eps = 15, 4, 3, 1e-3
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, 1)
    O, Vt, Z = oracle.decode(Q[None], Kx[None], V[None], mu, s2, lp, eps)
    t = np.arange(N)[:, None]
    assert np.max(np.abs(O[0] - np.cumsum(V, 0) / (t + 1 + eps))) < 1e-12
    assert abs(Z[0, 0] - N) < 1e-12 and np.max(np.abs(Vt[0, 0] - V.sum(0))) < 1e-12


def pin_latent_memory_mass_and_prior():
    """Rows of Gamma^K sum to one, so sum_k Z_k = N and sum_k Vt_k = sum_j V_j;
    with identical components gamma = pi, so Vt_k = pi_k sum_j V_j, Z_k = N pi_k."""
    rng = _rng(23)
    N, d_r, d_v, K = 31, 5, 3, 6
    _, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    Vt, Z = oracle.latent_memory(Kx, V, mu, s2, lp)
    assert abs(Z.sum() - N) < 1e-11
    assert np.max(np.abs(Vt.sum(0) - V.sum(0))) < 1e-11
    mu_same = np.tile(mu[:1], (K, 1)); s2_same = np.tile(s2[:1], (K, 1))
    pi = rng.dirichlet(np.ones(K))
    Vt, Z = oracle.latent_memory(Kx, V, mu_same, s2_same, np.log(pi))
    assert np.max(np.abs(Z - N * pi)) < 1e-11
    assert np.max(np.abs(Vt - pi[:, None] * V.sum(0)[None])) < 1e-11


def pin_latent_memory_read_gives_bidir_affinity():
    """Reading the latent memory with the query responsibilities (Eq. 7)
    equals the bidirectional output through the materialised affinity."""
    rng = _rng(24)
    N, d_r, d_v, K, eps = 27, 3, 4, 5, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    Vt, Z = oracle.latent_memory(Kx, V, mu, s2, lp)
    ref = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, eps, causal=False)
    assert _rel(oracle.read_memory(Q, mu, s2, lp, eps, Vt, Z), ref) < 1e-12


def pin_sharded_memories_add_up():
    """Latent memories of key/value shards add up to the memory of the whole
    sequence (the sums of Eqs. 5-6 split over N), so reading their sum gives the
    bidirectional output, and decoding a shard from the exclusive prefix of the
    shard memories gives that shard's causal rows."""
    rng = _rng(31)
    N, d_r, d_v, K, eps = 40, 3, 2, 4, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    cuts = [0, 9, 10, 31, 40]
    mems = [oracle.latent_memory(Kx[a:b], V[a:b], mu, s2, lp) for a, b in zip(cuts[:-1], cuts[1:])]
    Vt, Z = sum(m[0] for m in mems), sum(m[1] for m in mems)
    ref_b = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, eps, causal=False)
    assert _rel(oracle.read_memory(Q[:20], mu, s2, lp, eps, Vt, Z), ref_b[:20]) < 1e-12
    ref_c = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, eps, causal=True)
    carry_v, carry_z = np.zeros((K, d_v)), np.zeros(K)
    for (a, b), (mv, mz) in zip(zip(cuts[:-1], cuts[1:]), mems):
        O, _, _ = oracle.decode(Q[None, a:b], Kx[None, a:b], V[None, a:b], mu, s2, lp, eps, carry_v[None],
                                carry_z[None])
        assert _rel(O[0], ref_c[a:b]) < 1e-12
        carry_v, carry_z = carry_v + mv, carry_z + mz


def pin_decode_continues_a_prompt():
    """The memory of a prompt (latent memory of its keys) is the carried
    state: decoding the rest from it gives the causal rows after the prompt,
    and the final state is the latent memory of the whole sequence."""
    rng = _rng(25)
    N, N0, d_r, d_v, K, eps = 20, 13, 4, 3, 6, 1e-6
    Q, Kx, V, mu, s2, lp = random_head(rng, N, d_r, d_v, K)
    Vt0, Z0 = oracle.latent_memory(Kx[:N0], V[:N0], mu, s2, lp)
    O, Vt, Z = oracle.decode(Q[None, N0:], Kx[None, N0:], V[None, N0:], mu, s2, lp, eps,
                             Vt0[None], Z0[None])
    ref = oracle.affinity_forward(Q, Kx, V, mu, s2, lp, eps, causal=True)[N0:]
    assert _rel(O[0], ref) < 1e-12
    Vt_all, Z_all = oracle.latent_memory(Kx, V, mu, s2, lp)
    assert np.max(np.abs(Vt[0] - Vt_all)) < 1e-11 and np.max(np.abs(Z[0] - Z_all)) < 1e-11


# ---------------------------------------------------------------- component-usage diagnostics

def pin_stats_totals():
    """usage and counts each sum to N; used = number of non-empty counts;
    the normalised entropy lies in [0, 1]."""
    rng = _rng(26)
    for (N, d_r, K) in [(40, 3, 7), (5, 2, 9)]:
        X, _, _, mu, s2, lp = random_head(rng, N, d_r, 1, K)
        st = oracle.routing_stats(X, mu, s2, lp)
        assert abs(st["usage"].sum() - N) < 1e-11 and st["counts"].sum() == N
        assert st["used"] == np.count_nonzero(st["counts"])
        assert np.all(np.bincount(st["z"], minlength=K) == st["counts"])
        assert -1e-12 <= st["entropy_norm"] <= 1 + 1e-12


def pin_stats_match_sklearn_and_scipy():
    """Hard assignments equal scikit-learn's GaussianMixture.predict and the
    usage its predict_proba column sums (host only); the entropy equals
    scipy.stats.entropy of the usage, and the normalised one that over log K."""
    from scipy.stats import entropy
    rng = _rng(27)
    N, d_r, K = 60, 3, 6
    X, _, _, mu, s2, lp = random_head(rng, N, d_r, 1, K)
    pi = np.exp(lp); pi /= pi.sum()
    st = oracle.routing_stats(X, mu, s2, np.log(pi))
    H = entropy(st["usage"])
    assert abs(st["entropy"] - H) < 1e-12
    assert abs(st["entropy_norm"] - H / math.log(K)) < 1e-12
    try:
        from sklearn.mixture import GaussianMixture
    except ImportError:  # the GPU machine has no scikit-learn
        return
    gm = GaussianMixture(n_components=K, covariance_type="diag")
    gm.weights_, gm.means_, gm.covariances_ = pi, mu, s2
    gm.precisions_cholesky_ = 1.0 / np.sqrt(s2)
    assert np.all(st["z"] == gm.predict(X))
    assert np.max(np.abs(st["usage"] - gm.predict_proba(X).sum(0))) < 1e-10


def pin_stats_identical_components():
    """Identical components: gamma = pi on every row, so usage = N pi, every
    row is assigned to the largest prior, and uniform priors give H_norm = 1."""
    rng = _rng(28)
    N, d_r, K = 17, 4, 5
    X = rng.normal(size=(N, d_r))
    mu = np.tile(rng.normal(size=(1, d_r)), (K, 1)); s2 = np.tile(rng.uniform(0.5, 2, (1, d_r)), (K, 1))
    pi = rng.dirichlet(np.ones(K))
    st = oracle.routing_stats(X, mu, s2, np.log(pi))
    assert np.max(np.abs(st["usage"] - N * pi)) < 1e-11
    assert np.all(st["z"] == np.argmax(pi)) and st["used"] == 1
    st = oracle.routing_stats(X, mu, s2, np.full(K, -math.log(K)))
    assert abs(st["entropy_norm"] - 1.0) < 1e-12 and np.all(st["z"] == 0)


def pin_stats_rows_at_component_means():
    """Equal variances and priors, well-separated means, x_i placed exactly on
    the mean of component c_i: the hard assignment is c_i."""
    rng = _rng(29)
    N, d_r, K = 50, 3, 8
    mu = rng.normal(scale=5.0, size=(K, d_r))
    c = rng.integers(0, K, size=N)
    st = oracle.routing_stats(mu[c], mu, np.ones((K, d_r)), np.full(K, -math.log(K)))
    assert np.all(st["z"] == c)
    assert np.all(st["counts"] == np.bincount(c, minlength=K))


def pin_stats_single_component():
    """K = 1: usage = counts = N, entropy 0, normalised entropy 1, one used."""
    rng = _rng(30)
    X, _, _, mu, s2, lp = random_head(rng, 11, 2, 1, 1)
    st = oracle.routing_stats(X, mu, s2, lp)
    assert abs(st["usage"][0] - 11) < 1e-12 and st["counts"][0] == 11
    assert st["entropy"] == 0.0 and st["entropy_norm"] == 1.0 and st["used"] == 1


# ---------------------------------------------------------------- reparameterisation (Eqs. 14-15)

def pin_reparameterize_matches_torch_and_scipy():
    """sigma2 = torch softplus(omega) + eps (fp64) and log_pi = scipy
    log_softmax(alpha); extreme omega (+-80) neither overflows nor loses the
    identity softplus(w) - softplus(-w) = w."""
    import torch
    from scipy.special import log_softmax
    rng = _rng(40)
    omega = rng.normal(scale=3.0, size=(3, 5, 4))
    omega[0, 0, :2] = [80.0, -80.0]
    alpha = rng.normal(scale=4.0, size=(3, 5))
    s2, lp = oracle.reparameterize(omega, alpha, 1e-3)
    ref = torch.nn.functional.softplus(torch.from_numpy(omega)).numpy() + 1e-3
    assert np.max(np.abs(s2 - ref) / ref) < 1e-14
    assert np.max(np.abs(lp - log_softmax(alpha, axis=-1))) < 1e-13
    s2n, _ = oracle.reparameterize(-omega, alpha, 0.0)
    assert np.max(np.abs((s2 - 1e-3) - s2n - omega)) < 1e-12


def pin_reparameterize_gradient_by_finite_differences():
    """Chain rule through Eqs. 14-15 against central differences of a random
    linear functional L = <G1, sigma2> + <G2, log_pi>; the prior-logit gradient
    sums to zero (log_pi is invariant to a shift of alpha)."""
    rng = _rng(41)
    K, d_r, h = 6, 3, 1e-6
    omega, alpha = rng.normal(size=(K, d_r)), rng.normal(size=K)
    G1, G2 = rng.normal(size=(K, d_r)), rng.normal(size=K)
    dw, da = oracle.reparameterize_backward(omega, alpha, G1, G2)

    def L(w, a):
        s2, lp = oracle.reparameterize(w, a, 1e-3)
        return float((G1 * s2).sum() + (G2 * lp).sum())

    for idx in [(0, 0), (3, 2), (5, 1)]:
        e = np.zeros_like(omega); e[idx] = h
        assert abs((L(omega + e, alpha) - L(omega - e, alpha)) / (2 * h) - dw[idx]) < 1e-8
    for k in range(K):
        e = np.zeros(K); e[k] = h
        assert abs((L(omega, alpha + e) - L(omega, alpha - e)) / (2 * h) - da[k]) < 1e-8
    assert abs(da.sum()) < 1e-12


# ---------------------------------------------------------------- projections (Eq. 4)

def pin_project_matches_einsum_and_selects_heads():
    """Q_X[b, h, n, c] = sum_i X[b, n, i] W[h d + c, i] equals numpy's einsum; a
    weight that copies input column (h d + c) gives back the head-split input."""
    rng = _rng(50)
    B, N, D, H, d_r, d_v = 2, 7, 24, 3, 4, 8
    X = rng.normal(size=(B, N, D))
    Wq, Wk, Wv = rng.normal(size=(H * d_r, D)), rng.normal(size=(H * d_r, D)), rng.normal(size=(H * d_v, D))
    Q, K, V = oracle.project_qkv(X, Wq, Wk, Wv, H)
    for P, W, d in ((Q, Wq, d_r), (K, Wk, d_r), (V, Wv, d_v)):
        ref = np.einsum("bni,oi->bno", X, W).reshape(B, N, H, d).transpose(0, 2, 1, 3)
        assert P.shape == (B, H, N, d) and np.max(np.abs(P - ref)) < 1e-12
    sel = np.eye(H * d_v, D)
    _, _, V = oracle.project_qkv(X, Wq, Wk, sel, H)
    assert np.array_equal(V, X[:, :, :H * d_v].reshape(B, N, H, d_v).transpose(0, 2, 1, 3))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
