"""fp64 CPU oracle for the GMA forward pass and its gradients -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it imports nothing from the CUDA side.

The arithmetic lives in ``gma_oracle.c`` (plain C, fp64, single-threaded);
this module compiles it with gcc and exposes numpy wrappers that loop over
(batch, head).  Every definition cites "Gaussian Mixture Attention:
Linear-Time Sequence Mixing via Probabilistic Latent Routing" (arXiv
2606.18283), written [GMA, ...]:

* ``scores`` / ``responsibilities``  -- Eqs. (2)-(3) (reconstructed from prose)
* ``forward_bidir``                  -- Eqs. (5)-(7), footnote 4
* ``forward_causal``                 -- Eqs. (8a)/(8b), cumulative-sum remark
* ``affinity`` / ``affinity_forward`` -- Eqs. (9)-(11), brute force for tiny N
* ``bidir_rows`` / ``causal_rows``   -- the same definitions on selected rows
* ``backward_bidir`` / ``backward_causal`` -- gradients: gradient section,
  Eq. (18) (score gradient) and the chain rule through the score
* ``latent_memory``                  -- Eqs. (5)-(6): Vt, Z of a key/value sequence
* ``read_memory``                    -- Eq. (7) from a given memory (Vt, Z)
* ``decode_step`` / ``decode``        -- Eq. (8b) one position at a time (carried Vt, Z)
* ``project_qkv``                    -- Eq. (4): Q_X, K_X, V_X = X W^T, split into heads
* ``reparameterize`` (+ ``_backward``) -- Eqs. (14)-(15): sigma2 = softplus(omega) + eps,
  log pi = log_softmax(alpha), and the chain rule through them
* ``routing_stats``                  -- component usage, hard assignments, usage entropy
  (the introduction's usage / hard-assignment diagnostics)

Parity pins: see ``tests/test_oracle.py`` (closed forms, invariants, brute
force, scipy / scikit-learn textbook routines, hand-derived golden values)
and ``tests/test_oracle_backward.py`` (central finite differences of the
forward, shift and translation invariances, K = 1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gma_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict = {}
_ACTIVE = [0]  # which build the functions below call; 0 is the oracle

_D = ctypes.POINTER(ctypes.c_double)
_L = ctypes.POINTER(ctypes.c_long)


def _lib_path(mutant: int) -> str:
    name = "libgma_oracle.so" if mutant == 0 else f"libgma_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD_DIR, name)


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile gma_oracle.c with gcc (no fast-math, no FMA contraction).

    ``mutant`` != 0 builds a deliberately broken copy (see the list at the
    top of gma_oracle.c); only the pin-strength tests ask for one.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    path = _lib_path(mutant)
    stale = (not os.path.exists(path)) or (os.path.getmtime(path) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", f"-DGMA_ORACLE_MUTANT={int(mutant)}", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


def _load(mutant: int = 0):
    with _lock:
        lib = _libs.get(mutant)
        if lib is None:
            lib = ctypes.CDLL(build(mutant=mutant))
            common = [_D, _D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D, _D,
                      ctypes.c_int, ctypes.c_double]
            lib.gma_oracle_scores.argtypes = [_D, ctypes.c_int, ctypes.c_int, _D, _D, _D,
                                              ctypes.c_int, _D]
            lib.gma_oracle_responsibilities.argtypes = lib.gma_oracle_scores.argtypes
            lib.gma_oracle_bidir.argtypes = common + [_D]
            lib.gma_oracle_causal.argtypes = common + [_D]
            lib.gma_oracle_bidir_rows.argtypes = common + [_L, ctypes.c_int, _D]
            lib.gma_oracle_causal_rows.argtypes = common + [_L, ctypes.c_int, _D]
            lib.gma_oracle_causal_rows.restype = ctypes.c_int
            lib.gma_oracle_bidir_rows.restype = None
            lib.gma_oracle_affinity_forward.argtypes = common + [ctypes.c_int, _D]
            lib.gma_oracle_affinity.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, _D, _D,
                                                _D, ctypes.c_int, _D]
            lib.gma_oracle_bidir_backward.argtypes = common + [_D] * 7
            lib.gma_oracle_causal_backward.argtypes = common + [_D] * 7
            lib.gma_oracle_latent_memory.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, _D, _D, _D, ctypes.c_int,
                                                     _D, _D]
            lib.gma_oracle_latent_memory.restype = None
            lib.gma_oracle_decode_step.argtypes = [_D, _D, _D, ctypes.c_int, ctypes.c_int, _D,
                                                   _D, _D, ctypes.c_int, ctypes.c_double, _D,
                                                   _D, _D]
            lib.gma_oracle_decode_step.restype = None
            lib.gma_oracle_routing_stats.argtypes = [_D, ctypes.c_int, ctypes.c_int, _D, _D, _D,
                                                     ctypes.c_int, _D, _L, _L, _D]
            lib.gma_oracle_routing_stats.restype = None
            lib.gma_oracle_read_memory.argtypes = [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, _D, _D,
                                                   _D, ctypes.c_int, ctypes.c_double, _D, _D, _D]
            lib.gma_oracle_read_memory.restype = None
            lib.gma_oracle_project.argtypes = [_D, ctypes.c_int, ctypes.c_int, _D, ctypes.c_int, _D]
            lib.gma_oracle_project.restype = None
            lib.gma_oracle_reparameterize.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                      _D, _D]
            lib.gma_oracle_reparameterize.restype = None
            lib.gma_oracle_reparameterize_backward.argtypes = [_D, _D, ctypes.c_int, ctypes.c_int, _D, _D, _D,
                                                               _D]
            lib.gma_oracle_reparameterize_backward.restype = None
            _libs[mutant] = lib
    return lib


def _f64(a) -> np.ndarray:
    """Exact widening to a C-contiguous fp64 array (accepts numpy or torch)."""
    if hasattr(a, "detach"):  # torch tensor: widen on the CPU, exactly
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _heads(x: np.ndarray, nd: int):
    """View an array [..., rows, cols] as [(batch*heads), rows, cols]."""
    return x.reshape((-1,) + x.shape[-nd:])


def _params(mu, sigma2, log_pi):
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    if mu.ndim == 2:
        mu, sigma2, log_pi = mu[None], sigma2[None], log_pi[None]
    return mu, sigma2, log_pi


def _head_param(h_flat: int, H: int, mu, sigma2, log_pi):
    h = h_flat % H
    return (np.ascontiguousarray(mu[h]), np.ascontiguousarray(sigma2[h]),
            np.ascontiguousarray(log_pi[h]))


def scores(X, mu, sigma2, log_pi) -> np.ndarray:
    """Scores s_ik for X [..., N, d_r] with one head's params [K, d_r], [K]."""
    lib = _load(_ACTIVE[0])
    X = _f64(X)
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    N, d_r = X.shape[-2:]
    K = mu.shape[0]
    Xh = _heads(X, 2)
    out = np.empty(Xh.shape[:-1] + (K,), np.float64)
    for b in range(Xh.shape[0]):
        xb = np.ascontiguousarray(Xh[b])
        lib.gma_oracle_scores(_p(xb), N, d_r, _p(mu), _p(sigma2), _p(log_pi), K, _p(out[b]))
    return out.reshape(X.shape[:-1] + (K,))


def responsibilities(X, mu, sigma2, log_pi) -> np.ndarray:
    """Gamma [B, H, N, K] for X [B, H, N, d_r], per-head params [H, K, d_r] / [H, K].

    Two-dimensional X with [K, d_r] params is one head.
    """
    lib = _load(_ACTIVE[0])
    X = _f64(X)
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H = mu.shape[0]
    N, d_r = X.shape[-2:]
    K = mu.shape[1]
    Xh = _heads(X, 2)
    out = np.empty(Xh.shape[:-1] + (K,), np.float64)
    for b in range(Xh.shape[0]):
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        xb = np.ascontiguousarray(Xh[b])
        lib.gma_oracle_responsibilities(_p(xb), N, d_r, _p(m), _p(s), _p(lp), K, _p(out[b]))
    return out.reshape(X.shape[:-1] + (K,))


def _forward(fn_name, Q, K_, V, mu, sigma2, log_pi, eps, extra=None):
    lib = _load(_ACTIVE[0])
    fn = getattr(lib, fn_name)
    Q, K_, V = _f64(Q), _f64(K_), _f64(V)
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H = mu.shape[0]
    N, d_r = Q.shape[-2:]
    d_v = V.shape[-1]
    K = mu.shape[1]
    Qh, Kh, Vh = _heads(Q, 2), _heads(K_, 2), _heads(V, 2)
    out = np.empty(Vh.shape, np.float64)
    for b in range(Qh.shape[0]):
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        q, k, v = (np.ascontiguousarray(t[b]) for t in (Qh, Kh, Vh))
        args = [_p(q), _p(k), _p(v), N, d_r, d_v, _p(m), _p(s), _p(lp), K, float(eps)]
        if extra is not None:
            args.append(extra)
        fn(*args, _p(out[b]))
    return out.reshape(V.shape)


def forward_bidir(Q, K_, V, mu, sigma2, log_pi, eps) -> np.ndarray:
    """Bidirectional O [B, H, N, d_v] ([GMA, Eqs. 5-7])."""
    return _forward("gma_oracle_bidir", Q, K_, V, mu, sigma2, log_pi, eps)


def forward_causal(Q, K_, V, mu, sigma2, log_pi, eps) -> np.ndarray:
    """Causal O [B, H, N, d_v] ([GMA, Eq. 8b], j <= i inclusive)."""
    return _forward("gma_oracle_causal", Q, K_, V, mu, sigma2, log_pi, eps)


def affinity_forward(Q, K_, V, mu, sigma2, log_pi, eps, causal: bool) -> np.ndarray:
    """Brute force O = A^GMA V through the materialised N x N affinity (tiny N)."""
    return _forward("gma_oracle_affinity_forward", Q, K_, V, mu, sigma2, log_pi, eps,
                    extra=int(bool(causal)))


def affinity(Q, K_, mu, sigma2, log_pi) -> np.ndarray:
    """Un-normalised affinity Gamma^Q (Gamma^K)^T for one head ([GMA, Eq. 11])."""
    lib = _load(_ACTIVE[0])
    Q, K_ = _f64(Q), _f64(K_)
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    N, d_r = Q.shape
    A = np.empty((N, N), np.float64)
    lib.gma_oracle_affinity(_p(Q), _p(K_), N, d_r, _p(mu), _p(sigma2), _p(log_pi),
                            mu.shape[0], _p(A))
    return A


def _backward(fn_name, Q, K_, V, mu, sigma2, log_pi, eps, dO) -> dict:
    lib = _load(_ACTIVE[0])
    fn = getattr(lib, fn_name)
    Q, K_, V, dO = _f64(Q), _f64(K_), _f64(V), _f64(dO)
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H = mu.shape[0]
    N, d_r = Q.shape[-2:]
    d_v = V.shape[-1]
    K = mu.shape[1]
    Qh, Kh, Vh, dOh = _heads(Q, 2), _heads(K_, 2), _heads(V, 2), _heads(dO, 2)
    dQ, dK, dV = np.empty(Qh.shape), np.empty(Kh.shape), np.empty(Vh.shape)
    dmu, ds2, dlp = np.zeros(mu.shape), np.zeros(sigma2.shape), np.zeros(log_pi.shape)
    for b in range(Qh.shape[0]):
        h = b % H
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        q, k, v, g = (np.ascontiguousarray(t[b]) for t in (Qh, Kh, Vh, dOh))
        gm, gs, gl = np.zeros_like(m), np.zeros_like(s), np.zeros_like(lp)
        fn(_p(q), _p(k), _p(v), N, d_r, d_v, _p(m), _p(s), _p(lp), K, float(eps), _p(g),
           _p(dQ[b]), _p(dK[b]), _p(dV[b]), _p(gm), _p(gs), _p(gl))
        dmu[h] += gm
        ds2[h] += gs
        dlp[h] += gl
    return {"dQ": dQ.reshape(Q.shape), "dK": dK.reshape(K_.shape), "dV": dV.reshape(V.shape),
            "dmu": dmu, "dsigma2": ds2, "dlog_pi": dlp}


def backward_bidir(Q, K_, V, mu, sigma2, log_pi, eps, dO) -> dict:
    """Gradients of the bidirectional forward for upstream dO ([GMA, gradient
    section, Eq. 18 and the chain rule through the score]): dQ, dK, dV shaped
    like the inputs; dmu, dsigma2 [H, K, d_r] and dlog_pi [H, K] summed over
    the batch (per-head parameters; a single head's [K, d_r] params give a
    leading axis of 1)."""
    return _backward("gma_oracle_bidir_backward", Q, K_, V, mu, sigma2, log_pi, eps, dO)


def backward_causal(Q, K_, V, mu, sigma2, log_pi, eps, dO) -> dict:
    """Gradients of the causal forward ([GMA, Eq. 8b] differentiated: prefix
    memories forward, suffix sums backward); same outputs as backward_bidir."""
    return _backward("gma_oracle_causal_backward", Q, K_, V, mu, sigma2, log_pi, eps, dO)


def _rows(fn_name, q, k, v, mu_h, s2_h, lp_h, eps, rows):
    lib = _load(_ACTIVE[0])
    q, k, v = _f64(q), _f64(k), _f64(v)
    mu_h, s2_h, lp_h = _f64(mu_h), _f64(s2_h), _f64(lp_h)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    N, d_r = q.shape
    d_v = v.shape[1]
    out = np.empty((rows.shape[0], d_v), np.float64)
    rc = getattr(lib, fn_name)(_p(q), _p(k), _p(v), N, d_r, d_v, _p(mu_h), _p(s2_h),
                               _p(lp_h), mu_h.shape[0], float(eps),
                               rows.ctypes.data_as(_L), int(rows.shape[0]), _p(out))
    if rc not in (None, 0):
        raise ValueError("rows must be sorted ascending and within [0, N)")
    return out


def bidir_rows(q, k, v, mu_h, s2_h, lp_h, eps, rows) -> np.ndarray:
    """Bidirectional O rows of one head (q, k, v: [N, d]; params of that head)."""
    return _rows("gma_oracle_bidir_rows", q, k, v, mu_h, s2_h, lp_h, eps, rows)


def causal_rows(q, k, v, mu_h, s2_h, lp_h, eps, rows) -> np.ndarray:
    """Causal O rows of one head; ``rows`` sorted ascending."""
    return _rows("gma_oracle_causal_rows", q, k, v, mu_h, s2_h, lp_h, eps, rows)


def latent_memory(K_, V, mu, sigma2, log_pi):
    """Latent memory ([GMA, Eqs. 5-6]) of K_X [B, H, N, d_r], V_X [B, H, N, d_v]:
    returns (Vt [B, H, K, d_v], Z [B, H, K]).  Also the causal carried state
    after the last position."""
    lib = _load(_ACTIVE[0])
    K_, V = _f64(K_), _f64(V)
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H, K = mu.shape[0], mu.shape[1]
    N, d_r = K_.shape[-2:]
    d_v = V.shape[-1]
    Kh, Vh = _heads(K_, 2), _heads(V, 2)
    Vt = np.empty((Kh.shape[0], K, d_v))
    Z = np.empty((Kh.shape[0], K))
    for b in range(Kh.shape[0]):
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        k, v = np.ascontiguousarray(Kh[b]), np.ascontiguousarray(Vh[b])
        lib.gma_oracle_latent_memory(_p(k), _p(v), N, d_r, d_v, _p(m), _p(s), _p(lp), K,
                                     _p(Vt[b]), _p(Z[b]))
    lead = K_.shape[:-2]
    return Vt.reshape(lead + (K, d_v)), Z.reshape(lead + (K,))


def read_memory(Q, mu, sigma2, log_pi, eps, Vt, Z) -> np.ndarray:
    """O [B, H, N, d_v] = Gamma^Q Vt / (Gamma^Q Z + eps) ([GMA, Eq. 7]) for Q
    [B, H, N, d_r] and a given memory Vt [B, H, K, d_v], Z [B, H, K]."""
    lib = _load(_ACTIVE[0])
    Q, Vt, Z = _f64(Q), _f64(Vt), _f64(Z)
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H, K = mu.shape[0], mu.shape[1]
    N, d_r = Q.shape[-2:]
    d_v = Vt.shape[-1]
    Qh, Vth, Zh = _heads(Q, 2), Vt.reshape(-1, K, d_v), Z.reshape(-1, K)
    O = np.empty((Qh.shape[0], N, d_v))
    for b in range(Qh.shape[0]):
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        q, vt, z = (np.ascontiguousarray(t[b]) for t in (Qh, Vth, Zh))
        lib.gma_oracle_read_memory(_p(q), N, d_r, d_v, _p(m), _p(s), _p(lp), K, float(eps), _p(vt), _p(z),
                                   _p(O[b]))
    return O.reshape(Q.shape[:-1] + (d_v,))


def decode_step(q, k, v, mu, sigma2, log_pi, eps, Vt, Z):
    """One causal position ([GMA, Eq. 8b]) for every (b, h): q, k [B, H, d_r],
    v [B, H, d_v], carried Vt [B, H, K, d_v], Z [B, H, K].  Returns
    (o [B, H, d_v], Vt', Z'); the inputs are not modified."""
    lib = _load(_ACTIVE[0])
    q, k, v = _f64(q), _f64(k), _f64(v)
    Vt, Z = _f64(Vt).copy(), _f64(Z).copy()
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H, K = mu.shape[0], mu.shape[1]
    d_r, d_v = q.shape[-1], v.shape[-1]
    qh, kh, vh = q.reshape(-1, d_r), k.reshape(-1, d_r), v.reshape(-1, d_v)
    Vth, Zh = Vt.reshape(-1, K, d_v), Z.reshape(-1, K)
    o = np.empty((qh.shape[0], d_v))
    for b in range(qh.shape[0]):
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        qb, kb, vb = (np.ascontiguousarray(t[b]) for t in (qh, kh, vh))
        vt_b, z_b = np.ascontiguousarray(Vth[b]), np.ascontiguousarray(Zh[b])
        lib.gma_oracle_decode_step(_p(qb), _p(kb), _p(vb), d_r, d_v, _p(m), _p(s), _p(lp), K,
                                   float(eps), _p(vt_b), _p(z_b), _p(o[b]))
        Vth[b], Zh[b] = vt_b, z_b
    return o.reshape(v.shape), Vth.reshape(Vt.shape), Zh.reshape(Z.shape)


def decode(Q, K_, V, mu, sigma2, log_pi, eps, Vt=None, Z=None):
    """Run decode_step over the positions of Q, K_X, V_X [B, H, T, d] in order,
    starting from (Vt, Z) (zeros if None).  Returns (O [B, H, T, d_v], Vt, Z)."""
    Q, K_, V = _f64(Q), _f64(K_), _f64(V)
    K = _params(mu, sigma2, log_pi)[0].shape[1]
    lead, T, d_v = Q.shape[:-2], Q.shape[-2], V.shape[-1]
    Vt = np.zeros(lead + (K, d_v)) if Vt is None else _f64(Vt)
    Z = np.zeros(lead + (K,)) if Z is None else _f64(Z)
    O = np.empty(lead + (T, d_v))
    for t in range(T):
        O[..., t, :], Vt, Z = decode_step(Q[..., t, :], K_[..., t, :], V[..., t, :], mu, sigma2,
                                          log_pi, eps, Vt, Z)
    return O, Vt, Z


def routing_stats(X, mu, sigma2, log_pi) -> dict:
    """Component-usage diagnostics of X [B, H, N, d_r] per (b, h): usage
    [B, H, K] (sum of responsibilities), counts [B, H, K] and z [B, H, N] (hard
    assignments, smallest k on ties), entropy / entropy_norm / used [B, H]."""
    lib = _load(_ACTIVE[0])
    X = _f64(X)
    mu, sigma2, log_pi = _params(mu, sigma2, log_pi)
    H, K = mu.shape[0], mu.shape[1]
    N, d_r = X.shape[-2:]
    Xh = _heads(X, 2)
    nb = Xh.shape[0]
    usage = np.empty((nb, K))
    counts = np.empty((nb, K), np.int64)
    z = np.empty((nb, N), np.int64)
    st = np.empty((nb, 3))
    for b in range(nb):
        m, s, lp = _head_param(b, H, mu, sigma2, log_pi)
        xb = np.ascontiguousarray(Xh[b])
        u_b, c_b, z_b, s_b = usage[b], counts[b], z[b], st[b]
        lib.gma_oracle_routing_stats(_p(xb), N, d_r, _p(m), _p(s), _p(lp), K, _p(u_b),
                                     c_b.ctypes.data_as(_L), z_b.ctypes.data_as(_L), _p(s_b))
    lead = X.shape[:-2]
    return {"usage": usage.reshape(lead + (K,)), "counts": counts.reshape(lead + (K,)),
            "z": z.reshape(lead + (N,)), "entropy": st[:, 0].reshape(lead),
            "entropy_norm": st[:, 1].reshape(lead), "used": st[:, 2].astype(np.int64).reshape(lead)}


def project_qkv(X, W_q, W_k, W_v, H: int):
    """Q_X, K_X, V_X [B, H, N, d] of the layer input X [B, N, D] ([GMA, Eq. 4],
    Q_X = X W_Q^T with W_Q [H * d_r, D] stored one output feature per row;
    output feature h * d + c of a projection is column c of head h)."""
    lib = _load(_ACTIVE[0])
    X = _f64(X)
    B, N, D = X.shape
    outs = []
    for W in (W_q, W_k, W_v):
        W = _f64(W)
        O = W.shape[0]
        Y = np.empty((B * N, O))
        x = np.ascontiguousarray(X.reshape(B * N, D))
        lib.gma_oracle_project(_p(x), B * N, D, _p(W), O, _p(Y))
        outs.append(np.ascontiguousarray(Y.reshape(B, N, H, O // H).transpose(0, 2, 1, 3)))
    return tuple(outs)


def reparameterize(omega, alpha, eps_sigma=1e-3):
    """([GMA, Eqs. 14-15]) sigma2 = softplus(omega) + eps_sigma, log_pi =
    log_softmax(alpha), per head: omega [H, K, d_r], alpha [H, K] (a 2-D omega
    with a 1-D alpha is one head)."""
    lib = _load(_ACTIVE[0])
    omega, alpha = _f64(omega), _f64(alpha)
    one = omega.ndim == 2
    if one:
        omega, alpha = omega[None], alpha[None]
    H, K, d_r = omega.shape
    s2, lp = np.empty_like(omega), np.empty_like(alpha)
    for h in range(H):
        w, a = np.ascontiguousarray(omega[h]), np.ascontiguousarray(alpha[h])
        s_h, l_h = np.empty((K, d_r)), np.empty(K)
        lib.gma_oracle_reparameterize(_p(w), _p(a), K, d_r, float(eps_sigma), _p(s_h), _p(l_h))
        s2[h], lp[h] = s_h, l_h
    return (s2[0], lp[0]) if one else (s2, lp)


def reparameterize_backward(omega, alpha, dsigma2, dlog_pi):
    """Gradients of reparameterize: (domega, dalpha) for upstream (dsigma2, dlog_pi)."""
    lib = _load(_ACTIVE[0])
    omega, alpha, dsigma2, dlog_pi = _f64(omega), _f64(alpha), _f64(dsigma2), _f64(dlog_pi)
    one = omega.ndim == 2
    if one:
        omega, alpha, dsigma2, dlog_pi = omega[None], alpha[None], dsigma2[None], dlog_pi[None]
    H, K, d_r = omega.shape
    dw, da = np.empty_like(omega), np.empty_like(alpha)
    for h in range(H):
        w, a = np.ascontiguousarray(omega[h]), np.ascontiguousarray(alpha[h])
        gs, gl = np.ascontiguousarray(dsigma2[h]), np.ascontiguousarray(dlog_pi[h])
        dw_h, da_h = np.empty((K, d_r)), np.empty(K)
        lib.gma_oracle_reparameterize_backward(_p(w), _p(a), K, d_r, _p(gs), _p(gl), _p(dw_h), _p(da_h))
        dw[h], da[h] = dw_h, da_h
    return (dw[0], da[0]) if one else (dw, da)


class use_mutant:
    """Context manager: route the functions above to a planted-mistake build.

    For the pin-strength tests only; ``with use_mutant(3): ...``.
    """

    def __init__(self, mutant: int):
        self.mutant = int(mutant)

    def __enter__(self):
        self.prev = _ACTIVE[0]
        _ACTIVE[0] = self.mutant
        return self

    def __exit__(self, *exc):
        _ACTIVE[0] = self.prev
        return False
