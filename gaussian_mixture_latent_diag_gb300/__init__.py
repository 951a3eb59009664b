"""GMA forward hot path on GB300 (sm_103a): Python binding of libgma.so.

    import gaussian_mixture_latent_diag_gb300 as gma
    O = gma.forward_bidir(Q, K, V, mu, sigma2, log_pi, eps=1e-6)
    O = gma.forward_causal(Q, K, V, mu, sigma2, log_pi, eps=1e-6)
    G = gma.responsibilities(X, mu, sigma2, log_pi)
    Vt, Z = gma.latent_memory(K, V, mu, sigma2, log_pi)          # prompt -> carried state
    o = gma.decode_step(q, k, v, mu, sigma2, log_pi, Vt, Z)      # one position, state in place
    st = gma.routing_stats(X, mu, sigma2, log_pi)                 # usage, hard assignments, entropy

Tensors: Q, K, X [B, H, N, d_r], V [B, H, N, d_v] (CUDA, contiguous, fp32 or
bf16); mu, sigma2 [H, K, d_r] and log_pi [H, K] fp32 CUDA.  The functions
only marshal arguments; the arithmetic runs in libgma.so's CUDA kernels.
PyTorch provides device memory and the current stream.

Paper: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
Probabilistic Latent Routing" (arXiv 2606.18283).
"""
from __future__ import annotations

import ctypes

from ._native import (GMA_BF16, GMA_F32, PATH_AUTO, PATH_SIMT, PATH_TC, PATH_TC_SINGLE_PASS, GmaError,
                      load, options, status_string)

__all__ = ["forward_bidir", "forward_causal", "backward_bidir", "backward_causal", "responsibilities",
           "latent_memory", "read_memory", "forward_causal_carry", "decode_step", "routing_stats",
           "reparameterize", "reparameterize_backward", "project_qkv",
           "workspace_size",
           "selected_path", "last_device_status", "GmaError", "PATH_AUTO", "PATH_SIMT",
           "PATH_TC", "PATH_TC_SINGLE_PASS", "load"]


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return GMA_F32
    if t.dtype == torch.bfloat16:
        return GMA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _check_dev(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def workspace_size(B, H, N, d_r, d_v, K, dtype="bf16", causal=0, path=PATH_AUTO, splits=0) -> int:
    """Workspace bytes for a call (causal: 0 bidir, 1 causal, -1 responsibilities)."""
    code = GMA_F32 if dtype in ("f32", "float32") else GMA_BF16
    opt = options(path=path, splits=splits)
    return int(load().gma_workspace_size(B, H, N, d_r, d_v, K, code, causal, ctypes.byref(opt)))


def selected_path(N, d_r, d_v, K, dtype="bf16", causal=0, path=PATH_AUTO) -> int:
    code = GMA_F32 if dtype in ("f32", "float32") else GMA_BF16
    opt = options(path=path)
    return int(load().gma_selected_path(N, d_r, d_v, K, code, causal, ctypes.byref(opt)))


def _workspace(nbytes: int, device, workspace):
    import torch
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def last_device_status(workspace, stream=None) -> int:
    """Synchronise the stream; device-side status of the last call on `workspace`."""
    return int(load().gma_last_device_status(_ptr(workspace), _stream(stream)))


def responsibilities(X, mu, sigma2, log_pi, out=None, workspace=None, stream=None,
                     sync_status=False):
    """Gamma [B, H, N, K] fp32: posterior responsibilities of the rows of X."""
    import torch
    lib = load()
    _check_dev(X, mu, sigma2, log_pi)
    B, H, N, d_r = X.shape
    K = mu.shape[1]
    code = _dtype_code(X)
    if out is None:
        out = torch.empty(B, H, N, K, dtype=torch.float32, device=X.device)
    opt = options(sync_status=sync_status)
    nb = int(lib.gma_workspace_size(B, H, N, d_r, 16, K, code, -1, ctypes.byref(opt)))
    ws = _workspace(nb, X.device, workspace)
    st = lib.gma_responsibilities(_ptr(X), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(out),
                                  B, H, N, d_r, K, ctypes.byref(opt), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_responsibilities")
    return out


def _forward(fn_name, Q, K_, V, mu, sigma2, log_pi, eps, out, workspace, stream, path, splits,
             sync_status, o_bf16=False, chunk=0):
    import torch
    lib = load()
    _check_dev(Q, K_, V, mu, sigma2, log_pi)
    B, H, N, d_r = Q.shape
    d_v = V.shape[-1]
    K = mu.shape[1]
    if K_.shape != Q.shape or V.shape[:3] != Q.shape[:3]:
        raise ValueError("Q, K must be [B, H, N, d_r] and V [B, H, N, d_v]")
    if mu.shape != (H, K, d_r) or sigma2.shape != (H, K, d_r) or log_pi.shape != (H, K):
        raise ValueError("mu, sigma2 must be [H, K, d_r] and log_pi [H, K]")
    code = _dtype_code(Q)
    if K_.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K, V must share one dtype")
    odt = torch.bfloat16 if o_bf16 else torch.float32
    if out is None:
        out = torch.empty(B, H, N, d_v, dtype=odt, device=Q.device)
    elif out.dtype != odt or out.shape != V.shape:
        raise ValueError(f"out must be {odt} of shape {tuple(V.shape)}")
    causal = 1 if fn_name == "gma_forward_causal" else 0
    opt = options(path=path, chunk=chunk, splits=splits, sync_status=sync_status, o_bf16=o_bf16)
    nb = int(lib.gma_workspace_size(B, H, N, d_r, d_v, K, code, causal, ctypes.byref(opt)))
    if nb == 0:
        raise GmaError(2, fn_name)
    ws = _workspace(nb, Q.device, workspace)
    st = getattr(lib, fn_name)(_ptr(Q), _ptr(K_), _ptr(V), code, _ptr(mu), _ptr(sigma2),
                               _ptr(log_pi), float(eps), _ptr(out), B, H, N, d_r, d_v, K,
                               ctypes.byref(opt), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream))
    if st != 0:
        raise GmaError(st, fn_name)
    return out


def forward_bidir(Q, K, V, mu, sigma2, log_pi, eps=1e-6, out=None, workspace=None, stream=None,
                  path=PATH_AUTO, splits=0, sync_status=False, o_bf16=False):
    """Bidirectional GMA: O = Gamma^Q (Gamma^K)^T V / (Gamma^Q Z + eps); O fp32 (or bf16)."""
    return _forward("gma_forward_bidir", Q, K, V, mu, sigma2, log_pi, eps, out, workspace,
                    stream, path, splits, sync_status, o_bf16)


def forward_causal(Q, K, V, mu, sigma2, log_pi, eps=1e-6, out=None, workspace=None, stream=None,
                   path=PATH_AUTO, splits=0, sync_status=False, o_bf16=False, chunk=0):
    """Causal GMA: prefix memories over keys j <= i; O fp32 (or bf16).  ``chunk``:
    0 or the kernel family's chunk length (see gma_options.chunk)."""
    return _forward("gma_forward_causal", Q, K, V, mu, sigma2, log_pi, eps, out, workspace,
                    stream, path, splits, sync_status, o_bf16, chunk)


def backward_bidir(Q, K, V, mu, sigma2, log_pi, dO, eps=1e-6, workspace=None, stream=None,
                   splits=0, sync_status=False) -> dict:
    """Gradients of forward_bidir for upstream dO (fp32, like O): dict of dQ, dK, dV
    (fp32, shaped like Q, K, V) and dmu, dsigma2 [H, K, d_r], dlog_pi [H, K] summed
    over the batch and over the query and key rows."""
    return _backward("gma_backward_bidir", Q, K, V, mu, sigma2, log_pi, dO, eps, workspace, stream, splits,
                     sync_status)


def backward_causal(Q, K, V, mu, sigma2, log_pi, dO, eps=1e-6, workspace=None, stream=None,
                    sync_status=False) -> dict:
    """Gradients of forward_causal for upstream dO; same outputs as backward_bidir."""
    return _backward("gma_backward_causal", Q, K, V, mu, sigma2, log_pi, dO, eps, workspace, stream, 0,
                     sync_status)


def _backward(fn_name, Q, K, V, mu, sigma2, log_pi, dO, eps, workspace, stream, splits, sync_status) -> dict:
    import torch
    lib = load()
    _check_dev(Q, K, V, mu, sigma2, log_pi, dO)
    B, H, N, d_r = Q.shape
    d_v = V.shape[-1]
    Kc = mu.shape[1]
    if K.shape != Q.shape or V.shape[:3] != Q.shape[:3] or dO.shape != V.shape:
        raise ValueError("Q, K must be [B, H, N, d_r], V and dO [B, H, N, d_v]")
    if mu.shape != (H, Kc, d_r) or sigma2.shape != (H, Kc, d_r) or log_pi.shape != (H, Kc):
        raise ValueError("mu, sigma2 must be [H, K, d_r] and log_pi [H, K]")
    if dO.dtype != torch.float32:
        raise TypeError("dO must be fp32")
    code = _dtype_code(Q)
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K, V must share one dtype")
    dev = Q.device
    out = {"dQ": torch.empty(B, H, N, d_r, dtype=torch.float32, device=dev),
           "dK": torch.empty(B, H, N, d_r, dtype=torch.float32, device=dev),
           "dV": torch.empty(B, H, N, d_v, dtype=torch.float32, device=dev),
           "dmu": torch.empty(H, Kc, d_r, dtype=torch.float32, device=dev),
           "dsigma2": torch.empty(H, Kc, d_r, dtype=torch.float32, device=dev),
           "dlog_pi": torch.empty(H, Kc, dtype=torch.float32, device=dev)}
    opt = options(splits=splits, sync_status=sync_status)
    causal = 1 if fn_name == "gma_backward_causal" else 0
    nb = int(lib.gma_backward_workspace_size(B, H, N, d_r, d_v, Kc, code, causal, ctypes.byref(opt)))
    if nb == 0:
        raise GmaError(2, fn_name)
    ws = _workspace(nb, dev, workspace)
    st = getattr(lib, fn_name)(_ptr(Q), _ptr(K), _ptr(V), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi),
                                float(eps), _ptr(dO), _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]),
                                _ptr(out["dmu"]), _ptr(out["dsigma2"]), _ptr(out["dlog_pi"]),
                                B, H, N, d_r, d_v, Kc, ctypes.byref(opt), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, fn_name)
    return out


def _params_check(H, d_r, mu, sigma2, log_pi):
    K = mu.shape[1]
    if mu.shape != (H, K, d_r) or sigma2.shape != (H, K, d_r) or log_pi.shape != (H, K):
        raise ValueError("mu, sigma2 must be [H, K, d_r] and log_pi [H, K]")
    return K


def latent_memory(K, V, mu, sigma2, log_pi, workspace=None, stream=None, splits=0, sync_status=False,
                  path=PATH_AUTO):
    """Latent memory of a key/value sequence: (Vt [B, H, K, d_v], Z [B, H, K]) fp32,
    Vt = Gamma^K^T V, Z = Gamma^K^T 1.  It is also the causal state after the last
    position, i.e. what decode_step continues from after a prompt.  path=PATH_TC
    runs it on the tensor-core kernels (bf16, d_r in {32, 64}, d_v = 64, K <= 64)."""
    import torch
    lib = load()
    _check_dev(K, V, mu, sigma2, log_pi)
    B, H, N, d_r = K.shape
    d_v = V.shape[-1]
    if V.shape[:3] != K.shape[:3]:
        raise ValueError("K must be [B, H, N, d_r] and V [B, H, N, d_v]")
    Kc = _params_check(H, d_r, mu, sigma2, log_pi)
    code = _dtype_code(K)
    if V.dtype != K.dtype:
        raise TypeError("K, V must share one dtype")
    Vt = torch.empty(B, H, Kc, d_v, dtype=torch.float32, device=K.device)
    Z = torch.empty(B, H, Kc, dtype=torch.float32, device=K.device)
    opt = options(path=path, splits=splits, sync_status=sync_status)
    nb = int(lib.gma_latent_memory_workspace_size(B, H, N, d_r, d_v, Kc, code, ctypes.byref(opt)))
    if nb == 0:
        raise GmaError(2, "gma_latent_memory")
    ws = _workspace(nb, K.device, workspace)
    st = lib.gma_latent_memory(_ptr(K), _ptr(V), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(Vt), _ptr(Z),
                               B, H, N, d_r, d_v, Kc, ctypes.byref(opt), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_latent_memory")
    return Vt, Z


def decode_step(q, k, v, mu, sigma2, log_pi, Vt, Z, eps=1e-6, out=None, workspace=None, stream=None,
                sync_status=False):
    """One causal position for every (b, h): q, k [B, H, d_r], v [B, H, d_v]; the
    carried state Vt [B, H, K, d_v], Z [B, H, K] (fp32) is updated in place.
    Returns o [B, H, d_v] fp32."""
    import torch
    lib = load()
    _check_dev(q, k, v, mu, sigma2, log_pi, Vt, Z)
    B, H, d_r = q.shape
    d_v = v.shape[-1]
    Kc = _params_check(H, d_r, mu, sigma2, log_pi)
    if k.shape != q.shape or v.shape[:2] != q.shape[:2]:
        raise ValueError("q, k must be [B, H, d_r] and v [B, H, d_v]")
    if Vt.shape != (B, H, Kc, d_v) or Z.shape != (B, H, Kc) or Vt.dtype != torch.float32 \
            or Z.dtype != torch.float32:
        raise ValueError("Vt must be fp32 [B, H, K, d_v] and Z fp32 [B, H, K]")
    code = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        out = torch.empty(B, H, d_v, dtype=torch.float32, device=q.device)
    nb = int(lib.gma_decode_workspace_size(H, d_r, Kc))
    if nb == 0:
        raise GmaError(2, "gma_decode_step")
    ws = _workspace(nb, q.device, workspace)
    opt = options(sync_status=sync_status)
    st = lib.gma_decode_step(_ptr(q), _ptr(k), _ptr(v), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi), float(eps),
                             _ptr(Vt), _ptr(Z), _ptr(out), B, H, d_r, d_v, Kc, ctypes.byref(opt), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_decode_step")
    return out


def routing_stats(X, mu, sigma2, log_pi, want_z=True, workspace=None, stream=None, sync_status=False) -> dict:
    """Component-usage diagnostics per (b, h): usage [B, H, K] fp32 (sum of the
    responsibilities), counts [B, H, K] int32 (hard assignments), z [B, H, N] int32
    (if want_z), entropy [B, H] fp32 (usage entropy over log K), used [B, H]
    (non-empty counts, derived here from counts)."""
    import torch
    lib = load()
    _check_dev(X, mu, sigma2, log_pi)
    B, H, N, d_r = X.shape
    Kc = _params_check(H, d_r, mu, sigma2, log_pi)
    code = _dtype_code(X)
    dev = X.device
    usage = torch.empty(B, H, Kc, dtype=torch.float32, device=dev)
    counts = torch.empty(B, H, Kc, dtype=torch.int32, device=dev)
    z = torch.empty(B, H, N, dtype=torch.int32, device=dev) if want_z else None
    entropy = torch.empty(B, H, dtype=torch.float32, device=dev)
    nb = int(lib.gma_routing_stats_workspace_size(B, H, N, d_r, Kc, code))
    if nb == 0:
        raise GmaError(2, "gma_routing_stats")
    ws = _workspace(nb, dev, workspace)
    opt = options(sync_status=sync_status)
    st = lib.gma_routing_stats(_ptr(X), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(usage), _ptr(counts),
                               _ptr(z) if z is not None else None, _ptr(entropy), B, H, N, d_r, Kc,
                               ctypes.byref(opt), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_routing_stats")
    return {"usage": usage, "counts": counts, "z": z, "entropy": entropy, "used": (counts > 0).sum(-1)}


def read_memory(Q, mu, sigma2, log_pi, Vt, Z, eps=1e-6, out=None, workspace=None, stream=None, o_bf16=False,
                sync_status=False, path=PATH_AUTO):
    """O = Gamma^Q Vt / (Gamma^Q Z + eps) for Q [B, H, N, d_r] and a given latent
    memory Vt [B, H, K, d_v], Z [B, H, K] (fp32); O fp32 (or bf16)."""
    import torch
    lib = load()
    _check_dev(Q, mu, sigma2, log_pi, Vt, Z)
    B, H, N, d_r = Q.shape
    Kc = _params_check(H, d_r, mu, sigma2, log_pi)
    d_v = Vt.shape[-1]
    if Vt.shape != (B, H, Kc, d_v) or Z.shape != (B, H, Kc) or Vt.dtype != torch.float32 \
            or Z.dtype != torch.float32:
        raise ValueError("Vt must be fp32 [B, H, K, d_v] and Z fp32 [B, H, K]")
    code = _dtype_code(Q)
    odt = torch.bfloat16 if o_bf16 else torch.float32
    if out is None:
        out = torch.empty(B, H, N, d_v, dtype=odt, device=Q.device)
    nb = int(lib.gma_read_memory_workspace_size(B, H, N, d_r, d_v, Kc, code))
    if nb == 0:
        raise GmaError(2, "gma_read_memory")
    ws = _workspace(nb, Q.device, workspace)
    opt = options(path=path, sync_status=sync_status, o_bf16=o_bf16)
    st = lib.gma_read_memory(_ptr(Q), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi), float(eps), _ptr(Vt), _ptr(Z),
                             _ptr(out), B, H, N, d_r, d_v, Kc, ctypes.byref(opt), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_read_memory")
    return out


def forward_causal_carry(Q, K, V, mu, sigma2, log_pi, Vt_in=None, Z_in=None, eps=1e-6, want_state=True,
                         out=None, workspace=None, stream=None, o_bf16=False, sync_status=False, path=PATH_AUTO):
    """Causal forward whose prefix starts from (Vt_in, Z_in) (an empty prefix if
    None).  Returns (O, Vt_out, Z_out): the outputs and, if want_state, the
    prefix memory after the last position (else None, None)."""
    import torch
    lib = load()
    _check_dev(Q, K, V, mu, sigma2, log_pi)
    B, H, N, d_r = Q.shape
    d_v = V.shape[-1]
    Kc = _params_check(H, d_r, mu, sigma2, log_pi)
    if K.shape != Q.shape or V.shape[:3] != Q.shape[:3]:
        raise ValueError("Q, K must be [B, H, N, d_r] and V [B, H, N, d_v]")
    if (Vt_in is None) != (Z_in is None):
        raise ValueError("give both Vt_in and Z_in, or neither")
    if Vt_in is not None:
        _check_dev(Vt_in, Z_in)
        if Vt_in.shape != (B, H, Kc, d_v) or Z_in.shape != (B, H, Kc) or Vt_in.dtype != torch.float32 \
                or Z_in.dtype != torch.float32:
            raise ValueError("Vt_in must be fp32 [B, H, K, d_v] and Z_in fp32 [B, H, K]")
    code = _dtype_code(Q)
    if K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise TypeError("Q, K, V must share one dtype")
    dev = Q.device
    odt = torch.bfloat16 if o_bf16 else torch.float32
    if out is None:
        out = torch.empty(B, H, N, d_v, dtype=odt, device=dev)
    Vt_out = torch.empty(B, H, Kc, d_v, device=dev) if want_state else None
    Z_out = torch.empty(B, H, Kc, device=dev) if want_state else None
    nb = int(lib.gma_causal_carry_workspace_size(B, H, N, d_r, d_v, Kc, code))
    if nb == 0:
        raise GmaError(2, "gma_forward_causal_carry")
    ws = _workspace(nb, dev, workspace)
    opt = options(path=path, sync_status=sync_status, o_bf16=o_bf16)

    def p(t):
        return _ptr(t) if t is not None else None

    st = lib.gma_forward_causal_carry(_ptr(Q), _ptr(K), _ptr(V), code, _ptr(mu), _ptr(sigma2), _ptr(log_pi),
                                      float(eps), p(Vt_in), p(Z_in), p(Vt_out), p(Z_out), _ptr(out), B, H, N, d_r,
                                      d_v, Kc, ctypes.byref(opt), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_forward_causal_carry")
    return out, Vt_out, Z_out


def combine_memories(parts, count=None, out=None, stream=None):
    """Rank-order sum of latent memories (gma_combine_memories): ``parts`` is a
    [P, n] fp32 CUDA tensor, one row per sequence block in order; returns the
    [n] sum of rows 0..count-1 (count = P by default), summed in row order."""
    import torch
    _check_dev(parts)
    if parts.dim() != 2 or parts.dtype != torch.float32 or not parts.is_contiguous():
        raise ValueError("parts must be a contiguous fp32 [P, n] tensor")
    P, n = parts.shape
    count = P if count is None else int(count)
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=parts.device)
    st = load().gma_combine_memories(_ptr(parts), P, n, count, _ptr(out), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_combine_memories")
    return out


def reparameterize(omega, alpha, eps_sigma=1e-3, stream=None):
    """Eqs. (14)-(15): (sigma2 = softplus(omega) + eps_sigma, log_pi = log_softmax(alpha))
    for omega [H, K, d_r], alpha [H, K] fp32 CUDA tensors."""
    import torch
    _check_dev(omega, alpha)
    H, K, d_r = omega.shape
    if alpha.shape != (H, K) or omega.dtype != torch.float32 or alpha.dtype != torch.float32:
        raise ValueError("omega must be fp32 [H, K, d_r] and alpha fp32 [H, K]")
    sigma2, log_pi = torch.empty_like(omega), torch.empty_like(alpha)
    st = load().gma_reparameterize(_ptr(omega), _ptr(alpha), H, K, d_r, float(eps_sigma), _ptr(sigma2),
                                   _ptr(log_pi), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_reparameterize")
    return sigma2, log_pi


def reparameterize_backward(omega, alpha, dsigma2, dlog_pi, stream=None):
    """Chain rule through reparameterize: (domega, dalpha)."""
    import torch
    _check_dev(omega, alpha, dsigma2, dlog_pi)
    H, K, d_r = omega.shape
    if alpha.shape != (H, K) or dsigma2.shape != omega.shape or dlog_pi.shape != alpha.shape:
        raise ValueError("omega, dsigma2 must be [H, K, d_r] and alpha, dlog_pi [H, K]")
    domega, dalpha = torch.empty_like(omega), torch.empty_like(alpha)
    st = load().gma_reparameterize_backward(_ptr(omega), _ptr(alpha), _ptr(dsigma2), _ptr(dlog_pi), H, K, d_r,
                                            _ptr(domega), _ptr(dalpha), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_reparameterize_backward")
    return domega, dalpha


def project_qkv(X, W_q, W_k, W_v, H, out_dtype=None, workspace=None, stream=None, sync_status=False):
    """Eq. (4): Q_X, K_X, V_X [B, H, N, d] = X W^T split into heads, for X [B, N, D]
    and weights [H d, D] (bf16, one output feature per row); outputs bf16 by
    default (the forward's input type), or out_dtype=torch.float32."""
    import torch
    lib = load()
    _check_dev(X, W_q, W_k, W_v)
    if any(t.dtype != torch.bfloat16 for t in (X, W_q, W_k, W_v)):
        raise TypeError("X and the weights must be bfloat16")
    B, N, D = X.shape
    if W_q.shape[1] != D or W_k.shape != W_q.shape or W_v.shape[1] != D or W_q.shape[0] % H or W_v.shape[0] % H:
        raise ValueError("weights must be [H * d, D]")
    d_r, d_v = W_q.shape[0] // H, W_v.shape[0] // H
    odt = torch.bfloat16 if out_dtype is None else out_dtype
    code = GMA_BF16 if odt == torch.bfloat16 else GMA_F32
    Q = torch.empty(B, H, N, d_r, dtype=odt, device=X.device)
    K = torch.empty(B, H, N, d_r, dtype=odt, device=X.device)
    V = torch.empty(B, H, N, d_v, dtype=odt, device=X.device)
    ws = _workspace(int(lib.gma_project_workspace_size()), X.device, workspace)
    opt = options(sync_status=sync_status)
    st = lib.gma_project_qkv(_ptr(X), _ptr(W_q), _ptr(W_k), _ptr(W_v), _ptr(Q), _ptr(K), _ptr(V), code, B, N, D, H,
                             d_r, d_v, ctypes.byref(opt), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    if st != 0:
        raise GmaError(st, "gma_project_qkv")
    return Q, K, V
