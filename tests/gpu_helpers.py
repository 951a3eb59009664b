"""Helpers for the GPU parity tests: run the CUDA path through the C ABI
(via the Python binding) and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

# Tolerances on max |O - O_ref| / RMS(O_ref): 1e-4 for fp32 inputs, 1e-2 for
# bf16 inputs with fp32 accumulation.  Gamma rows must sum to 1 within 1e-5.
TOL = {"f32": 1e-4, "bf16": 1e-2}
ROWSUM_TOL = 1e-5


def to_dev(inp: dict, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_gpu(case: Case, dinp: dict, path=gma.PATH_AUTO, splits=0, o_bf16=False):
    fn = gma.forward_causal if case.causal else gma.forward_bidir
    O = fn(dinp["Q"], dinp["K"], dinp["V"], dinp["mu"], dinp["sigma2"], dinp["log_pi"],
           eps=case.eps, path=path, splits=splits, sync_status=True, o_bf16=o_bf16)
    torch.cuda.synchronize()
    return O


def oracle_full(case: Case, inp: dict) -> np.ndarray:
    import oracle
    fn = oracle.forward_causal if case.causal else oracle.forward_bidir
    return fn(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps)


def normalised_error(O_gpu, O_ref: np.ndarray, rms: float | None = None) -> float:
    g = O_gpu.detach().to("cpu", torch.float64).numpy()
    if rms is None:
        rms = float(np.sqrt(np.mean(O_ref ** 2)))
    return float(np.max(np.abs(g - O_ref)) / rms)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    m, e = np.frexp(np.abs(x))          # |x| = m 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 8)


def normalised_error_bf16_out(O_gpu, O_ref: np.ndarray) -> float:
    """As normalised_error for a bf16-rounded O: each element may also differ
    from the exact value by one bf16 ulp (the output rounding, which alone
    exceeds 1e-2 * RMS on heavy-tailed rows)."""
    g = O_gpu.detach().to("cpu", torch.float64).numpy()
    rms = float(np.sqrt(np.mean(O_ref ** 2)))
    excess = np.maximum(np.abs(g - O_ref) - bf16_ulp(O_ref), 0.0)
    return float(np.max(excess) / rms)
