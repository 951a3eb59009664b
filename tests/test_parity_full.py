"""GPU vs fp64 oracle on the five workloads at their full sizes, in the
launch configuration the benchmark times (default path and options).

The small fp32 workload is compared element by element.  For the large ones
the oracle computes sampled rows of a few heads one by one (all of the
latent memory / the whole prefix up to the row, exactly as defined), and the
GPU rows are compared element by element; the error is normalised by the RMS
of the GPU output over the whole tensor, and that RMS is checked against the
RMS of the oracle's sampled rows."""
import numpy as np
import pytest
import torch

from gaussian_mixture_latent_diag_gb300.synthetic import WORKLOADS, make_inputs
from gpu_helpers import TOL, normalised_error, oracle_full, run_gpu, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_rows(N, causal, rng):
    fixed = [0, 1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 127, 128, 129, 255, 256, N // 2, N - 2, N - 1]
    extra = rng.choice(N, size=24, replace=False).tolist()
    return np.unique(np.clip(np.array(fixed + extra), 0, N - 1))


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_full_size(name):
    import oracle
    case = WORKLOADS[name]
    inp = make_inputs(case, seed=0)
    O = run_gpu(case, to_dev(inp))
    if case.token_heads * case.d_v <= 1 << 16:
        err = normalised_error(O, oracle_full(case, inp))
        assert err <= TOL[case.dtype], f"{name}: {err:.3e}"
        return
    rms_gpu = float(O.float().pow(2).mean().sqrt())
    rng = np.random.default_rng(0)
    BH = case.B * case.H
    heads = sorted({0, BH - 1, int(rng.integers(BH))})
    worst = 0.0
    ref_sq, n_ref = 0.0, 0
    fn = oracle.causal_rows if case.causal else oracle.bidir_rows
    for bh in heads:
        b, h = divmod(bh, case.H)
        rows = _sample_rows(case.N, case.causal, rng)
        ref = fn(inp["Q"][b, h], inp["K"][b, h], inp["V"][b, h], inp["mu"][h], inp["sigma2"][h],
                 inp["log_pi"][h], case.eps, rows)
        got = O[b, h][torch.as_tensor(rows, device=O.device)].double().cpu().numpy()
        worst = max(worst, float(np.max(np.abs(got - ref))) / rms_gpu)
        if not case.causal:  # bidirectional rows are exchangeable: their RMS estimates the tensor's
            ref_sq += float((ref ** 2).sum()); n_ref += ref.size
    assert worst <= TOL[case.dtype], f"{name}: normalised max error {worst:.3e}"
    if n_ref:
        assert abs(np.sqrt(ref_sq / n_ref) / rms_gpu - 1.0) < 0.25
