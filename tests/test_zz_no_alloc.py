"""gma_forward_bidir_noalloc: the bidirectional forward for callers that
cannot allocate device memory (its scratch is a fixed device array inside
libgma.so).  Called through the C ABI and checked against the fp64 oracle and
against gma_forward_bidir, on two different inputs in a row, so that a result
that depended on what the previous call left in the shared array would show;
then in three CUDA contexts in a row (a child process), so that a stale device
address of the array would show.

This file is collected last on purpose; it must also pass on its own in a
fresh process."""
import ctypes
import json
import os
import subprocess
import sys

import pytest
import torch

from gaussian_mixture_latent_diag_gb300 import _native
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import TOL, normalised_error, oracle_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu

vp = ctypes.c_void_p
HERE = os.path.dirname(os.path.abspath(__file__))


def _noalloc(lib, case, d, O, o_bf16=False):
    opt = _native.options(sync_status=True, o_bf16=o_bf16)
    code = _native.GMA_F32 if case.dtype == "f32" else _native.GMA_BF16
    return lib.gma_forward_bidir_noalloc(
        vp(d["Q"].data_ptr()), vp(d["K"].data_ptr()), vp(d["V"].data_ptr()), code,
        vp(d["mu"].data_ptr()), vp(d["sigma2"].data_ptr()), vp(d["log_pi"].data_ptr()),
        float(case.eps), vp(O.data_ptr()), case.B, case.H, case.N, case.d_r, case.d_v, case.K,
        ctypes.byref(opt), vp(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_oracle_and_bidir_twice(dtype):
    lib = _native.load()
    case = Case("noalloc", False, 1, 2, 1000, 64, 64, 64, dtype)
    for seed in (11, 12):  # two calls in a row on different inputs
        inp = make_inputs(case, seed=seed)
        d = to_dev(inp)
        O = torch.full((case.B, case.H, case.N, case.d_v), float("nan"), dtype=torch.float32,
                       device="cuda")
        st = _noalloc(lib, case, d, O)
        assert st == 0, _native.status_string(st)
        torch.cuda.synchronize()
        ref_oracle = oracle_full(case, inp)
        err = normalised_error(O, ref_oracle)
        assert err <= TOL[dtype], f"seed {seed}: {err:.3e} against the oracle"
        ref = run_gpu(case, d)  # the existing entry point, caller-provided workspace
        err = normalised_error(O, ref.double().cpu().numpy())
        assert err <= TOL[dtype], f"seed {seed}: {err:.3e} against gma_forward_bidir"


def test_noalloc_does_not_allocate():
    lib = _native.load()
    case = Case("noalloc", False, 1, 2, 777, 32, 64, 32, "bf16")
    d = to_dev(make_inputs(case, seed=13))
    O = torch.empty(case.B, case.H, case.N, case.d_v, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, case, d, O) == 0  # first call in this context: the device code is loaded
    torch.cuda.synchronize()
    # The device's free memory is a whole-device reading: another process may
    # allocate between two readings, so one of a few tries must show no change.
    changes = []
    for _ in range(5):
        free_before, _ = torch.cuda.mem_get_info()
        for _ in range(3):
            assert _noalloc(lib, case, d, O) == 0
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        changes.append(free_before - free_after)
        if changes[-1] == 0:
            break
    assert 0 in changes, f"device free memory changed by {changes} bytes"


def test_noalloc_rejects_oversized_problem():
    lib = _native.load()
    case = Case("noalloc_big", False, 64, 64, 65536, 64, 64, 64, "bf16")
    opt = _native.options()
    need = lib.gma_workspace_size(case.B, case.H, case.N, case.d_r, case.d_v, case.K,
                                  _native.GMA_BF16, 0, ctypes.byref(opt))
    limit = 16 << 20
    assert need > limit
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    p = vp(dummy.data_ptr())
    st = lib.gma_forward_bidir_noalloc(p, p, p, _native.GMA_BF16, p, p, p, 1e-6, p, case.B,
                                       case.H, case.N, case.d_r, case.d_v, case.K, None, None)
    assert st == 3  # GMA_ERR_WORKSPACE_TOO_SMALL, nothing launched


def test_noalloc_in_three_contexts():
    """Primary context, a second context on the same device, the primary again:
    every call finds the array in the context current at the call."""
    r = subprocess.run([sys.executable, os.path.join(HERE, "noalloc_contexts.py")],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    calls = json.loads(r.stdout.strip().splitlines()[-1])["calls"]
    assert len(calls) == 3
    for i, c in enumerate(calls):
        assert c["status"] == 0 and c["status_ref"] == 0, (i, c)
        assert c["err"] <= TOL["bf16"], (i, c)
        assert c["same_as_bidir"], (i, c)
