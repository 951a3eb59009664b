"""Failure path of the bounded device waits: with the test hook
gma_options.test_stall the tensor-core key pass never loads its first key
tile, so the first wait on it runs out (4 s).  The call must report
GMA_ERR_TIMEOUT through the status word instead of hanging, and the stream
must stay usable: a normal call right after it matches the oracle.  No GPU
fault is involved -- every kernel returns after recording the status."""
import ctypes

import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300 import _native
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import TOL, normalised_error, oracle_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu

GMA_ERR_TIMEOUT = 5
vp = ctypes.c_void_p


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_forced_timeout_reports_status_and_recovers(causal):
    lib = _native.load()
    case = Case("stall", causal, 1, 2, 512, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=21)
    d = to_dev(inp)
    assert gma.selected_path(case.N, 64, 64, 64, "bf16", int(causal)) == gma.PATH_TC
    opt = _native.options(sync_status=True, test_stall=True)
    ws_bytes = gma.workspace_size(case.B, case.H, case.N, 64, 64, 64, "bf16", int(causal))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    O = torch.empty(case.B, case.H, case.N, 64, dtype=torch.float32, device="cuda")
    fn = lib.gma_forward_causal if causal else lib.gma_forward_bidir
    st = fn(vp(d["Q"].data_ptr()), vp(d["K"].data_ptr()), vp(d["V"].data_ptr()), _native.GMA_BF16,
            vp(d["mu"].data_ptr()), vp(d["sigma2"].data_ptr()), vp(d["log_pi"].data_ptr()), float(case.eps),
            vp(O.data_ptr()), case.B, case.H, case.N, 64, 64, 64, ctypes.byref(opt), vp(ws.data_ptr()),
            ws_bytes, vp(torch.cuda.current_stream().cuda_stream))
    assert st == GMA_ERR_TIMEOUT, _native.status_string(st)
    torch.cuda.synchronize()  # no sticky CUDA error
    # the stream still works: a normal call right after matches the oracle
    O2 = run_gpu(case, d)
    assert normalised_error(O2, oracle_full(case, inp)) <= TOL["bf16"]
