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


@pytest.mark.parametrize("causal,path", [(False, gma.PATH_TC), (True, gma.PATH_TC), (True, gma.PATH_TC_SINGLE_PASS)],
                         ids=["bidir", "causal", "causal1pass"])
def test_forced_timeout_reports_status_and_recovers(causal, path):
    lib = _native.load()
    case = Case("stall", causal, 1, 2, 512, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=21)
    d = to_dev(inp)
    assert gma.selected_path(case.N, 64, 64, 64, "bf16", int(causal), path=path) == path
    opt = _native.options(path=path, sync_status=True, test_stall=True)
    ws_bytes = gma.workspace_size(case.B, case.H, case.N, 64, 64, 64, "bf16", int(causal), path=path)
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
    O2 = run_gpu(case, d, path=path)
    assert normalised_error(O2, oracle_full(case, inp)) <= TOL["bf16"]


def test_projection_forced_timeout_reports_status_and_recovers():
    """The projection GEMM's bounded waits: with test_stall its first stage is
    never loaded, so the MMA issuer gives up after 4 s; the call reports
    GMA_ERR_TIMEOUT and a normal call right after is correct."""
    import numpy as np
    import oracle
    lib = _native.load()
    B, N, D, H, dh = 1, 300, 256, 2, 64
    g = torch.Generator().manual_seed(3)
    X = torch.randn(B, N, D, generator=g).to(torch.bfloat16).cuda()
    Ws = [(torch.randn(H * dh, D, generator=g) / 16).to(torch.bfloat16).cuda() for _ in range(3)]
    outs = [torch.empty(B, H, N, dh, dtype=torch.float32, device="cuda") for _ in range(3)]
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    opt = _native.options(sync_status=True, test_stall=True)
    st = lib.gma_project_qkv(*(vp(t.data_ptr()) for t in [X] + Ws + outs), _native.GMA_F32, B, N, D, H, dh, dh,
                             ctypes.byref(opt), vp(ws.data_ptr()), 256, vp(torch.cuda.current_stream().cuda_stream))
    assert st == GMA_ERR_TIMEOUT, _native.status_string(st)
    torch.cuda.synchronize()
    Q, K, V = gma.project_qkv(X, *Ws, H, out_dtype=torch.float32, sync_status=True)
    ref = oracle.project_qkv(X.cpu(), *(w.cpu() for w in Ws), H)
    assert np.max(np.abs(Q.double().cpu().numpy() - ref[0])) < 1e-3
