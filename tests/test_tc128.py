"""The causal and bidirectional forwards on the 128-wide tensor-core kernels
(d_r = d_v = 128, K <= 128, bf16): element by element against the fp64 oracle
on sizes the oracle finishes in seconds -- several 128-token chunks and a
ragged tail, padded components, one token, one component -- under every
partition of the chunks over CTAs (jobs that cross a head boundary, CTAs with
several jobs), fp32 and bf16 O, bitwise reproducibility, parameter errors and a
forced timeout."""
import zlib

import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import TOL, normalised_error, normalised_error_bf16_out, oracle_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def _case(B, H, N, K, causal=True, **kw):
    return Case(f"tc128_{'c' if causal else 'b'}_B{B}_H{H}_N{N}_K{K}", causal, B, H, N, 128, 128, K, "bf16", **kw)


def _inputs(case, salt=0):
    return make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000 + salt)


def test_selected_path_is_tensor_core():
    assert gma.selected_path(32768, 128, 128, 128, "bf16", 1) == gma.PATH_TC
    assert gma.selected_path(32768, 128, 128, 100, "bf16", 1) == gma.PATH_TC
    assert gma.selected_path(32768, 128, 128, 128, "bf16", 0) == gma.PATH_TC
    assert gma.selected_path(32768, 128, 128, 128, "f32", 1) == gma.PATH_SIMT
    assert gma.selected_path(32768, 128, 128, 129, "bf16", 1) == -1              # K > 128: no kernel
    assert gma.selected_path(32768, 128, 128, 128, "bf16", 1, path=gma.PATH_TC_SINGLE_PASS) == -1


@pytest.mark.parametrize("B,H,N,K", [(2, 3, 260, 128), (1, 2, 700, 100), (1, 1, 1, 128), (2, 1, 129, 1),
                                     (1, 2, 513, 64)], ids=lambda v: str(v))
@pytest.mark.parametrize("o_bf16", [False, True], ids=["o32", "o16"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "bidir"])
def test_matches_oracle(B, H, N, K, o_bf16, causal):
    case = _case(B, H, N, K, causal)
    inp = _inputs(case)
    O = run_gpu(case, to_dev(inp), path=gma.PATH_TC, o_bf16=o_bf16)
    ref = oracle_full(case, inp)
    err = normalised_error_bf16_out(O, ref) if o_bf16 else normalised_error(O, ref)
    assert err <= TOL["bf16"], f"{case.name}: normalised max error {err:.3e}"


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "bidir"])
@pytest.mark.parametrize("splits", [1, 2, 3, 5, 11, 0])
def test_every_partition_matches_oracle(splits, causal):
    """Six heads of eight chunks (the last ragged) cut into `splits` contiguous
    ranges: jobs start and end inside heads, a CTA may hold parts of several
    heads, and each job's carried-in prefix comes from the aggregation's
    combine (causal) or the head's whole memory (bidirectional)."""
    case = _case(2, 3, 1000, 128, causal)
    inp = _inputs(case, 3)
    O = run_gpu(case, to_dev(inp), path=gma.PATH_TC, splits=splits)
    err = normalised_error(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], f"splits={splits}: {err:.3e}"


def test_long_head_matches_oracle_rows():
    """One long head (32 chunks over 13 CTAs): early, boundary and last rows
    against the oracle's rows."""
    import oracle
    case = _case(1, 1, 4096 + 77, 128)
    inp = _inputs(case, 5)
    O = run_gpu(case, to_dev(inp), path=gma.PATH_TC, splits=13).double().cpu().numpy()[0, 0]
    rows = np.array(sorted({0, 1, 127, 128, 129, 1000, 2047, 2048, 4095, 4096, case.N - 1}))
    ref = oracle.causal_rows(inp["Q"][0, 0], inp["K"][0, 0], inp["V"][0, 0], inp["mu"][0], inp["sigma2"][0],
                             inp["log_pi"][0], case.eps, rows)
    rms = float(np.sqrt(np.mean(oracle_full(_case(1, 1, 600, 128), _inputs(_case(1, 1, 600, 128), 5)) ** 2)))
    err = float(np.max(np.abs(O[rows] - ref))) / max(rms, float(np.sqrt(np.mean(ref ** 2))))
    assert err <= TOL["bf16"], err


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "bidir"])
def test_deterministic(causal):
    case = _case(2, 2, 900, 128, causal)
    d = to_dev(_inputs(case, 8))
    a = run_gpu(case, d, path=gma.PATH_TC, splits=5)
    b = run_gpu(case, d, path=gma.PATH_TC, splits=5)
    assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "bidir"])
@pytest.mark.parametrize("bad", ["zero_var", "nan_mu", "inf_logpi"])
def test_invalid_parameters_reported(bad, causal):
    case = _case(1, 2, 300, 128, causal)
    d = to_dev(_inputs(case, 9))
    if bad == "zero_var":
        d["sigma2"][1, 100, 127] = 0.0
    elif bad == "nan_mu":
        d["mu"][0, 3, 64] = float("nan")
    else:
        d["log_pi"][1, 127] = float("-inf")
    with pytest.raises(gma.GmaError) as e:
        run_gpu(case, d, path=gma.PATH_TC)
    assert e.value.status == 6
    d2 = to_dev(_inputs(case, 9))
    O = run_gpu(case, d2, path=gma.PATH_TC)
    assert normalised_error(O, oracle_full(case, _inputs(case, 9))) <= TOL["bf16"]


def test_forced_timeout_reports_status_and_recovers():
    """The test hook skips the first key-tile load of the aggregation: its
    waits give up after ~4 s, the call reports GMA_ERR_TIMEOUT with no sticky
    CUDA error, and the next call on the same stream is correct."""
    import ctypes
    from gaussian_mixture_latent_diag_gb300 import _native
    vp = ctypes.c_void_p
    lib = _native.load()
    case = _case(1, 2, 700, 128)
    inp = _inputs(case, 11)
    d = to_dev(inp)
    opt = _native.options(path=gma.PATH_TC, sync_status=True, test_stall=True)
    ws_bytes = gma.workspace_size(case.B, case.H, case.N, 128, 128, 128, "bf16", 1, path=gma.PATH_TC)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    O = torch.empty(case.B, case.H, case.N, 128, dtype=torch.float32, device="cuda")
    st = lib.gma_forward_causal(vp(d["Q"].data_ptr()), vp(d["K"].data_ptr()), vp(d["V"].data_ptr()),
                                _native.GMA_BF16, vp(d["mu"].data_ptr()), vp(d["sigma2"].data_ptr()),
                                vp(d["log_pi"].data_ptr()), float(case.eps), vp(O.data_ptr()), case.B, case.H,
                                case.N, 128, 128, 128, ctypes.byref(opt), vp(ws.data_ptr()), ws_bytes,
                                vp(torch.cuda.current_stream().cuda_stream))
    assert st == 5, _native.status_string(st)  # GMA_ERR_TIMEOUT
    torch.cuda.synchronize()
    O2 = run_gpu(case, d, path=gma.PATH_TC)
    assert normalised_error(O2, oracle_full(case, inp)) <= TOL["bf16"]
