"""GPU vs fp64 oracle, element by element, on sizes the oracle finishes in
seconds: several 128-row tiles plus a ragged tail, every supported width,
both kernel families, fp32 and bf16, bidirectional and causal, and the
degenerate cases (N = 1, K = 1, identical components, peaked routing)."""
import zlib

import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import (TOL, ROWSUM_TOL, normalised_error, normalised_error_bf16_out,
                         oracle_full, run_gpu, to_dev)

pytestmark = pytest.mark.gpu

SHAPES = [  # (N, d_r, d_v, K)
    (300, 16, 32, 8),
    (300, 64, 64, 64),
    (417, 32, 64, 32),
    (260, 128, 128, 128),
    (129, 16, 128, 1),
    (1, 64, 64, 64),
    (200, 128, 16, 100),
]


def _case(causal, N, d_r, d_v, K, dtype, **kw):
    name = f"{'causal' if causal else 'bidir'}_{dtype}_N{N}_r{d_r}_v{d_v}_K{K}"
    return Case(name, causal, 2, 3, N, d_r, d_v, K, dtype, **kw)


@pytest.mark.parametrize("path", [gma.PATH_SIMT, gma.PATH_AUTO], ids=["simt", "auto"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "N%d_r%d_v%d_K%d" % s)
def test_forward_matches_oracle(shape, causal, dtype, path):
    case = _case(causal, *shape, dtype)
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000)
    O = run_gpu(case, to_dev(inp), path=path)
    ref = oracle_full(case, inp)
    err = normalised_error(O, ref)
    assert err <= TOL[dtype], f"{case.name}: normalised max error {err:.3e}"


@pytest.mark.parametrize("path", [gma.PATH_SIMT, gma.PATH_AUTO], ids=["simt", "auto"])
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_bf16_output(causal, path):
    """O requested in bf16: the fp32 result rounded to nearest even; same
    tolerance plus one bf16 ulp of the exact value per element."""
    case = _case(causal, 300, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=3)
    O = run_gpu(case, to_dev(inp), path=path, o_bf16=True)
    assert O.dtype == torch.bfloat16
    err = normalised_error_bf16_out(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], err


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_peaked_mixture_routing(causal):
    """Rows drawn from the mixture with well-separated means: near one-hot
    responsibilities (softmax underflow stress)."""
    case = Case("peaked", causal, 2, 2, 333, 32, 64, 32, "bf16", routing="mixture", mu_std=3.0)
    inp = make_inputs(case, seed=5)
    err = normalised_error(run_gpu(case, to_dev(inp)), oracle_full(case, inp))
    assert err <= TOL["bf16"], err


@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_identical_components(causal):
    case = Case("ident", causal, 1, 2, 190, 64, 64, 16, "f32")
    inp = make_inputs(case, seed=6)
    inp["mu"][:] = inp["mu"][:, :1]
    inp["sigma2"][:] = inp["sigma2"][:, :1]
    err = normalised_error(run_gpu(case, to_dev(inp)), oracle_full(case, inp))
    assert err <= TOL["f32"], err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_responsibilities(dtype):
    import oracle
    case = Case("resp", False, 2, 3, 300, 64, 16, 48, dtype)
    inp = make_inputs(case, seed=7)
    d = to_dev(inp)
    G = gma.responsibilities(d["Q"], d["mu"], d["sigma2"], d["log_pi"], sync_status=True)
    G = G.double().cpu().numpy()
    ref = oracle.responsibilities(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"])
    assert np.max(np.abs(G.sum(-1) - 1.0)) <= ROWSUM_TOL
    assert G.min() >= 0.0
    assert np.max(np.abs(G - ref)) <= 1e-4


@pytest.mark.parametrize("causal,path", [(False, gma.PATH_AUTO), (True, gma.PATH_AUTO),
                                         (True, gma.PATH_TC_SINGLE_PASS)], ids=["bidir", "causal", "causal1pass"])
def test_deterministic(causal, path):
    case = _case(causal, 700, 64, 64, 64, "bf16")
    d = to_dev(make_inputs(case, seed=8))
    a = run_gpu(case, d, path=path)
    b = run_gpu(case, d, path=path)
    assert torch.equal(a, b)


@pytest.mark.parametrize("shape", [(300, 64, 64, 64), (417, 32, 64, 32), (1, 64, 64, 64), (129, 64, 64, 17)],
                         ids=lambda s: "N%d_r%d_v%d_K%d" % s)
@pytest.mark.parametrize("o_bf16", [False, True], ids=["o32", "o16"])
def test_causal_single_pass_matches_oracle(shape, o_bf16):
    """The single-pass causal kernel (key responsibilities kept on chip, block
    look-back between chunks) against the oracle, ragged tails and padded
    components, fp32 and bf16 O."""
    case = _case(True, *shape, "bf16")
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000 + 7)
    O = run_gpu(case, to_dev(inp), path=gma.PATH_TC_SINGLE_PASS, o_bf16=o_bf16)
    ref = oracle_full(case, inp)
    err = normalised_error_bf16_out(O, ref) if o_bf16 else normalised_error(O, ref)
    assert err <= TOL["bf16"], f"{case.name}: normalised max error {err:.3e}"


@pytest.mark.parametrize("bad", ["zero_var", "neg_var", "nan_mu", "inf_logpi"])
def test_invalid_parameters_reported(bad):
    case = _case(False, 64, 16, 16, 4, "f32")
    d = to_dev(make_inputs(case, seed=9))
    if bad == "zero_var":
        d["sigma2"][1, 2, 3] = 0.0
    elif bad == "neg_var":
        d["sigma2"][0, 0, 0] = -1.0
    elif bad == "nan_mu":
        d["mu"][2, 1, 0] = float("nan")
    else:
        d["log_pi"][0, 3] = float("-inf")
    with pytest.raises(gma.GmaError) as e:
        run_gpu(case, d)
    assert e.value.status == 6
    # a clean call on the same workspace afterwards succeeds
    d2 = to_dev(make_inputs(case, seed=9))
    run_gpu(case, d2)


@pytest.mark.parametrize("path,chunk", [(gma.PATH_SIMT, 64), (gma.PATH_TC, 128), (gma.PATH_TC_SINGLE_PASS, 128)],
                         ids=["simt64", "tc128", "tc1pass128"])
def test_causal_each_supported_chunk(path, chunk):
    """options.chunk set to the kernel family's chunk length (the only one
    each family runs; other lengths are rejected on the host): the same
    result as the oracle, with ragged last chunks."""
    case = _case(True, 3 * chunk + 37, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=10)
    O = gma.forward_causal(*(to_dev(inp)[k] for k in ("Q", "K", "V", "mu", "sigma2", "log_pi")),
                           eps=case.eps, path=path, chunk=chunk, sync_status=True)
    torch.cuda.synchronize()
    err = normalised_error(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], err
    other = 256 if chunk == 128 else 128
    with pytest.raises(gma.GmaError) as e:
        gma.forward_causal(*(to_dev(inp)[k] for k in ("Q", "K", "V", "mu", "sigma2", "log_pi")),
                           eps=case.eps, path=path, chunk=other)
    assert e.value.status == 2
