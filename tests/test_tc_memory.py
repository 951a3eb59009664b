"""GPU vs fp64 oracle for the latent-memory calls on the tensor-core kernels
(GMA_PATH_TC: bf16 inputs, d_r in {32, 64}, d_v = 64, K <= 64):

* gma_latent_memory -- Vt = Gamma^K^T V and Z = Gamma^K^T 1 ("Gaussian Mixture
  Attention", Eqs. (5)-(6)) from the write kernel's per-head combine;
* gma_read_memory -- Eq. (7) from a caller's memory, packed into the read
  kernel's bf16 hi | lo operand;
* gma_forward_causal_carry -- Eq. (8) with the prefix started at a carried-in
  memory, and the prefix after the last position returned.

Bound: the stated 1e-2 on max |x - x_ref| / RMS(x_ref).  Where the two
families must agree exactly it is checked bitwise: the memory a tensor-core
latent_memory returns, read back by the tensor-core read_memory, gives the
tensor-core bidirectional forward's O bit for bit (same job partition, same
fp32 sums, same operand image), and an empty carried-in prefix gives the
tensor-core causal forward's O bit for bit."""
import zlib

import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import TOL, normalised_error_bf16_out, to_dev

pytestmark = pytest.mark.gpu

TC = gma.PATH_TC


def _rel(gpu, ref) -> float:
    g = gpu.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(g - ref)) / np.sqrt(np.mean(ref ** 2)))


SHAPES = [  # (B, H, N, d_r, d_v, K): one tile, ragged tails, heads spanning several CTAs, many heads per CTA
    (1, 1, 1, 64, 64, 64),
    (2, 3, 300, 64, 64, 64),
    (1, 2, 517, 32, 64, 17),
    (1, 1, 20000, 64, 64, 64),
    (4, 40, 130, 64, 64, 1),
]
IDS = ["B%d_H%d_N%d_r%d_v%d_K%d" % s for s in SHAPES]


def _case(shape, causal):
    B, H, N, d_r, d_v, K = shape
    return Case(f"tcmem_{int(causal)}_{B}_{H}_{N}_{d_r}_{K}", causal, B, H, N, d_r, d_v, K, "bf16")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_tc_latent_memory_matches_oracle(shape):
    import oracle
    case = _case(shape, False)
    assert gma.selected_path(case.N, case.d_r, case.d_v, case.K, "bf16", 0) == TC
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000)
    d = to_dev(inp)
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    Vt, Z = gma.latent_memory(d["K"], d["V"], *prm, path=TC, sync_status=True)
    Vt_ref, Z_ref = oracle.latent_memory(inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"])
    ev, ez = _rel(Vt, Vt_ref), _rel(Z, Z_ref)
    print(f"{case.name}: Vt {ev:.2e} Z {ez:.2e}")
    assert ev <= TOL["bf16"] and ez <= TOL["bf16"], (ev, ez)
    # the CUDA-core family gives the same memory to the same bound
    Vs, Zs = gma.latent_memory(d["K"], d["V"], *prm, path=gma.PATH_SIMT, sync_status=True)
    assert _rel(Vt, Vs.double().cpu().numpy()) <= TOL["bf16"]
    # reading it back is the tensor-core bidirectional forward, bit for bit
    O = gma.read_memory(d["Q"], *prm, Vt, Z, eps=case.eps, path=TC, sync_status=True)
    Of = gma.forward_bidir(d["Q"], d["K"], d["V"], *prm, eps=case.eps, path=TC, sync_status=True)
    assert torch.equal(O, Of)


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_tc_read_memory_matches_oracle(shape):
    import oracle
    case = _case(shape, False)
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000 + 5)
    d = to_dev(inp)
    g = torch.Generator().manual_seed(7)
    B, H, N, d_r, d_v, K = shape
    Vt = (torch.randn(B, H, K, d_v, generator=g, dtype=torch.float64) * 20).float()
    Z = (torch.rand(B, H, K, generator=g, dtype=torch.float64) * 40).float()
    O = gma.read_memory(d["Q"], d["mu"], d["sigma2"], d["log_pi"], Vt.cuda(), Z.cuda(), eps=case.eps, path=TC,
                        sync_status=True)
    ref = oracle.read_memory(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps, Vt, Z)
    err = _rel(O, ref)
    print(f"{case.name}: O {err:.2e}")
    assert err <= TOL["bf16"], err
    # bf16 output: the same bound beyond one bf16 unit of the exact value
    Ob = gma.read_memory(d["Q"], d["mu"], d["sigma2"], d["log_pi"], Vt.cuda(), Z.cuda(), eps=case.eps, path=TC,
                         o_bf16=True, sync_status=True)
    assert normalised_error_bf16_out(Ob, ref) <= TOL["bf16"]


@pytest.mark.parametrize("TC", [gma.PATH_TC, gma.PATH_TC_SINGLE_PASS], ids=["tc", "tc1pass"])
@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_tc_causal_carry_continues_a_prefix(shape, TC):
    """The first N0 positions from an empty prefix, the rest from the returned
    state, both on the tensor cores (either causal kernel): the two blocks equal
    the oracle's causal rows, the final state the oracle's latent memory."""
    import oracle
    case = _case(shape, True)
    assert gma.selected_path(case.N, case.d_r, case.d_v, case.K, "bf16", 1, path=TC) == TC
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000 + 1)
    d = to_dev(inp)
    N = shape[2]
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    ref = oracle.forward_causal(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps)
    Vt_ref, Z_ref = oracle.latent_memory(inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"])
    if N > 1:
        N0 = N // 3 + 1
        blk = lambda a, b: [d[n][:, :, a:b].contiguous() for n in ("Q", "K", "V")]  # noqa: E731
        O1, vt, z = gma.forward_causal_carry(*blk(0, N0), *prm, eps=case.eps, path=TC, sync_status=True)
        O2, vt2, z2 = gma.forward_causal_carry(*blk(N0, N), *prm, Vt_in=vt, Z_in=z, eps=case.eps, path=TC,
                                               sync_status=True)
        eo, ev, ez = _rel(torch.cat([O1, O2], dim=2), ref), _rel(vt2, Vt_ref), _rel(z2, Z_ref)
        print(f"{case.name}: O {eo:.2e} Vt {ev:.2e} Z {ez:.2e}")
        assert eo <= TOL["bf16"] and ev <= TOL["bf16"] and ez <= TOL["bf16"], (eo, ev, ez)
    # an empty carried-in prefix is the tensor-core causal forward, bit for bit
    O0, vt0, z0 = gma.forward_causal_carry(d["Q"], d["K"], d["V"], *prm, eps=case.eps, path=TC, sync_status=True)
    Of = gma.forward_causal(d["Q"], d["K"], d["V"], *prm, eps=case.eps, path=TC, sync_status=True)
    assert torch.equal(O0, Of)
    assert _rel(vt0, Vt_ref) <= TOL["bf16"] and _rel(z0, Z_ref) <= TOL["bf16"]


@pytest.mark.parametrize("P", [2, 5])
def test_tc_sharded_over_n_emulated_on_one_gpu(P):
    """Sequence sharding over N through sharded.CudaOps, which runs bf16
    d = K = 64 on the tensor cores: P uneven shards one after the other, their
    memories combined in shard order, against the unsharded oracle forward."""
    import oracle
    from gaussian_mixture_latent_diag_gb300 import sharded
    case = Case("tc_shard_gpu", True, 2, 2, 3000, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=23)
    d = to_dev(inp)
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    ops = sharded.CudaOps()
    assert ops._path(d["K"], d["V"], d["mu"]) == TC and ops._path(d["K"], d["V"], d["mu"], causal=1) == TC
    cuts = np.linspace(0, case.N, P + 1).astype(int)
    cuts[1] += 129  # uneven shards with ragged tails
    blocks = [[d[n][:, :, a:b].contiguous() for n in ("Q", "K", "V")] for a, b in zip(cuts[:-1], cuts[1:])]
    parts = [ops.latent_memory(k, v, *prm) for _, k, v in blocks]
    Vt, Z = sharded.combine_total(parts, ops)
    Ob = torch.cat([ops.read_memory(q, *prm, Vt, Z, case.eps) for q, _, _ in blocks], dim=2)
    Oc = torch.cat([ops.forward_causal_carry(q, k, v, *prm, *sharded.combine_exclusive(parts, r, ops), case.eps)
                    for r, (q, k, v) in enumerate(blocks)], dim=2)
    args = (inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps)
    eb, ec = _rel(Ob, oracle.forward_bidir(*args)), _rel(Oc, oracle.forward_causal(*args))
    print(f"P={P}: bidir {eb:.2e} causal {ec:.2e}")
    assert eb <= TOL["bf16"] and ec <= TOL["bf16"], (eb, ec)


def test_tc_memory_paths_reject_unsupported_sizes():
    """GMA_PATH_TC on sizes the tensor-core kernels do not take is refused with
    GMA_ERR_UNSUPPORTED_SHAPE (no silent switch to the other family)."""
    case = Case("tcmem_unsupported", False, 1, 1, 64, 64, 32, 8, "bf16")
    d = to_dev(make_inputs(case, seed=0))
    with pytest.raises(gma.GmaError):
        gma.latent_memory(d["K"], d["V"], d["mu"], d["sigma2"], d["log_pi"], path=TC)
    f = {k: (v.float() if k in ("Q", "K", "V") else v) for k, v in d.items()}
    with pytest.raises(gma.GmaError):
        gma.forward_causal_carry(f["Q"], f["K"], f["V"], f["mu"], f["sigma2"], f["log_pi"], path=TC)


def test_tc_memory_paths_report_invalid_parameters():
    """A non-positive sigma2 in one head: each of the three tensor-core calls
    reports GMA_ERR_NONFINITE_PARAM (the read from a memory, whose first kernel
    after the coefficient prep is the pack of the caller's memory, included),
    and a valid call on the same workspace afterwards matches a fresh one."""
    case = Case("tcmem_bad", True, 1, 2, 300, 64, 64, 64, "bf16")
    d = to_dev(make_inputs(case, seed=3))
    good = d["sigma2"].clone()
    bad = good.clone()
    bad[1, 5, 7] = -1.0
    prm_bad = (d["mu"], bad, d["log_pi"])
    prm = (d["mu"], good, d["log_pi"])
    Vt, Z = gma.latent_memory(d["K"], d["V"], *prm, path=TC, sync_status=True)
    import ctypes
    lib, shape = gma.load(), (1, 2, 300, 64, 64, 64, gma.GMA_BF16)
    nb = max(int(lib.gma_latent_memory_workspace_size(*shape, ctypes.byref(gma.options(path=TC)))),
             int(lib.gma_read_memory_workspace_size(*shape)), int(lib.gma_causal_carry_workspace_size(*shape)))
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    calls = [
        lambda p: gma.latent_memory(d["K"], d["V"], *p, path=TC, workspace=ws, sync_status=True),
        lambda p: gma.read_memory(d["Q"], *p, Vt, Z, eps=case.eps, path=TC, workspace=ws, sync_status=True),
        lambda p: gma.forward_causal_carry(d["Q"], d["K"], d["V"], *p, Vt, Z, eps=case.eps, path=TC, workspace=ws,
                                           sync_status=True),
    ]
    for call in calls:
        with pytest.raises(gma.GmaError) as e:
            call(prm_bad)
        assert e.value.status == 6
        first = call(prm)
        again = call(prm)
        for a, b in zip(first if isinstance(first, tuple) else (first,), again if isinstance(again, tuple) else (again,)):
            assert torch.equal(a, b)
