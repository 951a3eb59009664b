"""GPU vs fp64 oracle for the two entry points that split the forward at the
latent memory -- gma_read_memory (Eq. 7 from a given memory) and
gma_forward_causal_carry (causal forward from a carried-in prefix, returning
the prefix after its last position) -- and for sequence sharding over N
emulated on one GPU: P shards run one after the other through the CUDA path,
their memories combined in shard order by the functions the multi-rank path
uses, against the unsharded oracle forward."""
import zlib

import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300 import sharded
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-4  # fp32 arithmetic on exact inputs, max |x - x_ref| / RMS(x_ref)


def _rel(gpu, ref) -> float:
    g = gpu.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(g - ref)) / np.sqrt(np.mean(ref ** 2)))


SHAPES = [  # (B, H, N, d_r, d_v, K)
    (2, 3, 300, 16, 32, 8),
    (1, 2, 517, 64, 64, 64),
    (1, 1, 200, 128, 128, 128),
    (2, 1, 70, 32, 16, 1),
]


def _case(shape, dtype):
    B, H, N, d_r, d_v, K = shape
    return Case(f"carry_{dtype}_{B}_{H}_{N}_{d_r}_{d_v}_{K}", True, B, H, N, d_r, d_v, K, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_H%d_N%d_r%d_v%d_K%d" % s)
def test_read_memory_matches_oracle(shape, dtype):
    import oracle
    case = _case(shape, dtype)
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000)
    d = to_dev(inp)
    g = torch.Generator().manual_seed(3)
    B, H, N, d_r, d_v, K = shape
    Vt = torch.randn(B, H, K, d_v, generator=g, dtype=torch.float64) * 20
    Z = torch.rand(B, H, K, generator=g, dtype=torch.float64) * 40
    Vt32, Z32 = Vt.float(), Z.float()
    O = gma.read_memory(d["Q"], d["mu"], d["sigma2"], d["log_pi"], Vt32.cuda(), Z32.cuda(), eps=case.eps,
                        sync_status=True)
    ref = oracle.read_memory(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps, Vt32, Z32)
    assert _rel(O, ref) <= TOL


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_H%d_N%d_r%d_v%d_K%d" % s)
def test_causal_carry_continues_a_prefix(shape, dtype):
    """The first N0 positions through gma_forward_causal_carry from an empty
    prefix, the rest from the returned state: both blocks equal the oracle's
    causal rows and the final state equals the oracle's latent memory."""
    import oracle
    case = _case(shape, dtype)
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000 + 1)
    d = to_dev(inp)
    N = shape[2]
    N0 = N // 3 + 1
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    blk = lambda a, b: [d[n][:, :, a:b].contiguous() for n in ("Q", "K", "V")]  # noqa: E731
    O1, vt, z = gma.forward_causal_carry(*blk(0, N0), *prm, eps=case.eps, sync_status=True)
    O2, vt2, z2 = gma.forward_causal_carry(*blk(N0, N), *prm, Vt_in=vt, Z_in=z, eps=case.eps, sync_status=True)
    ref = oracle.forward_causal(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps)
    assert _rel(torch.cat([O1, O2], dim=2), ref) <= TOL
    Vt_ref, Z_ref = oracle.latent_memory(inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"])
    assert _rel(vt2, Vt_ref) <= TOL and _rel(z2, Z_ref) <= TOL
    # an empty carried-in prefix is the plain causal forward
    O0, _, _ = gma.forward_causal_carry(d["Q"], d["K"], d["V"], *prm, eps=case.eps, want_state=False,
                                        sync_status=True)
    Os = gma.forward_causal(d["Q"], d["K"], d["V"], *prm, eps=case.eps, path=gma.PATH_SIMT, sync_status=True)
    assert torch.equal(O0, Os)


@pytest.mark.parametrize("P", [2, 5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sharded_over_n_emulated_on_one_gpu(P, dtype):
    import oracle
    case = Case(f"shard_gpu_{dtype}", True, 2, 2, 700, 64, 64, 64, dtype)
    inp = make_inputs(case, seed=21)
    d = to_dev(inp)
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    cuts = np.linspace(0, case.N, P + 1).astype(int)
    cuts[1] += 3  # uneven shards
    ops = sharded.CudaOps()
    blocks = [[d[n][:, :, a:b].contiguous() for n in ("Q", "K", "V")] for a, b in zip(cuts[:-1], cuts[1:])]
    parts = [ops.latent_memory(k, v, *prm) for _, k, v in blocks]
    Vt, Z = sharded.combine_total(parts, ops)
    Ob = torch.cat([ops.read_memory(q, *prm, Vt, Z, case.eps) for q, _, _ in blocks], dim=2)
    Oc = torch.cat([ops.forward_causal_carry(q, k, v, *prm, *sharded.combine_exclusive(parts, r, ops), case.eps)
                    for r, (q, k, v) in enumerate(blocks)], dim=2)
    args = (inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], case.eps)
    tol = TOL if dtype == "f32" else 1e-2  # bf16 d = K = 64 runs on the tensor cores
    assert _rel(Ob, oracle.forward_bidir(*args)) <= tol
    assert _rel(Oc, oracle.forward_causal(*args)) <= tol


# ---------------------------------------------------------------- reparameterisation (Eqs. 14-15)

@pytest.mark.parametrize("shape", [(1, 1, 16), (3, 37, 32), (8, 128, 128)], ids=lambda s: "H%d_K%d_r%d" % s)
def test_reparameterize_matches_oracle(shape):
    """sigma2 = softplus(omega) + eps_sigma and log_pi = log_softmax(alpha) on the
    GPU against the fp64 oracle (fp32 rounding: 1e-6 relative on sigma2, 2e-6 on
    log_pi over max(1, |log_pi|)); extreme omega included.  The gradients of
    both against the oracle's chain rule."""
    import oracle
    H, K, d_r = shape
    g = torch.Generator().manual_seed(H * 1000 + K)
    omega = torch.randn(H, K, d_r, generator=g) * 3
    omega[0, 0, :2] = torch.tensor([60.0, -60.0])
    alpha = torch.randn(H, K, generator=g) * 4
    s2, lp = gma.reparameterize(omega.cuda(), alpha.cuda(), eps_sigma=1e-3)
    s2_ref, lp_ref = oracle.reparameterize(omega, alpha, 1e-3)
    s2g = s2.double().cpu().numpy()
    assert np.max(np.abs(s2g - s2_ref) / s2_ref) < 1e-6
    lpg = lp.double().cpu().numpy()
    assert np.max(np.abs(lpg - lp_ref) / np.maximum(1.0, np.abs(lp_ref))) < 2e-6
    ds2 = torch.randn(H, K, d_r, generator=g)
    dlp = torch.randn(H, K, generator=g)
    dw, da = gma.reparameterize_backward(omega.cuda(), alpha.cuda(), ds2.cuda(), dlp.cuda())
    dw_ref, da_ref = oracle.reparameterize_backward(omega, alpha, ds2, dlp)
    assert np.max(np.abs(dw.double().cpu().numpy() - dw_ref)) <= 1e-6 * np.max(np.abs(dw_ref))
    assert np.max(np.abs(da.double().cpu().numpy() - da_ref)) <= 2e-6 * np.max(np.abs(da_ref))


def test_reparameterized_parameters_drive_the_forward():
    """The reparameterisation's outputs are valid forward parameters: the forward
    from them equals the oracle forward from the oracle's reparameterisation."""
    import oracle
    case = Case("reparam_fwd", False, 1, 2, 300, 32, 32, 16, "f32")
    inp = make_inputs(case, seed=4)
    g = torch.Generator().manual_seed(9)
    omega, alpha = torch.randn(2, 16, 32, generator=g) * 0.7, torch.randn(2, 16, generator=g)
    s2, lp = gma.reparameterize(omega.cuda(), alpha.cuda())
    s2_ref, lp_ref = oracle.reparameterize(omega, alpha, 1e-3)
    d = to_dev(inp)
    O = gma.forward_bidir(d["Q"], d["K"], d["V"], d["mu"], s2, lp, eps=case.eps, sync_status=True)
    ref = oracle.forward_bidir(inp["Q"], inp["K"], inp["V"], inp["mu"], s2_ref, lp_ref, case.eps)
    assert _rel(O, ref) <= TOL


def test_combine_memories_rank_order():
    """gma_combine_memories sums rows 0..count-1 one after another in fp32,
    row 0 first: bitwise the same as that sequential sum on the host."""
    import gaussian_mixture_latent_diag_gb300 as gma
    g = torch.Generator().manual_seed(3)
    parts = torch.randn(5, 10001, generator=g) * torch.logspace(-3, 3, 10001)
    dparts = parts.cuda()
    for count in (1, 2, 5):
        want = parts[0].clone()
        for r in range(1, count):
            want += parts[r]
        got = gma.combine_memories(dparts, count)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu(), want), count
