"""GPU vs fp64 oracle for the latent memory, the one-position decode step and
the component-usage diagnostics, through the C ABI (Python binding), on seeded
inputs: several CTAs plus ragged tails (N not a multiple of 128, B not a
multiple of the decode kernel's 8 rows), every supported width, fp32 and bf16
inputs, and the degenerate cases (K = 1, exact ties, invalid parameters)."""
import zlib

import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

# fp32 arithmetic on exact inputs (bf16 inputs are widened exactly): the same
# 1e-4 bound as the fp32 forward, on max |x - x_ref| / RMS(x_ref).
TOL = 1e-4


def _rel(gpu, ref) -> float:
    g = gpu.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(g - ref)) / np.sqrt(np.mean(ref ** 2)))


def _case(B, H, N, d_r, d_v, K, dtype, **kw):
    name = f"aux_{dtype}_B{B}_H{H}_N{N}_r{d_r}_v{d_v}_K{K}_{kw.get('routing', 'iid')}"
    return Case(name, True, B, H, N, d_r, d_v, K, dtype, **kw)


def _seed(case):
    return zlib.crc32(case.name.encode()) % 1000


MEM_SHAPES = [  # (B, H, N, d_r, d_v, K)
    (2, 3, 300, 16, 32, 8),
    (1, 2, 1000, 64, 64, 64),
    (2, 1, 417, 128, 128, 128),
    (1, 2, 129, 32, 16, 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", MEM_SHAPES, ids=lambda s: "B%d_H%d_N%d_r%d_v%d_K%d" % s)
def test_latent_memory_matches_oracle(shape, dtype):
    import oracle
    case = _case(*shape, dtype)
    inp = make_inputs(case, seed=_seed(case))
    d = to_dev(inp)
    Vt, Z = gma.latent_memory(d["K"], d["V"], d["mu"], d["sigma2"], d["log_pi"], sync_status=True)
    Vt_ref, Z_ref = oracle.latent_memory(inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"])
    assert _rel(Vt, Vt_ref) <= TOL
    assert _rel(Z, Z_ref) <= TOL


DEC_SHAPES = [  # (B, H, N0 prompt, T steps, d_r, d_v, K)
    (11, 3, 0, 24, 16, 32, 8),
    (5, 2, 150, 12, 64, 64, 64),
    (9, 1, 40, 10, 128, 128, 128),
    (3, 2, 0, 9, 32, 16, 1),
    (17, 1, 70, 6, 64, 128, 37),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", DEC_SHAPES, ids=lambda s: "B%d_H%d_N0%d_T%d_r%d_v%d_K%d" % s)
def test_decode_continues_prompt_like_the_causal_forward(shape, dtype):
    """Prompt of N0 tokens through gma_latent_memory (or an empty state), then T
    decode steps: every step's o equals the oracle's causal row, and the final
    state equals the oracle's latent memory of all N0 + T tokens."""
    import oracle
    B, H, N0, T, d_r, d_v, K = shape
    case = _case(B, H, N0 + T, d_r, d_v, K, dtype)
    inp = make_inputs(case, seed=_seed(case))
    d = to_dev(inp)
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    if N0 > 0:
        Vt, Z = gma.latent_memory(d["K"][:, :, :N0].contiguous(), d["V"][:, :, :N0].contiguous(), *prm,
                                  sync_status=True)
    else:
        Vt = torch.zeros(B, H, K, d_v, device="cuda")
        Z = torch.zeros(B, H, K, device="cuda")
    outs = []
    for t in range(N0, N0 + T):
        q, k, v = (d[n][:, :, t].contiguous() for n in ("Q", "K", "V"))
        outs.append(gma.decode_step(q, k, v, *prm, Vt, Z, eps=case.eps, sync_status=True).clone())
    O = torch.stack(outs, dim=2)
    ref = oracle.forward_causal(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"],
                                case.eps)[:, :, N0:]
    assert _rel(O, ref) <= TOL
    Vt_ref, Z_ref = oracle.latent_memory(inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"])
    assert _rel(Vt, Vt_ref) <= TOL and _rel(Z, Z_ref) <= TOL


def test_decode_step_against_oracle_step_from_random_state():
    """One step from an arbitrary (non-negative) carried state, against the
    oracle's decode step directly; ragged batch (B = 13)."""
    import oracle
    B, H, d_r, d_v, K = 13, 4, 64, 64, 64
    g = torch.Generator().manual_seed(5)
    q, k = torch.randn(B, H, d_r, generator=g), torch.randn(B, H, d_r, generator=g)
    v = torch.randn(B, H, d_v, generator=g)
    Vt0 = torch.randn(B, H, K, d_v, generator=g) * 10
    Z0 = torch.rand(B, H, K, generator=g) * 50
    mu = torch.randn(H, K, d_r, generator=g)
    s2 = torch.nn.functional.softplus(torch.randn(H, K, d_r, generator=g) * 0.5 ** 0.5) + 1e-3
    lp = torch.log_softmax(torch.randn(H, K, generator=g), -1)
    Vt, Z = Vt0.cuda(), Z0.cuda()
    o = gma.decode_step(q.cuda(), k.cuda(), v.cuda(), mu.cuda(), s2.cuda(), lp.cuda(), Vt, Z, eps=1e-6,
                        sync_status=True)
    o_ref, Vt_ref, Z_ref = oracle.decode_step(q, k, v, mu, s2, lp, 1e-6, Vt0, Z0)
    assert _rel(o, o_ref) <= TOL
    assert _rel(Vt, Vt_ref) <= TOL and _rel(Z, Z_ref) <= TOL


def test_decode_invalid_parameters_leave_that_head_unchanged():
    """An invalid sigma2 in head 1: the call reports GMA_ERR_NONFINITE_PARAM and
    leaves head 1's rows untouched; head 0 is still updated.  The next valid
    call on the same workspace reports GMA_OK again."""
    B, H, d_r, d_v, K = 9, 2, 32, 32, 16
    q = torch.randn(B, H, d_r, device="cuda")
    v = torch.randn(B, H, d_v, device="cuda")
    mu = torch.randn(H, K, d_r, device="cuda")
    s2 = torch.ones(H, K, d_r, device="cuda")
    s2[1, 3, 5] = -1.0
    lp = torch.full((H, K), -float(np.log(K)), device="cuda")
    Vt = torch.randn(B, H, K, d_v, device="cuda")
    Z = torch.rand(B, H, K, device="cuda")
    Vt0, Z0 = Vt.clone(), Z.clone()
    with pytest.raises(gma.GmaError) as e:
        gma.decode_step(q, q.clone(), v, mu, s2, lp, Vt, Z, sync_status=True)
    assert e.value.status == 6
    assert torch.equal(Vt[:, 1], Vt0[:, 1]) and torch.equal(Z[:, 1], Z0[:, 1])
    assert not torch.equal(Z[:, 0], Z0[:, 0])
    ws = torch.empty(int(gma.load().gma_decode_workspace_size(H, d_r, K)), dtype=torch.uint8, device="cuda")
    with pytest.raises(gma.GmaError):
        gma.decode_step(q, q.clone(), v, mu, s2, lp, Vt, Z, workspace=ws, sync_status=True)
    s2[1, 3, 5] = 1.0
    gma.decode_step(q, q.clone(), v, mu, s2, lp, Vt, Z, workspace=ws, sync_status=True)


# ---------------------------------------------------------------- usage diagnostics

STAT_SHAPES = [  # (B, H, N, d_r, K, routing)
    (2, 3, 300, 16, 8, "iid"),
    (1, 2, 1000, 64, 64, "iid"),
    (2, 1, 257, 128, 128, "iid"),
    (1, 2, 129, 32, 1, "iid"),
    (2, 2, 700, 32, 32, "mixture"),
]


def check_stats(st, ref, scores, N, K):
    """usage / entropy within tolerance; hard assignments exact except where the
    fp64 top-two score gap is below 1e-3 (there the GPU's choice must be one of
    the near-maximal components); counts equal the histogram of z."""
    u = st["usage"].double().cpu().numpy()
    assert np.max(np.abs(u - ref["usage"])) <= 1e-5 * N
    assert np.max(np.abs(st["entropy"].double().cpu().numpy() - ref["entropy_norm"])) <= 1e-4
    z = st["z"].long().cpu().numpy()
    srt = np.sort(scores, axis=-1)
    gap = srt[..., -1] - srt[..., -2] if K > 1 else np.full(scores.shape[:-1], np.inf)
    clear = gap >= 1e-3
    assert np.all(z[clear] == ref["z"][clear])
    near = np.take_along_axis(scores, z[..., None], -1)[..., 0] >= srt[..., -1] - 1e-3
    assert np.all(near)
    counts = st["counts"].long().cpu().numpy()
    hist = np.stack([np.bincount(row, minlength=K) for row in z.reshape(-1, N)]).reshape(counts.shape)
    assert np.array_equal(counts, hist)
    assert np.array_equal(st["used"].cpu().numpy(), (counts > 0).sum(-1))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", STAT_SHAPES, ids=lambda s: "B%d_H%d_N%d_r%d_K%d_%s" % s)
def test_routing_stats_match_oracle(shape, dtype):
    import oracle
    B, H, N, d_r, K, routing = shape
    case = _case(B, H, N, d_r, 16, K, dtype, routing=routing, mu_std=3.0 if routing == "mixture" else 1.0)
    inp = make_inputs(case, seed=_seed(case))
    d = to_dev(inp)
    st = gma.routing_stats(d["Q"], d["mu"], d["sigma2"], d["log_pi"], sync_status=True)
    ref = oracle.routing_stats(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"])
    scores = np.stack([oracle.scores(inp["Q"][:, h], inp["mu"][h], inp["sigma2"][h], inp["log_pi"][h])
                       for h in range(H)], axis=1)
    check_stats(st, ref, scores, N, K)


def test_routing_stats_exact_ties_take_the_smallest_component():
    """Identical components with uniform priors: every score of a row is the
    same float, so every hard assignment is component 0; usage is N / K each and
    the normalised entropy is 1."""
    H, N, d_r, K = 2, 333, 32, 12
    X = torch.randn(1, H, N, d_r, device="cuda")
    mu = torch.randn(H, 1, d_r, device="cuda").expand(H, K, d_r).contiguous()
    s2 = (torch.rand(H, 1, d_r, device="cuda") + 0.5).expand(H, K, d_r).contiguous()
    lp = torch.full((H, K), -float(np.log(K)), device="cuda")
    st = gma.routing_stats(X, mu, s2, lp, sync_status=True)
    assert torch.all(st["z"] == 0)
    assert torch.all(st["counts"][..., 0] == N) and torch.all(st["counts"][..., 1:] == 0)
    assert torch.allclose(st["usage"], torch.full_like(st["usage"], N / K), rtol=1e-5)
    assert torch.allclose(st["entropy"], torch.ones_like(st["entropy"]), atol=1e-5)


def test_routing_stats_without_z():
    case = _case(1, 2, 500, 64, 16, 64, "bf16")
    inp = make_inputs(case, seed=1)
    d = to_dev(inp)
    a = gma.routing_stats(d["Q"], d["mu"], d["sigma2"], d["log_pi"], want_z=False, sync_status=True)
    b = gma.routing_stats(d["Q"], d["mu"], d["sigma2"], d["log_pi"], want_z=True, sync_status=True)
    assert a["z"] is None
    assert torch.equal(a["usage"], b["usage"]) and torch.equal(a["counts"], b["counts"])
