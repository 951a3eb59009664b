"""The decode step, the usage diagnostics and the projections at the full
sizes their benchmarks time, in the same launch configuration, against the
fp64 oracle on sampled outputs that it computes one by one:

* decode: one step over B=2048 x H=8 carried states (d_r = d_v = K = 64, bf16
  q, k, v), every output and state row of 24 sampled (b, h) pairs;
* diagnostics: the peaked-routing workload (B=16, H=4, N=16384, d_r = K = 32),
  usage, counts and hard assignments of 3 whole heads;
* projections: X [4, 16384, 1024] to three [4, 8, 16384, 64] bf16 tensors,
  64 sampled tokens, every output feature;
* the tensor-core latent memory, read from a memory and carried causal
  forward at B=4, H=8, N=16384, d = K = 64: 3 whole heads."""
import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import WORKLOADS, Case, make_inputs
from gpu_helpers import bf16_ulp, to_dev
from test_aux_paths import check_stats

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_decode_step_full_size():
    import oracle
    B, H, d, K = 2048, 8, 64, 64
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(B, H, d, generator=g).to(torch.bfloat16) for _ in range(3))
    mu = torch.randn(H, K, d, generator=g)
    s2 = torch.nn.functional.softplus(torch.randn(H, K, d, generator=g) * 0.5 ** 0.5) + 1e-3
    lp = torch.log_softmax(torch.randn(H, K, generator=g), -1)
    Vt0 = torch.randn(B, H, K, d, generator=g) * 30
    Z0 = torch.rand(B, H, K, generator=g) * 100
    Vt, Z = Vt0.cuda(), Z0.cuda()
    o = gma.decode_step(q.cuda(), k.cuda(), v.cuda(), mu.cuda(), s2.cuda(), lp.cuda(), Vt, Z, eps=1e-6,
                        sync_status=True)
    rng = np.random.default_rng(0)
    bs = np.unique(np.concatenate([[0, 7, 8, B - 1], rng.integers(0, B, 20)]))
    hs = rng.integers(0, H, bs.size)
    o_ref, vt_ref, z_ref = oracle.decode_step(q[bs, hs][:, None], k[bs, hs][:, None], v[bs, hs][:, None],
                                              np.stack([mu[h].numpy() for h in hs]),
                                              np.stack([s2[h].numpy() for h in hs]),
                                              np.stack([lp[h].numpy() for h in hs]), 1e-6,
                                              Vt0[bs, hs][:, None], Z0[bs, hs][:, None])
    # one head per sampled row: the oracle's per-head parameters are those rows' heads
    rms = float(o.float().pow(2).mean().sqrt())
    sel = (torch.as_tensor(bs), torch.as_tensor(hs))
    assert np.max(np.abs(o.cpu()[sel].double().numpy() - o_ref[:, 0])) / rms <= 1e-4
    vt_rms = float(Vt.float().pow(2).mean().sqrt())
    assert np.max(np.abs(Vt.cpu()[sel].double().numpy() - vt_ref[:, 0])) / vt_rms <= 1e-4
    assert np.max(np.abs(Z.cpu()[sel].double().numpy() - z_ref[:, 0])) / float(Z.float().pow(2).mean().sqrt()) <= 1e-4


def test_routing_stats_full_size():
    import oracle
    case = WORKLOADS["bidir_peaked_N16384_K32"]
    inp = make_inputs(case, seed=0)
    d = to_dev(inp)
    st = gma.routing_stats(d["Q"], d["mu"], d["sigma2"], d["log_pi"], sync_status=True)
    for bh in (0, 37, case.B * case.H - 1):
        b, h = divmod(bh, case.H)
        x = inp["Q"][b, h]
        ref = oracle.routing_stats(x, inp["mu"][h], inp["sigma2"][h], inp["log_pi"][h])
        scores = oracle.scores(x, inp["mu"][h], inp["sigma2"][h], inp["log_pi"][h])
        one = {k: v[b, h] for k, v in st.items()}
        check_stats(one, ref, scores, case.N, case.K)


def test_projection_full_size():
    import oracle
    B, N, D, H, dh = 4, 16384, 1024, 8, 64
    g = torch.Generator().manual_seed(12)
    X = torch.randn(B, N, D, generator=g).to(torch.bfloat16)
    Ws = [(torch.randn(H * dh, D, generator=g) / D ** 0.5).to(torch.bfloat16) for _ in range(3)]
    outs = gma.project_qkv(X.cuda(), *(w.cuda() for w in Ws), H, sync_status=True)
    rng = np.random.default_rng(1)
    toks = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 60)]))
    b = 2
    xs = X[b, toks][None]
    refs = oracle.project_qkv(xs, *Ws, H)
    absx = np.abs(xs.double().numpy())
    for P, R, W in zip(outs, refs, Ws):
        got = P[b][:, torch.as_tensor(toks, device=P.device)].double().cpu().numpy()
        mag = np.einsum("bni,oi->bno", absx, np.abs(W.double().numpy())).reshape(1, -1, H, dh).transpose(0, 2, 1, 3)
        bound = D * 2.0 ** -23 * mag[0] + bf16_ulp(R[0])
        assert np.all(np.abs(got - R[0]) <= bound)


def test_tc_memory_calls_full_size():
    """The three per-shard calls on the tensor cores at the size the shard
    benchmark times (B=4, H=8, N=16384, d_r = d_v = K = 64, bf16), against the
    fp64 oracle on 3 whole heads: the latent memory, the read of that memory
    (= the bidirectional forward), and the causal forward in two 8192-token
    pieces, the second carried from the first's returned state."""
    import oracle
    case = Case("tc_mem_full", True, 4, 8, 16384, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=5)
    d = to_dev(inp)
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    TC = gma.PATH_TC
    Vt, Z = gma.latent_memory(d["K"], d["V"], *prm, path=TC, sync_status=True)
    Ob = gma.read_memory(d["Q"], *prm, Vt, Z, eps=case.eps, path=TC, sync_status=True)
    half = case.N // 2
    blk = lambda a, b: [d[n][:, :, a:b].contiguous() for n in ("Q", "K", "V")]  # noqa: E731
    O1, vt1, z1 = gma.forward_causal_carry(*blk(0, half), *prm, eps=case.eps, path=TC, sync_status=True)
    O2, vt2, z2 = gma.forward_causal_carry(*blk(half, case.N), *prm, Vt_in=vt1, Z_in=z1, eps=case.eps, path=TC,
                                           sync_status=True)
    Oc = torch.cat([O1, O2], dim=2)
    for bh in (0, 13, case.B * case.H - 1):
        b, h = divmod(bh, case.H)
        one = lambda n: inp[n][b:b + 1, h:h + 1]  # noqa: E731
        p1 = (inp["mu"][h:h + 1], inp["sigma2"][h:h + 1], inp["log_pi"][h:h + 1])
        vt_ref, z_ref = oracle.latent_memory(one("K"), one("V"), *p1)
        rel = lambda g, r: float(np.max(np.abs(g - r)) / np.sqrt(np.mean(r ** 2)))  # noqa: E731
        assert rel(Vt[b, h].double().cpu().numpy(), vt_ref[0, 0]) <= 1e-2
        assert rel(Z[b, h].double().cpu().numpy(), z_ref[0, 0]) <= 1e-2
        assert rel(vt2[b, h].double().cpu().numpy(), vt_ref[0, 0]) <= 1e-2
        assert rel(z2[b, h].double().cpu().numpy(), z_ref[0, 0]) <= 1e-2
        ob_ref = oracle.forward_bidir(one("Q"), one("K"), one("V"), *p1, case.eps)[0, 0]
        assert rel(Ob[b, h].double().cpu().numpy(), ob_ref) <= 1e-2
        oc_ref = oracle.forward_causal(one("Q"), one("K"), one("V"), *p1, case.eps)[0, 0]
        assert rel(Oc[b, h].double().cpu().numpy(), oc_ref) <= 1e-2
