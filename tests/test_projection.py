"""The Q/K/V projections (gma_project_qkv, a tcgen05 GEMM) against the fp64
oracle, element by element.  Inputs and weights are bf16, so every product is
exact in fp32 and the only error is the fp32 accumulation: per element at most
D * 2^-23 * sum_i |x_i w_i|; a bf16 output may add one bf16 ulp of the exact
value (the final rounding).  Shapes cover ragged token tiles (B N not a
multiple of 128), D not a multiple of the 64-feature stage, projections
narrower than one 128-feature tile, and heads narrower than a 32-feature
store segment (d = 16)."""
import numpy as np
import pytest
import torch

import gaussian_mixture_latent_diag_gb300 as gma
from gpu_helpers import bf16_ulp

pytestmark = pytest.mark.gpu

SHAPES = [  # (B, N, D, H, d_r, d_v)
    (2, 300, 256, 3, 16, 32),
    (1, 129, 72, 2, 64, 128),
    (1, 1000, 512, 8, 64, 64),
    (3, 50, 8, 1, 16, 16),
    (1, 257, 1024, 4, 128, 32),
]


def _draw(shape, seed):
    B, N, D, H, d_r, d_v = shape
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(B, N, D, generator=g).to(torch.bfloat16)
    Wq = (torch.randn(H * d_r, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    Wk = (torch.randn(H * d_r, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    Wv = (torch.randn(H * d_v, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    return X, Wq, Wk, Wv


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_N%d_D%d_H%d_r%d_v%d" % s)
def test_projection_matches_oracle(shape, out):
    import oracle
    B, N, D, H, d_r, d_v = shape
    X, Wq, Wk, Wv = _draw(shape, seed=B * 1000 + N + D)
    odt = torch.float32 if out == "f32" else torch.bfloat16
    got = gma.project_qkv(X.cuda(), Wq.cuda(), Wk.cuda(), Wv.cuda(), H, out_dtype=odt, sync_status=True)
    ref = oracle.project_qkv(X, Wq, Wk, Wv, H)
    absx = np.abs(X.double().numpy())
    for P, R, W, d in zip(got, ref, (Wq, Wk, Wv), (d_r, d_r, d_v)):
        assert P.shape == (B, H, N, d) and P.dtype == odt
        mag = np.einsum("bni,oi->bno", absx, np.abs(W.double().numpy())).reshape(B, N, H, d).transpose(0, 2, 1, 3)
        bound = D * 2.0 ** -23 * mag + (bf16_ulp(R) if out == "bf16" else 0.0)
        err = np.abs(P.double().cpu().numpy() - R)
        assert np.all(err <= bound), float(np.max(err - bound))


def test_projection_feeds_the_forward():
    """The projected bf16 tensors are the forward's inputs as they are: the
    projection followed by the tensor-core forward runs end to end and equals
    the forward on the same tensors handed over explicitly."""
    B, N, D, H, d = 1, 512, 256, 2, 64
    X, Wq, Wk, Wv = _draw((B, N, D, H, d, d), seed=7)
    Q, K, V = gma.project_qkv(X.cuda(), Wq.cuda(), Wk.cuda(), Wv.cuda(), H, sync_status=True)
    g = torch.Generator().manual_seed(8)
    mu = (torch.randn(H, 64, d, generator=g) * 0.1).cuda()
    s2 = torch.full((H, 64, d), 0.05).cuda()
    lp = torch.full((H, 64), -float(np.log(64))).cuda()
    O1 = gma.forward_causal(Q, K, V, mu, s2, lp, sync_status=True)
    O2 = gma.forward_causal(Q.clone(), K.clone(), V.clone(), mu, s2, lp, sync_status=True)
    assert gma.selected_path(N, d, d, 64, "bf16", 1) == gma.PATH_TC
    assert torch.equal(O1, O2) and torch.isfinite(O1).all()
