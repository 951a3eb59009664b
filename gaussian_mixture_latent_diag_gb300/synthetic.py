"""Seeded synthetic inputs for the GMA forward pass.

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the attention arithmetic.  Both the CUDA path and
the CPU oracle are fed from it, so both see bit-identical inputs.

Recipe (one CPU ``torch.Generator`` per case, default seed 0):

* ``routing="iid"``: Q_X, K_X, V_X ~ N(0, 1) drawn in that order as fp32
  [B, H, N, d]; then mu [H, K, d_r] ~ N(0, mu_std^2), omega [H, K, d_r] ~
  N(0, 0.5) (variance 0.5) and alpha [H, K] ~ N(0, 1).
* ``routing="mixture"`` (rows drawn from the mixture itself): mu, omega, alpha
  first, then for Q and for K in turn a component z ~ Categorical(pi) per row
  and x = mu_z + sqrt(sigma2_z) * N(0, 1); V_X ~ N(0, 1) last.
* sigma2 = softplus(omega) + 1e-3 and log_pi = log_softmax(alpha), in fp32:
  the stated parameter distribution of the workloads (the covariance and prior
  parameterisations of the GMA paper, Eqs. (14)-(15)).
* bf16 cases round the fp32 draws to bfloat16 (round to nearest even).

N(m, v) in the workload descriptions names the variance v, so mu ~ N(0, 9)
has standard deviation 3.
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch


@dataclasses.dataclass(frozen=True)
class Case:
    name: str
    causal: bool
    B: int
    H: int
    N: int
    d_r: int
    d_v: int
    K: int
    dtype: str = "bf16"          # "f32" or "bf16" for Q_X, K_X, V_X and O
    routing: str = "iid"         # "iid" or "mixture"
    mu_std: float = 1.0
    eps: float = 1e-6

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.N

    def bytes_per_token_head(self) -> int:
        """Algorithmic HBM bytes per token and head: read Q_X, K_X, V_X, write O."""
        es = 4 if self.dtype == "f32" else 2
        return es * (2 * self.d_r + 2 * self.d_v)

    def replace(self, **kw) -> "Case":
        return dataclasses.replace(self, **kw)


# The five workloads: small fp32 bidirectional, mid-size bidirectional,
# long causal, long bidirectional with peaked (mixture-drawn) routing, and
# large-head causal.
WORKLOADS = {
    "bidir_f32_N256_K8": Case("bidir_f32_N256_K8", False, 1, 1, 256, 16, 32, 8, "f32"),
    "bidir_N4096_K64": Case("bidir_N4096_K64", False, 8, 8, 4096, 64, 64, 64),
    "causal_N16384_K64": Case("causal_N16384_K64", True, 4, 8, 16384, 64, 64, 64),
    "bidir_peaked_N16384_K32": Case("bidir_peaked_N16384_K32", False, 16, 4, 16384, 32, 64,
                                    32, routing="mixture", mu_std=3.0),
    "causal_N32768_K128": Case("causal_N32768_K128", True, 2, 32, 32768, 128, 128, 128),
}


def make_inputs(case: Case, seed: int = 0) -> dict:
    """Draw one case on the CPU.  Returns torch tensors:

    Q, K, V: [B, H, N, d] in ``case.torch_dtype``;
    mu, sigma2: [H, K, d_r] fp32; log_pi: [H, K] fp32; eps: float.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B, H, N, d_r, d_v, K = case.B, case.H, case.N, case.d_r, case.d_v, case.K

    def normal(*shape, std=1.0):
        t = torch.randn(*shape, generator=g, dtype=torch.float32)
        return t * std if std != 1.0 else t

    def params():
        mu = normal(H, K, d_r, std=case.mu_std)
        omega = normal(H, K, d_r, std=0.5 ** 0.5)
        alpha = normal(H, K)
        sigma2 = torch.nn.functional.softplus(omega) + 1e-3
        log_pi = torch.log_softmax(alpha, dim=-1)
        return mu, sigma2, log_pi

    if case.routing == "iid":
        Q = normal(B, H, N, d_r)
        Kx = normal(B, H, N, d_r)
        V = normal(B, H, N, d_v)
        mu, sigma2, log_pi = params()
    elif case.routing == "mixture":
        mu, sigma2, log_pi = params()
        pi = log_pi.double().exp()

        def rows():
            out = torch.empty(B, H, N, d_r, dtype=torch.float32)
            for h in range(H):
                z = torch.multinomial(pi[h], B * N, replacement=True, generator=g).view(B, N)
                noise = normal(B, N, d_r)
                out[:, h] = mu[h][z] + sigma2[h][z].sqrt() * noise
            return out

        Q = rows()
        Kx = rows()
        V = normal(B, H, N, d_v)
    else:
        raise ValueError(f"unknown routing {case.routing!r}")

    dt = case.torch_dtype
    return {"Q": Q.to(dt).contiguous(), "K": Kx.to(dt).contiguous(), "V": V.to(dt).contiguous(),
            "mu": mu.contiguous(), "sigma2": sigma2.contiguous(), "log_pi": log_pi.contiguous(),
            "eps": case.eps}


def input_digest(inp: dict) -> str:
    """SHA-256 over the raw bytes of every input tensor (logged with results)."""
    h = hashlib.sha256()
    for k in ("Q", "K", "V", "mu", "sigma2", "log_pi"):
        t = inp[k].contiguous()
        h.update(t.view(torch.uint8).numpy().tobytes() if t.dtype != torch.bfloat16
                 else t.view(torch.int16).numpy().tobytes())
    return h.hexdigest()
