"""Tensor-core path (bf16 inputs, d_r = d_v = 64, K <= 64) against the fp64
oracle, element by element, with the number of persistent CTAs forced so that
one CTA runs several multi-tile jobs whose ranges cross head boundaries: this
exercises the job partials, the fixed-order combine of the bidirectional
memory and the carried-in prefixes of the causal scan.  K below 64 exercises
the padded components (c_k = -inf); d_r = 32 the zero-padded routing columns."""
import zlib

import pytest

import gaussian_mixture_latent_diag_gb300 as gma
from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
from gpu_helpers import TOL, normalised_error, oracle_full, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("splits", [1, 5, 7, 48])
@pytest.mark.parametrize("d_r,K", [(64, 64), (64, 40), (32, 32)], ids=["r64K64", "r64K40", "r32K32"])
@pytest.mark.parametrize("causal", [False, True], ids=["bidir", "causal"])
def test_tc_partitions(causal, d_r, K, splits):
    # 6 heads x 8 tiles of 128 tokens (the last one ragged: 1000 = 7 x 128 + 104)
    case = Case(f"tcpart_{int(causal)}_{d_r}_{K}_{splits}", causal, 2, 3, 1000, d_r, 64, K, "bf16")
    assert gma.selected_path(case.N, d_r, 64, K, "bf16", int(causal)) == gma.PATH_TC
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000)
    O = run_gpu(case, to_dev(inp), splits=splits)
    err = normalised_error(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], f"{case.name}: normalised max error {err:.3e}"
