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


PATHS = [pytest.param((False, gma.PATH_TC), id="bidir"), pytest.param((True, gma.PATH_TC), id="causal"),
         pytest.param((True, gma.PATH_TC_SINGLE_PASS), id="causal1pass")]


@pytest.mark.parametrize("splits", [1, 5, 7, 48])
@pytest.mark.parametrize("d_r,K", [(64, 64), (64, 40), (32, 32)], ids=["r64K64", "r64K40", "r32K32"])
@pytest.mark.parametrize("variant", PATHS)
def test_tc_partitions(variant, d_r, K, splits):
    """The CTA count forced: job ranges that cross head boundaries (two-kernel
    paths), or chunks dealt round-robin to few CTAs (single-pass causal)."""
    causal, path = variant
    # 6 heads x 8 tiles of 128 tokens (the last one ragged: 1000 = 7 x 128 + 104)
    case = Case(f"tcpart_{int(causal)}_{path}_{d_r}_{K}_{splits}", causal, 2, 3, 1000, d_r, 64, K, "bf16")
    assert gma.selected_path(case.N, d_r, 64, K, "bf16", int(causal), path=path) == path
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000)
    O = run_gpu(case, to_dev(inp), splits=splits, path=path)
    err = normalised_error(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], f"{case.name}: normalised max error {err:.3e}"


@pytest.mark.parametrize("splits", [2, 3, 13, 0])
def test_tc_single_pass_long_heads(splits):
    """Single-pass causal kernel on heads of 40 chunks (the last one ragged):
    the block look-back chains many blocks, with 2 to 120 CTAs taking the
    chunks in turn (120: every chunk of every head in flight at once); bitwise
    reproducible from call to call."""
    case = Case(f"tclong_{splits}", True, 1, 3, 39 * 128 + 77, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=31 + splits)
    d = to_dev(inp)
    O = run_gpu(case, d, splits=splits, path=gma.PATH_TC_SINGLE_PASS)
    err = normalised_error(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], f"{case.name}: normalised max error {err:.3e}"
    O2 = run_gpu(case, d, splits=splits, path=gma.PATH_TC_SINGLE_PASS)
    assert (O == O2).all()


@pytest.mark.parametrize("splits", [2, 9, 0])
@pytest.mark.parametrize("variant", PATHS[:2])
def test_tc_many_one_tile_heads(variant, splits):
    """Forty heads of one ragged tile each: a CTA's range crosses a head boundary
    at every tile, so the time-balanced cuts (each boundary costs a job end and
    a job start) give CTAs many one-tile jobs and the job slots run deep; with
    the default CTA count every CTA holds at most one head."""
    causal, path = variant
    case = Case(f"tcsmall_{int(causal)}_{splits}", causal, 4, 10, 100, 64, 64, 64, "bf16")
    inp = make_inputs(case, seed=zlib.crc32(case.name.encode()) % 1000)
    O = run_gpu(case, to_dev(inp), splits=splits, path=path)
    err = normalised_error(O, oracle_full(case, inp))
    assert err <= TOL["bf16"], f"{case.name}: normalised max error {err:.3e}"
