"""The per-CTA tile ranges of the 64-wide tensor-core kernels, through the
host-only diagnostic gma_tc_partition (no GPU): every tile in exactly one
non-empty range, in order, within the CTA budget; the largest range cost
(tiles, plus the job-switch charge for every head boundary inside a range)
equal to the optimum of a brute-force dynamic programme over every way of
cutting the tiles into contiguous ranges; and argument errors reported."""
import ctypes

import pytest

from gaussian_mixture_latent_diag_gb300 import _native


@pytest.fixture(scope="module")
def lib():
    return _native.load()


def _cuts(lib, tiles_per_head, total, max_ctas):
    buf = (ctypes.c_int * 1024)()
    sw = ctypes.c_int(-1)
    n = lib.gma_tc_partition(tiles_per_head, total, max_ctas, buf, 1024, ctypes.byref(sw))
    assert n >= 1, n
    return list(buf[:n + 1]), sw.value


def _cost(a, b, tiles_per_head, sw):
    """Tiles a .. b - 1: their count plus sw per head boundary inside."""
    return (b - a) + sw * ((b - 1) // tiles_per_head - a // tiles_per_head)


def _optimum(total, tiles_per_head, max_ctas, sw):
    """Smallest largest-range cost over all cuts into at most max_ctas ranges."""
    inf = float("inf")
    best = [[inf] * (max_ctas + 1) for _ in range(total + 1)]  # best[b][c]: tiles 0 .. b-1 in c ranges
    best[0][0] = 0
    for b in range(1, total + 1):
        for c in range(1, max_ctas + 1):
            for a in range(b):
                if best[a][c - 1] < inf:
                    best[b][c] = min(best[b][c], max(best[a][c - 1], _cost(a, b, tiles_per_head, sw)))
    return min(best[total][1:])


@pytest.mark.parametrize("tiles_per_head,heads,max_ctas",
                         [(1, 1, 1), (1, 40, 2), (1, 40, 9), (3, 7, 4), (8, 6, 1), (8, 6, 5), (8, 6, 7),
                          (8, 6, 48), (5, 9, 6), (13, 3, 5), (2, 25, 11), (16, 3, 10)])
def test_partition_is_an_optimal_cover(lib, tiles_per_head, heads, max_ctas):
    total = tiles_per_head * heads
    st, sw = _cuts(lib, tiles_per_head, total, max_ctas)
    n = len(st) - 1
    assert sw >= 0
    assert n <= min(max_ctas, total)
    assert st[0] == 0 and st[-1] == total and all(st[i] < st[i + 1] for i in range(n))
    worst = max(_cost(st[i], st[i + 1], tiles_per_head, sw) for i in range(n))
    assert worst == _optimum(total, tiles_per_head, max_ctas, sw)


def test_ranges_that_cross_a_head_get_fewer_tiles(lib):
    """The bench shape (32 heads of 128 tiles on 152 SMs): every range that
    crosses a head boundary holds fewer tiles than the largest single-head one,
    and no range costs more than the largest single-head range."""
    st, sw = _cuts(lib, 128, 4096, 152)
    sizes = [(st[i + 1] - st[i], (st[i + 1] - 1) // 128 - st[i] // 128) for i in range(len(st) - 1)]
    single = max(t for t, crossings in sizes if crossings == 0)
    assert all(t < single for t, crossings in sizes if crossings > 0)
    assert max(t + sw * crossings for t, crossings in sizes) <= single


def test_rejects_bad_arguments(lib):
    buf = (ctypes.c_int * 4)()
    assert lib.gma_tc_partition(0, 8, 2, buf, 4, None) == -1   # no tiles per head
    assert lib.gma_tc_partition(3, 8, 2, buf, 4, None) == -1   # not whole heads
    assert lib.gma_tc_partition(2, 8, 0, buf, 4, None) == -1   # no CTA
    assert lib.gma_tc_partition(1, 8, 8, buf, 4, None) == -1   # 8 ranges need 9 entries
    assert lib.gma_tc_partition(2, 8, 2, None, 4, None) == -1
