"""The C-ABI library loads, exports every function include/*.h declares, and
rejects bad arguments on the host (before any CUDA call, so these run
without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

from gaussian_mixture_latent_diag_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(gma_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from gaussian_mixture_latent_diag_gb300 import build
    build.build()
    return _native.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gma_responsibilities", "gma_forward_bidir", "gma_forward_causal",
              "gma_workspace_size", "gma_status_string", "gma_last_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_binding_knows_every_symbol():
    assert set(declared_functions()) <= set(_native.EXPORTED)


def test_status_strings(lib):
    for code in range(7):
        s = lib.gma_status_string(code)
        assert s and s != b"unknown status"
    assert lib.gma_status_string(99) == b"unknown status"


FAKE = 1 << 40  # never dereferenced: every call below fails host validation first


def _fwd(lib, fn="gma_forward_bidir", **kw):
    a = dict(Q=FAKE, Kx=FAKE + (1 << 32), V=FAKE + (2 << 32), dtype=1, mu=FAKE + (3 << 32),
             s2=FAKE + (4 << 32), lp=FAKE + (5 << 32), eps=1e-6, O=FAKE + (6 << 32),
             B=1, H=1, N=64, d_r=64, d_v=64, K=64, opt=None, ws=FAKE + (7 << 32), wsb=0)
    a.update(kw)
    opt = ctypes.byref(a["opt"]) if a["opt"] is not None else None
    vp = ctypes.c_void_p
    return getattr(lib, fn)(vp(a["Q"]), vp(a["Kx"]), vp(a["V"]), a["dtype"], vp(a["mu"]),
                            vp(a["s2"]), vp(a["lp"]), a["eps"], vp(a["O"]), a["B"], a["H"],
                            a["N"], a["d_r"], a["d_v"], a["K"], opt, vp(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("fn", ["gma_forward_bidir", "gma_forward_causal"])
def test_host_validation(lib, fn):
    need = lib.gma_workspace_size(1, 1, 64, 64, 64, 64, 1, int(fn.endswith("causal")), None)
    assert need > 0
    ok = dict(wsb=need)
    assert _fwd(lib, fn, Q=0, **ok) == 1                       # null pointer
    assert _fwd(lib, fn, ws=0, **ok) == 1
    assert _fwd(lib, fn, dtype=7, **ok) == 1                   # bad dtype
    assert _fwd(lib, fn, eps=0.0, **ok) == 1                   # eps must be > 0
    assert _fwd(lib, fn, eps=float("nan"), **ok) == 1
    assert _fwd(lib, fn, ws=FAKE + (7 << 32) + 8, **ok) == 1   # misaligned workspace
    assert _fwd(lib, fn, O=FAKE, **ok) == 1                    # O aliases Q
    assert _fwd(lib, fn, d_r=48, **ok) == 2                    # unsupported sizes
    assert _fwd(lib, fn, d_v=8, **ok) == 2
    assert _fwd(lib, fn, K=129, **ok) == 2
    assert _fwd(lib, fn, K=0, **ok) == 2
    assert _fwd(lib, fn, N=0, **ok) == 2
    assert _fwd(lib, fn, B=0, **ok) == 2
    assert _fwd(lib, fn, wsb=need - 1) == 3                    # workspace too small
    bad = _native.Options(9, 0, 0, 0)
    assert _fwd(lib, fn, opt=bad, **ok) == 2                   # unknown path
    neg = _native.Options(0, 0, -1, 0)
    assert _fwd(lib, fn, opt=neg, **ok) == 1


def test_responsibilities_validation(lib):
    vp = ctypes.c_void_p
    need = lib.gma_workspace_size(1, 1, 64, 64, 0, 8, 0, -1, None)
    assert need > 0

    def call(X=FAKE, G=FAKE + (1 << 32), d_r=64, K=8, wsb=need, dtype=0):
        return lib.gma_responsibilities(vp(X), dtype, vp(FAKE + (2 << 32)), vp(FAKE + (3 << 32)),
                                        vp(FAKE + (4 << 32)), vp(G), 1, 1, 64, d_r, K, None,
                                        vp(FAKE + (5 << 32)), wsb, None)
    assert call(X=0) == 1
    assert call(G=FAKE) == 1
    assert call(d_r=12) == 2
    assert call(K=200) == 2
    assert call(wsb=need - 1) == 3


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.gma_workspace_size(1, 1, 64, 64, 64, 64, 1, 2, None) == 0
    assert lib.gma_workspace_size(1, 1, 64, 20, 64, 64, 1, 0, None) == 0
    assert lib.gma_workspace_size(1, 1, 64, 64, 64, 64, 1, 0, None) > 0


def test_path_selection(lib):
    simt = _native.Options(1, 0, 0, 0)
    assert lib.gma_selected_path(256, 16, 32, 8, 0, 0, ctypes.byref(simt)) == 1
    assert lib.gma_selected_path(256, 16, 32, 8, 0, 0, None) == 1   # fp32 runs on SIMT
    assert lib.gma_selected_path(256, 15, 32, 8, 0, 0, None) == -1


def test_noalloc_argument_errors_come_first(lib):
    """gma_forward_bidir_noalloc reports argument errors before the size
    check, as gma_forward_bidir does, and never touches the device for them."""
    vp = ctypes.c_void_p
    big = dict(B=64, H=64, N=65536)  # far beyond the fixed scratch array

    def call(Q=FAKE, O=FAKE + (6 << 32), dtype=1, opt=None, B=1, H=1, N=64, d_r=64):
        o = ctypes.byref(opt) if opt is not None else None
        return lib.gma_forward_bidir_noalloc(vp(Q), vp(FAKE + (1 << 32)), vp(FAKE + (2 << 32)), dtype,
                                             vp(FAKE + (3 << 32)), vp(FAKE + (4 << 32)),
                                             vp(FAKE + (5 << 32)), 1e-6, vp(O), B, H, N, d_r, 64, 64, o,
                                             None)
    assert call(Q=0, **big) == 1                               # null pointer, whatever the size
    assert call(O=0, **big) == 1
    assert call(dtype=7, **big) == 1                           # bad dtype
    assert call(opt=_native.Options(0, 0, -1, 0), **big) == 1  # negative splits
    assert call(opt=_native.Options(0, -2, 0, 0), **big) == 1  # negative chunk
    assert call(d_r=48) == 2                                   # unsupported sizes
    assert call(**big) == 3                                    # too large for the array


def test_chunk_option(lib):
    """Causal calls run only the kernel family's chunk length (tensor cores 128,
    CUDA cores 64); any other positive value is rejected, negative values are
    invalid, and the bidirectional call ignores the field."""
    def ws(causal, path, chunk):
        o = _native.Options(path, chunk, 0, 0)
        return lib.gma_workspace_size(1, 1, 512, 64, 64, 64, 1, causal, ctypes.byref(o))
    assert ws(1, 2, 0) > 0 and ws(1, 2, 128) > 0
    assert ws(1, 2, 64) == 0 and ws(1, 2, 256) == 0
    assert ws(1, 1, 64) > 0 and ws(1, 1, 128) == 0
    assert ws(0, 2, 256) > 0                                   # bidirectional: no chunks
    assert lib.gma_selected_path(512, 64, 64, 64, 1, 1, ctypes.byref(_native.Options(0, 256, 0, 0))) == -1
    need = ws(1, 2, 0)
    for chunk, code in ((256, 2), (64, 2), (-1, 1)):
        assert _fwd(lib, "gma_forward_causal", opt=_native.Options(2, chunk, 0, 0), wsb=need) == code


def test_single_pass_path_selection(lib):
    """GMA_PATH_TC_SINGLE_PASS: the single-pass kernel for causal calls on the
    tensor-core sizes, the tensor-core path for bidirectional calls, rejected
    elsewhere; two stages (prep, scan)."""
    o = ctypes.byref(_native.Options(3, 0, 0, 0))
    assert lib.gma_selected_path(16384, 64, 64, 64, 1, 1, o) == 3
    assert lib.gma_selected_path(16384, 64, 64, 64, 1, 0, o) == 2
    assert lib.gma_selected_path(16384, 128, 128, 128, 1, 1, o) == -1
    assert lib.gma_selected_path(16384, 64, 64, 64, 0, 1, o) == -1    # fp32 inputs
    assert _native.stage_names(3, 1) == ["prep", "tc_scan"]
    assert _native.stage_names(3, 8) == ["prep", "tc_scan"]
    assert _native.stage_names(2, 1) == ["prep", "tc_aggregate", "tc_causal"]
    assert lib.gma_workspace_size(4, 8, 16384, 64, 64, 64, 1, 1, o) > 0
