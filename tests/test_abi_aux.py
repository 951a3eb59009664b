"""Host-side argument checks of the entry points beyond the forward: latent
memory, read from a memory, carried-prefix causal forward, decode step, usage
diagnostics, reparameterisation and projections.  Every call below is
rejected before any CUDA call (null pointers, misalignment, unsupported sizes,
short workspace, aliasing), so these run without a GPU."""
import ctypes

import pytest

from gaussian_mixture_latent_diag_gb300 import _native

FAKE = 1 << 40  # never dereferenced
vp = ctypes.c_void_p


def P(i):
    return FAKE + (i << 32)


@pytest.fixture(scope="module")
def lib():
    from gaussian_mixture_latent_diag_gb300 import build
    build.build()
    return _native.load()


def test_workspace_queries(lib):
    assert lib.gma_latent_memory_workspace_size(1, 1, 64, 64, 64, 64, 1, None) > 0
    assert lib.gma_latent_memory_workspace_size(1, 1, 64, 48, 64, 64, 1, None) == 0
    assert lib.gma_decode_workspace_size(8, 64, 64) > 0
    assert lib.gma_decode_workspace_size(8, 64, 129) == 0
    assert lib.gma_routing_stats_workspace_size(1, 1, 64, 64, 64, 1) > 0
    assert lib.gma_routing_stats_workspace_size(1, 1, 0, 64, 64, 1) == 0
    assert lib.gma_read_memory_workspace_size(1, 1, 64, 64, 64, 64, 1) > 0
    assert lib.gma_causal_carry_workspace_size(1, 1, 64, 64, 64, 64, 9) == 0
    assert lib.gma_project_workspace_size() >= 4
    tc = _native.Options(2, 0, 0, 0)  # the tensor-core path: bf16, d_r in {32, 64}, d_v = 64, K <= 64
    assert lib.gma_latent_memory_workspace_size(1, 1, 64, 64, 64, 64, 1, ctypes.byref(tc)) > 0
    assert lib.gma_latent_memory_workspace_size(1, 1, 64, 64, 64, 64, 0, ctypes.byref(tc)) == 0
    assert lib.gma_latent_memory_workspace_size(1, 1, 64, 64, 64, 128, 1, ctypes.byref(tc)) == 0
    assert lib.gma_decode_workspace_size(8, 64, 64) > 0
    # the read and carried-prefix queries take no options, so their size covers either
    # kernel family: the tensor-core read and carried forward use the forward's
    # tensor-core workspace (0 where that path does not take the sizes), and the
    # CUDA-core carried forward the CUDA-core causal forward's
    for B, H, N, d_r, d_v, K, dt in [(4, 8, 16384, 64, 64, 64, 1), (2, 3, 1000, 32, 64, 17, 1),
                                      (1, 2, 517, 64, 32, 8, 0)]:
        cases = ((0, lib.gma_read_memory_workspace_size, (2,)), (1, lib.gma_causal_carry_workspace_size, (1, 2)))
        for causal, fn, paths in cases:
            got = fn(B, H, N, d_r, d_v, K, dt)
            assert got > 0
            for path in paths:
                opt = _native.Options(path, 0, 0, 0)
                assert got >= lib.gma_workspace_size(B, H, N, d_r, d_v, K, dt, causal, ctypes.byref(opt))


def test_stage_names(lib):
    assert _native.stage_names(1, 5) == ["prep", "step"]
    assert _native.stage_names(1, 6) == ["prep", "rows", "final"]
    assert _native.stage_names(1, 7) == ["prep", "resp_q", "pack", "read"]
    assert lib.gma_stage_count(2, 5) == 0 and lib.gma_stage_count(1, 9) == 0
    assert _native.stage_names(2, 4) == ["prep", "tc_write"]
    assert _native.stage_names(2, 7) == ["prep", "pack", "tc_read"]
    assert _native.stage_names(2, 8) == ["prep", "tc_aggregate", "tc_causal"]


def test_decode_validation(lib):
    need = lib.gma_decode_workspace_size(2, 64, 64)

    def call(q=P(1), k=P(2), v=P(3), Vt=P(7), Z=P(8), o=P(9), ws=P(10), wsb=need, eps=1e-6, d_r=64, K=64,
             opt=None):
        return lib.gma_decode_step(vp(q), vp(k), vp(v), 1, vp(P(4)), vp(P(5)), vp(P(6)), eps, vp(Vt), vp(Z),
                                   vp(o), 3, 2, d_r, 64, K, opt, vp(ws), wsb, None)
    assert call(q=0) == 1
    assert call(eps=-1.0) == 1
    assert call(Vt=P(7) + 4) == 1      # Vt must be 16-byte aligned
    assert call(o=P(9) + 4) == 1       # o is written as float4
    assert call(q=P(1) + 1) == 1       # bf16 inputs need 2-byte alignment
    assert call(Z=P(7)) == 1           # Z inside Vt
    assert call(o=P(1)) == 1           # o aliases q
    assert call(d_r=20) == 2
    assert call(K=0) == 2
    assert call(wsb=need - 1) == 3
    bf = _native.Options(0, 0, 0, 0, 1)
    assert call(opt=ctypes.byref(bf)) == 2  # bf16 output not offered


def test_latent_read_carry_validation(lib):
    need = lib.gma_latent_memory_workspace_size(1, 2, 64, 32, 32, 16, 1, None)

    def mem(Kx=P(1), Vt=P(6), Z=P(7), wsb=need, N=64):
        return lib.gma_latent_memory(vp(Kx), vp(P(2)), 1, vp(P(3)), vp(P(4)), vp(P(5)), vp(Vt), vp(Z), 1, 2, N,
                                     32, 32, 16, None, vp(P(8)), wsb, None)
    assert mem(Kx=0) == 1
    assert mem(Z=P(6)) == 1
    assert mem(Vt=P(1)) == 1
    assert mem(N=0) == 2
    assert mem(wsb=need - 1) == 3

    need = lib.gma_read_memory_workspace_size(1, 2, 64, 32, 32, 16, 1)

    def read(O=P(9), wsb=need, eps=1e-6):
        return lib.gma_read_memory(vp(P(1)), 1, vp(P(3)), vp(P(4)), vp(P(5)), eps, vp(P(6)), vp(P(7)), vp(O), 1, 2,
                                   64, 32, 32, 16, None, vp(P(8)), wsb, None)
    assert read(O=P(6)) == 1
    assert read(eps=0.0) == 1
    assert read(wsb=need - 1) == 3

    need = lib.gma_causal_carry_workspace_size(1, 2, 64, 32, 32, 16, 1)

    def carry(vin=P(10), zin=P(11), vout=P(12), zout=P(13), O=P(9), wsb=need):
        return lib.gma_forward_causal_carry(vp(P(1)), vp(P(2)), vp(P(3)), 1, vp(P(4)), vp(P(5)), vp(P(6)), 1e-6,
                                            vp(vin), vp(zin), vp(vout), vp(zout), vp(O), 1, 2, 64, 32, 32, 16,
                                            None, vp(P(8)), wsb, None)
    assert carry(zin=0) == 1            # carry-in given in half
    assert carry(vout=0) == 1           # carry-out given in half
    assert carry(vout=P(10)) == 1       # output aliases the carry-in
    assert carry(O=P(12)) == 1          # two outputs overlap
    assert carry(wsb=need - 1) == 3


def test_stats_validation(lib):
    need = lib.gma_routing_stats_workspace_size(1, 2, 64, 32, 16, 1)

    def call(X=P(1), usage=P(5), counts=P(6), z=P(7), ent=P(8), wsb=need, K=16):
        return lib.gma_routing_stats(vp(X), 1, vp(P(2)), vp(P(3)), vp(P(4)), vp(usage), vp(counts), vp(z), vp(ent),
                                     1, 2, 64, 32, K, None, vp(P(9)), wsb, None)
    assert call(usage=0) == 1
    assert call(counts=P(5)) == 1       # counts overlap usage
    assert call(z=P(1)) == 1            # z aliases X
    assert call(ent=P(8) + 2) == 1
    assert call(K=129) == 2
    assert call(wsb=need - 1) == 3


def test_reparameterize_and_projection_validation(lib):
    assert lib.gma_reparameterize(vp(P(1)), vp(P(2)), 2, 16, 32, 1e-3, vp(P(1)), vp(P(4)), None) == 1
    assert lib.gma_reparameterize(vp(P(1)), vp(P(2)), 2, 16, 32, 0.0, vp(P(3)), vp(P(4)), None) == 1
    assert lib.gma_reparameterize(vp(P(1)), vp(P(2)), 2, 16, 30, 1e-3, vp(P(3)), vp(P(4)), None) == 2
    assert lib.gma_reparameterize_backward(vp(P(1)), vp(P(2)), vp(P(3)), vp(P(4)), 2, 16, 32, vp(P(3)), vp(P(6)),
                                           None) == 1
    need = lib.gma_project_workspace_size()

    def proj(X=P(1), Q=P(5), D=256, d_r=64, wsb=need, out=1):
        return lib.gma_project_qkv(vp(X), vp(P(2)), vp(P(3)), vp(P(4)), vp(Q), vp(P(6)), vp(P(7)), out, 2, 100, D,
                                   4, d_r, 64, None, vp(P(8)), wsb, None)
    assert proj(X=0) == 1
    assert proj(Q=P(1)) == 1            # output aliases X
    assert proj(X=P(1) + 8) == 1        # 16-byte alignment
    assert proj(out=5) == 1
    assert proj(D=100) == 2             # D must be a multiple of 8
    assert proj(d_r=48) == 2
    assert proj(wsb=need - 1) == 3


def test_combine_memories_validation(lib):
    vp = ctypes.c_void_p
    F = 1 << 40
    n = 1000
    assert lib.gma_combine_memories(vp(0), 3, n, 3, vp(F), None) == 1          # null parts
    assert lib.gma_combine_memories(vp(F), 3, n, 3, vp(0), None) == 1          # null out
    assert lib.gma_combine_memories(vp(F + 2), 3, n, 3, vp(F << 1), None) == 1  # misaligned
    assert lib.gma_combine_memories(vp(F), 3, n, 4, vp(F << 1), None) == 2     # count > P
    assert lib.gma_combine_memories(vp(F), 3, n, 0, vp(F << 1), None) == 2     # count < 1
    assert lib.gma_combine_memories(vp(F), 0, n, 0, vp(F << 1), None) == 2     # no rows
    assert lib.gma_combine_memories(vp(F), 3, 0, 1, vp(F << 1), None) == 2     # empty rows
    assert lib.gma_combine_memories(vp(F), 3, n, 3, vp(F + 4 * n), None) == 1  # out inside parts
