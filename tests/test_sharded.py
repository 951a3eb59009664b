"""Sequence sharding over N (gaussian_mixture_latent_diag_gb300.sharded) on CPU
ranks joined by gloo: every rank holds one block of positions of the same
heads, the per-shard steps run through the fp64 oracle, and each rank's block of
O must equal the unsharded oracle forward on those rows.  The collectives and
the rank-order combination are the ones the CUDA path uses."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


class OracleOps:
    """The three per-shard steps of the sharded forward through the oracle."""

    def latent_memory(self, K, V, mu, sigma2, log_pi):
        import oracle
        vt, z = oracle.latent_memory(K, V, mu, sigma2, log_pi)
        return torch.from_numpy(vt), torch.from_numpy(z)

    def read_memory(self, Q, mu, sigma2, log_pi, Vt, Z, eps):
        import oracle
        return torch.from_numpy(oracle.read_memory(Q, mu, sigma2, log_pi, eps, Vt, Z))

    def forward_causal_carry(self, Q, K, V, mu, sigma2, log_pi, Vt_in, Z_in, eps):
        import oracle
        O, _, _ = oracle.decode(Q, K, V, mu, sigma2, log_pi, eps, Vt_in, Z_in)
        return torch.from_numpy(O)

    def combine(self, packed, count):
        """Rows 0..count-1 summed one after another in row order (the library's order)."""
        acc = packed[0].clone()
        for r in range(1, count):
            acc += packed[r]
        return acc


CUTS = {2: [0, 37, 90], 3: [0, 20, 21, 90]}


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from gaussian_mixture_latent_diag_gb300 import sharded
        from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

        case = Case("shard", False, 2, 2, 90, 16, 32, 8, "f32")
        inp = make_inputs(case, seed=11)  # every rank draws the same sequence
        a, b = CUTS[world][rank], CUTS[world][rank + 1]
        blk = {n: inp[n][:, :, a:b].double() for n in ("Q", "K", "V")}
        prm = (inp["mu"], inp["sigma2"], inp["log_pi"])
        Ob = sharded.forward_bidir_sharded(blk["Q"], blk["K"], blk["V"], *prm, eps=case.eps, ops=OracleOps())
        Oc = sharded.forward_causal_sharded(blk["Q"], blk["K"], blk["V"], *prm, eps=case.eps, ops=OracleOps())
        ref_b = oracle.forward_bidir(inp["Q"], inp["K"], inp["V"], *prm, case.eps)[:, :, a:b]
        ref_c = oracle.forward_causal(inp["Q"], inp["K"], inp["V"], *prm, case.eps)[:, :, a:b]
        eb = float(np.max(np.abs(Ob.numpy() - ref_b)) / np.sqrt(np.mean(ref_b ** 2)))
        ec = float(np.max(np.abs(Oc.numpy() - ref_c)) / np.sqrt(np.mean(ref_c ** 2)))
        out.put((rank, eb, ec))
    finally:
        dist.destroy_process_group()


def _run(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_forward_matches_unsharded(world):
    for rank, eb, ec in _run(world):
        assert eb < 1e-12, (rank, eb)
        assert ec < 1e-12, (rank, ec)


def test_rank_order_combination():
    from gaussian_mixture_latent_diag_gb300 import sharded
    ops = OracleOps()
    parts = [(torch.full((2, 3), float(r + 1)), torch.full((2,), 10.0 * (r + 1))) for r in range(4)]
    packed = sharded.pack_memories(parts)
    assert packed.shape == (4, 8) and torch.equal(packed[2], torch.tensor([3.0] * 6 + [30.0] * 2))
    Vt, Z = sharded.combine_total(parts, ops)
    assert torch.equal(Vt, torch.full((2, 3), 10.0)) and torch.equal(Z, torch.full((2,), 100.0))
    assert sharded.combine_exclusive(parts, 0, ops) == (None, None)
    Vt, Z = sharded.combine_exclusive(parts, 3, ops)
    assert torch.equal(Vt, torch.full((2, 3), 6.0)) and torch.equal(Z, torch.full((2,), 60.0))
    # the inputs are not modified
    assert torch.equal(parts[0][0], torch.full((2, 3), 1.0))


def test_cuda_ops_pick_the_unsharded_kernel_family():
    """sharded.CudaOps runs a shard on the tensor cores exactly where the
    memory calls have tensor-core kernels -- the sizes where the unsharded
    bidirectional forward runs there (bf16, d_r in {32, 64}, d_v = 64, K <= 64),
    so a sharded call has the unsharded call's accuracy; the 128-wide causal
    tensor-core kernels have no memory calls, so those sizes shard on the CUDA
    cores.  Host logic only: the choice comes from gma_selected_path, which
    needs no GPU."""
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300.sharded import CudaOps

    def pick(dtype, d_r, d_v, K, causal=0, n=300):
        X = torch.empty(1, 2, n, d_r, dtype=dtype)
        V = torch.empty(1, 2, n, d_v, dtype=dtype)
        mu = torch.empty(2, K, d_r)
        return CudaOps._path(X, V, mu, causal)

    bf, f32 = torch.bfloat16, torch.float32
    assert pick(bf, 64, 64, 64) == gma.PATH_TC
    assert pick(bf, 32, 64, 17, causal=1) == gma.PATH_TC
    assert pick(bf, 64, 64, 64, n=1) == gma.PATH_TC
    assert pick(f32, 64, 64, 64) == gma.PATH_SIMT
    assert pick(bf, 64, 32, 64) == gma.PATH_SIMT
    assert pick(bf, 128, 64, 64, causal=1) == gma.PATH_SIMT
    assert pick(bf, 64, 64, 128) == gma.PATH_SIMT
    for causal in (0, 1):  # the unsharded forward is on the tensor cores, the memory calls are not
        assert pick(bf, 128, 128, 128, causal=causal) == gma.PATH_SIMT
        assert gma.selected_path(300, 128, 128, 128, "bf16", causal) == gma.PATH_TC
    for dtype, d_r, d_v, K in [(bf, 64, 64, 64), (f32, 16, 32, 8)]:
        for causal in (0, 1):
            want = gma.selected_path(300, d_r, d_v, K, "bf16" if dtype == bf else "f32", causal)
            assert pick(dtype, d_r, d_v, K, causal) == want
