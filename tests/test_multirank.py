"""Host logic of the N > 1 bench path, on CPU with two gloo ranks.

Heads are independent, so N GPUs run N replicas of the workload shape with no
data-path exchange; the only cross-rank steps are the barrier, the maximum of
the step time over ranks and the whole-job throughput derived from it.  These
tests run that logic (bench.py's rank_seed / job_ms / job_throughput) in two
processes joined by a gloo process group on 127.0.0.1.
"""
import hashlib
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

        # each rank draws its own inputs of the same shape
        case = Case("t", False, 1, 2, 256, 16, 32, 8, "f32")
        d = make_inputs(case, seed=bench.rank_seed(rank, 0))
        digest = hashlib.sha256(d["Q"].numpy().tobytes() + d["K"].numpy().tobytes()).hexdigest()
        digests = [None] * world
        dist.all_gather_object(digests, digest)

        # the slowest rank sets the job's step time; every rank sees the same value
        dist.barrier()
        local_ms = 1.0 + 0.5 * rank
        ms = bench.job_ms(local_ms, world)
        value = bench.job_throughput(ms, world)
        out.put((rank, digests, local_ms, ms, value))
    finally:
        dist.destroy_process_group()


def _run(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_ranks_max_time_and_whole_job_throughput():
    import bench
    res = _run(2)
    w = bench.WORKLOAD
    slowest = max(r[2] for r in res)
    for rank, digests, local_ms, ms, value in res:
        assert ms == slowest == 1.5
        # two ranks x (one bidirectional + one causal forward) x B*H*N token*heads per step
        assert value == pytest.approx(2 * 2 * w["B"] * w["H"] * w["N"] / (1.5e-3))
        # replicas: each rank holds different data of the same shape
        assert len(set(digests)) == 2


def test_one_rank_is_local():
    import bench
    assert bench.job_ms(2.5, 1) == 2.5
    w = bench.WORKLOAD
    assert bench.job_throughput(2.5, 1) == pytest.approx(2 * w["B"] * w["H"] * w["N"] / 2.5e-3)
    assert len({bench.rank_seed(r, v) for r in range(8) for v in range(2)}) == 16
