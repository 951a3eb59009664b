"""Benchmark of the GMA forward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gma|reference]

One step = one bidirectional and one causal GMA forward (every step of the
hot path: coefficient prep, responsibilities, latent write, read, causal
scan) over a batch B=4, H=8, N=16384, d_r=d_v=K=64, bf16 inputs and fp32
output O, each variant on its own seeded synthetic input set.  The metric is forward token*heads per
second: 2 * B * H * N per step (both variants) divided by the step time.
The step moves 2 x 335 MB of algorithmic traffic (Q_X, K_X, V_X read, O
written), more than the 129 MB L2, so no separate L2 flush is done between
steps.

Prints ONE JSON line (rank 0).  With --impl reference the fp64 CPU oracle is
timed instead, on a bounded sample of the same workload (one head of each
variant per step), in the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(B=4, H=8, N=16384, d_r=64, d_v=64, K=64, dtype="bf16", eps=1e-6)
METRIC = "GMA fwd tokens*heads/s (bidir & causal, N=16K, K=64); % of GB300 HBM roofline"
UNIT = "token*heads/s"

# Algorithmic HBM bytes each stage accounts for, as the tensors of the path it
# reads or writes (Q_X, K_X, V_X read once, O written once per forward);
# intermediate scratch traffic is not algorithmic.  The single-pass tensor-core
# causal scan reads Q, K and V and writes O.
STAGE_TENSORS = {
    "prep": "", "reset": "", "reduce": "", "scan": "",
    "resp_q": "Q", "resp_k": "K", "write": "V", "read": "O", "causal": "VO",
    "tc_write": "KV", "tc_read": "QO", "tc_causal": "QVO", "tc_aggregate": "KV", "tc_scan": "QKVO",
}


def tensor_bytes(t: str, w=WORKLOAD, o_bytes: int = 4) -> int:
    """Bytes of the named path tensors; O is written in fp32 (o_bytes = 2: the
    byte count O would have in bf16, the metric's basis)."""
    es = 2 if w["dtype"] == "bf16" else 4
    per = {"Q": es * w["d_r"], "K": es * w["d_r"], "V": es * w["d_v"], "O": o_bytes * w["d_v"]}
    return sum(per[c] for c in t) * w["B"] * w["H"] * w["N"]


TC_SOURCES = ("gma_tc.cu", "gma_tc128.cu", "tc_common.cuh", "tc_ptx.cuh")


def source_digest() -> str:
    """Digest of the sources of the profiled tensor-core kernels."""
    h = hashlib.sha256()
    for name in TC_SOURCES:
        with open(os.path.join(ROOT, "gaussian_mixture_latent_diag_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def recorded_traffic(stage: str):
    """DRAM bytes per launch of `stage` from the committed ncu summary, if the
    kernels have not changed since it was taken (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_digest") != source_digest():
        return None
    v = d.get("stages", {}).get(stage)
    return None if v is None else float(v)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()
        return False

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ oracle (CPU)

def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def host_cpu_model() -> str:
    """CPU model of the host (lscpu's model name, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        return f"implementer {fields.get('cpu implementer', '?')} part {fields.get('cpu part', '?')}"
    except Exception:
        import platform
        return platform.processor() or platform.machine()


def _oracle_head(args):
    """One head of one variant through the fp64 oracle (runs in a worker); an
    optional fourth item sets the head's length (default: the workload's N)."""
    causal, seed, head = args[:3]
    n = args[3] if len(args) > 3 else WORKLOAD["N"]
    sys.path.insert(0, ROOT)
    import oracle
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
    w = WORKLOAD
    case = Case("sample", bool(causal), 1, 1, n, w["d_r"], w["d_v"], w["K"], w["dtype"])
    inp = make_inputs(case, seed=seed * 1000 + head)
    fn = oracle.forward_causal if causal else oracle.forward_bidir
    t = time.perf_counter()
    fn(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], w["eps"])
    return time.perf_counter() - t


def _oracle_backward_head(seed):
    """One head of the bidirectional backward through the fp64 oracle (single process)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
    w = WORKLOAD
    inp = make_inputs(Case("sample", False, 1, 1, w["N"], w["d_r"], w["d_v"], w["K"], w["dtype"]), seed=seed)
    dO = np.random.default_rng(seed).standard_normal((1, 1, w["N"], w["d_v"]))
    t = time.perf_counter()
    oracle.backward_bidir(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], w["eps"], dO)
    return time.perf_counter() - t


class OraclePool:
    """Spawned worker processes that run oracle heads (started once)."""

    def __init__(self, procs: int):
        import multiprocessing as mp
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(procs)
        self.pool.map(_oracle_head, [(0, 0, 0)] * procs)  # workers up, oracle loaded

    def sample(self, pairs: int, n: int = WORKLOAD["N"]):
        """Wall time and token*heads for `pairs` (bidir head, causal head) pairs of
        n tokens each."""
        jobs = [(c, 7, i, n) for i in range(pairs) for c in (0, 1)]
        t = time.perf_counter()
        self.pool.map(_oracle_head, jobs)
        return time.perf_counter() - t, len(jobs) * n

    def close(self):
        self.pool.close()
        self.pool.join()


def run_reference(args, rank: int):
    """The fp64 oracle on the host cores: one spawned process per core, each
    step one bidirectional and one causal head per process.  The heads are
    whole (N = 16384) unless that would make the run longer than about two and
    a half minutes; then every head of the run is the same shorter prefix of
    the workload's sequence length (the oracle's cost per token does not
    depend on N)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    steps = args.steps if args.steps is not None else 3
    procs = host_cores()
    pool = OraclePool(procs)
    # calibration (untimed): one pair of 2048-token heads per process
    wall, th = pool.sample(procs, 2048)
    per_token = wall / (th / procs)              # seconds per token*head on one process
    budget = 150.0 / (steps + args.warmup)       # seconds per step
    n = int(min(WORKLOAD["N"], max(256, budget / (2 * per_token))))
    n = 1 << (n.bit_length() - 1) if n < WORKLOAD["N"] else n
    times = []
    for s in range(args.warmup + steps):
        wall, th = pool.sample(procs, n)
        if s >= args.warmup:
            times.append(wall)
    pool.close()
    ms = 1e3 * statistics.mean(times)
    value = th / (ms / 1e3)
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": f"GMA forward, {procs} bidirectional + {procs} causal heads of N={n} per "
                                  "step (sample of B=4,H=8,N=16384,d_r=d_v=K=64)", **WORKLOAD},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": procs, "cpu_model": host_cpu_model(),
                            "kind": "oracle",
                            "sample": f"per step, one bidirectional + one causal head of N={n} tokens on "
                                      f"each of {procs} processes (one per host core), fp64 C oracle"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ GPU arm

BWD_METRIC = "GMA backward tokens*heads/s (bidir & causal, N=16K, K=64); % of GB300 HBM roofline"


def run_backward(args, rank: int, world: int, local_rank: int):
    """One bidirectional and one causal backward per step over the forward bench's
    workload: inputs Q, K, V (bf16) and dO (fp32) resident, gradients dQ, dK, dV
    (fp32) and the parameter gradients written every step.  Algorithmic bytes per
    token*head and variant: Q, K, V 2*64 each, dO 4*64, dQ, dK, dV 4*64 each = 1408 B."""
    import ctypes
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300 import _native
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOAD
    B, H, N, d_r, d_v, K = w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"]
    inp = make_inputs(Case("bwd", False, B, H, N, d_r, d_v, K, w["dtype"]), seed=rank_seed(rank, 2))
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = torch.Generator().manual_seed(rank_seed(rank, 3))
    dO = torch.randn(B, H, N, d_v, generator=g, dtype=torch.float32).to(dev)
    outs = [torch.empty(B, H, N, d_r, device=dev), torch.empty(B, H, N, d_r, device=dev),
            torch.empty(B, H, N, d_v, device=dev), torch.empty(H, K, d_r, device=dev),
            torch.empty(H, K, d_r, device=dev), torch.empty(H, K, device=dev)]
    lib = gma.load()
    opt0 = _native.options()
    nb = int(lib.gma_backward_workspace_size(B, H, N, d_r, d_v, K, _native.GMA_BF16, 0, ctypes.byref(opt0)))
    nb = max(nb, int(lib.gma_backward_workspace_size(B, H, N, d_r, d_v, K, _native.GMA_BF16, 1,
                                                     ctypes.byref(opt0))))
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    stages = [_native.stage_names(_native.PATH_SIMT, 2), _native.stage_names(_native.PATH_SIMT, 3)]
    stream = torch.cuda.current_stream()
    vp = ctypes.c_void_p

    def call1(fn, events=None):
        opt = _native.options(stage_events=events)
        st = getattr(lib, fn)(vp(d["Q"].data_ptr()), vp(d["K"].data_ptr()), vp(d["V"].data_ptr()),
                                    _native.GMA_BF16, vp(d["mu"].data_ptr()), vp(d["sigma2"].data_ptr()),
                                    vp(d["log_pi"].data_ptr()), float(w["eps"]), vp(dO.data_ptr()),
                                    *[vp(t.data_ptr()) for t in outs], B, H, N, d_r, d_v, K, ctypes.byref(opt),
                                    vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream))
        if st != 0:
            raise gma.GmaError(st, fn)

    def call(events=None):
        call1("gma_backward_bidir", events[0] if events else None)
        call1("gma_backward_causal", events[1] if events else None)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0.record(stream)
        for _ in range(args.steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = job_ms(t0.elapsed_time(t1) / args.steps, world, dev)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(stages[v]) + 1)] for v in range(2)]
          for _ in range(args.steps)]
    for s in range(args.steps):
        call(events=ev[s])
    torch.cuda.synchronize()
    stage_ms = {f"{('bidir', 'causal')[v]}:{name}": statistics.mean(ev[s][v][j].elapsed_time(ev[s][v][j + 1])
                                                                   for s in range(args.steps))
                for v in range(2) for j, name in enumerate(stages[v])}
    variant_ms = {("bidir", "causal")[v]: statistics.mean(ev[s][v][0].elapsed_time(ev[s][v][-1])
                                                         for s in range(args.steps)) for v in range(2)}
    units = world * 2 * B * H * N
    value = units / (ms / 1e3)
    peak, peak_src = measured_peaks()
    alg = 2 * B * H * N * (3 * 2 * 64 + 4 * 64 + 3 * 4 * 64)
    achieved = alg / (ms / 1e3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        secs = _oracle_backward_head(7)
        cpu = {"value": N / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "one bidirectional head of the same workload (N=16384, d=K=64) through the fp64 C "
                         f"oracle backward, {secs:.1f} s on one core"}
    if rank == 0:
        out = {"metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f32", "data": "synthetic",
               "config": {"workload": "GMA backward, bidirectional + causal, B=4 H=8 N=16384 d_r=d_v=K=64, bf16 "
                                      "inputs, fp32 dO and gradients (per GPU)", **{k: w[k] for k in ("B", "H", "N", "d_r",
                                                                                           "d_v", "K")},
                          "l2": "inputs larger than L2, no flush", "parallelism": f"replicas x{world}"},
               # bidirectional: prep, 2 responsibilities, write, reduce (state); upstream; ds_q;
               # colsum + reduce (dmem); ds_k + dV; dQ + dK; 2 statistics + final (params) = 16;
               # causal: prep, 2 responsibilities, write, scan (state); query; colsum + suffix;
               # key; dQ + dK; 2 statistics + final = 15
               "gpu_launches": (16 + 15) * args.steps,
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                            "frac": achieved / peak, "traffic": None, "kernel": "whole call (all stages)",
                            "algorithmic_bytes": alg, "peak_source": peak_src},
               "variants_ms": variant_ms, "stage_ms": stage_ms, "clocks": clocks.summary(), "cpu_baseline": cpu}
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ decode step and usage diagnostics

DEC_WORKLOAD = dict(B=2048, H=8, d_r=64, d_v=64, K=64, dtype="bf16", eps=1e-6)
DEC_METRIC = "GMA causal decode step token*heads/s (B=2048 x H=8, K=64); % of GB300 HBM roofline"
STAT_WORKLOAD = dict(B=16, H=4, N=16384, d_r=32, K=32, dtype="bf16")
STAT_METRIC = "GMA component-usage diagnostics token*heads/s (peaked routing, N=16K, K=32)"


def _oracle_decode_sample(pairs: int):
    """`pairs` (b, h) decode steps of the decode workload's shape through the fp64 oracle."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle
    w = DEC_WORKLOAD
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((pairs, 1, w["d_r"])), rng.standard_normal((pairs, 1, w["d_r"]))
    v = rng.standard_normal((pairs, 1, w["d_v"]))
    mu = rng.standard_normal((1, w["K"], w["d_r"]))
    s2 = np.log1p(np.exp(rng.standard_normal((1, w["K"], w["d_r"])) * 0.5 ** 0.5)) + 1e-3
    lp = np.log(np.full((1, w["K"]), 1.0 / w["K"]))
    Vt, Z = rng.standard_normal((pairs, 1, w["K"], w["d_v"])), rng.random((pairs, 1, w["K"])) * 50
    t = time.perf_counter()
    oracle.decode_step(q, k, v, mu, s2, lp, w["eps"], Vt, Z)
    return time.perf_counter() - t


def _oracle_stats_head(seed: int):
    """One head of the diagnostics workload through the fp64 oracle."""
    sys.path.insert(0, ROOT)
    import oracle
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs
    w = STAT_WORKLOAD
    inp = make_inputs(Case("stats", False, 1, 1, w["N"], w["d_r"], 16, w["K"], w["dtype"], routing="mixture",
                           mu_std=3.0), seed=seed)
    t = time.perf_counter()
    oracle.routing_stats(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"])
    return time.perf_counter() - t


def run_aux(args, rank: int, world: int, local_rank: int):
    """--workload decode: one gma_decode_step over B=2048 x H=8 carried states
    (K = d_v = 64, fp32 state of 272 MB, larger than L2) per step; algorithmic
    bytes per (b, h): q, k, v (bf16) 384 + state read and written 2 * 4 * K * (d_v + 1)
    + o (fp32) 256 = 33920 B.
    --workload stats: one gma_routing_stats over the peaked-routing workload
    (B=16, H=4, N=16384, d_r = K = 32, bf16, rows drawn from the mixture) per step,
    hard assignments written; it runs on the CUDA cores and is bound by their
    fp32 issue rate: 3 K d_r operations per row (difference, square, scaled
    accumulate per component and dimension) against 152 SMs x 128 lanes x the
    measured SM clock."""
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300 import _native
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    decode = args.workload == "decode"
    if decode:
        w = DEC_WORKLOAD
        B, H, d_r, d_v, K = w["B"], w["H"], w["d_r"], w["d_v"], w["K"]
        g = torch.Generator().manual_seed(rank_seed(rank, 4))
        q, k, v = (torch.randn(B, H, d, generator=g).to(torch.bfloat16).to(dev) for d in (d_r, d_r, d_v))
        mu = torch.randn(H, K, d_r, generator=g).to(dev)
        s2 = (torch.nn.functional.softplus(torch.randn(H, K, d_r, generator=g) * 0.5 ** 0.5) + 1e-3).to(dev)
        lp = torch.log_softmax(torch.randn(H, K, generator=g), -1).to(dev)
        Vt = torch.randn(B, H, K, d_v, device=dev)
        Z = torch.rand(B, H, K, device=dev) * 100
        o = torch.empty(B, H, d_v, device=dev)
        ws = torch.empty(int(gma.load().gma_decode_workspace_size(H, d_r, K)), dtype=torch.uint8, device=dev)
        stages = _native.stage_names(_native.PATH_SIMT, 5)
        units = B * H
        alg = B * H * (3 * 2 * 64 + 2 * 4 * K * (d_v + 1) + 4 * d_v)
        kernel_stage = "step"

        def call(events=None):
            gma.decode_step(q, k, v, mu, s2, lp, Vt, Z, eps=w["eps"], out=o, workspace=ws)
    else:
        w = STAT_WORKLOAD
        B, H, N, d_r, K = w["B"], w["H"], w["N"], w["d_r"], w["K"]
        inp = make_inputs(Case("stats", False, B, H, N, d_r, 16, K, w["dtype"], routing="mixture", mu_std=3.0),
                          seed=rank_seed(rank, 5))
        X, mu, s2, lp = (inp[n].to(dev) for n in ("Q", "mu", "sigma2", "log_pi"))
        ws = torch.empty(int(gma.load().gma_routing_stats_workspace_size(B, H, N, d_r, K, _native.GMA_BF16)),
                         dtype=torch.uint8, device=dev)
        stages = _native.stage_names(_native.PATH_SIMT, 6)
        units = B * H * N
        kernel_stage = "rows"

        def call(events=None):
            gma.routing_stats(X, mu, s2, lp, want_z=True, workspace=ws)

    def call_ev(events):
        # the binding builds its options itself; stage events go through the C ABI call here
        import ctypes
        opt = _native.options(stage_events=events)
        lib = gma.load()
        vp = ctypes.c_void_p
        if decode:
            st = lib.gma_decode_step(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), _native.GMA_BF16,
                                     vp(mu.data_ptr()), vp(s2.data_ptr()), vp(lp.data_ptr()), float(w["eps"]),
                                     vp(Vt.data_ptr()), vp(Z.data_ptr()), vp(o.data_ptr()), B, H, d_r, d_v, K,
                                     ctypes.byref(opt), vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream))
        else:
            st = lib.gma_routing_stats(vp(X.data_ptr()), _native.GMA_BF16, vp(mu.data_ptr()), vp(s2.data_ptr()),
                                       vp(lp.data_ptr()), vp(usage.data_ptr()), vp(counts.data_ptr()),
                                       vp(zbuf.data_ptr()), vp(ent.data_ptr()), B, H, N, d_r, K, ctypes.byref(opt),
                                       vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream))
        if st != 0:
            raise gma.GmaError(st, "stage-event pass")

    if not decode:
        usage = torch.empty(B, H, K, device=dev)
        counts = torch.empty(B, H, K, dtype=torch.int32, device=dev)
        zbuf = torch.empty(B, H, N, dtype=torch.int32, device=dev)
        ent = torch.empty(B, H, device=dev)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0.record(stream)
        for _ in range(args.steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = job_ms(t0.elapsed_time(t1) / args.steps, world, dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    for s in range(args.steps):
        call_ev(ev[s])
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(ev[s][j].elapsed_time(ev[s][j + 1]) for s in range(args.steps))
                for j, name in enumerate(stages)}
    value = world * units / (ms / 1e3)
    clk = clocks.summary()
    kms = stage_ms[kernel_stage]
    if decode:
        peak, peak_src = measured_peaks()
        achieved = alg / (kms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": None, "kernel": f"decode:{kernel_stage}", "algorithmic_bytes": alg, "peak_source": peak_src}
    else:
        mhz = (clk or {}).get("sm_mhz") or 2070.0
        peak = 152 * 128 * mhz * 1e6 / 1e12
        ops = units * 3 * K * d_r
        achieved = ops / (kms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Top/s", "frac": achieved / peak,
                "traffic": None, "kernel": f"stats:{kernel_stage}", "algorithmic_ops": ops,
                "peak_source": "152 SMs x 128 fp32 lanes x median SM clock under load"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        if decode:
            pairs = 2048
            secs = _oracle_decode_sample(pairs)
            cpu = {"value": pairs / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{pairs} (b, h) decode steps of the workload's shape through the fp64 C oracle, "
                             f"{secs:.2f} s on one core"}
        else:
            heads = 8
            secs = sum(_oracle_stats_head(7 + i) for i in range(heads))
            cpu = {"value": heads * STAT_WORKLOAD["N"] / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{heads} heads of the workload (N=16384, d_r=K=32, peaked) through the fp64 C "
                             f"oracle, {secs:.2f} s on one core"}
    if rank == 0:
        if decode:
            cfg = {"workload": "GMA causal decode step, B=2048 sequences x H=8 heads, d_r=d_v=K=64, bf16 q/k/v, "
                               "fp32 carried state (per GPU)", **{k_: w[k_] for k_ in ("B", "H", "d_r", "d_v", "K")},
                   "l2": "state (272 MB) larger than L2, no flush"}
        else:
            cfg = {"workload": "GMA component-usage diagnostics (usage, hard assignments, usage entropy), B=16 H=4 "
                               "N=16384 d_r=K=32 bf16, peaked routing (per GPU)",
                   **{k_: w[k_] for k_ in ("B", "H", "N", "d_r", "K")},
                   "l2": "inputs (67 MB) smaller than L2, compute-bound: no flush"}
        cfg["parallelism"] = f"replicas x{world}"
        out = {"metric": DEC_METRIC if decode else STAT_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
               "gpu_launches": (2 if decode else 3) * args.steps, "roofline": roof, "stage_ms": stage_ms,
               "clocks": clk, "cpu_baseline": cpu}
        print(json.dumps(out), flush=True)




def time_configs(args, rank: int, dev) -> dict:
    """One forward of each configured workload (the small fp32 bidirectional,
    bidirectional N=4096, causal N=16384, peaked bidirectional N=16384, causal
    large-head N=32768 K=d=128), each on the kernel family the library selects
    for it, timed with CUDA events on the launching stream after 3 untimed
    calls: as many calls as fill about 0.3 s (at least 5).  Per workload:
    token*heads/s and the whole call's algorithmic bytes (Q, K, V read, O
    written; O credited at 4 B, the fp32 it is written in, and at 2 B, the
    metric's basis) against the measured HBM peak."""
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300 import _native
    from gaussian_mixture_latent_diag_gb300.synthetic import WORKLOADS, make_inputs

    stream = torch.cuda.current_stream()
    peak, _ = measured_peaks()
    per = {}
    for name, case in WORKLOADS.items():
        inp = make_inputs(case, seed=rank_seed(rank, 8))
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        fn = gma.forward_causal if case.causal else gma.forward_bidir
        out = torch.empty(case.B, case.H, case.N, case.d_v, device=dev)
        code = "f32" if case.dtype == "f32" else "bf16"
        ws = torch.empty(gma.workspace_size(case.B, case.H, case.N, case.d_r, case.d_v, case.K, code,
                                            int(case.causal)), dtype=torch.uint8, device=dev)

        def call():
            fn(d["Q"], d["K"], d["V"], d["mu"], d["sigma2"], d["log_pi"], eps=case.eps, out=out, workspace=ws)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        call()
        t1.record(stream)
        torch.cuda.synchronize()
        steps = max(5, min(2000, int(300.0 / max(t0.elapsed_time(t1), 1e-3))))
        t0.record(stream)
        for _ in range(steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        es = 4 if case.dtype == "f32" else 2
        alg = case.token_heads * (es * (2 * case.d_r + case.d_v) + 4 * case.d_v)
        alg2 = case.token_heads * (es * (2 * case.d_r + case.d_v) + es * case.d_v)
        path = gma.selected_path(case.N, case.d_r, case.d_v, case.K, code, int(case.causal))
        launches = len(_native.stage_names(path, int(case.causal))) * steps
        per[name] = {"ms": ms, "token_heads_per_s": case.token_heads / (ms / 1e3),
                     "hbm_frac": alg / (ms / 1e3) / 1e9 / peak,
                     "hbm_frac_o_input_dtype_basis": alg2 / (ms / 1e3) / 1e9 / peak,
                     "path": "tc" if path == gma.PATH_TC else "simt", "algorithmic_bytes": alg,
                     "timed_calls": steps, "stages_launched": launches}
        del d, out, ws
    return per


CFG_METRIC = "GMA fwd tokens*heads/s on each of the five configured workloads; % of GB300 HBM roofline"


def run_configs(args, rank: int, world: int, local_rank: int):
    """--workload configs: the five configured workloads (time_configs) as a line of their own."""
    import torch
    from gaussian_mixture_latent_diag_gb300.synthetic import WORKLOADS

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peak, peak_src = measured_peaks()
    with ClockSampler(local_rank) as clocks:
        per = time_configs(args, rank, dev)
    if rank == 0:
        total = sum(v["ms"] for v in per.values())
        units = sum(WORKLOADS[n].token_heads for n in per)
        out = {"metric": CFG_METRIC, "value": world * units / (total / 1e3), "unit": UNIT, "n_gpus": world,
               "steps": None, "warmup": 3, "ms_per_step": total, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": "one forward of each of the five configured workloads per step",
                          "l2": "inputs at or above L2 size except the small fp32 case; no flush",
                          "parallelism": f"replicas x{world}"},
               "gpu_launches": sum(v["stages_launched"] for v in per.values()), "per_config": per,
               "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s", "peak_source": peak_src,
                            "note": "per workload in per_config.hbm_frac (whole call)"},
               "clocks": clocks.summary()}
        print(json.dumps(out), flush=True)


SHAPE_METRIC = "GMA fwd tokens*heads/s on a given shape; % of GB300 HBM roofline"


def run_shape(args, rank: int, world: int, local_rank: int):
    """--workload shape: one forward call (--causal 0/1) of the shape given by
    --shape B,H,N,d_r,d_v,K (bf16 inputs drawn as the configured workloads,
    fp32 O) on the kernel family the library selects, timed over --steps calls
    after the warm-up, with the per-stage times of a second pass (stage events
    between the kernels).  For sizes the five configured workloads do not
    cover, and for profiling one kernel on a smaller case."""
    import ctypes
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300 import _native
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

    B, H, N, d_r, d_v, K = (int(x) for x in args.shape.split(","))
    causal = int(args.causal)
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = Case("shape", bool(causal), B, H, N, d_r, d_v, K, "bf16")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(case, seed=rank_seed(rank, 9)).items()}
    path = gma.selected_path(N, d_r, d_v, K, "bf16", causal)
    ws = torch.empty(max(256, gma.workspace_size(B, H, N, d_r, d_v, K, "bf16", causal)), dtype=torch.uint8, device=dev)
    O = torch.empty(B, H, N, d_v, device=dev)
    names = _native.stage_names(path, causal)
    stream = torch.cuda.current_stream()
    lib = gma.load()
    vp = ctypes.c_void_p
    fn = lib.gma_forward_causal if causal else lib.gma_forward_bidir

    def call(events=None):
        opt = _native.options(stage_events=events)
        st = fn(vp(d["Q"].data_ptr()), vp(d["K"].data_ptr()), vp(d["V"].data_ptr()), _native.GMA_BF16,
                vp(d["mu"].data_ptr()), vp(d["sigma2"].data_ptr()), vp(d["log_pi"].data_ptr()), float(case.eps),
                vp(O.data_ptr()), B, H, N, d_r, d_v, K, ctypes.byref(opt), vp(ws.data_ptr()), ws.numel(),
                vp(stream.cuda_stream))
        if st != 0:
            raise gma.GmaError(st, "forward")

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    peak, peak_src = measured_peaks()
    with ClockSampler(local_rank) as clocks:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = job_ms(t0.elapsed_time(t1) / args.steps, world, dev)
    stage = [0.0] * len(names)
    reps = min(args.steps, 10)
    for _ in range(reps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        call(ev)
        torch.cuda.synchronize()
        for j in range(len(names)):
            stage[j] += ev[j].elapsed_time(ev[j + 1]) / reps
    th = B * H * N
    alg = th * (2 * (2 * d_r + d_v) + 4 * d_v)
    if rank == 0:
        out = {"metric": SHAPE_METRIC, "value": world * th / (ms / 1e3), "unit": UNIT, "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": f"GMA {'causal' if causal else 'bidirectional'} forward, B={B} H={H} N={N} "
                                      f"d_r={d_r} d_v={d_v} K={K} bf16, fp32 O (per GPU)",
                          "parallelism": f"replicas x{world}"},
               "gpu_launches": len(names) * args.steps, "path": {1: "simt", 2: "tc"}.get(path, str(path)),
               "stage_ms": dict(zip(names, stage)),
               "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                            "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": None, "kernel": "whole call",
                            "algorithmic_bytes": alg, "peak_source": peak_src},
               "clocks": clocks.summary()}
        print(json.dumps(out), flush=True)


SHARD_METRIC = "GMA per-shard steps of sequence sharding token*heads/s (N=16K, K=64); % of GB300 HBM roofline"


def run_shard(args, rank: int, world: int, local_rank: int):
    """--workload shard: the three per-shard steps of a sequence sharded over N
    (gaussian_mixture_latent_diag_gb300.sharded), each timed on the headline
    shape (B=4, H=8, N=16384, d_r=d_v=K=64, bf16): gma_latent_memory (reads K, V),
    gma_read_memory (reads Q, writes fp32 O) and gma_forward_causal_carry (reads
    Q, K, V, writes fp32 O and the final state).  One step = the three calls,
    on the kernel family sharded.CudaOps picks for the shape: the tensor-core
    kernels here (Gamma never leaves the SM).  per_call_simt times the same
    calls on the CUDA-core kernels for comparison."""
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    w = WORKLOAD
    B, H, N, d_r, d_v, K = w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"]
    inp = make_inputs(Case("shard", True, B, H, N, d_r, d_v, K, w["dtype"]), seed=rank_seed(rank, 9))
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    prm = (d["mu"], d["sigma2"], d["log_pi"])
    Vt, Z = gma.latent_memory(d["K"], d["V"], *prm)
    O = torch.empty(B, H, N, d_v, device=dev)
    import ctypes
    from gaussian_mixture_latent_diag_gb300.sharded import CudaOps
    path = CudaOps._path(d["K"], d["V"], d["mu"])
    ws = {}

    def wsp(name, nbytes):  # one workspace per call, allocated outside the timed region
        if name not in ws:
            ws[name] = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        return ws[name]

    code = gma.GMA_BF16
    nb_lm = lambda pth: int(gma.load().gma_latent_memory_workspace_size(  # noqa: E731
        B, H, N, d_r, d_v, K, code, ctypes.byref(gma.options(path=pth))))
    nb_rd = int(gma.load().gma_read_memory_workspace_size(B, H, N, d_r, d_v, K, code))
    nb_cc = int(gma.load().gma_causal_carry_workspace_size(B, H, N, d_r, d_v, K, code))

    def calls_for(pth):
        return {
            "latent_memory": lambda: gma.latent_memory(d["K"], d["V"], *prm, path=pth,
                                                       workspace=wsp(f"lm{pth}", nb_lm(pth))),
            "read_memory": lambda: gma.read_memory(d["Q"], *prm, Vt, Z, eps=w["eps"], out=O, path=pth,
                                                   workspace=wsp("rd", nb_rd)),
            "causal_carry": lambda: gma.forward_causal_carry(d["Q"], d["K"], d["V"], *prm, Vt, Z, eps=w["eps"],
                                                             out=O, path=pth, workspace=wsp("cc", nb_cc)),
        }

    es = 2
    alg = {"latent_memory": B * H * N * es * (d_r + d_v), "read_memory": B * H * N * (es * d_r + 4 * d_v),
           "causal_carry": B * H * N * (es * (2 * d_r + d_v) + 4 * d_v)}
    peak, peak_src = measured_peaks()

    def time_calls(calls):
        per = {}
        for name, fn in calls.items():
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(args.steps):
                fn()
            t1.record(stream)
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1) / args.steps
            per[name] = {"ms": ms, "hbm_frac": alg[name] / (ms / 1e3) / 1e9 / peak, "algorithmic_bytes": alg[name]}
        return per

    with ClockSampler(local_rank) as clocks:
        per = time_calls(calls_for(path))
    per_simt = time_calls(calls_for(gma.PATH_SIMT)) if path != gma.PATH_SIMT else None
    tc = path == gma.PATH_TC
    if rank == 0:
        total = sum(v["ms"] for v in per.values())
        out = {"metric": SHARD_METRIC, "value": world * 3 * B * H * N / (total / 1e3), "unit": UNIT,
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic",
               "config": {"workload": "latent memory + read from it + carried-prefix causal forward, B=4 H=8 "
                                      "N=16384 d_r=d_v=K=64 bf16 (per GPU)", **{k: w[k] for k in ("B", "H", "N", "K")},
                          "l2": "inputs larger than L2, no flush", "parallelism": f"replicas x{world}"},
               "path": "tc" if tc else "simt",
               "gpu_launches": ((2 + 3 + 3) if tc else (4 + 4 + 6)) * args.steps, "per_call": per,
               "per_call_simt": per_simt,
               "roofline": {"bound": "hbm", "peak": peak, "unit": "GB/s", "peak_source": peak_src,
                            "achieved": sum(alg.values()) / (total / 1e3) / 1e9,
                            "frac": sum(alg.values()) / (total / 1e3) / 1e9 / peak, "traffic": None,
                            "kernel": "the three calls together (" + ("tensor-core kernels" if tc else
                                      "CUDA-core stages, Gamma materialised") + ")"},
               "clocks": clocks.summary()}
        print(json.dumps(out), flush=True)


PROJ_WORKLOAD = dict(B=4, N=16384, D=1024, H=8, d_r=64, d_v=64)
PROJ_METRIC = "GMA Q/K/V projection (Eq. 4) token/s (B=4 N=16K D=1024 -> H=8 x (64+64+64)); % of GB300 bf16 peak"


def run_project(args, rank: int, world: int, local_rank: int):
    """--workload project: one gma_project_qkv per step, X [4, 16384, 1024] bf16 and
    the three weights [512, 1024] bf16 to Q_X, K_X, V_X [4, 8, 16384, 64] bf16.
    Algorithmic work 2 * B N * D * H (2 d_r + d_v) = 206 GFLOP per call (a dense
    contraction: tensor-bound against the measured bf16 peak); algorithmic bytes
    X 128 MB + W 3 MB + outputs 192 MB."""
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    w = PROJ_WORKLOAD
    B, N, D, H, d_r, d_v = w["B"], w["N"], w["D"], w["H"], w["d_r"], w["d_v"]
    g = torch.Generator().manual_seed(rank_seed(rank, 7))
    X = torch.randn(B, N, D, generator=g).to(torch.bfloat16).to(dev)
    Ws = [(torch.randn(H * d, D, generator=g) / D ** 0.5).to(torch.bfloat16).to(dev) for d in (d_r, d_r, d_v)]
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    outs = []

    def call():
        outs.clear()
        outs.extend(gma.project_qkv(X, *Ws, H, workspace=ws))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0.record(stream)
        for _ in range(args.steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = job_ms(t0.elapsed_time(t1) / args.steps, world, dev)
    flops = 2.0 * B * N * D * H * (2 * d_r + d_v)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, src = float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        peak, src = 1900.0, "fallback"
    achieved = flops / (ms / 1e3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        rows = 256
        xs = X[0, :rows].float().cpu().numpy()[None]
        t = time.perf_counter()
        oracle.project_qkv(xs, *(W.float().cpu().numpy() for W in Ws), H)
        secs = time.perf_counter() - t
        cpu = {"value": rows / secs, "unit": "token/s", "cores": 1, "kind": "oracle",
               "sample": f"{rows} tokens of the workload through the fp64 C oracle, {secs:.2f} s on one core"}
    if rank == 0:
        out = {"metric": PROJ_METRIC, "value": world * B * N / (ms / 1e3), "unit": "token/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": "GMA Q/K/V projection, X [4, 16384, 1024] bf16 -> Q_X, K_X, V_X "
                                      "[4, 8, 16384, 64] bf16 (fp32 accumulation)", **w,
                          "l2": "X (128 MB) and outputs (192 MB) larger than L2, no flush",
                          "parallelism": f"replicas x{world}"},
               "gpu_launches": args.steps,
               "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                            "frac": achieved / peak, "traffic": None, "kernel": "proj_kernel",
                            "algorithmic_flops": flops, "peak_source": src},
               "clocks": clocks.summary(), "cpu_baseline": cpu}
        print(json.dumps(out), flush=True)


PARAM_WORKLOAD = dict(H=32, K=128, d_r=128)
PARAM_METRIC = "GMA parameter reparameterisation + its gradient, elements/s (H=32, K=128, d_r=128)"


def run_params(args, rank: int, world: int, local_rank: int):
    """--workload params: one gma_reparameterize and one gma_reparameterize_backward
    (Eqs. 14-15 and their chain rule) per step over the largest parameter shape of
    the workloads (H=32, K=d_r=128: 524288 covariance elements).  Algorithmic bytes
    per covariance element: omega read and sigma2 written (8), then omega and
    dsigma2 read and domega written (12) = 20 B; the priors are K per head.  The
    two launches are latency-bound at this size."""
    import torch
    import gaussian_mixture_latent_diag_gb300 as gma

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    w = PARAM_WORKLOAD
    H, K, d_r = w["H"], w["K"], w["d_r"]
    g = torch.Generator().manual_seed(rank_seed(rank, 6))
    omega = torch.randn(H, K, d_r, generator=g).to(dev)
    alpha = torch.randn(H, K, generator=g).to(dev)
    ds2 = torch.randn(H, K, d_r, generator=g).to(dev)
    dlp = torch.randn(H, K, generator=g).to(dev)
    s2, lp = torch.empty_like(omega), torch.empty_like(alpha)
    dw, da = torch.empty_like(omega), torch.empty_like(alpha)
    lib = gma.load()
    import ctypes
    vp = ctypes.c_void_p

    def launch(strm):
        st = lib.gma_reparameterize(vp(omega.data_ptr()), vp(alpha.data_ptr()), H, K, d_r, 1e-3, vp(s2.data_ptr()),
                                    vp(lp.data_ptr()), vp(strm.cuda_stream))
        st |= lib.gma_reparameterize_backward(vp(omega.data_ptr()), vp(alpha.data_ptr()), vp(ds2.data_ptr()),
                                              vp(dlp.data_ptr()), H, K, d_r, vp(dw.data_ptr()), vp(da.data_ptr()),
                                              vp(strm.cuda_stream))
        if st != 0:
            raise gma.GmaError(st, "gma_reparameterize")

    # the two launches are a few microseconds each: replaying them from a CUDA
    # graph keeps the host's call overhead out of the measurement
    for _ in range(args.warmup):
        launch(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launch(torch.cuda.current_stream())

    def call():
        graph.replay()

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0.record(stream)
        for _ in range(args.steps):
            call()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = job_ms(t0.elapsed_time(t1) / args.steps, world, dev)
    units = H * K * d_r
    alg = units * 20 + H * K * 4 * 5
    peak, peak_src = measured_peaks()
    achieved = alg / (ms / 1e3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np
        import oracle
        oracle.build()
        o_np, a_np, d_np, l_np = (t.double().cpu().numpy() for t in (omega, alpha, ds2, dlp))
        t = time.perf_counter()
        oracle.reparameterize(o_np, a_np, 1e-3)
        oracle.reparameterize_backward(o_np, a_np, d_np, l_np)
        secs = time.perf_counter() - t
        cpu = {"value": units / secs, "unit": "elements/s", "cores": 1, "kind": "oracle",
               "sample": f"the whole parameter set (H=32, K=d_r=128) through the fp64 C oracle, {secs:.3f} s"}
    if rank == 0:
        out = {"metric": PARAM_METRIC, "value": world * units / (ms / 1e3), "unit": "elements/s", "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
               "config": {"workload": "GMA reparameterisation (Eqs. 14-15) forward + gradient, H=32 K=128 d_r=128",
                          **w, "l2": "2 MB parameter set, L2-resident (latency-bound launches)",
                          "launch": "both C-ABI calls captured once in a CUDA graph, replayed each step",
                          "parallelism": f"replicas x{world}"},
               "gpu_launches": 2 * args.steps,
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                            "frac": achieved / peak, "traffic": None, "kernel": "both launches",
                            "algorithmic_bytes": alg, "peak_source": peak_src},
               "clocks": clocks.summary(), "cpu_baseline": cpu}
        print(json.dumps(out), flush=True)


def rank_seed(rank: int, variant: int) -> int:
    """Input seed of one variant on one rank: each rank draws its own heads (replicas
    of the workload shape, no data shared between ranks)."""
    return 1000 * rank + variant


def job_ms(ms: float, world: int, device=None) -> float:
    """Step time of the whole job: the slowest rank's, every rank holding the same work."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ms: float, world: int, w=WORKLOAD) -> float:
    """token*heads/s of the whole job: per step every rank runs one bidirectional and
    one causal forward of the workload."""
    return world * 2 * w["B"] * w["H"] * w["N"] / (ms / 1e3)


def run_gma(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    import gaussian_mixture_latent_diag_gb300 as gma
    from gaussian_mixture_latent_diag_gb300 import _native
    from gaussian_mixture_latent_diag_gb300.synthetic import Case, make_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOAD
    cases = [Case("bidir", False, w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"], w["dtype"]),
             Case("causal", True, w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"], w["dtype"])]
    host = [make_inputs(c, seed=rank_seed(rank, i)) for i, c in enumerate(cases)]
    dinp = [{k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in h.items()} for h in host]
    outs = [torch.empty(w["B"], w["H"], w["N"], w["d_v"], dtype=torch.float32, device=dev) for _ in cases]
    paths = [gma.selected_path(w["N"], w["d_r"], w["d_v"], w["K"], w["dtype"], int(c.causal)) for c in cases]
    wss = [torch.empty(max(256, gma.workspace_size(w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"],
                                                   w["dtype"], int(c.causal))), dtype=torch.uint8, device=dev)
           for c in cases]
    stages = [_native.stage_names(p, int(c.causal)) for p, c in zip(paths, cases)]
    stream = torch.cuda.current_stream()
    lib = gma.load()

    ws1 = torch.empty(max(256, gma.workspace_size(w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"], w["dtype"], 1,
                                                  path=gma.PATH_TC_SINGLE_PASS)), dtype=torch.uint8, device=dev)

    def call(i, O=None, events=None, d=None, path=gma.PATH_AUTO):
        c = cases[i]
        d = dinp[i] if d is None else d
        fn = "gma_forward_causal" if c.causal else "gma_forward_bidir"
        opt = _native.options(stage_events=events, path=path)
        ws = ws1 if path == gma.PATH_TC_SINGLE_PASS else wss[i]
        import ctypes
        vp = ctypes.c_void_p
        st = getattr(lib, fn)(vp(d["Q"].data_ptr()), vp(d["K"].data_ptr()), vp(d["V"].data_ptr()),
                              _native.GMA_BF16, vp(d["mu"].data_ptr()), vp(d["sigma2"].data_ptr()),
                              vp(d["log_pi"].data_ptr()), float(w["eps"]),
                              vp((O if O is not None else outs[i]).data_ptr()),
                              w["B"], w["H"], w["N"], w["d_r"], w["d_v"], w["K"], ctypes.byref(opt),
                              vp(ws.data_ptr()), ws.numel(), vp(stream.cuda_stream))
        if st != 0:
            raise gma.GmaError(st, fn)

    for _ in range(args.warmup):
        call(0); call(1)
    torch.cuda.synchronize()
    if args.steps is None:  # enough steps for >= 1.2 s of device time (the clock sampler sees the run)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(20):
            call(0); call(1)
        c1.record(stream)
        torch.cuda.synchronize()
        est = c0.elapsed_time(c1) / 20
        steps = max(20, int(1200.0 / max(est, 1e-3)) + 1)
        if world > 1:  # every rank times the same number of steps
            t = torch.tensor([steps], dtype=torch.int64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            steps = int(t.item())
        args.steps = steps
    if world > 1:
        dist.barrier()

    # stage events: one list per (step, variant) of the breakdown pass
    nst = [len(s) + 1 for s in stages]
    nbreak = min(args.steps, 40)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(nst[i])] for i in range(2)]
          for _ in range(nbreak)]

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0.record(stream)
        for s in range(args.steps):
            call(0)
            call(1)
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps

    # per-stage breakdown: the same steps again with the library's stage events
    # (events between the kernels keep a kernel from starting before the previous
    # one ends, so they are kept out of the timed loop above)
    for s in range(nbreak):
        call(0, events=ev[s][0])
        call(1, events=ev[s][1])
    torch.cuda.synchronize()
    ms = job_ms(ms, world, dev)
    value = job_throughput(ms, world)

    # per-stage averages over the breakdown pass
    stage_ms = {}
    for i in range(2):
        for j, name in enumerate(stages[i]):
            key = f"{'causal' if cases[i].causal else 'bidir'}:{name}"
            stage_ms[key] = statistics.mean(ev[s][i][j].elapsed_time(ev[s][i][j + 1]) for s in range(nbreak))
    variant_ms = {("causal" if c.causal else "bidir"): statistics.mean(
        ev[s][i][0].elapsed_time(ev[s][i][-1]) for s in range(nbreak)) for i, c in enumerate(cases)}
    peak, peak_src = measured_peaks()
    dom = max(stage_ms, key=stage_ms.get)
    dom_stage = dom.split(":", 1)[1]
    dom_bytes = tensor_bytes(STAGE_TENSORS.get(dom_stage, ""))
    achieved = dom_bytes / (stage_ms[dom] / 1e3) / 1e9
    traffic = recorded_traffic(dom)
    dom_bytes_o2 = tensor_bytes(STAGE_TENSORS.get(dom_stage, ""), o_bytes=2)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "algorithmic_bytes": dom_bytes, "peak_source": peak_src,
                "o_bytes": 4,
                "frac_o_bf16_basis": dom_bytes_o2 / (stage_ms[dom] / 1e3) / 1e9 / peak,
                "note": "achieved / frac credit O at 4 B per element (the fp32 O the kernel writes); "
                        "frac_o_bf16_basis credits O at 2 B, the byte count of the metric's definition"}
    fwd_bytes, fwd_bytes_o2 = tensor_bytes("QKVO"), tensor_bytes("QKVO", o_bytes=2)
    variants = {k: {"ms": v, "token_heads_per_s": w["B"] * w["H"] * w["N"] / (v / 1e3),
                    "hbm_frac_of_" + peak_src: fwd_bytes / (v / 1e3) / 1e9 / peak,
                    "hbm_frac_o_bf16_basis": fwd_bytes_o2 / (v / 1e3) / 1e9 / peak,
                    "path": "tc" if paths[i] == gma.PATH_TC else "simt"}
                for i, (k, v) in enumerate(variant_ms.items())}
    # the single-pass causal kernel (GMA_PATH_TC_SINGLE_PASS), timed on its own; not part of the step
    if gma.selected_path(w["N"], w["d_r"], w["d_v"], w["K"], w["dtype"], 1, path=gma.PATH_TC_SINGLE_PASS) == \
            gma.PATH_TC_SINGLE_PASS:
        for _ in range(3):
            call(1, path=gma.PATH_TC_SINGLE_PASS)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 40
        s0.record(stream)
        for _ in range(reps):
            call(1, path=gma.PATH_TC_SINGLE_PASS)
        s1.record(stream)
        torch.cuda.synchronize()
        v = s0.elapsed_time(s1) / reps
        variants["causal_single_pass"] = {
            "ms": v, "token_heads_per_s": w["B"] * w["H"] * w["N"] / (v / 1e3),
            "hbm_frac_of_" + peak_src: fwd_bytes / (v / 1e3) / 1e9 / peak,
            "hbm_frac_o_bf16_basis": fwd_bytes_o2 / (v / 1e3) / 1e9 / peak, "path": "tc_single_pass",
            "note": "GMA_PATH_TC_SINGLE_PASS (Gamma^K kept on chip, one kernel after the prep); timed alone, "
                    "not part of the step"}

    # end to end through the public API: pinned host inputs; every step copies its inputs up and
    # its outputs down inside the timed region.  Host-to-device and device-to-host copies run on
    # their own streams and the device buffers are double-buffered across steps, so a step's
    # inputs travel while the previous step computes and its outputs return.
    pinned = [{k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in h.items()} for h in host]
    host_out = [torch.empty_like(o, device="cpu").pin_memory() for o in outs]
    h2d = sum(pinned[i][k].numel() * pinned[i][k].element_size() for i in range(2) for k in ("Q", "K", "V"))
    d2h = sum(o.numel() * o.element_size() for o in outs)
    dbuf = [dinp, [{k: (torch.empty_like(v) if isinstance(v, torch.Tensor) and k in ("Q", "K", "V") else v)
                    for k, v in d.items()} for d in dinp]]
    obuf = [outs, [torch.empty_like(o) for o in outs]]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]                          # inputs of set b on the device
    ev_read = [torch.cuda.Event() for _ in range(2)]                        # compute done with inputs of set b
    ev_done = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]    # output i of set b written
    ev_out = [torch.cuda.Event() for _ in range(2)]                         # outputs of set b copied out

    def e2e_step(j, start=None):
        b = j % 2
        with torch.cuda.stream(s_in):
            if start is not None:
                s_in.wait_event(start)
            s_in.wait_event(ev_read[b])
            for i in range(2):
                for k in ("Q", "K", "V"):
                    dbuf[b][i][k].copy_(pinned[i][k], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])
        for i in range(2):
            call(i, O=obuf[b][i], d=dbuf[b][i])
            ev_done[b][i].record(stream)
        ev_read[b].record(stream)
        with torch.cuda.stream(s_out):
            for i in range(2):
                s_out.wait_event(ev_done[b][i])
                host_out[i].copy_(obuf[b][i], non_blocking=True)
            ev_out[b].record(s_out)

    for j in range(max(2, args.warmup)):
        e2e_step(j)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the end-to-end leg is bound by the host link (milliseconds per step): it times as
    # many of the K steps as fill about 1.2 s, at least 20
    w0 = time.perf_counter()
    for j in range(4):
        e2e_step(j)
    torch.cuda.synchronize()
    e2e_est = (time.perf_counter() - w0) / 4
    e2e_steps = min(args.steps, max(20, int(1.2 / max(e2e_est, 1e-6)) + 1))
    if world > 1:
        t = torch.tensor([e2e_steps], dtype=torch.int64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_steps = int(t.item())
    e0.record(stream)
    for j in range(e2e_steps):
        e2e_step(j, start=e0 if j == 0 else None)
    stream.wait_event(ev_out[0])
    stream.wait_event(ev_out[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / e2e_steps
    e_ms = job_ms(e_ms, world, dev)
    e2e = {"value": job_throughput(e_ms, world), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "steps": e2e_steps,
           "schedule": "H2D and D2H on their own streams, device buffers double-buffered across steps"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        procs = host_cores()
        pairs = procs
        pool = OraclePool(procs)
        wall, th = pool.sample(pairs)
        pool.close()
        cpu = {"value": th / wall, "unit": UNIT, "cores": procs, "cpu_model": host_cpu_model(), "kind": "oracle",
               "sample": f"{pairs} bidirectional + {pairs} causal heads of N=16384, d=K=64 "
                         f"(fp64 C oracle, one spawned process per host core: {procs})"}

    per_config = time_configs(args, rank, dev) if not args.no_configs else None

    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": "GMA forward, bidirectional + causal, B=4 H=8 N=16384 "
                                      "d_r=d_v=K=64 bf16 (per GPU)",
                          "global_batch": world * w["B"], "seq_len": w["N"], "heads": w["H"],
                          "d_r": w["d_r"], "d_v": w["d_v"], "K": w["K"], "eps": w["eps"],
                          "l2": "inputs larger than L2 (201 MB read + 134 MB written per variant), no flush",
                          "output": "fp32 O",
                          "parallelism": f"replicas x{world}"},
               "gpu_launches": args.steps * sum(len([n for n in s if n != "reset"]) for s in stages),
               "roofline": roofline, "variants": variants, "stage_ms": stage_ms,
               "stage_note": "stage_ms / variants come from a second pass with stage events between the "
                             "kernels, which keep each kernel from starting before the previous one ends; "
                             "the timed loop has no events, so its step is shorter than their sum",
               "clocks": clocks.summary(), "e2e": e2e, "cpu_baseline": cpu, "configs": per_config}
        print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: as many as fill at least 1.2 s of device time)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gma", "reference"], default="gma")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave out the per-workload timings of the five configured workloads")
    ap.add_argument("--workload", choices=["forward", "backward", "decode", "stats", "params", "project",
                                           "configs", "shard", "shape"],
                    default="forward",
                    help="forward: the bidirectional + causal forward step (default); "
                         "backward: the bidirectional + causal backward; decode: one causal decode "
                         "step over B=2048 x H=8 carried states; stats: the component-usage diagnostics; "
                         "params: the reparameterisation and its gradient; project: the Q/K/V projections; "
                         "configs: each of the five configured workloads; shard: the per-shard steps of "
                         "sequence sharding; shape: one forward of --shape (B,H,N,d_r,d_v,K) --causal 0/1")
    ap.add_argument("--shape", default="1,8,32768,128,128,128", help="B,H,N,d_r,d_v,K of --workload shape")
    ap.add_argument("--causal", type=int, default=1, choices=[0, 1], help="direction of --workload shape")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.steps is None and args.workload != "forward":
        args.steps = 20  # the other legs time a fixed number of calls
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        if args.workload == "backward":
            run_backward(args, rank, world, local_rank)
        elif args.workload in ("decode", "stats"):
            run_aux(args, rank, world, local_rank)
        elif args.workload == "params":
            run_params(args, rank, world, local_rank)
        elif args.workload == "project":
            run_project(args, rank, world, local_rank)
        elif args.workload == "configs":
            run_configs(args, rank, world, local_rank)
        elif args.workload == "shard":
            run_shard(args, rank, world, local_rank)
        elif args.workload == "shape":
            run_shape(args, rank, world, local_rank)
        else:
            run_gma(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
