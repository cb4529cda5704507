#!/usr/bin/env python
"""Benchmark of the single-GPU collective datapath.

Default workload (one step = one all-reduce through the whole datapath:
stage as LL128 lines, validate + fold the partitions at their owners,
publish, validate + unpack at every rank):
    8 emulated ranks, 256 MiB of bf16 per rank (uniform[-4, 4], seeded),
    LL128 sequence-number lines, twoshot, one composed launch in which
    each CTA runs the stage, fold + publish and gather of one chunk of a
    partition at a time (``--path streamed``: the three stream-ordered
    launches).
The inputs (2 GiB) and staging (4.8 GiB) exceed the 126 MiB L2, so no L2
flush is needed between steps.

value = algorithmic bytes of one all-reduce / device time per step (GB/s),
summed over replicas for --gpus N (one independent replica per GPU: the
single-GPU emulation does not shard across GPUs).

The same JSON line carries the roofline of the dominant kernel (per-launch
CUDA events around each kernel of every timed step, with the DRAM-side rate
from the committed ncu traffic figure), the end-to-end number from pinned
host buffers, ``rows`` for the other collectives and paths (streamed
all-reduce, reduce-scatter, all-gather, all-to-all, MoE dispatch, the V
collectives, sentinel packs, fp32, bounded staging, and the pipeline-depth
ablation of the one-sided copy), the small-message latency sweep (8 ranks x
[T x 4096] bf16; warm = 128 ops per CUDA graph, cold = L2 flushed before
every op) and the CPU oracle timed on a bounded sample.  ``--impl
reference`` times the CPU oracle instead; ``--row``, ``--sweep-only`` and
``--atom-only`` run one part alone (profiling runs).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("all-reduce µs/op (1 KB–1 MB) and HBM GB/s vs 8 TB/s peak, "
          "N=8 emulated ranks")
N_RANKS = 8
EPS_LL128 = 128.0 / 120.0
EPS_LL8 = 2.0
L2_BYTES = 126.5 * 2**20


# ---- algorithmic bytes (per op, whole job of one GPU) ------------------------------

def bytes_allreduce_twoshot(n: int, s: float, eps: float) -> float:
    """stage NS read + NS*eps write; owners read NS*eps, publish S*eps; every
    rank reads N*S*eps lines and writes S."""
    return 2 * n * s + (3 * n + 1) * s * eps


def kernel_bytes_allreduce_twoshot(n: int, s: float, eps: float) -> list[float]:
    return [n * s + n * s * eps,          # stage
            n * s * eps + s * eps,        # reduce-scatter + publish
            n * s * eps + n * s]          # all-gather copy


def kernel_floor_bytes_allreduce_twoshot(n: int, s: float, eps: float) -> list[float]:
    """DRAM bytes each stream-ordered launch cannot avoid: the stage reads the
    inputs and writes the lines (the next launch reads them from HBM); the
    fold reads every rank's lines of its partition and publishes; the gather
    reads each published line once from HBM (its N readers share L2) and
    writes the outputs."""
    return [n * s + n * s * eps, n * s * eps + s * eps, s * eps + n * s]


def unique_bytes_allreduce(n: int, s: float) -> float:
    """DRAM floor of a one-launch all-reduce: every input read once, every
    output written once (staged and published lines never leave L2)."""
    return 2 * n * s


def bytes_allreduce_oneshot(n: int, s: float, eps: float) -> float:
    return 2 * n * s + n * s * eps + n * n * s * eps


def bytes_reduce_scatter(n: int, s: float, eps: float) -> float:
    return (n + 1) * s + 2 * n * s * eps


def bytes_all_gather(n: int, s: float, eps: float) -> float:
    """s = gathered output per rank; every rank contributes s / n."""
    return (n + 1) * s * (1 + eps)


# ---- helpers -----------------------------------------------------------------------

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d.get("hbm_gbs", 6800.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def l2_copy_peak(cd, stream) -> dict:
    """Copy throughput of buffers that stay in L2 (read + write bytes per
    second), the denominator of the issue-level figure, whose bytes are
    mostly served by L2.  The library's copy probe (coll_copy_passes: 64
    copies of a 16 MiB buffer into another in ONE launch, 16-byte accesses,
    4 or 8 CTAs per SM; source and destination, 32 MiB, stay in L2), best
    of 5 launches timed with CUDA events on `stream`.  torch's b.copy_(a) of
    the same buffers (a device-to-device cudaMemcpyAsync on a copy engine,
    one launch per copy) is recorded beside it."""
    import torch

    nbytes, passes = 16 << 20, 64
    a = torch.ones(nbytes // 2, dtype=torch.int16, device="cuda")
    b = torch.empty_like(a)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    res = {}
    with torch.cuda.stream(stream):
        for per_sm in (4, 8):
            op = lambda c=per_sm * sms: cd.coll_copy_passes(  # noqa: E731
                b, a, nbytes, passes, ctas=c, stream=stream)
            op()
            best = 0.0
            for _ in range(5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                op()
                e1.record(stream)
                stream.synchronize()
                best = max(best, 2 * nbytes * passes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
            res[f"coll_copy_passes, {per_sm * sms} CTAs, {passes} passes"] = round(best, 1)
        for _ in range(20):
            b.copy_(a)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(200):
            b.copy_(a)
        e1.record(stream)
        stream.synchronize()
        res["torch copy_ (copy engine, one launch per copy)"] = round(
            2 * nbytes * 200 / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    del a, b
    best = max(res, key=res.get)
    return {"gbs": res[best], "how": f"{best}: 16 MiB copied into another 16 MiB buffer (32 MiB "
                                     f"resident in L2), read + write bytes / CUDA-event time, "
                                     f"best of 5, measured in this run",
            "candidates": res}


class Clocks:
    """nvidia-smi sampler around the timed region (200 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier_max(value: float, world: int) -> float:
    """Max of a per-rank number over ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, bytes_per_replica: float, ms_max: float) -> float:
    """Whole-job GB/s: every replica moves the same bytes; the job takes the
    slowest replica's time."""
    return world * bytes_per_replica / (ms_max * 1e-3) / 1e9


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---- CPU baseline (the oracle, as it stands) ----------------------------------------

def host_cpu() -> dict:
    """The host's CPU model and logical core count (the oracle uses one)."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and not model:
                    model = ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return {"machine": platform.machine(), "model": model or platform.processor(),
            "nproc": os.cpu_count()}


def cpu_oracle_allreduce(per_rank_mib: int, seed: int = 4, runs: int = 1) -> dict:
    import oracle
    import synth

    count = per_rank_mib * 2**20 // 2
    xs = [synth.uniform_bf16(seed, count, -4.0, 4.0, 99, r) for r in range(N_RANKS)]
    times = []
    for _ in range(runs):
        t0 = time.perf_counter()
        oracle.allreduce(xs)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    s = count * 2.0
    gbs = bytes_allreduce_twoshot(N_RANKS, s, EPS_LL128) / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 3), "host": host_cpu(),
            "sample": f"all-reduce of {N_RANKS} ranks x {per_rank_mib} MiB bf16 by the "
                      f"plain C oracle (single thread), median of {runs} run(s); GB/s "
                      f"counted with the same algorithmic bytes as the GPU line"}


def _median_runs(fn, max_runs: int = 101, budget_s: float = 2.0, min_runs: int = 5) -> dict:
    """Median wall time of up to `max_runs` calls of fn (at least `min_runs`,
    stopping early once `budget_s` seconds have been spent)."""
    times = []
    t_start = time.perf_counter()
    while len(times) < max_runs:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
        if len(times) >= min_runs and time.perf_counter() - t_start > budget_s:
            break
    return {"median_s": statistics.median(times), "runs": len(times)}


def cpu_oracle_configs() -> dict:
    """The plain C oracle (single thread, called through ctypes, timed with
    time.perf_counter around each call) beside the small configurations:
    c1 (2 ranks x 512 bf16, one all-reduce), the decode-time sweep (8 ranks x
    [T x 4096] and 1 / 2 / 4 KiB per rank; all 8 output copies, as the GPU
    op writes them) and c3 (one epoch of 8 ranks x [16 x 7168]: the oracle's
    result for an epoch is the all-reduce of the published inputs).  Median
    of up to 101 runs per size, bounded at 2 s of runs per size."""
    import oracle
    import synth

    out = {}
    xs = [synth.uniform_bf16(0, 512, -1.0, 1.0, 1, r) for r in range(2)]
    m = _median_runs(lambda: oracle.allreduce(xs))
    out["c1_allreduce_2x512"] = {"us_per_op": round(m["median_s"] * 1e6, 2), "runs": m["runs"]}
    sweep = {}
    sizes = [(f"{kib}KiB", kib * 512) for kib in (1, 2, 4)]
    sizes += [(f"T={T}", T * 4096) for T in (1, 2, 4, 8, 16, 32, 64, 128)]
    for key, count in sizes:
        xs = [synth.normal_bf16(7, count, 0, r) for r in range(N_RANKS)]
        m = _median_runs(lambda: oracle.allreduce(xs))
        sweep[key] = {"bytes_per_rank": count * 2, "us_per_op": round(m["median_s"] * 1e6, 2),
                      "runs": m["runs"]}
    out["c2_allreduce_8x_Tx4096"] = sweep
    xs = [synth.normal_bf16(3, 16 * 7168, 1, r) for r in range(N_RANKS)]
    m = _median_runs(lambda: oracle.allreduce(xs))
    out["c3_epoch_allreduce_8x16x7168"] = {"us_per_op": round(m["median_s"] * 1e6, 2),
                                           "runs": m["runs"]}
    return out


def cpu_oracle_moe(ins_host, topk_host, experts: int) -> dict:
    """c5: the oracle's MoE dispatch of the bench's own inputs and routing,
    median of 3 runs (the first also touches the output pages)."""
    import oracle

    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        outs, _, _ = oracle.moe_dispatch(ins_host, topk_host, experts)
        times.append(time.perf_counter() - t0)
        del outs
    return {"s_per_op": round(statistics.median(times), 3),
            "runs_s": [round(t, 3) for t in times]}


def workload_config(mib: int, path: str, world: int) -> dict:
    """The bench workload, named the same way by both arms."""
    return {"workload": f"all-reduce, {N_RANKS} emulated ranks, {mib} MiB bf16 per rank, "
                        f"LL128 lines, twoshot (bandwidth regime)",
            "n_ranks": N_RANKS, "per_rank_mib": mib, "encoding": "LL128",
            "algorithm": "twoshot", "path": path, "parallelism": f"replicas{world}",
            "l2": _l2_note(N_RANKS * mib * 2**20)}


def _l2_note(input_bytes: int) -> str:
    """How the step treats L2: inputs (and the staging, at least as large)
    far larger than L2 need no flush; smaller ones are timed warm."""
    size = (f"{input_bytes / 2**30:g} GiB" if input_bytes >= 2**30
            else f"{input_bytes / 2**20:g} MiB")
    if input_bytes > 2 * L2_BYTES:
        return f"inputs ({size}) and staging larger than L2; no flush"
    return f"inputs ({size}) within twice L2: not flushed between steps (timed warm)"


def run_reference(args) -> int:
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    per_rank_mib = 8
    times = []
    for i in range(args.warmup + args.steps):
        r = cpu_oracle_allreduce(per_rank_mib, seed=100 + i)
        if i >= args.warmup:
            times.append(r["seconds"])
    sec = sum(times) / len(times)
    s = per_rank_mib * 2**20
    value = bytes_allreduce_twoshot(N_RANKS, s, EPS_LL128) / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args.mib, args.path, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "host": host_cpu(),
                         "sample": f"each step: the plain C oracle (single thread) on a "
                                   f"bounded sample of the workload, {N_RANKS} ranks x "
                                   f"{per_rank_mib} MiB bf16 instead of {args.mib} MiB; GB/s "
                                   f"counted with the same algorithmic bytes per element"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---- GPU measurements ---------------------------------------------------------------

def make_inputs(count: int, seed: int):
    """Seeded uniform[-4, 4] bf16 inputs, one per rank, drawn on the device;
    returns once they are written (they are drawn on torch's current stream,
    the collectives run on another)."""
    import torch

    xs = []
    for r in range(N_RANKS):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed * 1000 + r)
        u = torch.rand(count, generator=g, device="cuda", dtype=torch.float32)
        xs.append((u * 8.0 - 4.0).to(torch.bfloat16).view(torch.int16))
    torch.cuda.synchronize()
    return xs


def timed(step, k: int, w: int, stream, world: int) -> float:
    """ms for k steps after w warm-up steps (CUDA events on `stream`)."""
    import torch

    for i in range(w):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(k):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1)


def graph_us_per_op(g, stream) -> float:
    """Purlin's method for a captured graph of 128 ops: one warm-up replay,
    then 8 timed replays per measurement (CUDA events on `stream`), per op;
    the median of 5 such measurements, in microseconds."""
    import torch

    g.replay()
    reps = []
    for _ in range(5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(8):
            g.replay()
        e1.record(stream)
        stream.synchronize()
        reps.append(e0.elapsed_time(e1) * 1e3 / 1024)
    return statistics.median(reps)


def latency_sweep(cd, stream, only_T=None, only_variant=None, encoding=None) -> dict:
    """8 ranks x [T x 4096] bf16, LL8 (config of the decode-time sweep), or
    another readiness encoding; ahead of it 1, 2 and 4 KiB per rank, the
    low end of the all-reduce latency metric (1 KB - 1 MB).  A given T
    (--sweep-T) runs that size alone."""
    import torch

    enc = cd.COLL_LL8 if encoding is None else encoding

    out = {}
    flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device="cuda")
    sizes = [(f"{kib}KiB", kib * 512, 3 + kib) for kib in (1, 2, 4)]
    sizes += [(f"T={T}", T * 4096, 7 + T) for T in (1, 2, 4, 8, 16, 32, 64, 128)]
    for key, count, seed in sizes:
        if only_T is not None and key != f"T={only_T}":
            continue
        row = {}
        for algo, path, name in ((cd.COLL_ONESHOT, cd.COLL_PATH_FUSED, "oneshot_fused"),
                                 (cd.COLL_ONESHOT, cd.COLL_PATH_STREAMED, "oneshot_streamed"),
                                 (cd.COLL_TWOSHOT, cd.COLL_PATH_FUSED, "twoshot_fused"),
                                 (cd.COLL_TWOSHOT, cd.COLL_PATH_STREAMED, "twoshot_streamed"),
                                 (cd.COLL_ALGO_AUTO, cd.COLL_PATH_AUTO, "policy")):
            if only_variant is not None and name != only_variant:
                continue
            # "policy": encoding, algorithm and path from the calibrated table
            coll = cd.Collective(cd.ALLREDUCE, N_RANKS, count,
                                 encoding=cd.COLL_ENC_AUTO if name == "policy" else enc,
                                 algorithm=algo, path=path)
            ins = make_inputs(count, seed)
            outs = [torch.empty(count, dtype=torch.int16, device="cuda")
                    for _ in range(N_RANKS)]
            with torch.cuda.stream(stream):
                for _ in range(3):
                    coll.run(ins, outs, stream)
                # warm: 128 ops per graph, 1 warm-up replay, 8 timed replays
                g = torch.cuda.CUDAGraph()
                stream.synchronize()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(128):
                        coll.run(ins, outs, stream)
                warm = graph_us_per_op(g, stream)
                # the launch floor: an empty kernel in this run's one-launch
                # configuration, timed the same way (flash-comm Appendix A)
                floor = None
                pl = coll.plan()
                if pl["path"] in (cd.COLL_PATH_FUSED, cd.COLL_PATH_COMPOSED):
                    gf = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gf, stream=stream):
                        for _ in range(128):
                            cd.coll_launch_floor(coll.spec, stream)
                    floor = graph_us_per_op(gf, stream)
                    del gf
                # cold: L2 flushed (2x L2 written) before each op
                evs = []
                for _ in range(32):
                    flush.fill_(1)
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    coll.run(ins, outs, stream)
                    b.record(stream)
                    evs.append((a, b))
                stream.synchronize()
                cold = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)
            st = coll.status(stream)
            row[name] = {"warm_us": round(warm, 3), "cold_us": round(cold, 3),
                         "status": st[0]}
            if floor is not None:
                row[name]["floor_us"] = round(floor, 3)
                row[name]["excess_us"] = round(warm - floor, 3)
                row[name]["launch"] = ({"ctas": pl["ctas_per_rank"] * N_RANKS}
                                       if pl["path"] == cd.COLL_PATH_FUSED else
                                       {"columns": "composed"})
                row[name]["launch"]["dependent"] = pl["dependent_launch"]
            if name == "policy":
                row[name]["choice"] = {"encoding": pl["encoding"], "algorithm": pl["algorithm"],
                                       "path": pl["path"]}
            coll.close()
            del coll, ins, outs, g
        out[key] = {"bytes_per_rank": count * 2, **row}
    del flush
    torch.cuda.empty_cache()
    return out


def bandwidth_row(cd, triple, count_in_out, kind, stream, steps=5, path=None) -> dict:
    import torch

    n = N_RANKS
    count = count_in_out
    extra = {"algorithm": cd.COLL_TWOSHOT} if kind == "ar" else {}
    coll = cd.Collective(triple, n, count, encoding=cd.COLL_LL128,
                         path=cd.COLL_PATH_STREAMED if path is None else path, **extra)
    chosen = coll.plan()["path"]
    ins = make_inputs(max(coll.elems(r)[0] for r in range(n)), 11)
    ins = [x[:coll.elems(r)[0]] for r, x in enumerate(ins)]
    outs = [torch.empty(max(coll.elems(r)[1], 8), dtype=torch.int16, device="cuda")
            for r in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            coll.run(ins, outs, stream)
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    s = count * 2.0
    if kind == "ar":
        b = bytes_allreduce_twoshot(n, s, EPS_LL128)
    elif kind == "rs":
        b = bytes_reduce_scatter(n, s, EPS_LL128)
    elif kind == "a2a":
        b = 2 * n * s * (1 + EPS_LL128)
    else:
        b = bytes_all_gather(n, s, EPS_LL128)
    st = coll.status(stream)[0]
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "GB/s": round(b / ms / 1e6, 1), "algorithmic_bytes": b,
            "path": {1: "fused", 2: "streamed", 3: "composed"}.get(chosen, chosen),
            "status": st}


def sizes_row(cd, stream, sizes_mib=(32, 128)) -> dict:
    """The bandwidth regime at the smaller per-rank sizes: all-reduce (LL128
    twoshot), reduce-scatter and all-gather (gathered output per rank) at each
    size, each on the launch path AUTO picks."""
    out = {}
    for mib in sizes_mib:
        count = mib * 2**20 // 2
        out[f"{mib}MiB"] = {
            "allreduce": bandwidth_row(cd, cd.ALLREDUCE, count, "ar", stream,
                                       path=cd.COLL_PATH_AUTO),
            "reduce_scatter": bandwidth_row(cd, cd.REDUCE_SCATTER, count, "rs", stream,
                                            path=cd.COLL_PATH_AUTO),
            "all_gather": bandwidth_row(cd, cd.ALLGATHER, count, "ag", stream,
                                        path=cd.COLL_PATH_AUTO),
        }
    return out


def v_row(cd, name, total_bytes, stream, steps=5, path=None) -> dict:
    """Variable-length collective on a Zipf split (exponent 0.125) of a total
    of `total_bytes` over 8 ranks, LL128 lines, the composed launch by
    columns (or `path`).  all-to-all V rotates each source's split right by
    (source + 1).  `algbw` is the total T over the time, as the
    variable-length experiment reports it."""
    import torch

    import synth

    n = N_RANKS
    base = [b // 2 for b in synth.zipf_split(total_bytes, n)]
    if name == "ALLTOALL_V":
        v = [synth.rotate_right(base, p + 1) for p in range(n)]
        count = 0
    else:
        v, count = base, sum(base)
    coll = cd.Collective(getattr(cd, name), n, count, encoding=cd.COLL_LL128,
                         path=cd.COLL_PATH_COMPOSED if path is None else path, vcounts=v)
    ins = make_inputs(max(max(coll.elems(r)[0] for r in range(n)), 8), 12)
    ins = [x[:coll.elems(r)[0]] for r, x in enumerate(ins)]
    outs = [torch.empty(max(coll.elems(r)[1], 8), dtype=torch.int16, device="cuda")
            for r in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            coll.run(ins, outs, stream)
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    t = float(total_bytes)
    if name == "REDUCE_SCATTER_V":
        b = bytes_reduce_scatter(n, t, EPS_LL128)
    elif name == "ALLGATHER_V":
        b = bytes_all_gather(n, t, EPS_LL128)
    else:
        b = 2 * n * t * (1 + EPS_LL128)
    st = coll.status(stream)[0]
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "GB/s": round(b / ms / 1e6, 1), "algbw_GB/s": round(t / ms / 1e6, 1),
            "algorithmic_bytes": b, "status": st}


def streamed_row(cd, count, stream, steps=5) -> dict:
    """The same all-reduce through the three stream-ordered launches (stage,
    reduce-scatter fold + publish, all-gather copy), each timed with events
    recorded by the library."""
    import torch

    n = N_RANKS
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    ins = make_inputs(count, 4)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(n)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for ev in evs:
        for e in ev:
            e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        for i in range(steps):
            cd.coll_set_profile_events(coll.spec, evs[i])
            coll.run(ins, outs, stream)
        stream.synchronize()
    cd.coll_set_profile_events(coll.spec, [])
    s = count * 2.0
    kb = kernel_bytes_allreduce_twoshot(n, s, EPS_LL128)
    names = ["stage (LL128 encode)", "reduce-scatter fold + publish", "all-gather unpack"]
    dur = [statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(steps))
           for k in range(3)]
    total = statistics.mean(evs[i][0].elapsed_time(evs[i][3]) for i in range(steps))
    st = coll.status(stream)[0]
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()
    b = bytes_allreduce_twoshot(n, s, EPS_LL128)
    # run-only (inputs already staged, the analogue of Purlin's zero-staging
    # numbers): the fold and all-gather launches and their bytes
    run_ms = dur[1] + dur[2]
    return {"ms": round(total, 4), "GB/s": round(b / total / 1e6, 1), "status": st,
            "run_only": {"ms": round(run_ms, 4),
                         "GB/s": round((kb[1] + kb[2]) / run_ms / 1e6, 1)},
            "kernels": [{"name": names[k], "ms": round(dur[k], 4),
                         "GB/s": round(kb[k] / dur[k] / 1e6, 1),
                         "frac_of_hbm": round(kb[k] / dur[k] / 1e6 / load_peaks()["hbm_gbs"], 4)}
                        for k in range(3)]}


def f32_row(cd, nbytes, stream, steps=5) -> dict:
    """8 ranks x `nbytes` of fp32 per rank: twoshot all-reduce, LL128 lines,
    the composed launch (the bench workload with fp32 elements: the same
    bytes, folds in binary32 with no narrowing)."""
    import torch

    n = N_RANKS
    count = nbytes // 4
    coll = cd.Collective(cd.ALLREDUCE, n, count, dtype=cd.COLL_F32, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_COMPOSED)
    ins = [x.view(torch.int32) for x in make_inputs(2 * count, 14)]
    outs = [torch.empty(count, dtype=torch.int32, device="cuda") for _ in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            coll.run(ins, outs, stream)
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    b = bytes_allreduce_twoshot(n, float(nbytes), EPS_LL128)
    st = coll.status(stream)[0]
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "GB/s": round(b / ms / 1e6, 1), "algorithmic_bytes": b,
            "status": st}


def atom_ablation(cd, stream, nbytes=256 << 20, stage_bytes=16384, ctas_list=None,
                  steps=5, engines=("bulk", "lsu"), stages=range(1, 9)) -> dict:
    """Pipeline-depth ablation of the one-sided copy (Purlin §5.2, Figure 9;
    capacity Q_cap = C * S * B_stage of §3.3 Eq. (3)), against HBM: a copy of
    `nbytes` with the CTA count C fixed, S = 1..8 stages of `stage_bytes`,
    for both load engines.  copy_GBps = message bytes / time (the figure's
    quantity); hbm_GBps counts the read and the write (the HBM roofline);
    latency_ns = Q_cap / copy rate, the latency the bytes in flight cover by
    Little's law.  Median of `steps` launches, each timed alone."""
    import torch

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ctas_list = ctas_list or (16, 32, 64, sms)
    src = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=torch.int32, device="cuda")
    dst = torch.empty_like(src)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    out = {"bytes": nbytes, "stage_bytes": stage_bytes, "threads_per_cta": 256,
           "l2": "source and destination (512 MiB together) larger than L2; no flush"}
    for name, engine in (("bulk", cd.COLL_ATOM_BULK), ("lsu", cd.COLL_ATOM_LSU)):
        if name not in engines:
            continue
        for C in ctas_list:
            pts = []
            for S in stages:
                def launch():
                    cd.coll_atom_copy(dst, src, nbytes, engine=engine, ctas=C, stages=S,
                                      stage_bytes=stage_bytes, status=status, stream=stream)
                with torch.cuda.stream(stream):
                    for _ in range(2):
                        launch()
                    ms = []
                    for _ in range(steps):
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        launch()
                        e1.record(stream)
                        stream.synchronize()
                        ms.append(e0.elapsed_time(e1))
                t = statistics.median(ms)
                rate = nbytes / t / 1e6
                q = C * S * stage_bytes
                pts.append({"S": S, "q_cap_bytes": q, "ms": round(t, 4),
                            "copy_GBps": round(rate, 1), "hbm_GBps": round(2 * rate, 1),
                            "latency_ns": round(q / rate, 1)})
            out[f"{name}_C{C}"] = pts
    torch.cuda.synchronize()
    out["status"] = int(status.item())
    ok = bool(torch.equal(dst, src))
    out["last_copy_exact"] = ok
    del src, dst
    torch.cuda.empty_cache()
    return out


def bounded_staging_row(cd, count, stream, staging_mib=16, steps=5) -> dict:
    """The bench workload (8 ranks x 256 MiB, LL128 twoshot, composed launch)
    with each rank's staging image bounded to `staging_mib` MiB per slot:
    chunks cycle through the chunk slots that fit (Purlin §4.1)."""
    import torch

    n = N_RANKS
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_COMPOSED,
                         staging_bytes=staging_mib << 20)
    full = cd.coll_spec_create(*cd.ALLREDUCE, n, count, encoding=cd.COLL_LL128,
                               algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_COMPOSED)
    full_ws = cd.coll_workspace_bytes(full)
    cd.coll_destroy(full)
    ins = make_inputs(count, 4)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            coll.run(ins, outs, stream)
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    b = bytes_allreduce_twoshot(n, count * 2.0, EPS_LL128)
    st = coll.status(stream)[0]
    ws = cd.coll_workspace_bytes(coll.spec)
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "GB/s": round(b / ms / 1e6, 1), "algorithmic_bytes": b,
            "staging_mib_per_rank": staging_mib, "workspace_bytes": ws,
            "workspace_bytes_unbounded": full_ws, "status": st}


def sentinel_row(cd, count, stream, steps=5) -> dict:
    """8 ranks x `count` bf16 all-reduce, twoshot, sentinel packs, streamed.
    Algorithmic bytes are the LL form with epsilon = 1 (no readiness bytes);
    the re-arm writes (N S for the staging slot, S for the reduced
    partitions) are reported beside them, not in them."""
    import torch

    n = N_RANKS
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cd.COLL_SENT,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    ins = make_inputs(count, 13)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            coll.run(ins, outs, stream)
        e1.record(stream)
        stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    s = count * 2.0
    b = bytes_allreduce_twoshot(n, s, 1.0)
    st = coll.status(stream)[0]
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()
    return {"ms": round(ms, 4), "GB/s": round(b / ms / 1e6, 1), "algorithmic_bytes": b,
            "rearm_bytes": (n + 1) * s, "status": st}


def hbm_reference_row(stream, reps=10) -> dict:
    """Reference DRAM rates of plain torch kernels (not the library), for
    reading the write-heavy rows: a 2 GiB fill (writes only), a 2 GiB copy
    (half reads, half writes, like the measured copy peak) and eight copies
    fanning 256 MiB out into 2 GiB (the all-gather's traffic shape).  Every
    buffer is larger than L2; CUDA events on the timing stream."""
    import torch

    nb = 2 << 30
    a = torch.empty(nb, dtype=torch.uint8, device="cuda")
    b = torch.empty(nb, dtype=torch.uint8, device="cuda")
    src = torch.empty(nb // 8, dtype=torch.uint8, device="cuda")

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            stream.synchronize()
        return e0.elapsed_time(e1) / reps

    def fan():
        for k in range(8):
            a[k * (nb // 8):(k + 1) * (nb // 8)].copy_(src)

    fill_ms = timed(lambda: a.fill_(1))
    copy_ms = timed(lambda: b.copy_(a))
    fan_ms = timed(fan)
    del a, b, src
    torch.cuda.empty_cache()
    return {"fill_2GiB": {"ms": round(fill_ms, 4), "written_GB/s": round(nb / fill_ms / 1e6, 1)},
            "copy_2GiB": {"ms": round(copy_ms, 4), "read+written_GB/s": round(2 * nb / copy_ms / 1e6, 1)},
            "fan_out_256MiB_x8": {"ms": round(fan_ms, 4), "written_GB/s": round(nb / fan_ms / 1e6, 1)},
            "note": "torch kernels, not the library: the write side's ceiling for reading "
                    "write-heavy rows (all-gather, MoE dispatch)"}


def moe_row(cd, stream, steps=5, path=None, tokens=4096, cpu=False) -> dict:
    """MoE dispatch: 8 ranks x `tokens` tokens x 7168 bf16, top-8 of 256
    experts (routing drawn on the device from a seeded generator)."""
    import torch

    n, hidden, k, experts = N_RANKS, 7168, 8, 256
    coll = cd.Collective(cd.MOE_DISPATCH, n, 0, encoding=cd.COLL_LL128, tokens=tokens,
                         hidden=hidden, topk=k, experts=experts,
                         max_rows=(tokens * k * 40000 + 32767) // 32768,
                         path=cd.COLL_PATH_AUTO if path is None else path)
    composed = coll.plan()["path"] == cd.COLL_PATH_COMPOSED
    ins = make_inputs(tokens * hidden, 13)
    topk = []
    for r in range(n):
        g = torch.Generator(device="cuda")
        g.manual_seed(5000 + r)
        keys = torch.rand(tokens, experts, generator=g, device="cuda")
        topk.append(keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous())
        cd.coll_set_routing(coll.spec, r, topk[r])
    torch.cuda.synchronize()  # routing is drawn on torch's stream
    # staged rows: one per (token, destination rank holding one of its experts)
    el = experts // n
    staged = sum(int(torch.zeros(tokens, n, dtype=torch.bool, device="cuda")
                     .scatter_(1, topk[r].long() // el, True).sum()) for r in range(n))
    outs = [torch.empty(coll.elems(r)[1], dtype=torch.int16, device="cuda") for r in range(n)]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(2):
            coll.run(ins, outs, stream)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            coll.run(ins, outs, stream)
        e1.record(stream)
        stream.synchronize()
        # the split between the two launch groups, from events the library
        # records after each launch (separate runs, so the total above is
        # not perturbed)
        cd.coll_set_profile_events(coll.spec, ev)
        times = [0.0, 0.0]
        for _ in range(steps):
            coll.run(ins, outs, stream)
            stream.synchronize()
            times[0] += ev[0].elapsed_time(ev[1])
            times[1] += ev[1].elapsed_time(ev[2])
        cd.coll_set_profile_events(coll.spec, [])
    st = coll.status(stream)[0]
    rows = n * tokens * k
    row_b, line_b = hidden * 2, ((hidden + 59) // 60 + 3) // 4 * 4 * 128
    unique = n * tokens * row_b + staged * line_b + staged * line_b + rows * row_b
    issue = rows * row_b + rows * line_b + rows * line_b + rows * row_b  # a row per choice
    ms = e0.elapsed_time(e1) / steps
    coll.close()
    del coll, outs
    cpu_leg = None
    if cpu:
        import numpy as np

        ins_h = [x.cpu().numpy().view(np.uint16).reshape(tokens, hidden) for x in ins]
        topk_h = [t.cpu().numpy() for t in topk]
        cpu_leg = cpu_oracle_moe(ins_h, topk_h, experts)
        cpu_leg["GB/s"] = round(unique / (cpu_leg["s_per_op"] * 1e9), 4)
        del ins_h, topk_h
    del ins, topk
    torch.cuda.empty_cache()
    split = ({"routing_ms": round(times[0] / steps, 4),
              "stage_and_copy_ms": round(times[1] / steps, 4)} if composed else
             {"stage_ms": round(times[0] / steps, 4), "copy_ms": round(times[1] / steps, 4)})
    return {"ms": round(ms, 4), "GB/s": round(unique / ms / 1e6, 1),
            "path": "composed" if composed else "streamed",
            "algorithmic_bytes": unique, "issue_level_bytes": issue, "staged_rows": staged,
            "routed_rows": rows, **split,
            "note": "bytes: each token row read once, staged as LL128 once per destination "
                    "rank it is routed to, each staged row read once and unpacked into "
                    "every routed row", "status": st,
            **({"cpu_oracle": cpu_leg} if cpu_leg else {})}


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mib", type=int, default=256, help="per-rank MiB of the main workload")
    ap.add_argument("--path", default="composed", choices=["streamed", "composed"],
                    help="launch path of the main all-reduce")
    ap.add_argument("--quick", action="store_true", help="skip sweep, extra rows and CPU leg")
    ap.add_argument("--sweep-only", action="store_true",
                    help="only the small-message latency sweep (profiling runs)")
    ap.add_argument("--sweep-T", type=int, default=None, help="sweep only this T")
    ap.add_argument("--sweep-variant", default=None,
                    help="sweep only this variant, e.g. twoshot_fused")
    ap.add_argument("--sweep-enc", default="ll8", choices=["ll8", "ll128", "sent"],
                    help="readiness encoding of the sweep")
    ap.add_argument("--atom-only", action="store_true",
                    help="only the pipeline-depth ablation of the one-sided copy")
    ap.add_argument("--row", default=None,
                    help="run one extra row alone and print it (profiling runs): "
                         "moe, moe_streamed, rs, rs_composed, ag, a2a, a2a_composed, "
                         "sentinel, f32, staging16, sizes, rsv, agv, a2av (and their _streamed "
                         "forms), hbm_reference")
    ap.add_argument("--staging-mib", type=int, default=16,
                    help="staging MiB per rank of the bounded-staging row run alone")
    ap.add_argument("--moe-tokens", type=int, default=4096,
                    help="tokens per rank of the MoE rows (the bench line uses 4096)")
    ap.add_argument("--atom-case", default=None,
                    help="with --atom-only: one point ENGINE,C,S (e.g. bulk,16,8)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    args.warmup = max(args.warmup, 3)
    if not os.path.exists(os.path.join(ROOT, "collective_datapath_gb300", "libcoll.so")):
        import __graft_entry__

        __graft_entry__.build()
    import collective_datapath_gb300 as cd

    peaks = load_peaks()
    stream = torch.cuda.Stream()
    if args.sweep_only:
        enc = {"ll8": cd.COLL_LL8, "ll128": cd.COLL_LL128, "sent": cd.COLL_SENT}[args.sweep_enc]
        print(json.dumps({"encoding": args.sweep_enc,
                          "latency_us_per_op": latency_sweep(cd, stream, args.sweep_T,
                                                             args.sweep_variant, enc)}))
        return 0
    if args.atom_only:
        kw = {}
        if args.atom_case:
            eng, c, st = args.atom_case.split(",")
            kw = {"engines": (eng,), "ctas_list": (int(c),), "stages": (int(st),)}
        print(json.dumps({"pipeline_depth_ablation_256MiB": atom_ablation(cd, stream, **kw)}))
        return 0
    count = args.mib * 2**20 // 2
    if args.row:
        rows = {
            "moe": lambda: moe_row(cd, stream, tokens=args.moe_tokens),
            "moe_streamed": lambda: moe_row(cd, stream, path=cd.COLL_PATH_STREAMED,
                                            tokens=args.moe_tokens),
            "rs": lambda: bandwidth_row(cd, cd.REDUCE_SCATTER, count, "rs", stream),
            "rs_composed": lambda: bandwidth_row(cd, cd.REDUCE_SCATTER, count, "rs", stream,
                                                 path=cd.COLL_PATH_COMPOSED),
            "ag": lambda: bandwidth_row(cd, cd.ALLGATHER, count, "ag", stream),
            "ag_composed": lambda: bandwidth_row(cd, cd.ALLGATHER, count, "ag", stream,
                                                 path=cd.COLL_PATH_COMPOSED),
            "a2a": lambda: bandwidth_row(cd, cd.ALLTOALL, count, "a2a", stream),
            "a2a_composed": lambda: bandwidth_row(cd, cd.ALLTOALL, count, "a2a", stream,
                                                  path=cd.COLL_PATH_COMPOSED),
            "sentinel": lambda: sentinel_row(cd, count, stream),
            "f32": lambda: f32_row(cd, args.mib << 20, stream),
            "staging16": lambda: bounded_staging_row(cd, count, stream, args.staging_mib),
            "sizes": lambda: sizes_row(cd, stream),
            "rsv": lambda: v_row(cd, "REDUCE_SCATTER_V", args.mib << 20, stream),
            "agv": lambda: v_row(cd, "ALLGATHER_V", args.mib << 20, stream),
            "a2av": lambda: v_row(cd, "ALLTOALL_V", args.mib << 20, stream),
            "rsv_streamed": lambda: v_row(cd, "REDUCE_SCATTER_V", args.mib << 20, stream,
                                          path=cd.COLL_PATH_STREAMED),
            "agv_streamed": lambda: v_row(cd, "ALLGATHER_V", args.mib << 20, stream,
                                          path=cd.COLL_PATH_STREAMED),
            "a2av_streamed": lambda: v_row(cd, "ALLTOALL_V", args.mib << 20, stream,
                                           path=cd.COLL_PATH_STREAMED),
            "hbm_reference": lambda: hbm_reference_row(stream),
        }
        if args.row not in rows:
            raise SystemExit(f"unknown row {args.row}")
        print(json.dumps({"rows": {args.row: rows[args.row]()}}))
        return 0
    s_bytes = count * 2.0
    composed = args.path == "composed"
    coll = cd.Collective(cd.ALLREDUCE, N_RANKS, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT,
                         path=cd.COLL_PATH_COMPOSED if composed else cd.COLL_PATH_STREAMED)
    ins = make_inputs(count, 4)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N_RANKS)]
    K, W = args.steps, args.warmup
    nk = 1 if composed else 3
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
              for _ in range(W + K)]
    for evs in events:          # torch creates the CUDA event on first record
        for e in evs:
            e.record(stream)
    stream.synchronize()
    launches = [0]

    def step(i):
        cd.coll_set_profile_events(coll.spec, events[i % len(events)])
        coll.run(ins, outs, stream)
        launches[0] += cd.coll_last_launches(coll.spec)

    l2peak = l2_copy_peak(cd, stream)
    clocks = Clocks(local)
    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
        torch.cuda.synchronize()
        launches[0] = 0
        clocks.start()
        ms_total = timed(lambda i: step(W + i), K, 0, stream, world)
        clk = clocks.stop()
    cd.coll_set_profile_events(coll.spec, [])
    code = coll.status(stream)[0]
    if code != cd.COLL_OK:
        raise RuntimeError(f"device status {code} during the timed steps")
    ms_step = barrier_max(ms_total / K, world)
    algo_bytes = bytes_allreduce_twoshot(N_RANKS, s_bytes, EPS_LL128)
    value = replica_value(world, algo_bytes, ms_step)

    # per-kernel durations over the timed steps
    if composed:
        names = ["composed twoshot (columns: stage, fold + publish, gather of one chunk of a partition per CTA)"]
        kb = [bytes_allreduce_twoshot(N_RANKS, s_bytes, EPS_LL128)]
    else:
        names = ["stage (LL128 encode)", "reduce-scatter fold + publish", "all-gather unpack"]
        kb = kernel_bytes_allreduce_twoshot(N_RANKS, s_bytes, EPS_LL128)
    dur = [statistics.mean(events[W + i][k].elapsed_time(events[W + i][k + 1])
                           for i in range(K)) for k in range(nk)]
    kernels = [{"name": names[k], "ms": round(dur[k], 4), "bytes": kb[k],
                "GB/s": round(kb[k] / dur[k] / 1e6, 1)} for k in range(nk)]
    dom = max(range(nk), key=lambda k: dur[k])
    issue_gbs = kb[dom] / dur[dom] / 1e6
    floor_bytes = ([unique_bytes_allreduce(N_RANKS, s_bytes)] if composed
                   else kernel_floor_bytes_allreduce_twoshot(N_RANKS, s_bytes, EPS_LL128))
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.md")
    if os.path.exists(prof):
        key = f"allreduce_twoshot_ll128_{args.mib}mib"
        want = "composed" if composed else ["stage", "rs", "ag"][dom]
        with open(prof) as f:
            for ln in f:
                parts = ln.split()
                if len(parts) == 4 and parts[0] == "traffic" and parts[1] == key \
                        and parts[2] == want:
                    traffic = int(parts[3])

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args.mib, args.path, world),
        "roofline": {
            "bound": "hbm", "kernel": names[dom],
            # DRAM side: the kernel's ncu DRAM bytes per launch over this run's
            # launch time (CUDA events around every launch of the timed steps)
            "achieved": round(traffic / dur[dom] / 1e6, 1) if traffic else None,
            "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(traffic / dur[dom] / 1e6 / peaks["hbm_gbs"], 4) if traffic else None,
            "traffic": traffic, "peak_source": peaks["source"],
            "kernel_ms": round(dur[dom], 4),
            # speed of light: the DRAM bytes the launch cannot avoid
            "floor_bytes": floor_bytes[dom],
            "sol_frac": round(floor_bytes[dom] / dur[dom] / 1e6 / peaks["hbm_gbs"], 4),
            "issue_level": {"bytes": kb[dom], "achieved": round(issue_gbs, 1), "unit": "GB/s",
                            "l2_peak": l2peak["gbs"],
                            "frac_of_l2_peak": round(issue_gbs / l2peak["gbs"], 4),
                            "l2_peak_how": l2peak["how"],
                            "l2_peak_candidates": l2peak["candidates"]},
            "how": "achieved = traffic (ncu dram__bytes_read.sum + dram__bytes_write.sum per "
                   "launch, profiles/traffic.md) / kernel_ms; frac = achieved / peak; "
                   "sol_frac = floor_bytes / kernel_ms / peak; issue_level = every emulated "
                   "rank's reads and writes (mostly L2 hits in one launch) against an L2 "
                   "copy peak measured in this run"},
        "kernels": kernels,
        "gpu_launches": launches[0],
        "clocks": clk,
    }

    if not args.quick and rank == 0:
        # end to end from pinned host memory through coll_run_host
        host_in = [x.cpu().pin_memory() for x in ins]
        host_out = [torch.empty(count, dtype=torch.int16).pin_memory() for _ in range(N_RANKS)]
        with torch.cuda.stream(stream):
            cd.coll_run_host(coll.spec, host_in, ins, outs, host_out, stream)
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            ke = 3
            e0.record(stream)
            for _ in range(ke):
                cd.coll_run_host(coll.spec, host_in, ins, outs, host_out, stream)
            e1.record(stream)
            stream.synchronize()
        copy_ms = e0.elapsed_time(e1) / ke
        # the same call on pinned host buffers: the stage kernel reads the
        # inputs and the gather kernel writes the outputs across NVLink-C2C
        with torch.cuda.stream(stream):
            coll.run(host_in, host_out, stream)
            stream.synchronize()
            e0.record(stream)
            for _ in range(ke):
                coll.run(host_in, host_out, stream)
            e1.record(stream)
            stream.synchronize()
        direct_ms = e0.elapsed_time(e1) / ke
        code = coll.status(stream)[0]
        if code != cd.COLL_OK:
            raise RuntimeError(f"device status {code} in the end-to-end runs")
        e2e_ms = min(copy_ms, direct_ms)
        if world == 1:
            # c4 on the host: the oracle's reduce-scatter of these very inputs
            # (one fold per element in rank order, the all-reduce's arithmetic
            # without its 8 output copies), median of 3
            import numpy as np

            xs_h = [h.numpy().view(np.uint16) for h in host_in]
            import oracle

            ts = []
            for _ in range(3):
                t0 = time.perf_counter()
                oracle.reduce_scatter(xs_h)
                ts.append(time.perf_counter() - t0)
            rs_s = statistics.median(ts)
            cpu_c4 = {"s_per_op": round(rs_s, 3), "runs_s": [round(t, 3) for t in ts],
                      "GB/s": round(bytes_reduce_scatter(N_RANKS, s_bytes, EPS_LL128)
                                    / rs_s / 1e9, 4),
                      "what": f"reduce-scatter of the bench's own {N_RANKS} x {args.mib} MiB "
                              f"inputs (GB/s with the reduce-scatter's algorithmic bytes)"}
            del xs_h
        line["e2e"] = {"value": round(algo_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                       "h2d_bytes_per_step": int(N_RANKS * s_bytes),
                       "d2h_bytes_per_step": int(N_RANKS * s_bytes),
                       "ms_per_step": round(e2e_ms, 3),
                       "host_pointers_ms": round(direct_ms, 3),
                       "memcpy_ms": round(copy_ms, 3),
                       "how": "coll_run on pinned host buffers (kernels read/write host "
                              "memory over C2C) and coll_run_host (one cudaMemcpyAsync "
                              "per buffer); value = the faster"}
        del host_in, host_out
    coll.close()
    del coll, ins, outs
    torch.cuda.empty_cache()

    if not args.quick and rank == 0:
        line["rows"] = {
            **({"allreduce_256MiB_streamed_three_launches": streamed_row(cd, count, stream)}
               if composed else {}),
            "reduce_scatter_256MiB": bandwidth_row(cd, cd.REDUCE_SCATTER, count, "rs", stream),
            "reduce_scatter_256MiB_composed": bandwidth_row(cd, cd.REDUCE_SCATTER, count, "rs",
                                                            stream, path=cd.COLL_PATH_COMPOSED),
            "all_gather_256MiB": bandwidth_row(cd, cd.ALLGATHER, count, "ag", stream),
            "all_gather_256MiB_composed": bandwidth_row(cd, cd.ALLGATHER, count, "ag", stream,
                                                        path=cd.COLL_PATH_COMPOSED),
            "all_to_all_256MiB": bandwidth_row(cd, cd.ALLTOALL, count, "a2a", stream),
            "all_to_all_256MiB_composed": bandwidth_row(cd, cd.ALLTOALL, count, "a2a", stream,
                                                        path=cd.COLL_PATH_COMPOSED),
            "moe_dispatch_8x4096x7168_top8of256": moe_row(cd, stream, cpu=world == 1),
            "moe_dispatch_8x4096x7168_top8of256_streamed": moe_row(cd, stream,
                                                                   path=cd.COLL_PATH_STREAMED),
            "reduce_scatter_v_zipf_256MiB": v_row(cd, "REDUCE_SCATTER_V", 256 << 20, stream),
            "all_gather_v_zipf_256MiB": v_row(cd, "ALLGATHER_V", 256 << 20, stream),
            "all_to_all_v_zipf_256MiB": v_row(cd, "ALLTOALL_V", 256 << 20, stream),
            "allreduce_256MiB_sentinel_twoshot": sentinel_row(cd, count, stream),
            "allreduce_256MiB_f32_composed": f32_row(cd, 256 << 20, stream),
            "allreduce_256MiB_composed_staging_16MiB": bounded_staging_row(cd, count, stream),
            "bandwidth_regime_32_128MiB": sizes_row(cd, stream),
            "pipeline_depth_ablation_256MiB": atom_ablation(cd, stream),
            "hbm_reference_torch": hbm_reference_row(stream),
        }
        line["latency_us_per_op"] = latency_sweep(cd, stream)
        if world == 1:
            line["cpu_baseline"] = cpu_oracle_allreduce(64, runs=3)
            line["cpu_baselines"] = {
                "host": host_cpu(), "threads": 1,
                "how": "the plain C99 oracle (oracle/oracle.c) called through ctypes, one "
                       "thread, wall time by time.perf_counter around each call",
                **cpu_oracle_configs(),
                "c4_reduce_scatter_256MiB": cpu_c4,
                "c4_allreduce_64MiB_sample": line["cpu_baseline"],
                "c5_moe_dispatch_8x4096x7168_top8of256":
                    line["rows"]["moe_dispatch_8x4096x7168_top8of256"].get("cpu_oracle")}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
