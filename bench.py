#!/usr/bin/env python
"""Throughput of the SPME packet simulator on GB300.

Metric: simulated packet-hops per second over a batch of experiments (a
packet-hop is one packet placed on one link), plus the megakernel's achieved
bandwidth (algorithmic bytes over its device time) against the measured HBM
peak.

Default workload: config 3 (the GPT-13B 1F1B iteration on the k=16
fat-tree, 500 experiments over {ring, tree} x NC x chunk x duration seed), a
window of its data-parallel gradient all-reduce phase.  Every experiment is
first run untimed to the window's start tick (once; the simulator's whole
state is its workspace, so later steps restore that state with one device
copy).  One step = the whole path over the batch for the window's ticks: one
megakernel launch that advances all 500 experiments from the start tick to
start + ticks of their own clocks, inputs resident in HBM.  Steps are timed
with CUDA events on the simulator's stream; L2 is flushed (a 512 MiB write)
before each step.

``e2e`` repeats the step from host memory through the public API: the start
state (the workspace) is copied from pinned host memory to the device, the
window is run (mv_run) and the per-experiment counters are read back
(mv_results), timed by wall clock.  Whole-run workloads (configs 1 and 2)
instead time mv_reset + mv_run to completion, and their e2e creates the
simulator from the host arrays (mv_create), runs it and reads all results.

--impl reference, and the cpu_baseline leg, time the CPU oracle (the plain C
simulator, as it stands) on the host cores over a bounded sample of the
same workload: for a window, each worker runs one experiment to the start
tick untimed, then times the window from a copy of that state.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from experiment_network_simulation_gb300 import inputs as I  # noqa: E402

METRIC = "simulated packet-hops/s over experiment batch"
UNIT = "packet-hops/s"
# Algorithmic bytes: each packet-hop writes its 16-byte descriptor into the
# downstream queue and reads it back out (32 B); each packet also costs a
# sender flow-state read-modify-write (16 B) and a receiver update (8 B).
BYTES_PER_HOP, BYTES_PER_PKT = 32, 24

WORKLOADS = {
    "config1": (lambda seed: I.config1(),
                "ring all-reduce 16 MiB, 8 hosts, 2x2 leaf-spine, 400G, 16 experiments"),
    "config2": (lambda seed: I.config2(seed=seed),
                "pipelined broadcast 1-64 MiB over A in 2..16 hosts, K in 1..64, 10G, 256 experiments"),
    "config3": (lambda seed: I.config3(),
                "GPT-13B 1F1B iteration, 128 servers x 8 GPUs, TP8 PP4 DP32, k=16 fat-tree, 400G, "
                "500 experiments"),
    "config4": (lambda seed: I.config4(),
                "MoE dispatch/combine, 512 ranks, top-8 of 256, 4 fabrics x 256 router seeds, "
                "1,024 experiments"),
    "config5": (lambda seed: I.config5(n_exp=24),
                "topology search, GPT-13B at DP128 on 1,024-server 3-tier fabrics (24 of them)"),
    "gpt_small": (lambda seed: I.gpt_small(seeds=tuple(range(8))),
                  "the config-3 DAG shape at test size (8 servers x 2 GPUs, k=4 fat-tree), "
                  "8 experiments"),
}
DEFAULT = "config3"
# Default window (start tick, ticks) per workload; None = whole runs.  Config
# 3's window lies in the data-parallel all-reduce phase of all 500
# experiments: by tick 2.6 M every pipeline transfer has ended, the gradient
# all-reduces started from about 1.7 M on, and the iterations end between
# about 2.7 M (16 channels) and 4.5 M ticks (trees of 16 channels).
WINDOWS = {"config3": (2_600_000, 4_000), "config5": (300_000, 2_000), "gpt_small": (3_000, 2_000)}

# DRAM bytes (read + write) per megakernel launch from ncu captures of the
# current kernel, keyed by workload and window; each entry names the kernel
# source digest it was taken with, and is dropped (traffic: null) once the
# kernel source differs.
TRAFFIC: dict = {
    # ncu dram__bytes_read.sum + dram__bytes_write.sum of one window launch of
    # config 3's first 152 experiments (72,359,266,048 + 41,792,947,712 B for
    # 802,918,438 packet-hops); the 500-experiment step is too large to
    # capture, so its entry is that figure scaled by packet-hops
    # (2,344,660,048 a step): traffic grows with the hops.
    ("config3", (2_600_000, 4_000), 152): {"bytes_per_launch": 114_152_213_760,
                                           "kernel_digest": "2408b8ec10073668"},
    ("config3", (2_600_000, 4_000), 500): {"bytes_per_launch": 333_344_113_582,
                                           "kernel_digest": "2408b8ec10073668"},
}
KERNEL_SOURCES = ["experiment_network_simulation_gb300/csrc/mv_kernel.cu",
                  "experiment_network_simulation_gb300/csrc/mv_device.cuh"]


def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def make_batch(name: str, seed: int = 0, exps: int = 0):
    """The named workload; "+voq", "+dcqcn", "+dctcp" suffixes give every
    experiment virtual output queues or that congestion control (the
    generators' settings)."""
    base, *mods = name.split("+")
    b = WORKLOADS[base][0](seed)
    b = b.subset(range(min(exps, len(b)))) if exps else b
    for e in b.experiments:
        for m in mods:
            if m == "voq":
                e.voq = 1
            elif m == "dcqcn":
                e.cc = I.dcqcn(e.tick_ps, e.pkt)
            elif m == "dctcp":
                e.cc = I.DCTCP()
            else:
                raise ValueError(f"unknown workload variant {m!r}")
    return b


def batch_name(args) -> str:
    return args.workload + ("+voq" if args.voq else "") + \
        ("" if args.cc == "none" else "+" + args.cc)


def window_of(args):
    """(start tick, ticks) of the timed window, or None for whole runs."""
    if args.whole:
        return None
    if args.start_tick is not None or args.max_ticks is not None:
        d = WINDOWS.get(args.workload, (0, 0))
        s = d[0] if args.start_tick is None else args.start_tick
        n = d[1] if args.max_ticks is None else args.max_ticks
        return (s, n) if n > 0 else None
    return WINDOWS.get(args.workload)


# ----------------------------------------------------------------- oracle pool
def _oracle_worker(conn, name: str, seed: int, exps: int):
    """One host core: builds the batch, then serves commands.  A window's
    start state stays in this process, so its windows always run here."""
    sys.path.insert(0, ROOT)
    from oracle import oracle

    oracle.build()
    packed = make_batch(name, seed, exps).pack()
    paused = {}
    conn.send("ready")
    while True:
        cmd = conn.recv()
        if cmd[0] == "quit":
            break
        if cmd[0] == "whole":                 # one whole experiment
            e = cmd[1]
            t0 = time.perf_counter()
            r = oracle.run(packed, e, e + 1)
            conn.send((int(r["pkt_hops"][e]), time.perf_counter() - t0))
        elif cmd[0] == "prefix":              # untimed: to the window's start tick
            e, start = cmd[1], cmd[2]
            p = oracle.Paused(packed, e)
            p.advance(start)
            paused[e] = p
            conn.send(e)
        elif cmd[0] == "window":              # the window from a copy of the start state
            e, start, ticks = cmd[1], cmd[2], cmd[3]
            c = paused[e].clone()
            h0 = c.counters()["pkt_hops"]
            t0 = time.perf_counter()
            c.advance(start + ticks)
            dt = time.perf_counter() - t0
            h = c.counters()["pkt_hops"] - h0
            c.close()
            conn.send((int(h), dt))


class OraclePool:
    """The oracle on every host core: a process per core, one experiment per
    command.  For a window, each process holds the start state of one
    sampled experiment (computed untimed) and times the window from a copy."""

    def __init__(self, name: str, seed: int, exps: int, window, cores: int, wait: bool = True):
        from oracle import oracle

        oracle.build()
        self.n_exp = len(make_batch(name, seed, exps))
        self.order = [int(x) for x in np.random.default_rng(1234).permutation(self.n_exp)]
        self.window = window
        ctx = mp.get_context("spawn")
        self.workers = []
        for _ in range(min(cores, self.n_exp)):
            a, b = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(b, name, seed, exps), daemon=True)
            pr.start()
            self.workers.append((pr, a))
        for _, conn in self.workers:
            assert conn.recv() == "ready"
        self.sample = []
        self.pending = False
        if window:
            # each worker runs its experiment to the window's start; with
            # wait=False the caller does other work meanwhile (settle())
            self.sample = self.order[:len(self.workers)]
            for (_, conn), e in zip(self.workers, self.sample):
                conn.send(("prefix", e, window[0]))
            self.pending = True
            if wait:
                self.settle()

    def settle(self):
        """Wait for the start states of the sampled experiments."""
        if self.pending:
            for _, conn in self.workers[:len(self.sample)]:
                conn.recv()
            self.pending = False

    def _all(self, cmds):
        for (_, conn), cmd in zip(self.workers, cmds):
            conn.send(cmd)
        return [conn.recv() for (_, conn), _ in zip(self.workers, cmds)]

    def window_step(self):
        """Every sampled experiment's window once, in parallel: (hops, wall seconds)."""
        t0 = time.perf_counter()
        res = self._all([("window", e, self.window[0], self.window[1]) for e in self.sample])
        return sum(h for h, _ in res), time.perf_counter() - t0

    def whole_runs(self, budget_s: float):
        """Whole experiments in a seeded order, one per process at a time,
        until about budget_s of wall clock: (hops, wall seconds, done)."""
        hops, done, t0 = 0, 0, time.perf_counter()
        while done < self.n_exp and time.perf_counter() - t0 < budget_s:
            chunk = self.order[done:done + len(self.workers)]
            hops += sum(h for h, _ in self._all([("whole", e) for e in chunk]))
            done += len(chunk)
        return hops, time.perf_counter() - t0, done

    def close(self):
        for pr, conn in self.workers:
            try:
                conn.send(("quit",))
            except (BrokenPipeError, OSError):
                pass
        for pr, _ in self.workers:
            pr.join(timeout=5)
            if pr.is_alive():
                pr.terminate()


# ----------------------------------------------------------------- clocks
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l.split(",") for l in open(self.path).read().splitlines() if l.strip()]
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return None


def config_of(args, window, n_exp):
    cfg = {"workload": args.workload, "desc": WORKLOADS[args.workload][1],
           "experiments": n_exp}
    if args.voq:
        cfg["switch"] = "virtual output queues"
    if args.cc != "none":
        cfg["congestion_control"] = args.cc
    if window:
        cfg["window"] = {"start_tick": window[0], "ticks": window[1],
                         "note": "each step advances every experiment from start_tick to "
                                 "start_tick + ticks of its own clock; the run to start_tick "
                                 "is done once, untimed, and its state restored before each step"}
    return cfg


# ----------------------------------------------------------------- arms
def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    window = window_of(args)
    pool = OraclePool(batch_name(args), 0, args.exps, window, cores)
    try:
        if window:
            for _ in range(args.warmup):
                pool.window_step()
            hops, secs = 0, 0.0
            for _ in range(args.steps):
                h, dt = pool.window_step()
                hops += h
                secs += dt
            sample = (f"{len(pool.sample)} of {pool.n_exp} experiments (seeded permutation), "
                      f"ticks [{window[0]}, {window[0] + window[1]}) of each, one experiment per "
                      f"process, each window from a copy of its start state")
        else:
            per_step = max(1.0, args.cpu_budget_s / max(1, args.steps + args.warmup))
            for _ in range(args.warmup):
                pool.whole_runs(min(per_step, 5.0))
            pool.order = pool.order[len(pool.workers):] + pool.order[:len(pool.workers)]
            hops, secs, n_done = 0, 0.0, 0
            for _ in range(args.steps):
                h, dt, done = pool.whole_runs(per_step)
                hops += h
                secs += dt
                n_done += done
            sample = (f"{n_done // max(1, args.steps)} of {pool.n_exp} experiments per step "
                      f"(seeded permutation), whole runs, one experiment per process")
    finally:
        pool.close()
    value = hops / secs
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic", "config": config_of(args, window, pool.n_exp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def cpu_leg(args, window, pool=None):
    """cpu_baseline of the GPU arm: the oracle on the same workload (`pool`:
    one started earlier, whose start states may still be on their way)."""
    cores = os.cpu_count() or 1
    if pool is None:
        pool = OraclePool(batch_name(args), 0, args.exps, window, cores)
    try:
        pool.settle()
        if window:
            h, dt = pool.window_step()
            sample = (f"{len(pool.sample)} of {pool.n_exp} experiments (seeded permutation), "
                      f"ticks [{window[0]}, {window[0] + window[1]}) of each from its start "
                      f"state, {dt:.1f} s wall, one experiment per process")
        else:
            h, dt, done = pool.whole_runs(args.cpu_budget_s)
            sample = (f"{done} of {pool.n_exp} experiments (seeded permutation), whole runs, "
                      f"{dt:.1f} s wall, one experiment per process")
    finally:
        pool.close()
    return {"value": h / dt, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}


def run_gpu(args, rank: int, world: int):
    # the CPU baseline's processes start first (spawned, before any GPU
    # call) and run their experiments to the window's start while the GPU
    # does the same; the timed GPU steps wait until they are done
    import torch

    from experiment_network_simulation_gb300 import mv

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py: the GPU arm needs a CUDA device")
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = OraclePool(batch_name(args), 0, args.exps, window_of(args), os.cpu_count() or 1,
                          wait=False)

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    window = window_of(args)
    batch = make_batch(batch_name(args), seed=rank, exps=args.exps)   # each rank: its own shard
    packed = batch.pack()
    stream = torch.cuda.Stream(dev)
    sim = mv.Simulator(packed, device=str(dev), stream=stream)
    n_levels = int(packed["sw_level"].max())
    # our kernels a step launches: the megakernel; whole runs also reset
    # (routes per level, up lists, 2 init)
    launches_per_step = 1 if window else n_levels + 4
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    budget = window[1] if window else mv.UNSET - 1

    snap = {}
    if window:
        # untimed: every experiment to the window's start tick, once
        sim.reset()
        rc = sim.run(max_ticks=window[0], variant=args.variant, block_warps=args.block_warps)
        assert rc in (mv.MV_OK, mv.MV_INCOMPLETE), rc
        c = sim.counters()
        snap["ws"] = sim.ws.clone()
        snap["h"] = (int(c["pkt_hops"].sum()), int(c["pkts_injected"].sum()))
        snap["running"] = int((c["status"] == mv.EXP_RUNNING).sum())

    def prefix():
        if window:
            with torch.cuda.stream(stream):
                sim.ws.copy_(snap["ws"])
        with torch.cuda.stream(stream):
            flush.zero_()                             # L2 flush between steps
        return snap.get("h", (0, 0))

    def timed():
        if not window:
            sim.reset()
        rc = sim.run(max_ticks=budget, variant=args.variant, block_warps=args.block_warps)
        assert rc in ((mv.MV_OK, mv.MV_INCOMPLETE) if window else (mv.MV_OK,)), rc

    if pool is not None:
        pool.settle()                                 # the host cores are quiet from here on
    for _ in range(args.warmup):
        prefix()
        timed()
    res = sim.counters()
    if not window:
        assert (res["status"] == mv.EXP_DONE).all(), "warm-up did not finish every experiment"

    clocks = Clocks(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    total_ms, kernel_ms, steps_grid, hops_l, pkts_l = 0.0, [], [], [], []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.steps):
        h0, p0 = prefix()
        ev0.record(stream)
        timed()
        ev1.record(stream)
        ev1.synchronize()
        total_ms += ev0.elapsed_time(ev1)
        kernel_ms.append(sim.last_run_ms())
        steps_grid.append(sim.steps)
        c = sim.counters()
        hops_l.append(int(c["pkt_hops"].sum()) - h0)
        pkts_l.append(int(c["pkts_injected"].sum()) - p0)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    res = sim.counters()
    if not window:
        assert (res["status"] == mv.EXP_DONE).all()
    assert len(set(hops_l)) == 1, "a step simulated different work"
    hops_step, pkts_step = hops_l[0], pkts_l[0]

    ms_step = total_ms / args.steps
    t = torch.tensor([ms_step, float(hops_step), float(len(batch))], dtype=torch.float64)
    if world > 1:
        tt = t.to(dev)
        mx = tt.clone()
        torch.distributed.all_reduce(mx, op=torch.distributed.ReduceOp.MAX)
        sm = tt.clone()
        torch.distributed.all_reduce(sm, op=torch.distributed.ReduceOp.SUM)
        ms_max, hops_all, exps_all = float(mx[0]), float(sm[1]), float(sm[2])
    else:
        ms_max, hops_all, exps_all = ms_step, float(hops_step), float(len(batch))
    value = hops_all / (ms_max / 1000.0)

    # e2e through the public API from host memory
    e2e = None
    if args.e2e_steps > 0:
        e2e_s, h2d, d2h = [], 0, 0
        if window:
            host = torch.empty(snap["ws"].numel(), dtype=torch.uint8, pin_memory=True)
            host.copy_(snap["ws"])
            del snap["ws"]
            for _ in range(args.e2e_steps):
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                with torch.cuda.stream(stream):
                    sim.ws.copy_(host, non_blocking=True)     # the start state, host -> device
                sim.run(max_ticks=budget, variant=args.variant, block_warps=args.block_warps)
                c = sim.counters()                            # per-experiment results, device -> host
                e2e_s.append(time.perf_counter() - t0)
            h2d = int(host.numel())
            d2h = sum(int(v.nbytes) for v in c.values())
            del host
        else:
            h2d = sum(int(np.asarray(v).nbytes) for k, v in packed.items() if k != "version")
            for _ in range(args.e2e_steps):
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                s2 = mv.Simulator(packed, device=str(dev), stream=stream)
                s2.run(variant=args.variant, block_warps=args.block_warps)
                r2 = s2.results()
                s2.close()
                e2e_s.append(time.perf_counter() - t0)
                d2h = sum(int(v.nbytes) for k, v in r2.items() if isinstance(v, np.ndarray)
                          and not k.endswith("_offset"))
                del s2
        e2e = {"value": hops_step / statistics.mean(e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks = load_peaks()
    km = statistics.mean(kernel_ms)
    alg_bytes = BYTES_PER_HOP * hops_step + BYTES_PER_PKT * pkts_step
    achieved = alg_bytes / (km / 1000.0) / 1e9
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    key = (batch_name(args), tuple(window) if window else None, len(batch))
    tr = TRAFFIC.get(key)
    traffic = tr["bytes_per_launch"] if tr and tr["kernel_digest"] == kernel_digest() else None
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": "measured" if peaks else "fallback",
            "kernel": "k_megakernel", "kernel_ms": km, "alg_bytes_per_launch": alg_bytes}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_leg(args, window, pool)

    if rank == 0:
        cfg = config_of(args, window, int(exps_all))
        cfg.update({"kernel_build": args.variant or "automatic",
                    "packet_hops_per_step": int(hops_all),
                    "l2": "flushed between steps (512 MiB write)",
                    "grid_steps_per_run": int(statistics.mean(steps_grid))})
        if window:
            cfg["window"]["running_at_start"] = snap["running"]
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u32", "data": "synthetic", "config": cfg,
            "experiments_per_hour": None if window else exps_all / (ms_max / 1000.0) * 3600.0,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clk,
            "gpu_launches": launches_per_step * args.steps,
        }
        print(json.dumps(out), flush=True)
    sim.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--exps", type=int, default=0, help="first N experiments of the batch")
    ap.add_argument("--start-tick", type=int, default=None,
                    help="window start (default: the workload's window)")
    ap.add_argument("--max-ticks", type=int, default=None,
                    help="window length in ticks of each experiment's clock (0: whole runs)")
    ap.add_argument("--whole", action="store_true", help="time whole runs, no window")
    ap.add_argument("--variant", type=int, default=0, help="kernel build (0: automatic)")
    ap.add_argument("--voq", action="store_true", help="switches with virtual output queues")
    ap.add_argument("--cc", default="none", choices=["none", "dcqcn", "dctcp"],
                    help="congestion control of every experiment")
    ap.add_argument("--block-warps", type=int, default=0, help="warps a block (0: automatic)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch

        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
