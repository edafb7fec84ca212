#!/usr/bin/env python
"""Throughput of the SPME packet simulator on GB300.

Metric: simulated packet-hops per second over a batch of experiments (a
packet-hop is one packet placed on one link), plus experiments per hour and
the megakernel's achieved HBM bandwidth against the measured peak.

One step = the whole path over the batch: mv_reset (back to tick 0,
routing tables, memory check) + mv_run to completion, inputs resident in HBM.
Steps are timed with CUDA events on the simulator's stream; L2 is flushed
(a 512 MiB write) between steps.  ``e2e`` repeats the step through the
public API from host buffers: mv_create (upload), mv_run, mv_results
(download), timed by wall clock.

--impl reference times the CPU oracle (the plain C simulator, as it stands)
on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
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
# DRAM bytes (read + write) of one megakernel launch of the whole-run
# workload, from an ncu capture of the current kernel (see profiles/).
TRAFFIC = {"config2": 6724608}

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
}
DEFAULT = "config2"


def make_batch(name: str, seed: int = 0, exps: int = 0):
    b = WORKLOADS[name][0](seed)
    return b.subset(range(min(exps, len(b)))) if exps else b


# ----------------------------------------------------------------- oracle pool
_W = {}


def _worker_init(name: str, seed: int, exps: int, limit: int):
    sys.path.insert(0, ROOT)
    from oracle import oracle

    oracle.build()
    _W["packed"] = make_batch(name, seed, exps).pack()
    _W["oracle"] = oracle
    _W["limit"] = limit


def _worker_run(e: int):
    r = _W["oracle"].run(_W["packed"], e, e + 1, _W["limit"])
    return int(r["pkt_hops"][e])


def oracle_sample(name: str, seed: int, budget_s: float, cores: int, exps: int = 0,
                  limit: int = 0xFFFFFFFE):
    """Time the oracle over a seeded sample of experiments, all host cores in
    parallel (one experiment per task, each to completion or to `limit`
    ticks), until about budget_s of wall clock."""
    from oracle import oracle

    oracle.build()
    n_exp = len(make_batch(name, seed, exps))
    order = np.random.default_rng(1234).permutation(n_exp)
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_worker_init, initargs=(name, seed, exps, limit)) as pool:
        pool.map(_worker_run, [int(order[0])] * cores)          # warm the workers
        hops, done, t0 = 0, 0, time.perf_counter()
        while done < n_exp and time.perf_counter() - t0 < budget_s:
            chunk = [int(e) for e in order[done:done + cores]]
            hops += sum(pool.map(_worker_run, chunk))
            done += len(chunk)
        dt = time.perf_counter() - t0
    return hops, dt, done, n_exp


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


# ----------------------------------------------------------------- arms
def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    name = args.workload
    per_step = max(1.0, args.cpu_budget_s / max(1, args.steps + args.warmup))
    lim = args.start_tick + args.max_ticks if (args.start_tick or args.max_ticks) else 0xFFFFFFFE
    for _ in range(args.warmup):
        oracle_sample(name, 0, min(per_step, 5.0), cores, args.exps, lim)
    hops, secs, n_done = 0, 0.0, 0
    for _ in range(args.steps):
        h, dt, done, n_exp = oracle_sample(name, 0, per_step, cores, args.exps, lim)
        hops += h
        secs += dt
        n_done += done
    value = hops / secs
    sample = (f"{n_done // max(1, args.steps)} of {n_exp} experiments per step "
              f"(seeded permutation), one experiment per process")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic", "config": {"workload": name, "desc": WORKLOADS[name][1]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_gpu(args, rank: int, world: int):
    import torch

    from experiment_network_simulation_gb300 import mv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    batch = make_batch(args.workload, seed=rank, exps=args.exps)   # each rank: its own shard
    packed = batch.pack()
    stream = torch.cuda.Stream(dev)
    sim = mv.Simulator(packed, device=str(dev), stream=stream)
    n_levels = int(packed["sw_level"].max())
    launches_per_step = n_levels + 4                  # routes per level, up lists, 2 init, megakernel
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    window = args.start_tick > 0 or args.max_ticks > 0
    budget = args.max_ticks if args.max_ticks > 0 else mv.UNSET - 1

    snap = {}

    def prefix():
        """Untimed: back to tick 0 and, for a window, on to its start tick.
        The simulator's whole state is its workspace, so the window's start
        state is computed once and then restored by a device copy."""
        if args.start_tick:
            if not snap:
                sim.reset()
                rc = sim.run(max_ticks=args.start_tick)
                assert rc in (mv.MV_OK, mv.MV_INCOMPLETE), rc
                c = sim.counters()
                snap["ws"] = sim.ws.clone()
                snap["h"] = (int(c["pkt_hops"].sum()), int(c["pkts_injected"].sum()))
            with torch.cuda.stream(stream):
                sim.ws.copy_(snap["ws"])
        with torch.cuda.stream(stream):
            flush.zero_()                             # L2 flush between steps
        return snap.get("h", (0, 0))

    def timed():
        """The timed region: reset (unless a window) + one megakernel run."""
        if not args.start_tick:
            sim.reset()
        rc = sim.run(max_ticks=budget)
        assert rc in ((mv.MV_OK, mv.MV_INCOMPLETE) if window else (mv.MV_OK,)), rc

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
        with torch.cuda.stream(stream):
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

    # e2e through the public API from host buffers: create (upload), run,
    # results (download); whole runs only
    e2e = None
    if not window and args.e2e_steps > 0:
        h2d = sum(int(np.asarray(v).nbytes) for k, v in packed.items() if k != "version")
        e2e_s, d2h = [], 0
        for _ in range(args.e2e_steps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            s2 = mv.Simulator(packed, device=str(dev), stream=stream)
            s2.run()
            r2 = s2.results()
            s2.close()
            e2e_s.append(time.perf_counter() - t0)
            d2h = sum(int(v.nbytes) for k, v in r2.items() if isinstance(v, np.ndarray)
                      and k not in ("node_offset", "rec_offset"))
            del s2
        e2e = {"value": hops_step / statistics.mean(e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks = load_peaks()
    km = statistics.mean(kernel_ms)
    alg_bytes = BYTES_PER_HOP * hops_step + BYTES_PER_PKT * pkts_step
    achieved = alg_bytes / (km / 1000.0) / 1e9
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": TRAFFIC.get(args.workload) if not window else None,
            "peak_source": "measured" if peaks else "fallback",
            "kernel": "k_megakernel", "kernel_ms": km,
            "alg_bytes_per_launch": alg_bytes}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        lim = args.start_tick + args.max_ticks if window else 0xFFFFFFFE
        h, dt, done, n_exp = oracle_sample(args.workload, 0, args.cpu_budget_s, cores,
                                           args.exps, lim)
        what = f"first {lim} ticks of " if window else ""
        cpu = {"value": h / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{what}{done} of {n_exp} experiments (seeded permutation), "
                         f"{dt:.1f} s wall, one experiment per process"}

    if rank == 0:
        cfg = {"workload": args.workload, "desc": WORKLOADS[args.workload][1],
               "experiments": int(exps_all), "packet_hops_per_step": int(hops_all),
               "l2": "flushed between steps (512 MiB write)",
               "grid_steps_per_run": int(statistics.mean(steps_grid))}
        if window:
            cfg["window"] = {"start_tick": args.start_tick, "max_ticks": args.max_ticks,
                             "note": "each step times ticks [start, start + max) of every "
                                     "experiment's clock; the prefix runs untimed"}
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
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--exps", type=int, default=0, help="first N experiments of the batch")
    ap.add_argument("--start-tick", type=int, default=0,
                    help="run every experiment to this tick before the timed region")
    ap.add_argument("--max-ticks", type=int, default=0,
                    help="timed run budget in ticks of each experiment's clock (0 = to the end)")
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
