"""Simulator-driven search of the collective parameters <algorithm, NC, C>.

AutoCCL (NSDI'25), section 4.1: the implementation parameters (algorithm,
protocol, transport) split the space into subspaces, searched one by one
(Algorithm 1); inside a subspace the resource parameters are tuned by
coordinate descent (Algorithm 2), which section 4.2 justifies by the
unimodality of bandwidth in each resource parameter when the others are
fixed.  Here the "profile" of a configuration is a packet-level simulation
of the collective: every step of every running search becomes one
experiment, and the experiments of one step are simulated together as one
batch (a wave), which is what the single-process multi-experiment design is
for.

Readings (the listing of Algorithm 2 leaves them open):
  - Subspaces are the algorithms ring and tree (protocol and transport are
    not modelled by the simulator); the resource parameters are NC
    (channels) and C (chunk bytes); the thread count NT has no counterpart.
  - A configuration holds grid indices: NC on GRID_NC, C on GRID_C.  Adding
    the learning rate lr to coordinate `dim` moves it by max(1, ceil(lr *
    grid length)) grid points, clamped to the grid, in the increasing
    direction, as the listing adds lr.
  - lr starts at 0.01 and, after an improvement, becomes the improvement
    relative to the previous optimum (the prose of section 4.3; the listing's
    line is garbled); the coordinate index wraps around the M coordinates.
    The start is the first optimum, so its own profile counts as no
    improvement and the first move is along the second coordinate, as the
    listing runs.  The search of a subspace ends once M + 1 profiles in a
    row did not improve (the loop runs while tuned_dim <= M).
  - Bandwidth is the collective's bytes over its simulated completion time
    (its end tick + 1), kept as an exact fraction, so the decisions do not
    depend on floating-point rounding; a configuration that the simulator
    stops with an error or a table overflow has bandwidth 0.
  - The random start of each search (Algorithm 2's line "randomly generate a
    config") comes from a seeded generator; several starts per subspace may
    run side by side in the same waves.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from fractions import Fraction

import numpy as np

from . import inputs as I

GRID_NC = list(range(1, 33))                       # channels
GRID_C = [4096 << k for k in range(11)]            # 4 KiB .. 4 MiB chunks
GRIDS = (GRID_NC, GRID_C)
M = len(GRIDS)                                     # resource parameters tuned


@dataclass
class Task:
    """One collective to tune: `kind` over `members` of `topo`, `nbytes`."""
    topo: I.Topology
    n_ranks: int
    kind: int
    nbytes: int
    members: list
    name: str = ""

    def workload(self) -> I.Workload:
        return I.single_collective(self.n_ranks, self.kind, self.nbytes, members=self.members)


@dataclass
class Chain:
    """Algorithm 2 on one subspace (algorithm) of one task, from one start."""
    task: int
    algo: int
    p: list                                        # grid indices of the config to profile next
    opt: list = None
    opt_bw: Fraction = Fraction(-1)
    dim: int = 0
    tuned: int = 0
    lr: Fraction = Fraction(1, 100)
    done: bool = False
    trail: list = field(default_factory=list)      # (config, bandwidth) in profile order

    def config(self, idx=None) -> tuple:
        i = self.p if idx is None else idx
        return (self.algo, GRID_NC[i[0]], GRID_C[i[1]])

    def observe(self, bw: Fraction):
        """One pass of Algorithm 2's loop for the profiled config self.p."""
        self.trail.append((self.config(), bw))
        if self.opt is None:                       # the random start is the first optimum
            self.opt, self.opt_bw = list(self.p), bw
        if bw - self.opt_bw > 0:                   # better: keep going along this coordinate
            # (from a configuration the simulator refused, any working one is
            # an unbounded improvement: the largest step)
            self.lr = (bw - self.opt_bw) / self.opt_bw if self.opt_bw > 0 else Fraction(1)
            self.opt, self.opt_bw, self.tuned = list(self.p), bw, 0
        else:                                      # not better: the next coordinate
            self.tuned += 1
            self.dim = (self.dim + 1) % M
            self.lr = Fraction(1, 100)
        if self.tuned > M:
            self.done = True
            return
        q = list(self.opt)
        n = len(GRIDS[self.dim])
        q[self.dim] = min(n - 1, q[self.dim] + max(1, math.ceil(self.lr * n)))
        self.p = q


def bandwidth(nbytes: int, status: int, end_tick: int) -> Fraction:
    if status != 0:
        return Fraction(0)
    return Fraction(max(1, nbytes), end_tick + 1)


def wave_batch(tasks, configs, tick_ps: int, pkt: int = 4096, cap: int = 64) -> I.Batch:
    """One experiment per (task index, algorithm, NC, C)."""
    works = {}
    exps = []
    for ti, (algo, nc, c) in configs:
        t = tasks[ti]
        if ti not in works:
            works[ti] = t.workload()
        exps.append(I.Experiment(t.topo, works[ti], algo, nc, c, pkt, cap, tick_ps,
                                 label=dict(task=ti, algo=algo, nc=nc, chunk=c)))
    return I.Batch(exps, "autoccl-wave")


def search(tasks, simulate, starts: int = 1, seed: int = 0, tick_ps: int = 81920,
           algos=(I.RING, I.TREE), max_waves: int = 1000) -> dict:
    """Algorithm 1 over every task: a coordinate-descent chain per (task,
    algorithm, start), all chains stepped together, one wave of
    experiments per step.  `simulate(packed)` returns per-experiment
    (status, end_tick) arrays for a packed batch -- the CUDA library or the
    oracle.  Profiles are memoised per (task, config).  Returns the best
    config per task, the chains and the waves' sizes."""
    rng = np.random.default_rng(seed)
    chains = []
    for ti in range(len(tasks)):
        for algo in algos:
            for _ in range(starts):
                p = [int(rng.integers(len(g))) for g in GRIDS]
                chains.append(Chain(ti, algo, p))
    memo: dict = {}
    waves = []
    for _ in range(max_waves):
        live = [c for c in chains if not c.done]
        if not live:
            break
        want = []
        for c in live:
            key = (c.task, c.config())
            if key not in memo and key not in want:
                want.append(key)
        if want:
            r = simulate(wave_batch(tasks, want, tick_ps).pack())
            for j, key in enumerate(want):
                memo[key] = bandwidth(tasks[key[0]].nbytes, int(r["status"][j]),
                                      int(r["end_tick"][j]))
        waves.append(len(want))
        for c in live:
            c.observe(memo[(c.task, c.config())])
    best = {}
    for c in chains:
        if c.opt is None:
            continue
        cur = best.get(c.task)
        cand = (c.opt_bw, c.config(c.opt))
        if cur is None or cand[0] > cur[0]:
            best[c.task] = cand
    return {"best": best, "chains": chains, "waves": waves, "profiles": len(memo)}
