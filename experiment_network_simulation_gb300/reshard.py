"""Cross-mesh resharding workloads (AlpaComm, "On Optimizing the
Communication of Model Parallelism", MLSys'23), built for the simulator.

  - Unit-task decomposition (appendix B.2): the tensor is cut at every
    shard boundary of the source and the destination layouts, dimension by
    dimension; each cell of the cut is a data slice, and its unit task
    sends it from the source devices that hold it to the destination devices
    that need it (section 2.2).
  - Host-level load balancing and scheduling (section 3.2): each task gets
    one sender host among the hosts holding its slice and a start time, so
    that tasks sharing a host do not overlap and the last task ends as early
    as possible.  Four algorithms: the naive one (lowest sender, task order),
    load balance only (longest task first onto the least loaded sender), a
    depth-first search with pruning, and the randomized greedy search.
  - A task is a pipelined broadcast (section 3.1): the slice cut into K
    partitions relayed along the sender and the receiving hosts, which the
    simulator runs packet by packet (RELAY collectives); a schedule becomes
    per-host chains of memberships in the workload DAG.
  - Eager-1F1B (section 4): stage i (counted from 1) runs 2 (stages - i) + 1
    warm-up forward micro-batches instead of 1F1B's stages - i, so that a
    stage's cross-mesh communication overlaps later micro-batches' compute.

Readings where the page leaves a step open:
  - A mesh is a 2-D array of devices numbered row-major; a dimension sharded
    over several mesh axes (S^01) is split in the product of their sizes,
    indexed row-major over those axes; device d sits on host d // g.
  - Source and destination meshes use disjoint hosts; a task's receiving
    hosts are the hosts of its receiving devices (intra-host copies are
    ignored, as section 3.1 neglects intra-node time).
  - A task's duration is the pipelined-broadcast time t (K + A - 1) / K
    (section 3.1) rounded up, with t its packet count (one tick a packet)
    and A its receiving hosts.
  - A schedule is a priority order of tasks plus a sender per task; a task
    starts when its sender and all its receivers are free (list
    scheduling).  The depth-first search explores orders and senders (the
    task that can start earliest first, then the sender giving the earliest
    start), and prunes a branch once the larger of its makespan so far and,
    for every host, its free time plus the remaining tasks it must take
    part in (as a receiver, or as the only possible sender: the per-device
    sum of durations of the page's bound) reaches the best makespan found;
    it stops after a budget of expanded nodes.
  - The randomized greedy search repeats: shuffle the remaining tasks
    (seeded), take each task in turn with the first of its senders whose
    hosts do not meet those already taken, keep the shuffle whose set spans
    the most hosts; that set is the next round, in the priority order.
"""
from __future__ import annotations

import itertools
import math
from dataclasses import dataclass

import numpy as np

from . import inputs as I


# --------------------------------------------------------------------------
# Unit-task decomposition
# --------------------------------------------------------------------------
@dataclass
class Mesh:
    shape: tuple                 # (m1, m2)
    first_device: int = 0        # devices first_device .. first_device + m1*m2 - 1, row-major

    @property
    def size(self) -> int:
        return self.shape[0] * self.shape[1]

    def device(self, idx: int) -> int:
        return self.first_device + idx

    def coord(self, idx: int) -> tuple:
        return (idx // self.shape[1], idx % self.shape[1])


def held(shape, mesh: Mesh, spec, idx: int) -> list:
    """The [lo, hi) interval of each tensor dimension that mesh device idx
    holds under `spec` (per dimension: None = replicated, or the tuple of
    mesh axes the dimension is sharded over)."""
    c = mesh.coord(idx)
    out = []
    for d, axes in enumerate(spec):
        n = shape[d]
        if not axes:
            out.append((0, n))
            continue
        k, pos = 1, 0
        for a in axes:
            k *= mesh.shape[a]
            pos = pos * mesh.shape[a] + c[a]
        out.append((pos * n // k, (pos + 1) * n // k))
    return out


def cuts(shape, spec, mesh: Mesh, d: int) -> set:
    axes = spec[d]
    k = 1
    for a in (axes or ()):
        k *= mesh.shape[a]
    return {j * shape[d] // k for j in range(k + 1)}


@dataclass
class UnitTask:
    box: tuple                   # per dimension [lo, hi)
    senders: list                # source devices holding the slice
    receivers: list              # destination devices needing it
    nbytes: int


def unit_tasks(shape, src: Mesh, src_spec, dst: Mesh, dst_spec, elem_bytes: int = 2) -> list:
    """Appendix B.2: cut points per dimension from both layouts, slices = the
    Cartesian product of the intervals, one task per slice."""
    ivs = []
    for d in range(len(shape)):
        pts = sorted(cuts(shape, src_spec, src, d) | cuts(shape, dst_spec, dst, d))
        ivs.append(list(zip(pts[:-1], pts[1:])))
    out = []
    for box in itertools.product(*ivs):
        def inside(h):
            return all(a >= lo and b <= hi for (a, b), (lo, hi) in zip(box, h))
        snd = [src.device(i) for i in range(src.size) if inside(held(shape, src, src_spec, i))]
        rcv = [dst.device(i) for i in range(dst.size) if inside(held(shape, dst, dst_spec, i))]
        vol = 1
        for a, b in box:
            vol *= b - a
        out.append(UnitTask(tuple(box), snd, rcv, vol * elem_bytes))
    return out


# --------------------------------------------------------------------------
# Host-level scheduling
# --------------------------------------------------------------------------
@dataclass
class HostTask:
    senders: list                # candidate sender hosts (ascending)
    receivers: list              # receiving hosts (ascending)
    nbytes: int
    dur: int                     # ticks


def host_tasks(tasks, gpus_per_host: int, parts: int, pkt: int = 4096) -> list:
    out = []
    for t in tasks:
        s = sorted({d // gpus_per_host for d in t.senders})
        r = sorted({d // gpus_per_host for d in t.receivers})
        n = max(1, -(-t.nbytes // pkt))
        A = len(r)
        out.append(HostTask(s, r, t.nbytes, -(-n * (parts + A - 1) // parts)))
    return out


@dataclass
class Schedule:
    order: list                  # task indices in priority order
    sender: dict                 # task -> sender host
    start: dict                  # task -> start tick
    makespan: int


def list_schedule(tasks, order, sender) -> Schedule:
    """Each task starts when its sender and every receiver are free."""
    free: dict = {}
    start = {}
    span = 0
    for i in order:
        t = tasks[i]
        hosts = [sender[i]] + t.receivers
        s = max(free.get(h, 0) for h in hosts)
        start[i] = s
        for h in hosts:
            free[h] = s + t.dur
        span = max(span, s + t.dur)
    return Schedule(list(order), dict(sender), start, span)


def naive(tasks) -> Schedule:
    """The lowest-index sender for every task, tasks in their own order."""
    return list_schedule(tasks, range(len(tasks)), {i: t.senders[0] for i, t in enumerate(tasks)})


def load_balance(tasks) -> Schedule:
    """Longest task first, each onto the least loaded of its senders (lowest
    host on ties); tasks then run in that order."""
    order = sorted(range(len(tasks)), key=lambda i: (-tasks[i].dur, i))
    load: dict = {}
    sender = {}
    for i in order:
        h = min(tasks[i].senders, key=lambda x: (load.get(x, 0), x))
        sender[i] = h
        load[h] = load.get(h, 0) + tasks[i].dur
    return list_schedule(tasks, order, sender)


def dfs(tasks, budget: int = 200_000) -> Schedule:
    """Depth-first search over priority orders and senders, pruned by the
    per-host lower bound; the best schedule found within `budget` expanded
    nodes (exact when the search completes)."""
    n = len(tasks)
    best = load_balance(tasks)
    best_span = [best.makespan]
    best_pick = [None]
    expanded = [0]
    recv_left: dict = {}          # per host: durations it must still take part in
    for t in tasks:
        for h in t.receivers + (t.senders if len(t.senders) == 1 else []):
            recv_left[h] = recv_left.get(h, 0) + t.dur

    def go(order, sender, free, span, left):
        if expanded[0] >= budget:
            return
        expanded[0] += 1
        if not left:
            if span < best_span[0]:
                best_span[0] = span
                best_pick[0] = (list(order), dict(sender))
            return
        bound = span
        for h, w in recv_left.items():
            if w:
                bound = max(bound, free.get(h, 0) + w)
        if bound >= best_span[0]:
            return
        # the task that can start earliest first (longest on ties), each
        # sender in the order of the start it gives: good schedules come
        # early, so the bound prunes more
        def start_with(t, h):
            return max(free.get(x, 0) for x in [h] + t.receivers)

        def key(x):
            return (min(start_with(tasks[x], h) for h in tasks[x].senders), -tasks[x].dur, x)
        for i in sorted(left, key=key):
            t = tasks[i]
            for h in sorted(t.senders, key=lambda x: (start_with(t, x), x)):
                hosts = [h] + t.receivers
                s = max(free.get(x, 0) for x in hosts)
                saved = {x: free.get(x, 0) for x in hosts}
                fixed = t.receivers + (t.senders if len(t.senders) == 1 else [])
                for x in hosts:
                    free[x] = s + t.dur
                for x in fixed:
                    recv_left[x] -= t.dur
                order.append(i)
                sender[i] = h
                left.remove(i)
                go(order, sender, free, max(span, s + t.dur), left)
                left.add(i)
                del sender[i]
                order.pop()
                for x in fixed:
                    recv_left[x] += t.dur
                for x, v in saved.items():
                    free[x] = v

    go([], {}, {}, 0, set(range(n)))
    if best_pick[0] is None:
        return best
    return list_schedule(tasks, *best_pick[0])


def randomized_greedy(tasks, tries: int = 16, seed: int = 0) -> Schedule:
    """Rounds of non-overlapping tasks: each round keeps, of `tries` seeded
    shuffles, the greedy set spanning the most hosts."""
    rng = np.random.default_rng(seed)
    left = list(range(len(tasks)))
    order, sender = [], {}
    while left:
        best = None
        for _ in range(tries):
            perm = [left[j] for j in rng.permutation(len(left))]
            used, pick = set(), []
            for i in perm:
                t = tasks[i]
                for h in t.senders:
                    hosts = {h, *t.receivers}
                    if not hosts & used:
                        used |= hosts
                        pick.append((i, h))
                        break
            if best is None or len(used) > best[0]:
                best = (len(used), pick)
        for i, h in best[1]:
            order.append(i)
            sender[i] = h
        taken = {i for i, _ in best[1]}
        left = [i for i in left if i not in taken]
    return list_schedule(tasks, order, sender)


def valid(tasks, sch: Schedule) -> bool:
    """Every task once, its sender one of its candidates, and no two tasks
    that share a host overlapping in time."""
    if sorted(sch.order) != list(range(len(tasks))):
        return False
    iv = {}
    for i, t in enumerate(tasks):
        if sch.sender[i] not in t.senders:
            return False
        for h in [sch.sender[i]] + t.receivers:
            iv.setdefault(h, []).append((sch.start[i], sch.start[i] + t.dur))
    for spans in iv.values():
        spans.sort()
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            if b0 < a1:
                return False
    return True


# --------------------------------------------------------------------------
# Simulation of a schedule
# --------------------------------------------------------------------------
def schedule_workload(tasks, sch: Schedule, n_hosts: int, parts: int) -> I.Workload:
    """One pipelined broadcast (RELAY collective over the sender, then the
    receiving hosts in ascending order, `parts` partitions) per task; on
    every host the memberships follow the schedule's order."""
    w = I.Workload(n_hosts, "reshard")
    last: dict = {}
    for i in sch.order:
        t = tasks[i]
        members = [sch.sender[i]] + t.receivers
        ids = w.collective(I.RELAY, members, t.nbytes, parts=parts)
        for h, u in zip(members, ids):
            if h in last:
                w.edge(last[h], u)
            last[h] = u
    return w


# --------------------------------------------------------------------------
# Eager-1F1B
# --------------------------------------------------------------------------
def warmup_forwards(stages: int, i: int, micro: int, eager: bool) -> int:
    """Forward micro-batches stage i (1-based) runs before its first backward."""
    w = 2 * (stages - i) + 1 if eager else stages - i
    return min(w, micro)


def stage_program(stages: int, i: int, micro: int, eager: bool) -> list:
    """(F|B, micro-batch) in execution order on stage i (1-based): warm-up
    forwards, then one forward and one backward alternately, then the
    remaining backwards."""
    wu = warmup_forwards(stages, i, micro, eager)
    prog = [("F", j) for j in range(wu)]
    f, b = wu, 0
    while b < micro:
        if f < micro:
            if b < f:
                prog.append(("B", b))
                b += 1
            prog.append(("F", f))
            f += 1
        else:
            prog.append(("B", b))
            b += 1
    return prog


def pipeline_workload(stages: int, micro: int, fwd_ns: int, bwd_ns: int, act_bytes: int,
                      eager: bool, parts: int = 1) -> I.Workload:
    """One host per stage.  Stage s's forward of micro-batch j waits for the
    activation of stage s-1 (a point-to-point transfer of act_bytes, or a
    pipelined broadcast of `parts` partitions); its backward waits for the
    gradient of stage s+1.  Transfers are posted when their producer ends
    and do not block the producer's next compute."""
    w = I.Workload(stages, "eager-1f1b" if eager else "1f1b")
    node = {}
    for s in range(stages):
        for fb, j in stage_program(stages, s + 1, micro, eager):
            node[(s, fb, j)] = w.compute(s, fwd_ns if fb == "F" else bwd_ns)
    for s in range(stages):
        prog = stage_program(stages, s + 1, micro, eager)
        w.chain(*[node[(s, fb, j)] for fb, j in prog])
    for j in range(micro):
        for s in range(stages - 1):
            a = w.collective(I.P2P if parts == 1 else I.RELAY, [s, s + 1], act_bytes,
                             parts=0 if parts == 1 else parts)
            w.edge(node[(s, "F", j)], a[0])
            w.edge(a[1], node[(s + 1, "F", j)])
            g = w.collective(I.P2P if parts == 1 else I.RELAY, [s + 1, s], act_bytes,
                             parts=0 if parts == 1 else parts)
            w.edge(node[(s + 1, "B", j)], g[0])
            w.edge(g[1], node[(s, "B", j)])
    return w
