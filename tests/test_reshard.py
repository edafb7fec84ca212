"""Cross-mesh resharding (AlpaComm sections 2.2, 3.1, 3.2, 4 and appendix
B.2) on the CPU: unit tasks of hand-derived layouts, the four host-level
schedulers against hand-worked cases and brute force, the schedules run on
the oracle simulator, and the eager-1F1B program."""
import itertools

import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from experiment_network_simulation_gb300 import reshard as R
from oracle import oracle as O


# ---------------------------------------------------------------- unit tasks
def test_unit_tasks_rows_to_row_pairs():
    """A 4x4 tensor from S^01 R on a 2x2 mesh (devices 0-3, one row each)
    to S^0 R on another 2x2 mesh (devices 4-7: rows 0-1 on 4 and 5, rows 2-3
    on 6 and 7): the cuts are the four rows, so four tasks, each one row
    (4 elements of 2 bytes) from one source device to two destination
    devices."""
    t = R.unit_tasks((4, 4), R.Mesh((2, 2), 0), [(0, 1), None], R.Mesh((2, 2), 4),
                     [(0,), None])
    assert [(x.box, x.senders, x.receivers, x.nbytes) for x in t] == [
        (((0, 1), (0, 4)), [0], [4, 5], 8), (((1, 2), (0, 4)), [1], [4, 5], 8),
        (((2, 3), (0, 4)), [2], [6, 7], 8), (((3, 4), (0, 4)), [3], [6, 7], 8)]


def test_unit_tasks_rows_to_columns():
    """S^0 R (row halves, replicated along mesh axis 1) to R S^1 (column
    halves, replicated along mesh axis 0): cuts at 2 in both dimensions, so
    four 2x2 blocks; block (rows 0-1, cols 0-1) is held by source devices 0
    and 1 and needed by destination devices 4 and 6."""
    t = R.unit_tasks((4, 4), R.Mesh((2, 2), 0), [(0,), None], R.Mesh((2, 2), 4),
                     [None, (1,)])
    got = {x.box: (x.senders, x.receivers) for x in t}
    assert got == {((0, 2), (0, 2)): ([0, 1], [4, 6]), ((0, 2), (2, 4)): ([0, 1], [5, 7]),
                   ((2, 4), (0, 2)): ([2, 3], [4, 6]), ((2, 4), (2, 4)): ([2, 3], [5, 7])}


def _spec(rng):
    """A layout of a 3-D tensor that uses each mesh axis at most once."""
    while True:
        s = [[None, (0,), (1,), (0, 1), (1, 0)][int(rng.integers(5))] for _ in range(3)]
        axes = [a for x in s if x for a in x]
        if len(axes) == len(set(axes)):
            return s


def test_unit_tasks_cover_the_tensor_once():
    """Over random layouts, the slices partition the tensor and each has a
    holder and a consumer."""
    rng = np.random.default_rng(0)
    for _ in range(30):
        src, dst = R.Mesh((2, 4), 0), R.Mesh((4, 2), 8)
        ss, ds = _spec(rng), _spec(rng)
        t = R.unit_tasks((8, 16, 8), src, ss, dst, ds, elem_bytes=1)
        assert sum(x.nbytes for x in t) == 8 * 16 * 8
        assert all(x.senders and x.receivers for x in t)


# ---------------------------------------------------------------- schedulers
def HT(s, r, d):
    return R.HostTask(s, r, 0, d)


def test_duration_is_the_pipelined_broadcast_time():
    """t (K + A - 1) / K rounded up: 10 packets, 3 receiving hosts, K = 4:
    ceil(10 * 6 / 4) = 15."""
    ut = R.UnitTask(((0, 1),), [0], [4, 8, 12], 10 * 4096)
    (h,) = R.host_tasks([ut], gpus_per_host=4, parts=4)
    assert (h.senders, h.receivers, h.dur) == ([0], [1, 2, 3], 15)


def test_naive_and_load_balance_hand_cases():
    """Tasks (senders, receivers, duration): a ({0,1} -> {5}, 5),
    b ({0,1} -> {6}, 4), c ({0} -> {7}, 3).  Naive: all from host 0, in
    order: 0-5, 5-9, 9-12.  Load balance: longest first onto the least
    loaded sender: a on 0, b on 1, c on 0 (load 5 vs 4: 1 is lighter but c
    can only use 0); so a 0-5, b 0-4, c 5-8: makespan 8."""
    ts = [HT([0, 1], [5], 5), HT([0, 1], [6], 4), HT([0], [7], 3)]
    nv = R.naive(ts)
    assert (nv.start, nv.makespan) == ({0: 0, 1: 5, 2: 9}, 12)
    lb = R.load_balance(ts)
    assert lb.sender == {0: 0, 1: 1, 2: 0} and lb.start == {0: 0, 1: 0, 2: 5}
    assert lb.makespan == 8 and R.valid(ts, nv) and R.valid(ts, lb)


def brute(ts):
    best = None
    for order in itertools.permutations(range(len(ts))):
        for snd in itertools.product(*[t.senders for t in ts]):
            sch = R.list_schedule(ts, order, dict(enumerate(snd)))
            if best is None or sch.makespan < best:
                best = sch.makespan
    return best


@pytest.mark.parametrize("seed", range(12))
def test_dfs_is_exact_and_others_are_valid(seed):
    """On small random instances the pruned search reaches the brute-force
    optimum, and every scheduler's schedule is valid."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 6))
    ts = []
    for _ in range(n):
        k = int(rng.integers(1, 3))
        s = sorted(rng.choice(3, k, replace=False).tolist())
        r = sorted((3 + rng.choice(3, int(rng.integers(1, 3)), replace=False)).tolist())
        ts.append(HT(s, r, int(rng.integers(1, 9))))
    d = R.dfs(ts)
    assert R.valid(ts, d) and d.makespan == brute(ts)
    for f in (R.naive, R.load_balance, lambda x: R.randomized_greedy(x, seed=seed)):
        sch = f(ts)
        assert R.valid(ts, sch) and sch.makespan >= d.makespan


def test_randomized_greedy_rounds_do_not_overlap():
    """Eight identical tasks, each from host 0 or 1 to a receiver of its own:
    rounds of two, so four rounds and a makespan of 4 durations."""
    ts = [HT([0, 1], [2 + i], 3) for i in range(8)]
    g = R.randomized_greedy(ts, seed=4)
    assert R.valid(ts, g) and g.makespan == 12


# ---------------------------------------------------------------- simulation
def test_schedule_runs_in_order_on_the_simulator():
    """The schedule as a workload: on every host, memberships start in the
    schedule's order, and every task's broadcast completes."""
    ut = R.unit_tasks((8, 64, 64), R.Mesh((2, 4), 0), [(0,), (1,), None], R.Mesh((2, 4), 8),
                      [None, (0,), (1,)], elem_bytes=2)
    hts = R.host_tasks(ut, gpus_per_host=4, parts=4)
    sch = R.load_balance(hts)
    w = R.schedule_workload(hts, sch, n_hosts=4, parts=4)
    r = O.run(I.Batch([I.Experiment(I.single_switch(4, 1, 0), w, tick_ps=1000)]).pack())
    assert r["status"][0] == O.ST_DONE
    starts = r["node_start"]
    arrs = w.arrays()
    host_of = np.repeat(np.arange(4), arrs["rank_nnodes"])
    for h in range(4):
        s = starts[host_of == h]
        assert list(s) == sorted(s)        # nodes of a host are in schedule order


# ---------------------------------------------------------------- eager-1F1B
def test_eager_warmup_counts():
    """1F1B's stage i (from 1) runs stages - i warm-up forwards; eager-1F1B
    runs 2 (stages - i) + 1, capped by the micro-batches."""
    assert [R.warmup_forwards(4, i, 16, False) for i in (1, 2, 3, 4)] == [3, 2, 1, 0]
    assert [R.warmup_forwards(4, i, 16, True) for i in (1, 2, 3, 4)] == [7, 5, 3, 1]
    assert R.warmup_forwards(4, 1, 5, True) == 5


@pytest.mark.parametrize("eager", [False, True])
def test_stage_program_shape(eager):
    for st, i, m in ((4, 1, 8), (4, 4, 8), (3, 2, 2), (2, 1, 6)):
        prog = R.stage_program(st, i, m, eager)
        assert sorted(prog) == sorted([("F", j) for j in range(m)] + [("B", j) for j in range(m)])
        for j in range(m):
            assert prog.index(("F", j)) < prog.index(("B", j))
        wu = R.warmup_forwards(st, i, m, eager)
        assert all(x[0] == "F" for x in prog[:wu])


def test_eager_overlaps_communication():
    """With transfers as long as a compute step, eager-1F1B ends no later
    than 1F1B on the simulator (section 4: it puts other micro-batches'
    compute between two dependent tasks)."""
    ends = {}
    for eager in (False, True):
        w = R.pipeline_workload(4, 6, 40_000, 80_000, 32 * 4096, eager)
        e = I.Experiment(I.single_switch(4, 1, 0), w, chunk=1 << 30, tick_ps=81920)
        r = O.run(I.Batch([e]).pack())
        assert r["status"][0] == O.ST_DONE
        ends[eager] = int(r["end_tick"][0])
    assert ends[True] <= ends[False]
