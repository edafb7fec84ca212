"""CUDA path vs the CPU oracle, element by element (all results are integers,
so the bar is bit-exact): per-experiment counters, per-node start and end
ticks, per-collective first start and last end, and, where an experiment
keeps them, its per-message completion records (sender node, connection
key, delivery tick), compared as sorted lists since the order in which
records are produced is not a result.  Every call goes through the C ABI."""
import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from experiment_network_simulation_gb300 import mv  # noqa: E402

KEYS = ["status", "end_tick", "now", "pkts_injected", "pkt_hops", "pkts_delivered",
        "msgs_delivered", "digest", "rec_count"]


def records(res, e, cap):
    a = res["rec_offset"][e]
    n = min(int(res["rec_count"][e]), cap)
    return sorted(zip(res["rec_sender"][a:a + n].tolist(), res["rec_key"][a:a + n].tolist(),
                      res["rec_tick"][a:a + n].tolist()))


def assert_same(got, want, exps=None):
    E = len(want["status"])
    idx = range(E) if exps is None else exps
    for k in KEYS:
        g = np.array([got[k][e] for e in idx])
        w = np.array([want[k][e] for e in idx])
        bad = np.nonzero(g != w)[0]
        assert bad.size == 0, f"{k}: first mismatch at exp {list(idx)[bad[0]]}: {g[bad[0]]} != {w[bad[0]]}"
    for e in idx:
        a, b = want["node_offset"][e], want["node_offset"][e + 1]
        for k in ("node_start", "node_end"):
            g, w = got[k][a:b], want[k][a:b]
            bad = np.nonzero(g != w)[0]
            assert bad.size == 0, f"{k} exp {e} node {bad[0]}: {g[bad[0]]} != {w[bad[0]]}"
        a, b = want["coll_offset"][e], want["coll_offset"][e + 1]
        assert got["coll_offset"][e] == a and got["coll_offset"][e + 1] == b
        for k in ("coll_start", "coll_end"):
            g, w = got[k][a:b], want[k][a:b]
            bad = np.nonzero(g != w)[0]
            assert bad.size == 0, f"{k} exp {e} coll {bad[0]}: {g[bad[0]]} != {w[bad[0]]}"
        cap = int(want["rec_offset"][e + 1] - want["rec_offset"][e])
        if cap:
            assert records(got, e, cap) == records(want, e, cap), f"records of exp {e}"


def every_record(batch, cap):
    """Keep up to `cap` per-message records in every experiment."""
    for x in batch.experiments:
        x.rec_cap = cap
    return batch


def pin_batch():
    """The oracle's pin scenarios, in one batch of mixed topologies."""
    ex = []
    for d in (0, 1, 12):
        for n in (1, 7, 40):
            t = I.single_switch(2, 1, d)
            ex.append(I.Experiment(t, I.lone_message(2, 0, 1, n * 4096), chunk=1 << 30, tick_ps=1000))
            t = I.fat_tree(4, d)
            ex.append(I.Experiment(t, I.lone_message(16, 0, 15, n * 4096), chunk=1 << 30,
                                   tick_ps=1000, rec_cap=4))
    # incast with tight credit
    t = I.single_switch(3, 1, 1)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 3 * 4096)
    w.collective(I.P2P, [1, 2], 3 * 4096)
    ex.append(I.Experiment(t, w, chunk=1 << 20, cap=2, tick_ps=1000, rec_cap=8))
    # trees with internal members: depth 2 with one and with two channels
    ex.append(I.Experiment(I.single_switch(4, 1, 0), I.single_collective(4, I.AR, 2 * 4096),
                           algo=I.TREE, nc=1, chunk=4096, tick_ps=1000, rec_cap=64))
    for t in (I.single_switch(7, 1, 3), I.leaf_spine(2, 2, 4, 2)):
        ex.append(I.Experiment(t, I.single_collective(7, I.AR, 4 * 4096), algo=I.TREE, nc=2,
                               chunk=4096, tick_ps=1000, rec_cap=64))
    # the largest legal switch and link delay: 64 ports, delta 63
    ex.append(I.Experiment(I.single_switch(64, 1, 63), I.single_collective(64, I.AR, 64 * 4096),
                           nc=2, chunk=8192, cap=130, tick_ps=1000))
    # pipelined broadcast
    for A, K, npk in ((1, 3, 2), (3, 5, 3), (7, 16, 1)):
        ex.append(I.Experiment(I.single_switch(A + 1, 1, 0), I.relay_chain(A + 1, K * npk * 4096, K),
                               tick_ps=1000))
    # rings, trees, all-to-all
    for kind in (I.AR, I.RS, I.AG):
        ex.append(I.Experiment(I.single_switch(5, 1, 2), I.single_collective(5, kind, 3 * I.MIB + 777),
                               nc=3, chunk=100_000, tick_ps=1000))
    ex.append(I.Experiment(I.single_switch(7, 1, 1), I.single_collective(7, I.AR, 64 * 4096),
                           algo=I.TREE, nc=2, chunk=8 * 4096, tick_ps=1000))
    ex.append(I.Experiment(I.leaf_spine(2, 2, 4, 3), I.single_collective(8, I.AR, I.MIB + 5),
                           algo=I.TREE, nc=4, chunk=16 * 4096, tick_ps=1000))
    w = I.Workload(4)
    rng = np.random.default_rng(3)
    m = {(i, j): int(rng.integers(0, 9)) * 4096 + int(rng.integers(0, 3)) for i in range(4)
         for j in range(4) if i != j}
    w.collective(I.A2A, [0, 1, 2, 3], 0, a2a=m)
    ex.append(I.Experiment(I.leaf_spine(2, 2, 2, 1), w, nc=2, chunk=3 * 4096, tick_ps=1000))
    # compute DAG + analytic intra-server collective + memory check
    w = I.Workload(4)
    pre = [w.compute(r, 1000 * (3 + 2 * r), 1000 * (9 + 2 * r), key=r) for r in range(4)]
    ids = w.collective(I.AR, [0, 1, 2, 3], 8000, intra=True, alpha=7, beta=(1, 1000))
    for p_, u in zip(pre, ids):
        w.edge(p_, u)
    ex.append(I.Experiment(I.single_switch(4, 1, 0), w, tick_ps=1000, dur_seed=5))
    w = I.Workload(1)
    w.compute(0, 5)
    w.set_memory_model(13_000_000_000, 8, 4, 10, 8, 2048, 1, 5120, 40)
    ex.append(I.Experiment(I.single_switch(1, 1, 0), w, tick_ps=1000, gpu_mem=12_476_883_199))
    # deadlock
    w = I.Workload(2)
    a = w.collective(I.P2P, [0, 1], 4096)
    b = w.collective(I.P2P, [1, 0], 4096)
    w.edge(b[1], a[0])
    w.edge(a[1], b[0])
    ex.append(I.Experiment(I.single_switch(2, 1, 0), w, tick_ps=1000, chunk=1 << 20))
    return I.Batch(ex, "pins")


def test_pin_scenarios_bit_exact():
    p = pin_batch().pack()
    got, want = mv.simulate(p), O.run(p)
    assert_same(got, want)
    assert (want["status"] != O.ST_RUNNING).all()
    assert O.ST_OOM in want["status"] and O.ST_DEADLOCK in want["status"]


def test_config1_bit_exact():
    """Config 1 whole, every message's completion record included."""
    p = every_record(I.config1(), 1 << 14).pack()
    got, want = mv.simulate(p), O.run(p)
    assert (want["rec_count"] <= 1 << 14).all() and (want["rec_count"] > 0).all()
    assert_same(got, want)
    assert (got["status"] == mv.EXP_DONE).all()


def test_config2_bit_exact():
    """Config 2 whole, every message's completion record included."""
    p = every_record(I.config2(), 1 << 11).pack()
    got, want = mv.simulate(p), O.run(p)
    assert (want["rec_count"] <= 1 << 11).all() and (want["rec_count"] > 0).all()
    assert_same(got, want)
    assert (got["status"] == mv.EXP_DONE).all()


def test_batch_composition_invariance():
    """SPME correctness: an experiment's results do not depend on which
    other experiments share the batch or on its position in it."""
    b = I.config1()
    full = mv.simulate(b.pack())
    for idx in ([5], [15, 2], [3, 9, 0]):
        sub = mv.simulate(b.subset(idx).pack())
        for j, e in enumerate(idx):
            for k in KEYS:
                assert sub[k][j] == full[k][e], (k, e)
            a, z = full["node_offset"][e], full["node_offset"][e + 1]
            a2, z2 = sub["node_offset"][j], sub["node_offset"][j + 1]
            assert np.array_equal(sub["node_end"][a2:z2], full["node_end"][a:z])


def test_resume_equals_one_run():
    """State stays on the device: run(a) then run(b)... equals one run."""
    p = I.config2(n_exp=24).pack()
    once = mv.simulate(p)
    sim = mv.Simulator(p)
    calls = 0
    while sim.run(max_ticks=3000) == mv.MV_INCOMPLETE:
        calls += 1
        assert calls < 10_000
    got = sim.results()
    sim.close()
    assert calls > 3
    assert_same(got, once)


def test_tick_budget_reports_incomplete():
    p = I.config1().pack()
    sim = mv.Simulator(p)
    assert sim.run(max_ticks=100) == mv.MV_INCOMPLETE
    r = sim.results()
    assert (r["status"] == mv.EXP_RUNNING).all()
    assert (r["now"] >= 100).all()
    sim.close()


def test_repeatable():
    p = I.config2(n_exp=40, seed=3).pack()
    a, b = mv.simulate(p), mv.simulate(p)
    assert_same(a, b)


def test_watchdog_stops_at_a_tick_boundary_and_resumes():
    """The run watchdog fires: every block stops its experiment at a tick
    boundary, the call returns MV_ETIMEOUT (no hang, no fault), and a later
    run continues from the saved state to the oracle's exact results."""
    p = I.config1().pack()
    sim = mv.Simulator(p)
    with pytest.raises(mv.MVError) as ei:
        sim.run(watchdog_ns=1)
    assert ei.value.code == mv.MV_ETIMEOUT
    mid = sim.results()
    assert (mid["status"] == mv.EXP_RUNNING).any()
    assert sim.run() == mv.MV_OK
    got = sim.results()
    sim.close()
    assert_same(got, O.run(p))


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("stage", [mv.STAGE_AUTO, mv.STAGE_WAKE, mv.STAGE_NONE])
def test_every_build_and_staging_bit_exact(stage, variant):
    """The same batches through the four kernel builds (one block an SM
    with a register copy of the view and one switch a pass; two 8-warp blocks
    an SM, one 16-warp block or one 32-warp block, with the shared view and
    up to four switches a pass), with the state staged in shared memory by
    priority, only the wake table staged, or nothing staged, and other block
    shapes."""
    for p in (pin_batch().pack(), I.config1().pack(), I.gpt_small(seeds=(4,)).pack()):
        want = O.run(p)
        for warps in (0, 1, 3, 16, 32):
            got = mv.simulate(p, run_opts=dict(stage=stage, block_warps=warps, variant=variant))
            assert_same(got, want)


@pytest.mark.parametrize("variant", [1, 2])
def test_table_limits_match_oracle(variant):
    """At and one past each per-rank table limit, in both register builds
    (their per-rank table strides are sized from the DAG, so this pins that
    the overflow status appears exactly where the fixed-size tables put it)."""
    p = I.table_limits().pack()
    got = mv.simulate(p, run_opts=dict(variant=variant))
    assert_same(got, O.run(p))


@pytest.mark.parametrize("algo", [I.RING, I.TREE])
def test_gpt_small_bit_exact(algo):
    """The config-3 DAG shape (1F1B, analytic TP all-reduces, pipeline p2p,
    chained DP all-reduces) at test size, three duration seeds."""
    p = I.gpt_small(algo=algo, seeds=(0, 1, 2)).pack()
    got, want = mv.simulate(p), O.run(p)
    assert_same(got, want)
    assert (got["status"] == mv.EXP_DONE).all()
