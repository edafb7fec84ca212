"""Degenerate and boundary scenarios pinned on the oracle, bit-exact through
the CUDA path, and the oracle pins' seeded random collectives on small fabrics
through every kernel build."""
import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from experiment_network_simulation_gb300 import mv  # noqa: E402
from test_gpu_parity import assert_same, records  # noqa: E402


def degenerate_batch():
    ex = []
    ex.append(I.Experiment(I.single_switch(2, 1, 3), I.lone_message(2, 0, 1, 0), chunk=1 << 20,
                           tick_ps=1000, rec_cap=4))                       # zero-byte message
    ex.append(I.Experiment(I.single_switch(2, 1, 0), I.lone_message(2, 0, 1, 5 * 4096 + 100),
                           chunk=8192, tick_ps=1000, rec_cap=8))          # p2p chunks
    ex.append(I.Experiment(I.single_switch(3, 1, 0), I.single_collective(3, I.AR, 4096),
                           algo=I.TREE, nc=1, chunk=4096, tick_ps=1000))  # 3-member tree
    ex.append(I.Experiment(I.single_switch(1, 1, 0), I.single_collective(1, I.AR, 4096),
                           tick_ps=1000))                                  # 1-member collective
    t = I.Topology("leaves-linked")
    l0, l1, sp = t.add_switch(1), t.add_switch(1), t.add_switch(2)
    hs = t.add_hosts(16)
    for h in hs[:8]:
        t.attach_host(h, l0)
    for h in hs[8:]:
        t.attach_host(h, l1)
    t.link(l0, sp)
    t.link(l1, sp)
    t.link(l0, l1)
    w = I.Workload(16)
    for i in range(8):
        w.collective(I.P2P, [i, 8 + i], 2 * 4096)
        w.collective(I.P2P, [8 + i, i], 2 * 4096)
    ex.append(I.Experiment(t, w, chunk=1 << 20, tick_ps=1000))          # same-level link
    for d in (0xFFF00000 - 1, 0xFFF00000):                               # tick limit boundary
        w = I.Workload(1)
        w.compute(0, d)
        ex.append(I.Experiment(I.single_switch(1, 1, 0), w, tick_ps=1000))
    w = I.Workload(3)                                                      # failure tick (R31)
    w.collective(I.P2P, [0, 1], 4096)
    c = w.compute(2, 2)
    for _ in range(17):
        u = w.collective(I.AR, [2], 1000, intra=True, alpha=5, beta=(1, 1))[0]
        w.edge(c, u)
    ex.append(I.Experiment(I.single_switch(3, 1, 0), w, chunk=1 << 20, tick_ps=1000, rec_cap=4))
    ex.append(I.Experiment(I.single_switch(2, 1, 0), I.Workload(2), tick_ps=1000))   # no nodes
    w = I.Workload(4)                                  # ranks 1 and 3 have no nodes
    w.collective(I.P2P, [0, 2], 3 * 4096)
    ex.append(I.Experiment(I.single_switch(4, 1, 1), w, chunk=1 << 20, tick_ps=1000))
    return I.Batch(ex, "degenerate")


def test_degenerate_scenarios_bit_exact():
    p = degenerate_batch().pack()
    got, want = mv.simulate(p), O.run(p)
    assert_same(got, want)
    for e in range(len(want["status"])):
        cap = int(p["exp_rec_cap"][e])
        if cap:
            assert records(got, e, cap) == records(want, e, cap)


def random_batch(seed=2024, n=200):
    """The oracle pins' seeded random collectives on small fabrics."""
    rng = np.random.default_rng(seed)
    ex = []
    for _ in range(n):
        fab = int(rng.integers(3))
        delta, sigma = int(rng.integers(0, 4)), int(rng.integers(1, 3))
        if fab == 0:
            t = I.single_switch(6, sigma, delta)
        elif fab == 1:
            t = I.leaf_spine(2, 2, 3, delta, sigma=sigma)
        else:
            t = I.fat_tree(4, delta, sigma=sigma)
        H = t.n_hosts
        kind = int(rng.choice([I.AR, I.RS, I.AG, I.RELAY, I.P2P, I.A2A]))
        k = 2 if kind == I.P2P else int(rng.integers(2, min(H, 6) + 1))
        ranks = [int(x) for x in rng.choice(H, k, replace=False)]
        w = I.Workload(H)
        nbytes = int(rng.choice([0, 1, 4095, 4096, 4097,
                                 int(rng.integers(1, 40)) * 4096 + int(rng.integers(0, 4096))]))
        if kind == I.A2A:
            m = {(i, j): int(rng.integers(0, 5)) * 4096 + int(rng.integers(0, 100))
                 for i in range(k) for j in range(k) if i != j}
            w.collective(I.A2A, ranks, 0, a2a=m)
        elif kind == I.RELAY:
            w.collective(I.RELAY, ranks, nbytes, parts=int(rng.integers(1, 6)))
        else:
            w.collective(kind, ranks, nbytes)
        ex.append(I.Experiment(t, w, algo=int(rng.integers(2)), nc=int(rng.integers(1, 5)),
                               chunk=int(rng.choice([4096, 8192, 3 * 4096 + 7, 1 << 20])),
                               cap=int(rng.integers(2, 17)), tick_ps=1000,
                               ecmp_seed=int(rng.integers(1 << 30)), rec_cap=16))
    return I.Batch(ex, "random")


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_random_scenarios_bit_exact(variant):
    p = random_batch().pack()
    want = O.run(p)
    sim = mv.Simulator(p)
    sim.run(variant=variant)
    got = sim.results()
    sim.close()
    assert_same(got, want)
    for e in range(len(want["status"])):
        assert records(got, e, 16) == records(want, e, 16)
