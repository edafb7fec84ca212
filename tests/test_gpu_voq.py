"""Switches with virtual output queues (the VOQ variant of the pull-based
forwarding of Multiverse section 4.2) on the CUDA path, bit-exact against
the oracle: the VOQ pin traffic, random collectives on small fabrics in every
kernel build, the GPT DAG at test size and config 1 with VOQs."""
import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from experiment_network_simulation_gb300 import mv  # noqa: E402
from test_gpu_parity import assert_same  # noqa: E402


def voq_batch(seed=17, n=60):
    rng = np.random.default_rng(seed)
    ex = []
    w = I.Workload(5)
    for a, b in ((0, 1), (0, 3), (2, 1), (4, 1)):
        w.collective(I.P2P, [a, b], 8 * 4096)
    ex.append(I.Experiment(I.single_switch(5, 1, 0), w, chunk=1 << 20, cap=4, tick_ps=1000,
                           voq=1, rec_cap=64))
    for _ in range(n):
        delta = int(rng.integers(0, 3))
        t = [I.single_switch(6, 1, delta), I.leaf_spine(2, 2, 3, delta),
             I.fat_tree(4, delta)][int(rng.integers(3))]
        H = t.n_hosts
        kind = int(rng.choice([I.AR, I.RS, I.AG, I.RELAY, I.P2P, I.A2A]))
        k = 2 if kind == I.P2P else int(rng.integers(2, min(H, 6) + 1))
        ranks = [int(x) for x in rng.choice(H, k, replace=False)]
        w = I.Workload(H)
        if kind == I.A2A:
            w.collective(I.A2A, ranks, 0, a2a={(i, j): int(rng.integers(0, 5)) * 4096 + 7
                                              for i in range(k) for j in range(k) if i != j})
        elif kind == I.RELAY:
            w.collective(I.RELAY, ranks, int(rng.integers(1, 30)) * 4096 + 11,
                         parts=int(rng.integers(1, 5)))
        else:
            w.collective(kind, ranks, int(rng.integers(1, 30)) * 4096 + 11)
        ex.append(I.Experiment(t, w, algo=int(rng.integers(2)), nc=int(rng.integers(1, 4)),
                               chunk=int(rng.choice([4096, 3 * 4096, 1 << 20])),
                               cap=int(rng.integers(2, 9)), tick_ps=1000, voq=1,
                               ecmp_seed=int(rng.integers(1 << 20)), rec_cap=64))
    return I.Batch(ex, "voq")


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_voq_scenarios_bit_exact(variant):
    p = voq_batch().pack()
    want = O.run(p)
    assert (want["status"] == O.ST_DONE).all()
    assert_same(mv.simulate(p, run_opts=dict(variant=variant)), want)


def test_voq_gpt_small_and_config1_bit_exact():
    b = I.gpt_small(seeds=(0, 1))
    c = I.config1()
    for x in b.experiments + c.experiments:
        x.voq = 1
    for batch in (b, c):
        p = batch.pack()
        want = O.run(p)
        assert (want["status"] == O.ST_DONE).all()
        assert_same(mv.simulate(p), want)
