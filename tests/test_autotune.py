"""The <algorithm, NC, C> search (AutoCCL sections 4.1-4.3) on the CPU: its
coordinate descent against a hand-traced run on a separable bandwidth
function, its convergence on unimodal functions, its choice of subspace,
and one search driven by the oracle simulator end to end."""
from fractions import Fraction

import numpy as np
import pytest

from experiment_network_simulation_gb300 import autotune as A
from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O


def fake(time_of):
    """A stand-in simulator: each experiment 'ends' at time_of(algo, NC grid
    index, C grid index)."""
    def sim(packed):
        E = len(packed["exp_topo"])
        end = np.zeros(E, np.uint32)
        for e in range(E):
            nc, c = int(packed["exp_nc"][e]), int(packed["exp_chunk"][e])
            end[e] = time_of(int(packed["exp_algo"][e]), A.GRID_NC.index(nc), A.GRID_C.index(c))
        return {"status": np.zeros(E, np.uint32), "end_tick": end}
    return sim


def one_task():
    return [A.Task(I.single_switch(2, 1, 0), 2, I.AR, 1 << 20, [0, 1])]


def test_coordinate_descent_hand_trace():
    """time = 1000 + 10 (n - 2)^2 + 10 (k - 2)^2 with n, k the NC and C grid
    indices, started at (0, 0).  The start's own profile is no improvement,
    so the first move is along C (lr 0.01: one grid point): C 8K improves
    (1081 -> 1051: lr 30/1051, still one point), 16K improves, 32K does not;
    then NC: 2 improves (lr 30/1011), 3 improves, 4 does not; then C 32K at
    NC 3 does not, and NC 4 (already profiled) does not: three misses in a
    row end it at NC 3, C 16K."""
    def t(algo, n, k):
        return 1000 + 10 * (n - 2) ** 2 + 10 * (k - 2) ** 2
    ch = A.Chain(0, I.RING, [0, 0])
    sim = fake(t)
    while not ch.done:
        r = sim(A.wave_batch(one_task(), [(0, ch.config())], 1000).pack())
        ch.observe(A.bandwidth(1 << 20, int(r["status"][0]), int(r["end_tick"][0])))
    K = 4096
    assert [c[1:] for c, _ in ch.trail] == [(1, K), (1, 2 * K), (1, 4 * K), (1, 8 * K),
                                            (2, 4 * K), (3, 4 * K), (4, 4 * K), (3, 8 * K),
                                            (4, 4 * K)]
    assert ch.config(ch.opt) == (I.RING, 3, 4 * K) and ch.opt_bw == Fraction(1 << 20, 1001)


def test_large_improvement_takes_a_large_step():
    """lr is the improvement relative to the previous optimum: halving the
    time (lr 1) moves the coordinate by the whole grid, clamped to its end."""
    ch = A.Chain(0, I.RING, [0, 0])
    ch.observe(Fraction(1, 100))          # the start: no improvement, next coordinate (C)
    assert ch.p == [0, 1]
    ch.observe(Fraction(2, 100))          # doubled: lr = 1
    assert ch.lr == 1 and ch.p == [0, len(A.GRID_C) - 1]


@pytest.mark.parametrize("peak", [(3, 4), (10, 2), (20, 8)])
def test_converges_on_separable_unimodal_functions(peak):
    """Started below the peak in both coordinates, with gentle slopes (every
    step is one grid point), the search ends at the peak."""
    def t(algo, n, k):
        return 100_000 + 3 * (n - peak[0]) ** 2 + 3 * (k - peak[1]) ** 2
    r = A.search(one_task(), fake(t), starts=1, seed=5, algos=(I.RING,))
    ch = r["chains"][0]
    if ch.trail[0][0][1] - 1 <= peak[0] and A.GRID_C.index(ch.trail[0][0][2]) <= peak[1]:
        assert r["best"][0][1] == (I.RING, peak[0] + 1, A.GRID_C[peak[1]])


def test_subspace_choice_and_memoised_waves():
    """Algorithm 1 keeps the best subspace's optimum; waves simulate each
    distinct (task, config) once."""
    def t(algo, n, k):
        return 5000 + (n - 5) ** 2 + (k - 3) ** 2 + (0 if algo == I.TREE else 700)
    r = A.search(one_task(), fake(t), starts=3, seed=1)
    assert r["best"][0][1][0] == I.TREE
    total = sum(len(c.trail) for c in r["chains"])
    assert r["profiles"] == sum(r["waves"]) <= total


def test_search_driven_by_the_oracle():
    """End to end on the oracle: ring and tree all-reduce of 2 MiB over the
    8 hosts of config 1's leaf-spine fabric; every chain ends, the only
    refused profiles are trees of more than 21 channels (3 send lanes a
    channel exceed the 64 a rank has), and the best has the highest
    bandwidth seen."""
    topo = I.leaf_spine(2, 2, 4, delta=12)
    tasks = [A.Task(topo, 8, I.AR, 2 << 20, list(range(8)), "ar2m")]
    r = A.search(tasks, lambda p: O.run(p), starts=2, seed=3)
    assert all(c.done for c in r["chains"])
    seen = [(cfg, bw) for c in r["chains"] for cfg, bw in c.trail]
    for (algo, nc, _), bw in seen:
        assert (bw == 0) == (algo == I.TREE and nc > 21)
    assert r["best"][0][0] == max(bw for _, bw in seen)
