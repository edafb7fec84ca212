"""Congestion control (DCQCN and DCTCP) on the CUDA path, bit-exact against
the oracle: the oracle's pin scenarios, seeded random collectives with
aggressive settings in every kernel build, the GPT DAG at test size and
config 1 with the generators' settings."""
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
from test_oracle_cc import _random_batch, cc, tcp  # noqa: E402


def pin_batch():
    ex = []
    t = I.single_switch(3, 1, 0)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 120 * 4096)
    w.collective(I.P2P, [1, 2], 120 * 4096)
    ex.append(I.Experiment(t, w, cap=4, cc=cc(kmin=1, kmax=1), chunk=1 << 30, tick_ps=1000,
                           rec_cap=512))
    for delta in (0, 1, 12):
        ex.append(I.Experiment(I.single_switch(2, 1, delta), I.lone_message(2, 0, 1, 40 * 4096),
                               cc=cc(kmin=1, kmax=1, n=5, k=7, t=9, f=2, rai=100, rhai=100,
                                     rmin=100), chunk=1 << 30, tick_ps=1000, rec_cap=64))
    ex.append(I.Experiment(I.single_switch(2, 64, 0), I.lone_message(2, 0, 1, 400 * 4096),
                           cc=cc(kmin=0, kmax=0, t=300, f=100), chunk=1 << 30, tick_ps=1000,
                           rec_cap=512))
    ex.append(I.Experiment(I.single_switch(2, 1, 0), I.lone_message(2, 0, 1, 300 * 4096),
                           cc=cc(kmin=0, kmax=0, n=50, k=30), chunk=1 << 30, tick_ps=1000,
                           rec_cap=512))
    ex.append(I.Experiment(I.single_switch(2, 1, 0), I.lone_message(2, 0, 1, 300 * 4096),
                           cc=cc(kmin=0, kmax=0, n=25, k=400, t=7, b=3, f=2, rai=1 << 9,
                                 rhai=1 << 10, rmin=1 << 12, gshift=4),
                           chunk=1 << 30, tick_ps=1000, rec_cap=512))
    return I.Batch(ex, "dcqcn-pins")


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_dcqcn_pins_and_random_traffic_bit_exact(variant):
    for b in (pin_batch(), _random_batch(11, 80, cc(kmin=1, kmax=4, pmax=30000, n=5, k=7, t=11,
                                                    b=6, f=2, rai=3000, rhai=20000, rmin=5000))):
        p = b.pack()
        want = O.run(p)
        assert (want["status"] == O.ST_DONE).all()
        assert_same(mv.simulate(p, run_opts=dict(variant=variant)), want)


def test_dcqcn_gpt_small_and_config1_bit_exact():
    b = I.gpt_small(seeds=(0, 1))
    c = I.config1()
    for x in b.experiments + c.experiments:
        x.cc = I.dcqcn(x.tick_ps, x.pkt)
    for batch in (b, c):
        p = batch.pack()
        want = O.run(p)
        assert (want["status"] == O.ST_DONE).all()
        assert_same(mv.simulate(p), want)


def tcp_pin_batch():
    ex = []
    for delta, w in ((0, 2), (0, 3), (2, 2), (1, 5)):
        ex.append(I.Experiment(I.single_switch(2, 1, delta), I.lone_message(2, 0, 1, 24 * 4096),
                               cc=tcp(w0=w, wmax=w), chunk=1 << 30, tick_ps=1000, rec_cap=64))
    ex.append(I.Experiment(I.single_switch(2, 1, 0), I.lone_message(2, 0, 1, 60 * 4096),
                           cc=tcp(w0=1, wmax=4), chunk=1 << 30, tick_ps=1000, rec_cap=64))
    ex.append(I.Experiment(I.single_switch(2, 1, 0), I.lone_message(2, 0, 1, 60 * 4096),
                           cc=tcp(kmark=0, w0=8, wmax=8), chunk=1 << 30, tick_ps=1000, rec_cap=64))
    t = I.single_switch(3, 1, 0)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 150 * 4096)
    w.collective(I.P2P, [1, 2], 150 * 4096)
    ex.append(I.Experiment(t, w, cap=8, cc=tcp(kmark=1, gshift=4, w0=10, wmax=64),
                           chunk=1 << 30, tick_ps=1000, rec_cap=512))
    return I.Batch(ex, "dctcp-pins")


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_dctcp_pins_and_random_traffic_bit_exact(variant):
    for b in (tcp_pin_batch(), _random_batch(13, 80, tcp(kmark=2, gshift=3, w0=2, wmax=12))):
        p = b.pack()
        want = O.run(p)
        assert (want["status"] == O.ST_DONE).all()
        assert_same(mv.simulate(p, run_opts=dict(variant=variant)), want)


def test_dctcp_gpt_small_and_config1_bit_exact():
    b = I.gpt_small(seeds=(0, 1))
    c = I.config1()
    for x in b.experiments + c.experiments:
        x.cc = I.DCTCP()
    for batch in (b, c):
        p = batch.pack()
        want = O.run(p)
        assert (want["status"] == O.ST_DONE).all()
        assert_same(mv.simulate(p), want)


@pytest.mark.parametrize("which", ["dcqcn", "dctcp"])
def test_congestion_control_resumes_and_repeats(which):
    """The congestion-control state (rates, windows, notification rings)
    lives in the workspace: a run in pieces of 50 ticks, stopped at tick
    boundaries, equals one run, which equals the oracle; a second run
    repeats it bit for bit."""
    if which == "dcqcn":
        b = _random_batch(21, 40, cc(kmin=1, kmax=4, pmax=30000, n=5, k=7, t=11, b=6, f=2,
                                     rai=3000, rhai=20000, rmin=5000))
    else:
        b = _random_batch(21, 40, tcp(kmark=2, gshift=3, w0=2, wmax=12))
    p = b.pack()
    once = mv.simulate(p)
    assert_same(once, O.run(p))
    sim = mv.Simulator(p)
    calls = 0
    while sim.run(max_ticks=50) == mv.MV_INCOMPLETE:
        calls += 1
        assert calls < 100_000
    got = sim.results()
    sim.close()
    assert calls > 3
    assert_same(got, once)
    assert_same(mv.simulate(p), once)
