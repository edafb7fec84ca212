"""The oracle's pausable run (used to time a window of ticks on the CPU)
gives the same results as one uninterrupted run: advancing in pieces, and
advancing a copy of a paused state, change nothing."""
import numpy as np

from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O


def test_pieces_and_copies_equal_one_run():
    p = I.gpt_small(seeds=(0, 3)).pack()
    whole = O.run(p)
    for e in (0, 1):
        a = O.Paused(p, e)
        a.advance(2_500)
        b = a.clone()
        a.advance(5_000)
        c = a.clone()
        for x in (a, b, c):
            x.advance(O.UNSET - 1)
            r = x.counters()
            assert r["status"] == O.ST_DONE
            for k in ("pkts_injected", "pkt_hops", "pkts_delivered", "msgs_delivered"):
                assert r[k] == int(whole[k][e]), (e, k)
        for x in (c, b, a):
            x.close()


def test_a_paused_run_stops_at_its_limit():
    p = I.config1().pack()
    r = O.run(p, 0, 1, limit=1000)
    a = O.Paused(p, 0)
    assert a.advance(1000) == O.ST_RUNNING
    got = a.counters()
    for k in ("pkts_injected", "pkt_hops", "pkts_delivered", "msgs_delivered"):
        assert got[k] == int(r[k][0]), k
    assert got["clock"] == int(r["now"][0])
    a.close()
