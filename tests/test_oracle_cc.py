"""Pins of the oracle's congestion control (DCQCN) against things other than
itself: parameters that never mark change nothing; hand-derived cut
values, notification timing and pacing gaps; the closed form of fast
recovery; invariants and tick-by-tick stepping over seeded random traffic.

DCQCN is Zhu et al., SIGCOMM 2015 (an outside source: the Multiverse page
names it in its implementation section without parameters).  Rates are in
units of 2^-20 of the line rate (LINE = 2^20)."""
import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O

LINE = 1 << 20
NEVER = 0xFFFFFFFF                 # a threshold, gap or timer that is never reached


def cc(**kw):
    base = dict(kmin=NEVER, kmax=NEVER, pmax=0, gshift=8, n=NEVER, k=NEVER, t=NEVER, b=NEVER,
                f=5, rai=0, rhai=0, rmin=1)
    base.update(kw)
    return I.DCQCN(**base)


def traced(topo, work, **kw):
    kw.setdefault("tick_ps", 1000)
    kw.setdefault("chunk", 1 << 30)
    r = O.run(I.Batch([I.Experiment(topo, work, **kw)]).pack(), 0, 1, trace_cap=200_000)
    assert r["status"][0] == O.ST_DONE and r["trace_total"] == len(r["trace"])
    assert r["violations"][0] == 0
    return r, r["trace"]


def of_kind(ev, kind, a=None):
    x = ev[ev["kind"] == kind]
    return x if a is None else x[x["a"] == a]


# ---------------------------------------------------------------- inert
def _random_batch(seed, n, ccfg):
    rng = np.random.default_rng(seed)
    ex = []
    for _ in range(n):
        delta, sigma = int(rng.integers(0, 3)), int(rng.integers(1, 3))
        t = [I.single_switch(6, sigma, delta), I.leaf_spine(2, 2, 3, delta, sigma=sigma),
             I.fat_tree(4, delta, sigma=sigma)][int(rng.integers(3))]
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
                               cap=int(rng.integers(2, 9)), tick_ps=1000, cc=ccfg,
                               ecmp_seed=int(rng.integers(1 << 20)), rec_cap=64))
    return I.Batch(ex, "cc")


def test_parameters_that_never_mark_change_nothing():
    """With thresholds no queue reaches, no packet is marked, so no
    notification is sent and every lane keeps the line rate: pacing at the
    line rate is exactly the NIC's one packet per serialisation time, so
    every result equals the run without congestion control."""
    on = _random_batch(5, 60, cc(rai=77, rhai=99, k=3, t=5, b=2, f=1)).pack()
    off = _random_batch(5, 60, None).pack()
    a, b = O.run(on), O.run(off)
    for key in ("status", "end_tick", "pkts_injected", "pkt_hops", "pkts_delivered",
                "msgs_delivered", "digest", "node_start", "node_end", "rec_tick", "rec_key"):
        assert (a[key] == b[key]).all(), key


@pytest.mark.parametrize("delta", [0, 1, 12])
def test_lone_flow_is_never_marked(delta):
    """A lone flow at line rate never has more than one arrived packet in a
    switch ingress queue (the packet leaves in the tick it arrives; those
    still on the wire have not arrived), so even marking everything above
    one packet marks nothing and the lone-message closed form holds:
    (1 + delta) + (n - 1) + L (1 + delta) for the receiver."""
    n = 40
    t = I.single_switch(2, 1, delta)
    r, ev = traced(t, I.lone_message(2, 0, 1, n * 4096),
                   cc=cc(kmin=1, kmax=1, n=5, k=7, t=9, f=2, rai=100, rhai=100, rmin=100))
    assert len(of_kind(ev, O.EV_CNP)) == 0 and len(of_kind(ev, O.EV_CUT)) == 0
    assert r["node_end"][1] == (1 + delta) + (n - 1) + 2 * (1 + delta)


# ---------------------------------------------------------------- incast: one cut a flow
def test_incast_cut_timing_value_and_pacing():
    """Hosts 0 and 1 send to host 2 through one switch (sigma 1, delta 0).
    The egress to host 2 is the bottleneck, so both ingress queues fill;
    marking at more than one arrived packet in the queue and a notification
    gap no flow reaches give exactly one notification a flow.  Each reaches
    its sender three ticks after the receiver generated it (one tick in the
    receiver's notification ring, then two hops of sigma + delta = 1 with
    nothing else on the way back) and halves the rate (alpha is still 1):
    from then on the sender's packets leave every 2 ticks."""
    t = I.single_switch(3, 1, 0)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 120 * 4096)
    w.collective(I.P2P, [1, 2], 120 * 4096)
    r, ev = traced(t, w, cap=4, cc=cc(kmin=1, kmax=1))
    gen = of_kind(ev, O.EV_CNP)
    cuts = of_kind(ev, O.EV_CUT)
    assert len(gen) == 2 and len(cuts) == 2
    assert (gen["a"] == 2).all()                         # generated by the receiver
    assert sorted(cuts["a"].tolist()) == [0, 1]
    assert (cuts["b"] == LINE // 2).all()
    assert sorted((cuts["tick"] - gen["tick"]).tolist()) == [3, 3]
    for sender in (0, 1):
        y = int(cuts[cuts["a"] == sender]["tick"][0])
        inj = of_kind(ev, O.EV_INJECT, sender)["tick"].astype(np.int64)
        after = inj[inj > y]
        gaps = np.diff(after)
        assert (gaps >= 2).all()                         # paced at half rate
        assert (gaps[-20:] == 2).all()                   # the queues drained: exactly the rate


# ---------------------------------------------------------------- fast recovery closed form
def test_fast_recovery_closed_form():
    """A lone flow with every forwarded packet marked (kmin = kmax = 0) and a
    notification gap it never reaches gets one notification, which halves
    its rate: RC = 2^19, RT = 2^20.  Every T ticks after the cut the rate
    timer fires a fast-recovery step RC <- ceil((RT + RC) / 2), so after j
    steps RC = 2^20 - 2^(19 - j) (and 2^20 from j = 20 on).  With sigma = 64
    a packet sent at tick s while j steps have fired is followed by the
    next after ceil(64 * 2^20 / RC_j) ticks: 128, 86, 74, 69, 67, 66, 65,
    ..., 65, then 64 once the line rate is back."""
    sig, T = 64, 300
    t = I.single_switch(2, sig, 0)
    r, ev = traced(t, I.lone_message(2, 0, 1, 400 * 4096),
                   cc=cc(kmin=0, kmax=0, t=T, f=100))
    cuts = of_kind(ev, O.EV_CUT)
    assert len(cuts) == 1 and cuts["b"][0] == LINE // 2
    y = int(cuts["tick"][0])
    inj = of_kind(ev, O.EV_INJECT, 0)["tick"].astype(np.int64)
    sends = inj[inj >= y]
    seen_j = set()
    for s0, s1 in zip(sends[:-1], sends[1:]):
        j = (s0 - y) // T
        rc = LINE if j >= 20 else LINE - (1 << (19 - j))
        want = -(-sig * LINE // rc)
        assert s1 - s0 == want, (s0, j, s1 - s0, want)
        seen_j.add(int(j))
    assert set(range(22)) <= seen_j                       # every step, and the line rate again
    assert [-(-sig * LINE // (LINE - (1 << (19 - j)))) for j in range(4)] == [128, 86, 74, 69]


# ---------------------------------------------------------------- alpha
def test_alpha_decay_between_two_cuts():
    """A lone flow, every forwarded packet marked, notifications at most one
    per N = 50 ticks, the alpha timer K = 30, no rate timer or byte counter.
    First cut (before alpha's first decay): alpha = 1, RC = 2^20 / 2 = 2^19;
    alpha then moves to (1 - 1/256) + 1/256 = 1.  One decay later (30 ticks
    on) alpha = 1 - 1/256 = (2^20 - 2^12) / 2^20, and the second cut leaves
    RC = 2^19 - 2^19 (2^20 - 2^12) / 2^21 = 2^18 + 2^10.  The receiver's
    second notification comes from the first delivery of the flow at least
    N ticks after the first."""
    t = I.single_switch(2, 1, 0)
    r, ev = traced(t, I.lone_message(2, 0, 1, 300 * 4096),
                   cc=cc(kmin=0, kmax=0, n=50, k=30))
    cuts = of_kind(ev, O.EV_CUT)
    gen = of_kind(ev, O.EV_CNP)
    y1, y2 = int(cuts["tick"][0]), int(cuts["tick"][1])
    assert y1 < 30 and 30 <= y2 - y1 < 60                 # the premises: one decay between
    assert cuts["b"][0] == 1 << 19
    assert cuts["b"][1] == (1 << 18) + (1 << 10)
    g1, g2 = int(gen["tick"][0]), int(gen["tick"][1])
    dl = of_kind(ev, O.EV_DELIVER, 1)["tick"].astype(np.int64)
    assert g2 == dl[dl >= g1 + 50][0]


# ---------------------------------------------------------------- every rule at once
def test_reaction_point_replays_the_published_rules():
    """A lone flow, every forwarded packet marked, notifications at most one
    per 25 ticks (so the rate never recovers fully and the target stays below
    the line rate), a short rate timer (T = 7), a byte counter of 3 packets,
    F = 2, gain 1/16 and small increase steps, so that fast recovery,
    additive and hyper increase (with unequal event counts) and the byte
    counter all occur; alpha decays over K = 400 ticks.  Replaying the
    published rules (timer events in time order, alpha first on a tie; each
    packet sent, then any notification taken in that tick; RC <- ceil((RT +
    RC) / 2) after each increase) from the lane's join over the ticks the
    oracle logged predicts every cut value and every gap between packets."""
    sig, gs, N, K, T, B, F = 1, 4, 25, 400, 7, 3, 2
    rai, rhai, rmin = 1 << 9, 1 << 10, 1 << 12
    t = I.single_switch(2, sig, 0)
    r, ev = traced(t, I.lone_message(2, 0, 1, 300 * 4096),
                   cc=cc(kmin=0, kmax=0, n=N, k=K, t=T, b=B, f=F, rai=rai, rhai=rhai, rmin=rmin,
                         gshift=gs))
    t0 = int(ev[(ev["kind"] == O.EV_START) & (ev["b"] == 0)]["tick"][0])
    cuts = {int(x["tick"]): int(x["b"]) for x in of_kind(ev, O.EV_CUT, 0)}
    sends = [int(x) for x in of_kind(ev, O.EV_INJECT, 0)["tick"]]
    assert len(cuts) >= 5
    st = dict(rc=LINE, rt=LINE, alpha=LINE, abase=t0, rbase=t0, tc=0, bc=0, sent=0)
    modes, hyper_below_line = set(), []

    def increase():
        mx, mn = max(st["tc"], st["bc"]), min(st["tc"], st["bc"])
        if mx < F:
            modes.add("fast recovery")
        elif mn > F:
            modes.add("hyper")
            if st["rt"] < LINE and st["tc"] != st["bc"]:
                hyper_below_line.append(1)
            st["rt"] = min(LINE, st["rt"] + (mn - F) * rhai)
        else:
            modes.add("additive")
            st["rt"] = min(LINE, st["rt"] + rai)
        st["rc"] = (st["rt"] + st["rc"] + 1) // 2

    def timers(now):
        while True:
            ta, tr = st["abase"] + K, st["rbase"] + T
            if ta > now and tr > now:
                return
            if ta <= tr:
                st["alpha"] -= st["alpha"] >> gs
                st["abase"] = ta
            else:
                st["rbase"] = tr
                st["tc"] += 1
                increase()

    gaps = {}
    for now in sorted(set(sends) | set(cuts)):
        timers(now)
        if now in sends:
            st["sent"] += 1
            if st["sent"] >= B:
                st["sent"] = 0
                st["bc"] += 1
                increase()
            gaps[now] = -(-sig * LINE // st["rc"])
        if now in cuts:
            st["rt"] = st["rc"]
            st["rc"] = max(rmin, st["rc"] - ((st["rc"] * st["alpha"]) >> 21))
            st["alpha"] = min(LINE, st["alpha"] - (st["alpha"] >> gs) + (LINE >> gs))
            st["abase"] = st["rbase"] = now
            st["tc"] = st["bc"] = st["sent"] = 0
            assert cuts[now] == st["rc"], now
    for a, b in zip(sends[:-1], sends[1:]):
        assert b - a == gaps[a], (a, b - a, gaps[a])
    assert modes == {"fast recovery", "additive", "hyper"}
    assert hyper_below_line                              # a hyper step that moved the target


# ---------------------------------------------------------------- random traffic
def test_random_congestion_controlled_traffic_keeps_invariants():
    """Seeded random collectives with aggressive settings (marking from two
    packets, notifications every 5 ticks, short timers, every branch of the
    rate increase): every run ends, delivers every packet, breaks no
    run-time invariant, sends notifications, and gives the same results
    stepped tick by tick (so the idle-tick skip sees the pacing and the
    notifications)."""
    p = _random_batch(11, 80, cc(kmin=1, kmax=4, pmax=30000, n=5, k=7, t=11, b=6, f=2,
                                 rai=3000, rhai=20000, rmin=5000)).pack()
    a, b = O.run(p), O.run(p, no_skip=True)
    assert (a["status"] == O.ST_DONE).all()
    assert (a["violations"] == 0).all()
    assert (a["pkts_injected"] == a["pkts_delivered"]).all()
    for k in ("end_tick", "pkts_injected", "pkt_hops", "msgs_delivered", "digest", "node_end"):
        assert (a[k] == b[k]).all(), k
    off = O.run(_random_batch(11, 80, None).pack())
    assert (a["pkt_hops"] > off["pkt_hops"]).any()        # notifications travelled
    assert (a["end_tick"] != off["end_tick"]).any()


def test_parameter_limits_are_refused():
    """Malformed settings are refused: kmin above kmax, pmax above 1, gain
    shift 0 or above 16, zero gaps, timers or counters, a zero minimum rate,
    and congestion control together with virtual output queues."""
    t = I.single_switch(2, 1, 0)
    w = I.lone_message(2, 0, 1, 4096)
    ok = I.Experiment(t, w, tick_ps=1000, chunk=1 << 20, cc=cc())
    assert O.run(I.Batch([ok]).pack())["status"][0] == O.ST_DONE
    for bad in (dict(kmin=5, kmax=4), dict(pmax=65537), dict(gshift=0), dict(gshift=17),
                dict(n=0), dict(k=0), dict(t=0), dict(b=0), dict(rmin=0), dict(rmin=LINE + 1)):
        e = I.Experiment(t, w, tick_ps=1000, chunk=1 << 20, cc=cc(**bad))
        with pytest.raises(Exception):
            O.run(I.Batch([e]).pack())
    e = I.Experiment(t, w, tick_ps=1000, chunk=1 << 20, cc=cc(), voq=1)
    with pytest.raises(Exception):
        O.run(I.Batch([e]).pack())


# ================================================================ DCTCP
# DCTCP is Alizadeh et al., SIGCOMM 2010 (an outside source: the Multiverse
# page names it without parameters).  Windows are in units of 2^-10 packets.
W1 = 1 << 10


def tcp(**kw):
    base = dict(kmark=NEVER, gshift=4, w0=10, wmax=256)
    base.update(kw)
    return I.DCTCP(**base)


@pytest.mark.parametrize("delta,w", [(0, 2), (0, 3), (2, 2), (1, 5)])
def test_window_limited_lone_flow_closed_form(delta, w):
    """A lone flow whose window is fixed at w packets (w0 = wmax, nothing
    marked) sends w packets back to back, then waits for acknowledgements:
    a packet sent at t is delivered at t + L (1 + delta), its
    acknowledgement leaves the receiver's NIC the next tick and is taken off
    the sender's downlink at t + 2 L (1 + delta) + 1, which frees the window
    for a packet at t + 2 L (1 + delta) + 2.  So packet k leaves at
    t0 + (2 L (1 + delta) + 2) floor(k / w) + k mod w (while w is below that
    round trip), and every packet is acknowledged (one acknowledgement
    packet each, L hops) but those still on their way when the last message
    completes the run."""
    n, L = 24, 2
    t = I.single_switch(2, 1, delta)
    r, ev = traced(t, I.lone_message(2, 0, 1, n * 4096), cc=tcp(w0=w, wmax=w))
    inj = of_kind(ev, O.EV_INJECT, 0)["tick"].astype(np.int64)
    rtt = 2 * L * (1 + delta) + 2
    assert w < rtt
    want = inj[0] + rtt * (np.arange(n) // w) + np.arange(n) % w
    assert (inj == want).all()
    acks = of_kind(ev, O.EV_ACK, 0)
    assert (acks["b"] & 0xFF == 1).all() and n - w <= len(acks) < n
    assert r["pkt_hops"][0] >= n * L + len(acks) * L


def test_window_grows_one_packet_a_window_until_wmax():
    """Nothing marked: each closed observation window adds one packet to the
    window, up to wmax (1, 2, 3, 4, 4, ... packets)."""
    t = I.single_switch(2, 1, 0)
    r, ev = traced(t, I.lone_message(2, 0, 1, 60 * 4096), cc=tcp(w0=1, wmax=4))
    w = of_kind(ev, O.EV_WINDOW, 0)["b"].tolist()
    assert w[:4] == [2 * W1, 3 * W1, 4 * W1, 4 * W1]
    assert max(w) == 4 * W1


def test_window_halves_while_everything_is_marked():
    """Every forwarded packet marked (threshold 0): each window's marked
    fraction is 1, so alpha stays 1 ((1 - g) + g) and each closed window
    halves the window, down to one packet: 8 -> 4 -> 2 -> 1 -> 1."""
    t = I.single_switch(2, 1, 0)
    r, ev = traced(t, I.lone_message(2, 0, 1, 60 * 4096), cc=tcp(kmark=0, w0=8, wmax=8))
    w = of_kind(ev, O.EV_WINDOW, 0)["b"].tolist()
    assert w[:5] == [4 * W1, 2 * W1, 1 * W1, 1 * W1, 1 * W1]


def test_window_updates_follow_the_acknowledgement_stream():
    """A two-sender incast with marking above one queued packet: from the
    acknowledgements each sender received (packets and marks, in order) and
    the packets it had sent by then, the published update (close the window
    once every packet sent before the last update is acknowledged; alpha <-
    (1 - g) alpha + g F; the window shrinks by alpha / 2 if F > 0, else
    grows one packet) gives every window the oracle logged."""
    t = I.single_switch(3, 1, 0)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 150 * 4096)
    w.collective(I.P2P, [1, 2], 150 * 4096)
    gs, w0, wmax = 4, 10, 64
    r, ev = traced(t, w, cap=8, cc=tcp(kmark=1, gshift=gs, w0=w0, wmax=wmax))
    saw_partial = False
    for sender in (0, 1):
        mine = ev[ev["a"] == sender]
        wnd, alpha, acked, wend, wa, wm, sent = w0 * W1, LINE, 0, w0, 0, 0, 0
        got = []
        for x in mine:
            if x["kind"] == O.EV_INJECT:
                sent += 1
            elif x["kind"] == O.EV_ACK:
                n, m = int(x["b"]) & 0xFF, (int(x["b"]) >> 8) & 0xFF
                acked, wa, wm = acked + n, wa + n, wm + m
                if acked >= wend:
                    F = (wm << 20) // wa
                    saw_partial |= 0 < wm < wa
                    alpha = alpha - (alpha >> gs) + (F >> gs)
                    if wm:
                        wnd = max(W1, wnd - ((wnd * alpha) >> 21))
                    else:
                        wnd = min(wmax * W1, wnd + W1)
                    wa = wm = 0
                    wend = sent
                    got.append(wnd)
        logged = of_kind(ev, O.EV_WINDOW, sender)["b"].tolist()
        assert got == logged and len(logged) > 5
    assert saw_partial                                   # some window was partly marked


def test_dctcp_random_traffic_keeps_invariants():
    """Seeded random collectives under DCTCP (threshold two packets, small
    windows): every run ends, every packet is delivered and acknowledged,
    no run-time invariant breaks, and stepping tick by tick changes
    nothing."""
    p = _random_batch(13, 80, tcp(kmark=2, gshift=3, w0=2, wmax=12)).pack()
    a, b = O.run(p), O.run(p, no_skip=True)
    assert (a["status"] == O.ST_DONE).all()
    assert (a["violations"] == 0).all()
    assert (a["pkts_injected"] == a["pkts_delivered"]).all()
    for k in ("end_tick", "pkts_injected", "pkt_hops", "msgs_delivered", "digest", "node_end"):
        assert (a[k] == b[k]).all(), k
    off = O.run(_random_batch(13, 80, None).pack())
    assert (a["end_tick"] >= off["end_tick"]).mean() > 0.5   # windows slow most runs


def test_dctcp_parameter_limits_are_refused():
    """DCTCP needs one marking threshold (kmin = kmax), a gain shift of
    1..16, an initial window of at least one packet and wmax between w0 and
    65,535; with VOQs it is refused."""
    t = I.single_switch(2, 1, 0)
    wl = I.lone_message(2, 0, 1, 4096)
    ok = I.Experiment(t, wl, tick_ps=1000, chunk=1 << 20, cc=tcp())
    assert O.run(I.Batch([ok]).pack())["status"][0] == O.ST_DONE
    for bad in (dict(gshift=0), dict(gshift=17), dict(w0=0), dict(w0=5, wmax=4),
                dict(wmax=65536)):
        e = I.Experiment(t, wl, tick_ps=1000, chunk=1 << 20, cc=tcp(**bad))
        with pytest.raises(Exception):
            O.run(I.Batch([e]).pack())
    c = tcp()
    wds = c.words()
    wds[2] -= 1                                          # kmin != kmax
    e = I.Experiment(t, wl, tick_ps=1000, chunk=1 << 20, cc=c)
    p = I.Batch([e]).pack()
    p["exp_cc"][:16] = wds
    with pytest.raises(Exception):
        O.run(p)
    e = I.Experiment(t, wl, tick_ps=1000, chunk=1 << 20, cc=tcp(), voq=1)
    with pytest.raises(Exception):
        O.run(I.Batch([e]).pack())
