"""Pins of the CPU oracle against things other than itself.

Each test states what fixes the expected value: a published constant, a
closed form from the pages, a hand-traced tick table, or an independent
evaluator (a longest-path recurrence with no queues in it).
"""
import os

import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run1(topo, work, **kw):
    kw.setdefault("tick_ps", 1000)
    e = I.Experiment(topo, work, **kw)
    r = O.run(I.Batch([e]).pack())
    assert r["status"][0] == O.ST_DONE, r["status"]
    return r


# ---------------------------------------------------------------- hash
def test_mix64_published_splitmix64_outputs():
    """splitmix64 (Vigna) seeded with 0 yields 0xe220a8397b1dcdaf,
    0x6e789e6aa1b965f4, 0x06c45d188009454f: the finaliser applied to
    k * 0x9e3779b97f4a7c15 for k = 1, 2, 3."""
    g = 0x9E3779B97F4A7C15
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [O.mix64((k * g) % 2 ** 64) for k in (1, 2, 3)] == want


# ---------------------------------------------------------------- lone message
def chain_topology(n_switch_hops: int, sigmas, deltas):
    """hosts 0 and 1 joined through a chain of switches; link j has
    (sigmas[j], deltas[j]); link 0 is host 0's uplink, the last link is the
    downlink to host 1.  Levels rise along the chain so up/down routing
    follows it (the last switch reaches host 1 downward)."""
    t = I.Topology("chain")
    nsw = n_switch_hops
    sws = [t.add_switch(nsw - i) for i in range(nsw)]
    h0, h1 = t.add_hosts(2)
    # switch levels: host 0 attaches to the top of a descending chain so that
    # every switch reaches host 1 downward
    t.attach_host(h0, sws[0], sigmas[0], deltas[0], sigmas[0], deltas[0])
    for j in range(nsw - 1):
        t.link(sws[j], sws[j + 1], sigmas[j + 1], deltas[j + 1])
    t.attach_host(h1, sws[-1], sigmas[-1], deltas[-1], sigmas[-1], deltas[-1])
    return t


@pytest.mark.parametrize("n", [1, 2, 7, 40])
@pytest.mark.parametrize("delta", [0, 1, 12])
@pytest.mark.parametrize("topo", ["switch", "leafspine", "fattree"])
def test_lone_message_closed_form(n, delta, topo):
    """A lone message of n packets over L links of one tick each: the last
    packet reaches the receiver (n-1) + L*(1+delta) ticks after the first
    injection (serialisation of the packets behind the head plus, per hop,
    propagation and per-packet serialisation).  Both ends join at tick 0 and
    the join reaches the sender 1 + delta ticks later, so the first injection
    is at tick 1 + delta.  The sender's acknowledgement arrives L*(delta+1)
    ticks after delivery."""
    if topo == "switch":
        t, src, dst, L = I.single_switch(2, 1, delta), 0, 1, 2
    elif topo == "leafspine":
        t, src, dst, L = I.leaf_spine(2, 2, 2, delta), 0, 3, 4
    else:
        t, src, dst, L = I.fat_tree(4, delta), 0, 15, 6
    w = I.lone_message(t.n_hosts, src, dst, n * 4096)
    r = run1(t, w, chunk=1 << 30)
    done = (1 + delta) + (n - 1) + L * (1 + delta)
    ends = dict(zip(["send", "recv"], r["node_end"][[0, 1]] if src < dst else r["node_end"][[1, 0]]))
    assert ends["recv"] == done
    assert ends["send"] == done + L * (delta + 1)
    assert r["pkts_injected"][0] == n and r["pkts_delivered"][0] == n
    assert r["pkt_hops"][0] == n * L


@pytest.mark.parametrize("n", [1, 5, 30])
@pytest.mark.parametrize("sig", [[1, 3, 2, 1], [3, 1, 2, 1]])
def test_heterogeneous_path_closed_form(n, sig):
    """Per-link serialisation differs: the bottleneck spaces the packets, so
    delivery = first injection + (n-1)*max(sigma) + sum(sigma + delta).  The
    bottleneck is a switch link, or the sender's own uplink."""
    dl = [2, 0, 5, 1]
    t = chain_topology(3, sig, dl)
    w = I.lone_message(2, 0, 1, n * 4096)
    r = run1(t, w, chunk=1 << 30)
    assert r["node_end"][1] == 1 + (n - 1) * max(sig) + sum(s + d for s, d in zip(sig, dl))


def test_credit_loop_needs_two_delta_plus_two():
    """A slot is held from the push until the pop's credit is back: sigma +
    delta to reach the head, delta + 1 for the credit to return.  Line rate
    therefore needs queue capacity >= 2*delta + 2; one slot fewer must make
    the message slower."""
    delta, n = 4, 30
    t = I.single_switch(2, 1, delta)
    w = I.lone_message(2, 0, 1, n * 4096)
    full = run1(t, w, chunk=1 << 30, cap=2 * delta + 2)["node_end"][1]
    short = run1(t, w, chunk=1 << 30, cap=2 * delta + 1)["node_end"][1]
    assert full == (1 + delta) + (n - 1) + 2 * (1 + delta)
    assert short > full


# ---------------------------------------------------------------- hand trace
def _incast_gold():
    gold = {}
    for line in open(os.path.join(GOLDEN, "incast_cap2_delta1.txt")):
        if line.strip() and not line.startswith("#"):
            k, *v = line.split()
            gold[k] = [int(x) for x in v]
    return gold


def test_incast_hand_trace():
    gold = _incast_gold()
    t = I.single_switch(3, 1, 1)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 3 * 4096)
    w.collective(I.P2P, [1, 2], 3 * 4096)
    r = run1(t, w, chunk=1 << 20, cap=2, rec_cap=8)
    assert list(r["node_end"][:4]) == gold["node_end"]
    assert sorted(r["rec_tick"][: r["rec_count"][0]]) == gold["delivery_ticks"]
    assert r["pkts_injected"][0] == gold["packets"][0]
    assert r["pkt_hops"][0] == gold["packet_hops"][0]


def test_incast_event_trace_matches_hand_trace():
    """The oracle's event trace reproduces the hand-traced table tick by tick:
    every injection, switch hop and delivery of A's and B's packets."""
    gold = _incast_gold()
    t = I.single_switch(3, 1, 1)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 3 * 4096)
    w.collective(I.P2P, [1, 2], 3 * 4096)
    p = I.Batch([I.Experiment(t, w, tick_ps=1000, chunk=1 << 20, cap=2)]).pack()
    r = O.run(p, 0, 1, trace_cap=1000)
    ev = r["trace"]
    assert r["trace_total"] == len(ev)
    sender_node = {"A": 0, "B": 1}          # node order: A's send, B's send, C's receives
    for who, h in (("A", 0), ("B", 1)):
        inj = ev[(ev["kind"] == O.EV_INJECT) & (ev["a"] == h)]["tick"]
        hop = ev[(ev["kind"] == O.EV_HOP) & (ev["b"] == h)]["tick"]        # ingress queue = port h
        dlv = ev[(ev["kind"] == O.EV_DELIVER) & (ev["b"] == sender_node[who])]["tick"]
        assert list(inj) == gold[f"inject_ticks_{who}"]
        assert list(hop) == gold[f"hop_ticks_{who}"]
        assert list(dlv) == gold[f"deliver_ticks_{who}"]
    assert (np.diff(ev["tick"].astype(np.int64)) >= 0).all()
    ends = ev[ev["kind"] == O.EV_END]
    assert sorted(zip(ends["a"], ends["b"])) == list(enumerate(gold["node_end"]))


def test_first_divergence_finds_the_earliest_difference():
    b = I.config1()
    p = b.pack()
    mine = O.run(p)
    assert O.first_divergence(p, mine, 3) is None
    other = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in mine.items()}
    e, n0 = 3, int(mine["node_offset"][3])
    other["node_end"][n0 + 5] += 7
    d = O.first_divergence(p, other, e)
    assert d["what"] == "node_end" and d["node"] == 5
    assert d["tick"] == int(mine["node_end"][n0 + 5])
    other = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in mine.items()}
    import dataclasses
    p2 = I.Batch([dataclasses.replace(b.experiments[0], rec_cap=64)]).pack()
    mine2 = O.run(p2)
    other2 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in mine2.items()}
    j = int(np.argsort(mine2["rec_tick"][:64])[10])
    other2["rec_tick"][j] += 1
    d = O.first_divergence(p2, other2, 0)
    assert d["what"] == "message" and d["tick"] <= int(mine2["rec_tick"][j])


# ---------------------------------------------------------------- pipelined broadcast
@pytest.mark.parametrize("A", [1, 2, 3, 7])
@pytest.mark.parametrize("K", [1, 2, 5, 16])
@pytest.mark.parametrize("np_", [1, 3, 8])
def test_pipelined_broadcast_closed_form(A, K, np_):
    """AlpaComm section 3.1: with the slice cut in K partitions of t/K each,
    the broadcast over A receivers takes T_bc = t/K * (K + A - 1).  In ticks
    (t = K*n_p packets) the last receiver holds the slice at exactly
    T_bc + A * L*(1+delta): each of the A relay hops adds its path latency
    L*(1+delta) on top of the page's serialisation-only count (the one-tick
    dependency and the one-tick rendezvous cancel the -1 of the last packet).
    A=1 is a lone message; K=1 is store-and-forward."""
    delta, L = 0, 2
    t = I.single_switch(A + 1, 1, delta)
    w = I.relay_chain(A + 1, K * np_ * 4096, K)
    r = run1(t, w)
    last = r["node_end"][A]
    T_bc = np_ * (K + A - 1)
    assert last == T_bc + A * L * (1 + delta)
    if A == 1:
        assert last == 1 + (K * np_ - 1) + L * (1 + delta)
    assert r["pkt_hops"][0] == A * K * np_ * L


def test_pipelined_broadcast_tends_to_t():
    """T_bc -> t as the per-partition size grows (the page's K >> A regime
    with hop latency negligible): ratio of simulated time to t = K*n_p."""
    A, K = 4, 100
    ratios = []
    for np_ in (1, 4, 16):
        t = I.single_switch(A + 1, 1, 0)
        w = I.relay_chain(A + 1, K * np_ * 4096, K)
        last = run1(t, w)["node_end"][A]
        ratios.append(last / (K * np_))
    assert ratios[0] > ratios[1] > ratios[2]
    assert ratios[2] < 1 + (A - 1) / K + 0.15


# ---------------------------------------------------------------- ring all-reduce
def ring_longest_path(N, loops, steps, n, lat, first=1):
    """Independent evaluator of a contention-free ring (one channel): message
    (l,k) of member i starts after its previous message finished injecting and
    one tick after member i received (l,k-1); the first message starts at
    `first` (when the joins have reached the senders); it injects n packets on
    consecutive ticks and reaches member i+1 lat[i] ticks after its last
    packet.  Returns each member's last delivery tick."""
    M = loops * steps
    start = [[0] * M for _ in range(N)]
    recv = [[0] * M for _ in range(N)]  # recv[i][m]: member i got message m from i-1
    for m in range(M):
        k = m % steps
        for i in range(N):
            s = first if m == 0 else start[i][m - 1] + n
            if k >= 1:
                s = max(s, recv[i][m - 1] + 1)
            start[i][m] = s
        for i in range(N):
            recv[(i + 1) % N][m] = start[i][m] + n - 1 + lat[i]
    return [recv[i][M - 1] for i in range(N)]


@pytest.mark.parametrize("kind,steps_of", [(I.AR, lambda N: 2 * (N - 1)),
                                            (I.RS, lambda N: N - 1),
                                            (I.AG, lambda N: N - 1)])
@pytest.mark.parametrize("N,loops,blk", [(2, 1, 3), (4, 2, 2), (8, 3, 5)])
def test_ring_contention_free_longest_path(kind, steps_of, N, loops, blk):
    """Ring collectives with one channel on a single switch (every ingress
    feeds one egress): timing equals the longest path of the message DAG.
    Sizes make every block equal (S = N * C * loops, C = blk packets)."""
    delta = 2
    C = blk * 4096
    S = N * C * loops
    t = I.single_switch(N, 1, delta)
    w = I.single_collective(N, kind, S)
    r = run1(t, w, nc=1, chunk=C)
    steps = steps_of(N)
    got = list(r["node_end"][:N])
    lat = [2 * (1 + delta)] * N
    recv = ring_longest_path(N, loops, steps, blk, lat, first=1 + delta)
    # a member finishes at max(last delivery to it, ack of its own last message)
    want = [max(recv[i], recv[(i + 1) % N] + 2 * (delta + 1)) for i in range(N)]
    assert got == want
    assert r["pkts_injected"][0] == N * loops * steps * blk


def test_ring_leafspine_paths_of_two_lengths():
    """config-1 fabric with one channel: hosts 0-3 on leaf 0, 4-7 on leaf 1;
    only 3->4 and 7->0 cross a spine (4 links), the rest use 2 links; each
    directed link carries one connection, so the longest path is exact."""
    N, loops, blk, delta = 8, 2, 4, 12
    C = blk * 4096
    t = I.leaf_spine(2, 2, 4, delta)
    w = I.single_collective(N, I.AR, N * C * loops)
    r = run1(t, w, nc=1, chunk=C)
    lat = [(4 if i in (3, 7) else 2) * (1 + delta) for i in range(N)]
    recv = ring_longest_path(N, loops, 2 * (N - 1), blk, lat, first=1 + delta)
    ack = [(4 if i in (3, 7) else 2) * (delta + 1) for i in range(N)]
    want = [max(recv[i], recv[(i + 1) % N] + ack[i]) for i in range(N)]
    assert list(r["node_end"][:N]) == want


def test_ring_allreduce_bandwidth_term():
    """AutoCCL's ring cost: each rank sends 2(N-1)/N * S bytes, so the
    all-reduce cannot finish before 2(N-1)/N * S / B; with one chunk per
    block and growing S the ratio to that bound tends to 1."""
    N, delta = 8, 1
    ratios = []
    for mib in (1, 4, 16):
        S = mib * I.MIB
        t = I.single_switch(N, 1, delta)
        w = I.single_collective(N, I.AR, S)
        r = run1(t, w, nc=1, chunk=S // N)
        bound = 2 * (N - 1) * S // N // 4096
        assert r["pkts_injected"][0] == N * bound
        end = int(r["node_end"][:N].max())
        assert end >= bound
        ratios.append(end / bound)
    assert ratios[0] > ratios[1] > ratios[2] and ratios[2] < 1.05


def test_ring_packet_totals_uneven_sizes():
    """2(N-1) block sends per loop per rank cover 2(N-1)/N of every loop's
    bytes; with partial packets rounding up, the total packet count per rank
    is at least the byte bound and every partition is moved."""
    N, S = 5, 3 * I.MIB + 12345
    t = I.single_switch(N, 1, 0)
    for nc, C in [(1, 64 * I.KIB), (3, 100000), (4, 1 << 20)]:
        w = I.single_collective(N, I.AR, S)
        r = run1(t, w, nc=nc, chunk=C)
        assert r["pkts_injected"][0] >= N * -(-2 * (N - 1) * S // (N * 4096))
        assert r["pkts_injected"][0] == r["pkts_delivered"][0]


# ---------------------------------------------------------------- tree
@pytest.mark.parametrize("n", [1, 6])
def test_tree_two_members_closed_form(n):
    """Binary tree over 2 members (root 0, leaf 1), one chunk: the leaf's
    chunk goes up (reduce), then the root sends it down (broadcast)."""
    delta, L = 3, 2
    t = I.single_switch(2, 1, delta)
    w = I.single_collective(2, I.AR, n * 4096)
    r = run1(t, w, algo=I.TREE, nc=1, chunk=1 << 30)
    up = (1 + delta) + (n - 1) + L * (1 + delta)
    down = up + 1 + (n - 1) + L * (1 + delta)
    assert r["node_end"][1] == down
    assert r["node_end"][0] == down + L * (delta + 1)


def test_tree_packet_totals():
    """Each non-root member sends every chunk up once and receives it down
    once: 2(N-1) * S / pkt packets in all."""
    N, S = 7, 64 * 4096
    t = I.single_switch(N, 1, 1)
    w = I.single_collective(N, I.AR, S)
    r = run1(t, w, algo=I.TREE, nc=2, chunk=8 * 4096)
    assert r["pkts_injected"][0] == 2 * (N - 1) * S // 4096


# ---------------------------------------------------------------- all-to-all
@pytest.mark.parametrize("N,n", [(2, 5), (3, 4), (4, 2)])
def test_alltoall_rotation_closed_form(N, n):
    """Equal sizes, one channel, one switch: in rotation order every phase is
    a permutation, so no link is shared; each member's last delivery is
    (N-1)*n - 1 + L*(1+delta) ticks after the first injection at tick 1+delta."""
    delta, L = 1, 2
    t = I.single_switch(N, 1, delta)
    w = I.Workload(N)
    m = {(i, j): n * 4096 for i in range(N) for j in range(N) if i != j}
    w.collective(I.A2A, list(range(N)), 0, a2a=m)
    r = run1(t, w, nc=1, chunk=1 << 30)
    recv = (1 + delta) + (N - 1) * n - 1 + L * (1 + delta)
    assert list(r["node_end"][:N]) == [recv + L * (delta + 1)] * N
    assert r["pkts_injected"][0] == N * (N - 1) * n


# ---------------------------------------------------------------- DAG
def test_compute_dag_critical_path():
    """Compute-only DAGs: the iteration ends at the longest path, each node
    adding its duration and each edge one tick (topological DP)."""
    rng = np.random.default_rng(7)
    R = 3
    w = I.Workload(R)
    ids, dur = [], {}
    for r in range(R):
        nodes = []
        for k in range(12):
            d = int(rng.integers(0, 20))
            u = w.compute(r, d)     # tick_ps = 1000: ns == ticks
            dur[u] = d
            for p in nodes:
                if rng.random() < 0.3:
                    w.edge(p, u)
            nodes.append(u)
        ids += nodes
    t = I.single_switch(R, 1, 0)
    r = run1(t, w)
    fin = {}
    preds = {u: [a for a, b in w.edges if b == u] for u in ids}
    for u in ids:   # creation order is a topological order
        st = max([fin[p] + 1 for p in preds[u]], default=0)
        fin[u] = st + dur[u]
    order = sorted(range(len(w.nodes)), key=lambda i: (w.nodes[i]["rank"], i))
    assert [int(x) for x in r["node_end"][: len(order)]] == [fin[u] for u in order]
    assert r["end_tick"][0] == max(fin.values())


def test_compute_duration_units_and_hash_range():
    """Durations in ns become ceil(ns * 1000 / tick_ps) ticks: 50,000 ns at
    81,920 ps per tick is 610.35 -> 611 ticks.  Hashed durations stay in
    [lo, hi] (the U[50,500] us range) and vary with the seed."""
    w = I.Workload(1)
    w.compute(0, 50_000)
    t = I.single_switch(1, 1, 0)
    assert run1(t, w, tick_ps=81920)["node_end"][0] == 611
    w = I.Workload(1)
    us = [w.compute(0, 50_000, 500_000, key=k) for k in range(200)]
    w.chain(*us)   # one at a time: at most 64 nodes may wait to start per rank
    ends = []
    for seed in (1, 2):
        r = run1(t, w, tick_ps=1_000_000, dur_seed=seed)   # 1 tick = 1 us
        d = r["node_end"][: len(us)].astype(np.int64) - r["node_start"][: len(us)]
        assert d.min() >= 50 and d.max() <= 500
        ends.append(d)
    assert (ends[0] != ends[1]).any()
    assert 200 < ends[0].mean() < 350


def test_intra_server_analytic_model():
    """Multiverse section 4.1: an intra-server collective takes alpha +
    bytes/beta once its last member has joined.  alpha=7 ticks, beta = 1
    tick per 1000 bytes; all-reduce over g=4 moves 2*3/4*S bytes per GPU:
    S=8000 -> 12000 bytes -> 12 ticks.  Members join at 3, 9, 5, 0."""
    w = I.Workload(4)
    pre = [w.compute(r, d) for r, d in enumerate([3, 9, 5, 0])]
    ids = w.collective(I.AR, [0, 1, 2, 3], 8000, intra=True, alpha=7, beta=(1, 1000))
    for p, u in zip(pre, ids):
        w.edge(p, u)
    t = I.single_switch(4, 1, 0)
    r = run1(t, w)
    order = sorted(range(len(w.nodes)), key=lambda i: (w.nodes[i]["rank"], i))
    end = dict(zip(order, r["node_end"]))
    # preds end at 3,9,5,0 -> joins at 4,10,6,1; last join 10 -> 10 + 7 + 12
    assert [end[u] for u in ids] == [29] * 4
    # reduce-scatter moves half of the all-reduce's bytes: 6000 -> 6 ticks
    w2 = I.Workload(4)
    ids2 = w2.collective(I.RS, [0, 1, 2, 3], 8000, intra=True, alpha=7, beta=(1, 1000))
    r2 = run1(t, w2)
    assert list(r2["node_end"][:4]) == [0 + 7 + 6] * 4


# ---------------------------------------------------------------- memory check
def test_memory_check_worked_example():
    """GPT-3 13B, TP 8, PP 4, 10 layers per stage, 8 micro-batches, s=2048,
    b=1, h=5120, a=40.  By hand: weights+grads+Adam 16 * 13e9 / 32 =
    6,500,000,000 bytes; activations per layer 2048*5120*(34 + 5*40*2048/5120)
    = 10,485,760 * 114 = 1,195,376,640 bytes, times 10 layers times min(8,4)
    in-flight micro-batches / TP 8 = 5,976,883,200 bytes.  Total
    12,476,883,200 bytes: fits in exactly that much memory, not one byte less."""
    w = I.Workload(1)
    w.compute(0, 5)
    w.set_memory_model(13_000_000_000, 8, 4, 10, 8, 2048, 1, 5120, 40)
    t = I.single_switch(1, 1, 0)
    ok = I.Experiment(t, w, tick_ps=1000, gpu_mem=12_476_883_200)
    oom = I.Experiment(t, w, tick_ps=1000, gpu_mem=12_476_883_199)
    r = O.run(I.Batch([ok, oom]).pack())
    assert list(r["status"]) == [O.ST_DONE, O.ST_OOM]
    assert r["node_end"][1] == O.UNSET


# ---------------------------------------------------------------- invariants
def test_config1_invariants():
    """Config 1: 7,168 packets per rank (2*7/8 * 16 MiB / 4 KiB) whatever NC
    and chunk; 6 ring connections use 2 links and 2 use 4 links, so
    packet-hops are 2.5 per packet."""
    b = I.config1()
    r = O.run(b.pack())
    assert (r["status"] == O.ST_DONE).all()
    assert (r["pkts_injected"] == 8 * 7168).all()
    assert (r["pkts_delivered"] == r["pkts_injected"]).all()
    assert (r["pkt_hops"] == 8 * 7168 * 5 // 2).all()
    assert (r["end_tick"] >= 7168).all()


def test_config2_invariants():
    b = I.config2(n_exp=24)
    r = O.run(b.pack())
    assert (r["status"] == O.ST_DONE).all()
    for e, ex in enumerate(b.experiments):
        A, K, mib = ex.label["A"], ex.label["K"], ex.label["mib"]
        S = mib * I.MIB
        per_part = [-(-(S // K + (k < S % K)) // 4096) for k in range(K)]
        assert r["pkts_injected"][e] == A * sum(per_part)
        assert r["pkt_hops"][e] == 2 * r["pkts_injected"][e]
        # at least t = the slice's serialisation, and within the pipelined bound
        assert r["end_tick"][e] >= sum(per_part)


def test_deadlock_is_detected():
    """A collective whose receiver never joins (its predecessor is a member
    of a collective that the other side never reaches) is a deadlock, not a
    hang: two ranks each wait in a different order."""
    w = I.Workload(2)
    a = w.collective(I.P2P, [0, 1], 4096)
    b = w.collective(I.P2P, [1, 0], 4096)
    w.edge(b[1], a[0])   # rank 0: receive b before sending a
    w.edge(a[1], b[0])   # rank 1: receive a before sending b
    t = I.single_switch(2, 1, 0)
    r = O.run(I.Batch([I.Experiment(t, w, tick_ps=1000, chunk=1 << 20)]).pack())
    assert r["status"][0] == O.ST_DEADLOCK


def test_table_limits_overflow_exactly_one_past_the_limit():
    """Each per-rank table (send lanes 64, receive counters 128, pending
    nodes 64, running collectives 16) holds its limit and fails one past it
    with the overflow status (the limits the C ABI documents)."""
    b = I.table_limits()
    r = O.run(b.pack())
    for e, x in enumerate(b.experiments):
        over = x.label["n"] in (65, 129, 17)
        assert r["status"][e] == (O.ST_OVERFLOW if over else O.ST_DONE), x.label


# ---------------------------------------------------------------- invariants
def _incast(n_pkts: int, sigma: int = 1):
    """Hosts 0 and 1 each send n_pkts packets to host 2 through one switch
    with 2-slot queues: the egress to host 2 is the bottleneck, so both
    ingress queues run full and the credit rule is what holds them."""
    t = I.single_switch(3, sigma, 1)
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], n_pkts * 4096)
    w.collective(I.P2P, [1, 2], n_pkts * 4096)
    return I.Batch([I.Experiment(t, w, tick_ps=1000, chunk=1 << 20, cap=2)]).pack()


def _planted(tmp_path, name: str, old: str, new: str) -> str:
    """A copy of the oracle with one planted mistake, built with gcc."""
    src = open(O.SRC).read()
    assert src.count(old) == 1, old
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    import subprocess
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", str(lib), str(c)])
    return str(lib)


def test_invariants_hold():
    """Lossless credit (no queue beyond cap), one packet per serialisation
    time on every link, and delivery at the addressed host, over ring, tree,
    relay, point-to-point and incast traffic."""
    for packed in (I.config1().pack(), I.config2(n_exp=8).pack(), _incast(20), _incast(9, 3),
                   I.gpt_small(algo=I.TREE, seeds=(0,)).pack()):
        r = O.run(packed)
        assert (r["violations"] == 0).all()
        assert (r["status"] == O.ST_DONE).all()


def test_invariant_checks_catch_planted_mistakes(tmp_path):
    """Each check fails on an oracle with the matching mistake planted: credit
    always granted (queues overflow), the egress busy time not kept (a link
    outruns its serialisation time), routing by the wrong destination."""
    no_credit = _planted(tmp_path, "no_credit", "return s->tail[f] - (h - back) < s->cap;",
                         "return 1;")
    assert O.run(_incast(20), lib_path=no_credit)["violations"][0] > 0
    no_busy = _planted(tmp_path, "no_busy", "s->eg_busy[qe] = t + s->port_sigma[qe];", "")
    assert O.run(_incast(9, 3), lib_path=no_busy)["violations"][0] > 0
    # (the planted copies run in this process, so each mistake stays in bounds)
    bad_route = _planted(tmp_path, "bad_route", "s->route[(size_t)w * s->H + p->dst]",
                         "s->route[(size_t)w * s->H + (p->dst + 1) % s->H]")
    assert O.run(_incast(3), lib_path=bad_route)["violations"][0] > 0


# ---------------------------------------------------------------- schedule details, by trace
def _per_message(ev, sender):
    """Packets of each message from node `sender`, in delivery order."""
    out, n = [], 0
    for x in ev:
        if x["kind"] == O.EV_DELIVER and x["b"] == sender:
            n += 1
        elif x["kind"] == O.EV_MESSAGE and x["b"] == sender:
            out.append(n)
            n = 0
    return out


def _traced(topo, work, **kw):
    kw.setdefault("tick_ps", 1000)
    r = O.run(I.Batch([I.Experiment(topo, work, **kw)]).pack(), 0, 1, trace_cap=100_000)
    assert r["status"][0] == O.ST_DONE and r["trace_total"] == len(r["trace"])
    return r["trace"]


def test_ring_step_sends_block_i_minus_k():
    """Ring schedule (the NCCL ring named in Multiverse section 5, cut per
    AutoCCL section 2.3): at step k member i sends block (i - k) mod N.  Reduce-scatter
    of 12,289 B over 3 ranks, one loop: blocks of ceil(12289/3) = 4,097 B, the
    last 4,095 B, so 2, 2 and 1 packets.  Member 0 sends blocks 0 then 2 (2, 1
    packets), member 1 blocks 1 then 0 (2, 2), member 2 blocks 2 then 1 (1, 2)."""
    w = I.Workload(3)
    ids = w.collective(I.RS, [0, 1, 2], 12289)
    ev = _traced(I.single_switch(3, 1, 0), w, nc=1, chunk=1 << 20)
    assert [_per_message(ev, ids[i]) for i in range(3)] == [[2, 1], [2, 2], [1, 2]]


def test_nic_round_robin_and_partition_extra_byte():
    """A NIC serves its send lanes round-robin from its pointer (Multiverse
    section 3.2, NIC send), and of AutoCCL's NC partitions (section 2.3) the
    first S mod NC carry one byte more.  Reduce-scatter of
    16,385 B over 2 ranks with NC = 2: channel 0's partition is 8,193 B, so
    member 0's block on channel 0 is 4,097 B (2 packets) and on channel 1
    4,096 B (1 packet).  Member 0 injects on channel 0, channel 1, channel 0."""
    w = I.Workload(2)
    w.collective(I.RS, [0, 1], 16385)
    ev = _traced(I.single_switch(2, 1, 0), w, nc=2, chunk=1 << 20)
    keys = ev[(ev["kind"] == O.EV_INJECT) & (ev["a"] == 0)]["b"]
    assert len(keys) == 3 and keys[0] == keys[2] and keys[0] != keys[1]


def test_alltoall_chunks_stripe_over_lanes():
    """All-to-all chunk j goes on lane j mod NC, destinations in rotation
    order from the next rank.  Rank 0 sends two chunks to rank 1 and one each
    to ranks 2 and 3 (a packet a chunk), NC = 2: lane 0 carries chunks 0 and 2
    (to ranks 1 and 2), lane 1 chunks 1 and 3 (to ranks 1 and 3), so the
    NIC's round robin delivers to ranks 1, 1, 2, 3."""
    w = I.Workload(4)
    ids = w.collective(I.A2A, [0, 1, 2, 3], 0, a2a={(0, 1): 8192, (0, 2): 4096, (0, 3): 4096})
    ev = _traced(I.single_switch(4, 1, 0), w, nc=2, chunk=4096)
    recv = ev[(ev["kind"] == O.EV_DELIVER) & (ev["b"] == ids[0])]["a"]
    assert list(recv) == [1, 1, 2, 3]


def test_duration_range_includes_both_ends():
    """Compute durations drawn from U[lo, hi] include hi.  With hi = lo + 1 ns
    and 1 tick = 1 ns, 64
    hashed compute nodes take both 1,000 and 1,001 ticks."""
    w = I.Workload(1)
    us = [w.compute(0, 1000, 1001, key=k) for k in range(64)]
    w.chain(*us)
    r = run1(I.single_switch(1, 1, 0), w, tick_ps=1000)
    d = r["node_end"][:64].astype(np.int64) - r["node_start"][:64]
    assert set(d.tolist()) == {1000, 1001}


def test_ecmp_one_path_per_connection_spread_over_up_ports():
    """ECMP (Multiverse section 5): the up port is a hash of the connection,
    so all packets of a
    connection take one path (in order), and connections spread over the up
    ports.  Eight 3-packet messages from leaf 0's hosts to leaf 1's over four
    spines: each ingress port of leaf 0 forwards up on exactly one port, and
    more than one up port is used."""
    t = I.leaf_spine(2, 4, 8)
    w = I.Workload(16)
    for i in range(8):
        w.collective(I.P2P, [i, 8 + i], 3 * 4096)
    ev = _traced(t, w, chunk=1 << 20)
    hops = ev[ev["kind"] == O.EV_HOP]
    up = {}
    for x in hops:
        if x["b"] < 8:                     # leaf 0's host-facing ingress queues 0..7
            up.setdefault(int(x["b"]), set()).add(int(x["a"]))
    assert sorted(up) == list(range(8))
    assert all(len(v) == 1 for v in up.values())
    assert all(min(v) >= 8 for v in up.values())           # ports 8..11 face the spines
    assert len(set().union(*up.values())) > 1


def test_same_tick_starts_go_in_node_order():
    """Nodes of a rank due at one tick start in node order, so the
    lower node's send lane takes the lower lane slot and the NIC's round robin
    (pointer 0) serves it first.  Rank 0's two root sends, to rank 1 (the
    lower node) and to rank 2: the first delivery is at rank 1."""
    w = I.Workload(3)
    w.collective(I.P2P, [0, 1], 2 * 4096)
    w.collective(I.P2P, [0, 2], 2 * 4096)
    ev = _traced(I.single_switch(3, 1, 0), w, chunk=1 << 20)
    recv = ev[ev["kind"] == O.EV_DELIVER]["a"]          # rank 0 is the only sender
    assert list(recv) == [1, 2, 1, 2]


def test_relay_partitions_first_get_the_extra_byte():
    """The pipelined broadcast (On Optimizing the Communication of Model
    Parallelism, section 3.1) cuts its slice like NC partitions: the first
    S mod K partitions carry one
    byte more.  S = 3*4096 + 1 in K = 3 partitions over one hop: the first
    partition is 4,097 B (2 packets), the others 4,096 B (1 packet)."""
    w = I.relay_chain(2, 3 * 4096 + 1, 3)
    ev = _traced(I.single_switch(2, 1, 0), w)
    sender = int(ev[ev["kind"] == O.EV_DELIVER]["b"][0])
    assert _per_message(ev, sender) == [2, 1, 1]


def test_zero_byte_message_is_one_packet():
    """A message of no bytes still costs one packet (a synchronisation
    message): a 0-byte point-to-point send behaves as the 1-packet lone
    message, (n-1) + L(1+delta) = 2(1+delta) ticks from its first injection."""
    delta = 3
    r = run1(I.single_switch(2, 1, delta), I.lone_message(2, 0, 1, 0), chunk=1 << 20)
    assert r["pkts_injected"][0] == 1 and r["msgs_delivered"][0] == 1
    first = 1 + delta                       # the join reaches the sender 1 + delta later
    assert r["node_end"][1] == first + 2 * (1 + delta)


def test_point_to_point_splits_into_chunks():
    """A point-to-point send is a train of messages of at most C bytes:
    S = 5*4096 + 100 with C = 8192 is 3 messages (8192, 8192, 4196 B) of
    2 + 2 + 2 = 6 packets."""
    r = run1(I.single_switch(2, 1, 0), I.lone_message(2, 0, 1, 5 * 4096 + 100), chunk=8192)
    assert r["msgs_delivered"][0] == 3 and r["pkts_injected"][0] == 6


def test_digest_depends_on_completion_ticks():
    """The per-experiment digest covers every message's completion tick: the
    same messages on links one tick slower give another digest."""
    d = [run1(I.single_switch(3, 1, delta), I.lone_message(3, 0, 2, 3 * 4096),
              chunk=4096)["digest"][0] for delta in (0, 1)]
    assert d[0] != d[1]


def test_down_route_takes_the_lowest_port():
    """A switch sends a packet down the lowest port under which its
    destination sits.  Leaf-spine with two parallel links per leaf-spine
    pair: the spine reaches leaf 1 on its ports 2 and 3 and uses port 2."""
    t = I.leaf_spine(2, 1, 1, links_per_pair=2)
    ev = _traced(t, I.lone_message(2, 0, 1, 4 * 4096), chunk=1 << 20)
    nports = t.arrays()["sw_nports"]
    spine_base = int(nports[0] + nports[1])        # switches: leaf 0, leaf 1, spine
    at_spine = {int(x["a"]) - spine_base for x in ev[ev["kind"] == O.EV_HOP]
                if spine_base <= x["a"] < spine_base + nports[2]}
    assert at_spine == {2}



def test_skipping_idle_ticks_changes_nothing():
    """Jumping the clock over ticks in which nothing can change gives the
    same results as stepping every tick one by one (brute force), over
    bottlenecked senders, credit stalls, incast, relays, rings and trees, and
    200 seeded small paths and incasts of random link times and capacities."""
    ex = []
    for sig in ([1, 3, 2, 1], [3, 1, 2, 1]):
        ex.append(I.Experiment(chain_topology(3, sig, [2, 0, 5, 1]),
                               I.lone_message(2, 0, 1, 9 * 4096), chunk=1 << 30, tick_ps=1000))
    for cap in (2, 5, 10):                         # credit loop 2*4+2 = 10
        ex.append(I.Experiment(I.single_switch(2, 1, 4), I.lone_message(2, 0, 1, 30 * 4096),
                               chunk=1 << 30, cap=cap, tick_ps=1000))
    w = I.Workload(3)
    w.collective(I.P2P, [0, 2], 7 * 4096)
    w.collective(I.P2P, [1, 2], 5 * 4096)
    ex.append(I.Experiment(I.single_switch(3, 2, 3), w, chunk=8192, cap=3, tick_ps=1000))
    ex.append(I.Experiment(I.single_switch(5, 1, 2), I.relay_chain(5, 9 * 4096, 3), tick_ps=1000))
    for algo in (I.RING, I.TREE):
        ex.append(I.Experiment(I.leaf_spine(2, 2, 3, 3),
                               I.single_collective(6, I.AR, 48 * 4096 + 5), algo=algo, nc=2,
                               chunk=16384, cap=8))
    rng = np.random.default_rng(11)              # seeded small paths and incasts
    for _ in range(150):
        nsw = int(rng.integers(1, 4))
        sig, dl = rng.integers(1, 5, nsw + 1).tolist(), rng.integers(0, 5, nsw + 1).tolist()
        ex.append(I.Experiment(chain_topology(nsw, sig, dl),
                               I.lone_message(2, 0, 1, int(rng.integers(1, 13)) * 4096),
                               chunk=int(rng.choice([4096, 8192, 1 << 30])),
                               cap=int(rng.integers(2, 7)), tick_ps=1000))
    for _ in range(50):
        w = I.Workload(3)
        w.collective(I.P2P, [0, 2], int(rng.integers(1, 9)) * 4096)
        w.collective(I.P2P, [1, 2], int(rng.integers(1, 9)) * 4096)
        ex.append(I.Experiment(I.single_switch(3, int(rng.integers(1, 4)), int(rng.integers(0, 4))),
                               w, chunk=int(rng.choice([4096, 1 << 20])),
                               cap=int(rng.integers(2, 6)), tick_ps=1000))
    p = I.Batch(ex).pack()
    a, b = O.run(p), O.run(p, no_skip=True)
    for k in ("status", "end_tick", "now", "pkts_injected", "pkt_hops", "pkts_delivered",
              "msgs_delivered", "digest", "node_start", "node_end", "violations"):
        assert (a[k] == b[k]).all(), k
    assert (a["status"] == O.ST_DONE).all()
    assert (a["ticks_active"] < b["ticks_active"]).any()      # skipping did skip


def test_tree_waits_for_both_children():
    """A tree member sends chunk j on (up, or down from the root) only
    after chunk j arrived from every child.  Three members on one switch,
    sigma 1, delta 0, one 1-packet chunk: both leaves send at tick 1 (the
    joins of tick 0 reach them one tick later); their packets are ready at
    the switch at 2, which forwards the left child's first (round robin
    from port 0) and the right child's at 3; the root receives them at 3
    and 4, and its first broadcast goes at 5 (a receipt counts from the next
    tick)."""
    ev = _traced(I.single_switch(3, 1, 0), I.single_collective(3, I.AR, 4096),
                 algo=I.TREE, nc=1, chunk=4096)
    inj = ev[ev["kind"] == O.EV_INJECT]
    assert sorted(int(x["tick"]) for x in inj if x["a"] != 0) == [1, 1]
    dl = ev[(ev["kind"] == O.EV_DELIVER) & (ev["a"] == 0)]["tick"]
    assert list(dl) == [3, 4]
    assert int(inj[inj["a"] == 0]["tick"].min()) == 5


def test_tree_depth_two_hand_trace():
    """A tree deep enough to have an internal member: 4 members on one
    switch (root 0; children 1 and 2; member 1's child 3), sigma 1, delta 0,
    one channel, two 1-packet chunks.  Traced by hand: a packet injected at
    t is at the switch at t+1 and delivered at t+2; a receipt counts from the
    next tick; acknowledgements take 2 ticks.  Leaves 2 and 3 send chunks 0,
    1 up at 1, 2 (delivered 3, 4).  Internal member 1 sends chunk j up only
    after it holds chunk j from child 3: at 4 and 5 (delivered at the root at
    6, 7).  The root broadcasts chunk 0 at 7 (to 1) and 8 (to 2), once both
    children's chunk 0 arrived, then chunk 1 at 9 and 10, round-robin over
    its two down lanes.  Member 1 forwards chunk j down only after the
    root's chunk j arrived: delivered at 9 and 11, so sent at 10 and 12
    (delivered at 3 at 12, 14).  Ends: root 14 (last acknowledgement of its
    chunk 1 to member 2), member 1 16 (acknowledgement of its last send to
    3), member 2 12, member 3 14."""
    w = I.single_collective(4, I.AR, 2 * 4096)
    e = I.Experiment(I.single_switch(4, 1, 0), w, algo=I.TREE, nc=1, chunk=4096,
                     tick_ps=1000, rec_cap=64)
    r = O.run(I.Batch([e]).pack(), 0, 1, trace_cap=10_000)
    assert r["status"][0] == O.ST_DONE
    assert list(r["node_end"][:4]) == [14, 16, 12, 14]
    ev = r["trace"]
    inj = ev[ev["kind"] == O.EV_INJECT]
    ticks = {m: [int(x["tick"]) for x in inj if x["a"] == m] for m in range(4)}
    assert ticks == {0: [7, 8, 9, 10], 1: [4, 5, 10, 12], 2: [1, 2], 3: [1, 2]}
    msg = ev[ev["kind"] == O.EV_MESSAGE]
    got = sorted((int(x["tick"]), int(x["a"]), int(x["b"])) for x in msg)
    # (delivery tick, receiving rank, sending node); node = rank here
    assert got == [(3, 0, 2), (3, 1, 3), (4, 0, 2), (4, 1, 3), (6, 0, 1), (7, 0, 1),
                   (9, 1, 0), (10, 2, 0), (11, 1, 0), (12, 2, 0), (12, 3, 1), (14, 3, 1)]


def _conn_key(node, chan, kind, drank):
    """The 24-bit connection identifier a packet carries (R10/R11 layout)."""
    return O.mix64(node | ((chan * 4 + kind) << 32) | (drank << 44)) & 0xFFFFFF


@pytest.mark.parametrize("topo", ["switch", "switch_delta", "leafspine"])
def test_tree_seven_members_data_dependencies(topo):
    """A reduction cannot send what it has not received: in a 7-member tree
    (depth 2; members 1 and 2 internal), with 2 channels of 2 one-packet
    chunks each, every member sends chunk j of channel c up only after
    chunk j of channel c arrived from each of its children, the root sends
    it down only after both children's arrived, and an internal member
    forwards it down only after the root's (its parent's) arrived.  Every
    member receives each chunk once from each child and once from its
    parent, in chunk order on each connection."""
    N, nc, chunks = 7, 2, 2
    t = {"switch": I.single_switch(N, 1, 0), "switch_delta": I.single_switch(N, 1, 3),
         "leafspine": I.leaf_spine(2, 2, 4, 2)}[topo]
    w = I.single_collective(N, I.AR, nc * chunks * 4096)
    e = I.Experiment(t, w, algo=I.TREE, nc=nc, chunk=4096, tick_ps=1000, rec_cap=1024)
    r = O.run(I.Batch([e]).pack(), 0, 1, trace_cap=100_000)
    assert r["status"][0] == O.ST_DONE and r["trace_total"] == len(r["trace"])
    ev = r["trace"]
    inj = ev[ev["kind"] == O.EV_INJECT]
    n = int(r["rec_count"][0])
    rec = sorted(zip(r["rec_key"][:n].tolist(), r["rec_sender"][:n].tolist(),
                     r["rec_tick"][:n].tolist()), key=lambda x: x[2])
    assert n == 2 * (N - 1) * nc * chunks

    def sends(node, key):          # injection tick of each chunk, in order
        return [int(x["tick"]) for x in inj if x["a"] == node and x["b"] == key]

    def delivered(node, key):      # delivery tick of each chunk, in order
        return [tk for k, s, tk in rec if k == key and s == node]

    kids = {i: [c for c in (2 * i + 1, 2 * i + 2) if c < N] for i in range(N)}
    for ch in range(nc):
        up_in = {i: [delivered(c, _conn_key(c, ch, 0, i)) for c in kids[i]] for i in range(N)}
        for i in range(N):
            for d in up_in[i]:
                assert len(d) == chunks
        for i in range(1, N):
            par = (i - 1) // 2
            up = sends(i, _conn_key(i, ch, 0, par))
            assert len(up) == chunks
            for j in range(chunks):
                for d in up_in[i]:
                    assert up[j] > d[j], (topo, ch, i, j)
            down_in = delivered(par, _conn_key(par, ch, 1 + (i - 2 * par - 1), i))
            assert len(down_in) == chunks
            for k, c in enumerate(kids[i]):
                down = sends(i, _conn_key(i, ch, 1 + k, c))
                assert len(down) == chunks
                for j in range(chunks):
                    assert down[j] > down_in[j], (topo, ch, i, j)
        for k, c in enumerate(kids[0]):
            down = sends(0, _conn_key(0, ch, 1 + k, c))
            for j in range(chunks):
                for d in up_in[0]:
                    assert down[j] > d[j], (topo, ch, j)


def test_failure_tick_completes_for_every_other_rank():
    """The tick in which one rank's table overflows still completes for
    the other ranks.  Rank 2 finishes a 2-tick compute node at tick 2, and 17
    intra-server collectives (one more than the 16 running collectives a rank
    may hold) become due at tick 3, so its table overflows at tick 3.  In the
    same tick rank 1 receives the one packet of rank 0's lone message
    (injected at 1, at the switch at 2, at rank 1 at 3): that delivery and
    its message still count."""
    w = I.Workload(3)
    w.collective(I.P2P, [0, 1], 4096)
    c = w.compute(2, 2)
    for _ in range(17):
        u = w.collective(I.AR, [2], 1000, intra=True, alpha=5, beta=(1, 1))[0]
        w.edge(c, u)
    r = O.run(I.Batch([I.Experiment(I.single_switch(3, 1, 0), w, chunk=1 << 20,
                                    tick_ps=1000, rec_cap=4)]).pack())
    assert r["status"][0] == O.ST_OVERFLOW
    assert r["node_end"][2] == 2                 # rank 2's compute node (rank-major order)
    assert r["pkts_delivered"][0] == 1 and r["msgs_delivered"][0] == 1
    assert list(r["rec_tick"][: r["rec_count"][0]]) == [3]


def test_intra_server_time_rounds_up():
    """The analytic model (Multiverse section 4.1) rounds bytes/beta up to
    whole ticks.  All-reduce over g = 4 of
    S = 8,001 B moves ceil(2*3*8001/4) = 12,002 B per GPU: at 1 tick per
    1,000 B that is 13 ticks (12.002 rounded up), after alpha = 7."""
    w = I.Workload(4)
    w.collective(I.AR, [0, 1, 2, 3], 8001, intra=True, alpha=7, beta=(1, 1000))
    r = run1(I.single_switch(4, 1, 0), w)
    assert list(r["node_end"][:4]) == [7 + 13] * 4


def test_tick_limit_is_exclusive():
    """Ticks stop at 0xFFF00000: a node that would end there overflows,
    one that ends a tick earlier completes (1 tick = 1 ns)."""
    limit = 0xFFF00000
    st = []
    for d in (limit - 1, limit):
        w = I.Workload(1)
        w.compute(0, d)
        st.append(O.run(I.Batch([I.Experiment(I.single_switch(1, 1, 0), w,
                                               tick_ps=1000)]).pack())["status"][0])
    assert st == [O.ST_DONE, O.ST_OVERFLOW]


def test_receive_counters_are_freed():
    """A membership's receive counters return to the rank when it completes:
    130 one-after-another point-to-point receives at rank 1 (more than its
    128 counters) complete."""
    w = I.Workload(2)
    prev = None
    for _ in range(130):
        a, b = w.collective(I.P2P, [0, 1], 4096)
        if prev is not None:
            w.edge(prev[0], a)
            w.edge(prev[1], b)
        prev = (a, b)
    r = run1(I.single_switch(2, 1, 0), w, chunk=1 << 20)
    assert r["msgs_delivered"][0] == 130


def test_routes_use_no_same_level_link():
    """Routes go up then down; a link between two switches of one level
    is neither, so no packet crosses it.  Two leaves under one spine, wired
    to each other too: eight connections each way between leaf 0's hosts
    and leaf 1's all pass the spine."""
    t = I.Topology("leaves-linked")
    l0, l1, sp = t.add_switch(1), t.add_switch(1), t.add_switch(2)
    hs = t.add_hosts(16)
    for h in hs[:8]:
        t.attach_host(h, l0)
    for h in hs[8:]:
        t.attach_host(h, l1)
    t.link(l0, sp)
    t.link(l1, sp)
    t.link(l0, l1)                         # leaf 0's port 9, leaf 1's port 9
    w = I.Workload(16)
    for i in range(8):
        w.collective(I.P2P, [i, 8 + i], 2 * 4096)
        w.collective(I.P2P, [8 + i, i], 2 * 4096)
    ev = _traced(t, w, chunk=1 << 20)
    hops = ev[ev["kind"] == O.EV_HOP]
    assert not np.isin(hops["a"], [9, 10 + 9]).any()       # the leaf-leaf ports (global index)
    assert (hops["a"] == 8).sum() == 8 * 2                  # leaf 0 sends everything up
    assert (hops["a"] == 10 + 8).sum() == 8 * 2             # and so does leaf 1


def test_ecmp_depends_on_seed_and_switch():
    """The up port hashes the connection with the experiment's ECMP seed
    and the switch.  Another seed moves some connections to other up ports.
    In a k=4 fat-tree the edge and the aggregation switches both have their
    up ports at local ports 2 and 3, so a hash blind to the switch would
    take the same local port at both; over eight one-packet connections
    across pods, some take different ones."""
    t = I.fat_tree(4)
    base = np.concatenate([[0], np.cumsum(t.arrays()["sw_nports"])])
    local = lambda q: int(q - base[np.searchsorted(base, q, "right") - 1])
    firsts = []
    for src, dst in [(0, 15), (1, 14), (2, 13), (3, 12), (4, 11), (5, 10), (6, 9), (7, 8)]:
        w = I.lone_message(16, src, dst, 4096)
        ev = _traced(t, w, chunk=1 << 20)
        hops = ev[ev["kind"] == O.EV_HOP]["a"]
        assert len(hops) == 5                       # edge, aggregation, core, aggregation, edge
        firsts.append((local(hops[0]), local(hops[1])))
    assert all(a in (2, 3) and b in (2, 3) for a, b in firsts)
    assert any(a != b for a, b in firsts)
    paths = []
    for sd in (0, 1):
        w = I.Workload(16)
        for src, dst in [(0, 15), (1, 14), (2, 13), (3, 12), (4, 11), (5, 10), (6, 9), (7, 8)]:
            w.collective(I.P2P, [src, dst], 4096)
        ev = _traced(t, w, chunk=1 << 20, ecmp_seed=sd)
        paths.append(sorted((int(x["b"]), int(x["a"])) for x in ev[ev["kind"] == O.EV_HOP]))
    assert paths[0] != paths[1]


def test_random_scenarios_keep_invariants():
    """Seeded random collectives on random small fabrics: every run ends
    DONE, delivers every packet it injected, breaks no run-time invariant
    (queue within cap, links within their rate, delivery at the addressed
    host) and gives the same results stepped tick by tick."""
    rng = np.random.default_rng(2024)
    ex = []
    for _ in range(200):
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
        n = 2 if kind == I.P2P else int(rng.integers(2, min(H, 6) + 1))
        ranks = [int(x) for x in rng.choice(H, n, replace=False)]
        w = I.Workload(H)
        nbytes = int(rng.choice([0, 1, 4095, 4096, 4097, int(rng.integers(1, 40)) * 4096 + int(rng.integers(0, 4096))]))
        if kind == I.A2A:
            m = {(i, j): int(rng.integers(0, 5)) * 4096 + int(rng.integers(0, 100))
                 for i in range(n) for j in range(n) if i != j}
            w.collective(I.A2A, ranks, 0, a2a=m)
        elif kind == I.RELAY:
            w.collective(I.RELAY, ranks, nbytes, parts=int(rng.integers(1, 6)))
        else:
            w.collective(kind, ranks, nbytes)
        ex.append(I.Experiment(t, w, algo=int(rng.integers(2)), nc=int(rng.integers(1, 5)),
                               chunk=int(rng.choice([4096, 8192, 3 * 4096 + 7, 1 << 20])),
                               cap=int(rng.integers(2, 17)), tick_ps=1000,
                               ecmp_seed=int(rng.integers(1 << 30))))
    p = I.Batch(ex).pack()
    a, b = O.run(p), O.run(p, no_skip=True)
    assert (a["status"] == O.ST_DONE).all()
    assert (a["violations"] == 0).all()
    assert (a["pkts_injected"] == a["pkts_delivered"]).all()
    for k in ("end_tick", "pkts_injected", "pkt_hops", "msgs_delivered", "digest", "node_end"):
        assert (a[k] == b[k]).all(), k


def test_ingress_queue_is_fifo_with_head_of_line_blocking():
    """An ingress port is one FIFO (the per-ingress to-do list of Multiverse
    section 4.2); its packets leave in arrival order,
    so a packet for a free egress waits behind a head whose egress is busy
    (head-of-line blocking).  Rank 0 alternates packets to ranks 1 and 3
    (lanes in node order) while ranks 2 and 4 also send to rank 1: port
    1 serves ingress 0 a third of the time but rank 0 offers it half its
    packets, so ingress 0 backs up.  Its packets still leave in exactly the
    order rank 0 injected them, and packets for the idle port 3 wait
    behind them (leave later than the tick after they arrived)."""
    w = I.Workload(5)
    w.collective(I.P2P, [0, 1], 8 * 4096)
    w.collective(I.P2P, [0, 3], 8 * 4096)
    w.collective(I.P2P, [2, 1], 8 * 4096)
    w.collective(I.P2P, [4, 1], 8 * 4096)
    ev = _traced(I.single_switch(5, 1, 0), w, chunk=1 << 20, cap=4)
    inj = ev[(ev["kind"] == O.EV_INJECT) & (ev["a"] == 0)]
    dst_of = {int(inj["b"][0]): 1, int(inj["b"][1]): 3}      # lane 0 -> rank 1, lane 1 -> rank 3
    want = [dst_of[int(k)] for k in inj["b"]]
    hops = ev[(ev["kind"] == O.EV_HOP) & (ev["b"] == 0)]
    assert [int(x) for x in hops["a"]] == want                 # egress port p faces host p
    ready = inj["tick"] + 1                                    # sigma 1, delta 0: at the switch next tick
    assert any(int(h["tick"]) > int(r) for h, r, d in zip(hops, ready, want) if d == 3)


def test_virtual_output_queues_remove_head_of_line_blocking():
    """With virtual output queues (the VOQ variant of the forwarding of
    Multiverse section 4.2) and the same traffic as the FIFO pin above, a
    packet for the idle port 3 no longer waits behind packets for port 1: it
    leaves the tick it is ready at the switch (one tick after its injection:
    sigma 1, delta 0), or the tick after when ingress 0 already sent a packet
    to port 1 in that tick (an ingress sends at most one packet a tick, and
    egresses take their turn in index order).  Rank 0's packets for port 1
    still leave in their injection order."""
    w = I.Workload(5)
    w.collective(I.P2P, [0, 1], 8 * 4096)
    w.collective(I.P2P, [0, 3], 8 * 4096)
    w.collective(I.P2P, [2, 1], 8 * 4096)
    w.collective(I.P2P, [4, 1], 8 * 4096)
    ev = _traced(I.single_switch(5, 1, 0), w, chunk=1 << 20, cap=4, voq=1)
    inj = ev[(ev["kind"] == O.EV_INJECT) & (ev["a"] == 0)]
    dst_of = {int(inj["b"][0]): 1, int(inj["b"][1]): 3}
    dst = [dst_of[int(k)] for k in inj["b"]]
    hops = ev[(ev["kind"] == O.EV_HOP) & (ev["b"] == 0)]
    to3 = [int(h["tick"]) for h in hops if h["a"] == 3]
    ready3 = [int(x["tick"]) + 1 for x, d in zip(inj, dst) if d == 3]
    to1 = [int(h["tick"]) for h in hops if h["a"] == 1]
    assert len(to1) == 8 and to1 == sorted(to1) and len(to3) == 8
    for left, ready in zip(to3, ready3):
        assert left == ready or (left == ready + 1 and ready in to1), (left, ready)
    assert any(left > ready for left, ready in zip(to3, ready3))     # the rule is exercised
    allh = ev[ev["kind"] == O.EV_HOP]
    pairs = [(int(h["tick"]), int(h["b"])) for h in allh]
    assert len(pairs) == len(set(pairs))          # one packet an ingress a tick


def test_virtual_output_queues_lone_message_and_invariants():
    """A lone message sees no difference (one packet an ingress a tick, no
    other traffic): the lone-message closed form holds with VOQs; incast and
    random collectives keep every invariant and deliver every packet, and
    stepping every tick gives the same results as skipping idle ticks."""
    for n, delta in ((1, 0), (7, 3), (40, 12)):
        t = I.fat_tree(4, delta)
        r = run1(t, I.lone_message(16, 0, 15, n * 4096), chunk=1 << 30, voq=1)
        assert r["node_end"][1] == (1 + delta) + (n - 1) + 6 * (1 + delta)
    rng = np.random.default_rng(17)
    exps = []
    for _ in range(40):
        delta = int(rng.integers(0, 3))
        t = [I.single_switch(6, 1, delta), I.leaf_spine(2, 2, 3, delta), I.fat_tree(4, delta)][int(rng.integers(3))]
        H = t.n_hosts
        kind = int(rng.choice([I.AR, I.RS, I.AG, I.P2P, I.A2A]))
        k = 2 if kind == I.P2P else int(rng.integers(2, min(H, 6) + 1))
        ranks = [int(x) for x in rng.choice(H, k, replace=False)]
        w = I.Workload(H)
        if kind == I.A2A:
            w.collective(I.A2A, ranks, 0, a2a={(i, j): int(rng.integers(0, 5)) * 4096 + 7
                                              for i in range(k) for j in range(k) if i != j})
        else:
            w.collective(kind, ranks, int(rng.integers(1, 30)) * 4096 + 11)
        exps.append(I.Experiment(t, w, algo=int(rng.integers(2)), nc=int(rng.integers(1, 4)),
                                 chunk=int(rng.choice([4096, 3 * 4096, 1 << 20])),
                                 cap=int(rng.integers(2, 9)), tick_ps=1000, voq=1,
                                 ecmp_seed=int(rng.integers(1 << 20))))
    p = I.Batch(exps).pack()
    a, b = O.run(p), O.run(p, no_skip=True)
    assert (a["status"] == O.ST_DONE).all() and (a["violations"] == 0).all()
    assert (a["pkts_injected"] == a["pkts_delivered"]).all()
    for k in ("end_tick", "pkt_hops", "digest", "node_end"):
        assert (a[k] == b[k]).all(), k
