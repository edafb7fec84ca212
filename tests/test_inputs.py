"""The seeded input generators build the workloads the configurations name:
unit conversions, fabric sizes, experiment sweeps and DAG shapes, each
checked against the numbers stated for it (figures derived by hand from the
configuration text and the pages)."""
import collections

import numpy as np

from experiment_network_simulation_gb300 import inputs as I


def test_tick_and_delay_units():
    """One tick is a 4 KiB packet's serialisation: 81,920 ps at 400 Gbps,
    3,276,800 ps at 10 Gbps; 1 us of propagation rounds half-up to 12 ticks
    and to 0 ticks."""
    assert I.tick_ps(4096, 400) == 81_920
    assert I.tick_ps(4096, 10) == 3_276_800
    assert I.delay_ticks(1_000_000, 81_920) == 12
    assert I.delay_ticks(1_000_000, 3_276_800) == 0


def test_config1_sweep_and_fabric():
    """16 MiB ring all-reduce over 8 hosts, 2 leaves x 2 spines, 16
    experiments = NC {1,2,4,8} x chunk {128K,512K,1M,4M}."""
    b = I.config1()
    assert len(b) == 16
    assert {(e.nc, e.chunk) for e in b.experiments} == {
        (nc, c) for nc in (1, 2, 4, 8) for c in (128 << 10, 512 << 10, 1 << 20, 4 << 20)}
    t = b.experiments[0].topo
    a = t.arrays()
    assert t.n_hosts == 8 and collections.Counter(a["sw_level"].tolist()) == {1: 2, 2: 2}
    assert set(a["port_delta"].tolist()) == {12} and set(a["host_delta"].tolist()) == {12}
    w = b.experiments[0].work
    assert [(c.kind, c.nbytes, c.ranks) for c in w.colls] == [(I.AR, 16 << 20, list(range(8)))]
    assert {(e.pkt, e.cap, e.tick_ps, e.algo) for e in b.experiments} == {(4096, 64, 81_920, I.RING)}


def test_config2_sweep():
    """256 distinct (A, K) pairs, A in 2..16, K in 1..64, a whole number of
    MiB in [1, 64], A+1 hosts on one 10 Gbps switch with no propagation
    delay in ticks."""
    b = I.config2()
    assert len(b) == 256
    ak = [(e.label["A"], e.label["K"]) for e in b.experiments]
    assert len(set(ak)) == 256
    assert all(2 <= A <= 16 and 1 <= K <= 64 for A, K in ak)
    assert all(1 <= e.label["mib"] <= 64 for e in b.experiments)
    for e in b.experiments:
        assert e.topo.n_hosts == e.label["A"] + 1 and e.tick_ps == 3_276_800
        c = e.work.colls[0]
        assert (c.kind, c.nbytes, c.parts) == (I.RELAY, e.label["mib"] << 20, e.label["K"])
        assert set(e.topo.arrays()["port_delta"].tolist()) == {0}


def test_config3_dag_shape_and_sweep():
    """GPT-13B on 128 servers x 8 GPUs (TP 8, PP 4, DP 32), 40
    layers (10 a stage), 8 micro-batches.  Per collective kind:
    - DP all-reduce of 12*h^2/TP*2 B = 78,643,200 B over 32 ranks, one per
      layer and (stage, TP rank): 10 * 32 = 320;
    - TP all-reduce (intra-server) of s*b*h*2 B = 20,971,520 B over 8 GPUs,
      four per layer and micro-batch: 4 * 10 * 8 * 128 groups = 40,960;
    - pipeline point-to-point of s*b*h*2/TP B = 2,621,440 B: 8 micro-batches
      x 3 boundaries x 2 directions x 256 (TP, DP) pairs = 12,288.
    Nodes: per GPU 4 computes + 4 TP joins per layer and micro-batch (640),
    10 DP joins and 16 (end stages) or 32 (middle stages) pipeline nodes:
    1,024 GPUs average 674, 690,176 in all.  Fabric: k=16 fat-tree, 128 edge,
    128 aggregation, 64 core switches, 1,024 NICs.  500 experiments =
    {ring, tree} x NC {1,2,4,8,16} x chunk {64K..1M} x duration seeds 0..9."""
    b = I.config3()
    w = b.experiments[0].work
    got = collections.Counter((c.kind, c.intra, c.nbytes, len(c.ranks)) for c in w.colls)
    assert got == {(I.AR, False, 78_643_200, 32): 320, (I.AR, True, 20_971_520, 8): 40_960,
                   (I.P2P, False, 2_621_440, 2): 12_288}
    assert len(w.nodes) == 690_176
    t = b.experiments[0].topo
    assert t.n_hosts == 1024
    assert collections.Counter(t.arrays()["sw_level"].tolist()) == {1: 128, 2: 128, 3: 64}
    assert len(b) == 500
    assert collections.Counter((e.algo, e.nc, e.chunk, e.dur_seed) for e in b.experiments) == {
        (a, nc, c << 10, s): 1 for a in (I.RING, I.TREE) for nc in (1, 2, 4, 8, 16)
        for c in (64, 128, 256, 512, 1024) for s in range(10)}


def test_config4_router_traffic():
    """512 ranks, 128 tokens each, top-8 distinct experts of 256 (expert
    e on rank 2e), 7,168 x 2 B a token copy.  Every rank sends 128 * 8 copies,
    only even ranks receive, an expert gets a token at most once, and the
    Zipf(1.2) popularity makes the busiest expert far busier than the
    median."""
    byte = I.moe_traffic(0)
    assert byte.shape == (512, 512)
    assert (byte.sum(axis=1) == 128 * 8 * 14_336).all()
    assert not byte[:, 1::2].any()
    assert (byte[:, ::2] <= 128 * 14_336).all()
    load = byte[:, ::2].sum(axis=0)
    assert load.max() > 4 * np.median(load)
    assert not (I.moe_traffic(1) == byte).all()
    b = I.config4(n_seeds=2)
    assert len(b) == 8 and len({id(e.topo) for e in b.experiments}) == 4
    assert all(e.topo.n_hosts == 512 and (e.nc, e.chunk) == (4, 512 << 10) for e in b.experiments)


def test_config5_fabrics():
    """24 three-tier fabrics of {32, 48, 64}-port switches x
    oversubscription {1..4}:1 x {plain, rail-optimised}, each with 8,192
    NICs, no switch beyond its radix; ring, NC 8, chunk 256 KiB; the DAG is
    config 3's at DP 128 on the first 512 servers."""
    topos = I.config5_topologies()
    assert len(topos) == 24
    for t in topos:
        a = t.arrays()
        assert t.n_hosts == 8192
        assert set(a["sw_level"].tolist()) == {1, 2, 3}
        assert a["sw_nports"].max() <= 64
    b = I.config5(n_exp=48, wave=(0, 2))
    w = b.experiments[0].work
    dp = [c for c in w.colls if c.kind == I.AR and not c.intra]
    assert {len(c.ranks) for c in dp} == {128}
    assert max(max(c.ranks) for c in w.colls) == 4095
    assert {(e.algo, e.nc, e.chunk) for e in b.experiments} == {(I.RING, 8, 256 << 10)}


def test_moe_workload_shape():
    """Dispatch then combine.  Same GPU: no traffic; same server: one
    analytic exchange per server whose size is the largest per-GPU share;
    other servers: one network all-to-all.  Combine uses the transposed
    sizes, and each rank's combine waits for both of its dispatch parts."""
    R, gpus = 16, 8
    rng = np.random.default_rng(5)
    byte = rng.integers(0, 4, (R, R)) * 14_336
    w = I.moe_workload(byte, gpus, alpha=3)
    net = [c for c in w.colls if c.kind == I.A2A and not c.intra]
    intra = [c for c in w.colls if c.kind == I.A2A and c.intra]
    assert len(net) == 2 and len(intra) == 2 * (R // gpus)
    srv = np.arange(R) // gpus
    for c, M in zip(net, (byte, byte.T)):
        want = {(i, j): int(M[i, j]) for i in range(R) for j in range(R)
                if srv[i] != srv[j] and M[i, j]}
        assert {k: v for k, v in c.a2a.items() if v} == want
    for c, M in zip(intra, [byte] * (R // gpus) + [byte.T] * (R // gpus)):
        members = c.ranks
        share = np.where(np.eye(gpus, dtype=bool), 0, M[np.ix_(members, members)]).sum(axis=1)
        assert c.nbytes == int(share.max())
    preds = collections.defaultdict(set)
    for u, v in w.edges:
        preds[v].add(u)
    for r in range(R):
        disp = {net[0].nodes[r]} | {n for c in intra[: R // gpus] for n, rr in zip(c.nodes, c.ranks) if rr == r}
        comb = [net[1].nodes[r]] + [n for c in intra[R // gpus:] for n, rr in zip(c.nodes, c.ranks) if rr == r]
        assert all(preds[v] == disp for v in comb)


def test_gpt_1f1b_schedule_and_branches():
    """Each GPU's chain runs 1F1B -- stage i does min(PP - i - 1, m)
    warm-up forwards, then alternates one forward and one backward, then
    drains the backwards; a pipeline receive sits in the chain, a send
    branches off it; each layer's DP all-reduce follows that layer's last
    backward and the previous layer's all-reduce.  PP 3, 4 micro-batches,
    one layer a stage, 2 GPUs a server (TP 2), DP 1."""
    pp, micro = 3, 4
    w = I.gpt_1f1b(3, 2, pp, 3, micro, 16, 8, 2, 1000, 1000)
    nk = [n["kind"] for n in w.nodes]
    succ = collections.defaultdict(list)
    for u, v in w.edges:
        succ[u].append(v)
    indeg = collections.Counter(v for _, v in w.edges)
    coll_of = {n: (c, i) for c in w.colls for i, n in enumerate(c.nodes)}
    for st in range(pp):
        r = st * 2                                   # GPU 0 of the stage's one server
        root = [u for u, n in enumerate(w.nodes) if n["rank"] == r and indeg[u] == 0]
        assert len(root) == 1
        seq, u = [], root[0]
        while True:
            if nk[u] == I.COMPUTE:
                key = w.nodes[u]["key"]
                part, isb, j = key & 1, (key >> 1) & 1, key >> 2   # one layer a stage
                assert (j // micro) == st
                if part == 0:
                    seq.append(("B" if isb else "F", j % micro))
            nxt = []
            for v in succ[u]:
                c, i = coll_of.get(v, (None, None))
                if c is not None and c.kind == I.P2P and i == 0:
                    continue                          # a send: a branch off the chain
                if c is not None and c.kind == I.AR and not c.intra:
                    continue                          # the DP all-reduce: a branch
                nxt.append(v)
            assert len(nxt) <= 1
            if not nxt:
                break
            u = nxt[0]
        wu = min(pp - st - 1, micro)
        want = [("F", j) for j in range(wu)]
        for j in range(micro - wu):
            want += [("F", wu + j), ("B", j)]
        want += [("B", j) for j in range(micro - wu, micro)]
        assert seq == want, (st, seq)
    dp = [c for c in w.colls if c.kind == I.AR and not c.intra]
    assert len(dp) == pp * 2                          # per stage and GPU, one layer each
    for c in dp:
        (u,) = c.nodes                                # DP 1: one member
        preds = [a for a, b in w.edges if b == u]
        assert len(preds) == 1 and nk[preds[0]] == I.INTRA   # after the last backward's TP step
