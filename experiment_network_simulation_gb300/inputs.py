"""Seeded synthetic inputs: topologies, workload DAGs and experiment batches.

This module only builds the integer tables that describe a batch of
experiments (who is wired to whom, which DAG node waits on which, which ranks
take part in which collective, and the per-experiment parameters).  It holds
none of the simulation's arithmetic: no routing, no collective decomposition,
no timing, no hashing.  Both the CUDA library and the CPU oracle consume the
flat arrays that :meth:`Batch.pack` returns.

Units follow the Multiverse page (section 5, "simulation step"): one tick is
one packet serialisation time on the experiment's base link rate, so a
400 Gbps link carrying 4 KiB packets has sigma = 1 tick of 81,920 ps, and a
propagation delay is rounded half-up to whole ticks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# DAG node kinds (Multiverse, section 3.2: Task entities are compute or comm).
COMPUTE, INTRA, NET = 0, 1, 2
# Collective kinds.  AR/RS/AG follow NCCL's ring (Multiverse section 5,
# AutoCCL section 2.3); RELAY is AlpaComm's pipelined broadcast (section 3.1);
# P2P is a pipeline-parallel send; A2A is the MoE dispatch/combine exchange.
AR, RS, AG, RELAY, P2P, A2A = 0, 1, 2, 3, 4, 5
KIND_NAMES = {AR: "allreduce", RS: "reducescatter", AG: "allgather",
              RELAY: "relay", P2P: "p2p", A2A: "alltoall"}
# Collective algorithm (AutoCCL's A parameter).
RING, TREE = 0, 1

KIB = 1024
MIB = 1024 * 1024
FORMAT_VERSION = 1


def tick_ps(pkt_bytes: int, gbps: int) -> int:
    """Serialisation time of one packet at ``gbps``, in picoseconds, rounded up."""
    return -(-pkt_bytes * 8 * 1000 // gbps)


def delay_ticks(prop_ps: int, tick: int) -> int:
    """Propagation delay in whole ticks, rounded half-up."""
    return (2 * prop_ps + tick) // (2 * tick)


# --------------------------------------------------------------------------
# Topology
# --------------------------------------------------------------------------
class Topology:
    """Hosts (one NIC each) and switches joined by bidirectional links.

    Switch ports are numbered in the order links are attached.  Each switch
    has a tier level (edge = 1, aggregation = 2, core = 3); hosts are level 0.
    """

    def __init__(self, name: str = ""):
        self.name = name
        self.n_hosts = 0
        self.sw_level: list[int] = []
        self.sw_ports: list[list[tuple]] = []   # per switch: [(peer, sigma, delta)]
        self.host_att: list[tuple | None] = []  # per host: (switch, port, sigma, delta)
        self._edits, self._arrays = 0, None     # arrays() is cached until the next edit

    def add_switch(self, level: int) -> int:
        self._edits += 1
        self.sw_level.append(level)
        self.sw_ports.append([])
        return len(self.sw_level) - 1

    def add_hosts(self, n: int) -> list[int]:
        self._edits += 1
        ids = list(range(self.n_hosts, self.n_hosts + n))
        self.n_hosts += n
        self.host_att.extend([None] * n)
        return ids

    def attach_host(self, h: int, s: int, sigma: int = 1, delta: int = 0,
                    sigma_down: int | None = None, delta_down: int | None = None):
        """Link host ``h`` to a new port of switch ``s``.  ``sigma``/``delta``
        describe the NIC uplink; the ``*_down`` values the switch-to-host link."""
        assert self.host_att[h] is None
        self._edits += 1
        p = len(self.sw_ports[s])
        self.sw_ports[s].append((("h", h),
                                 sigma if sigma_down is None else sigma_down,
                                 delta if delta_down is None else delta_down))
        self.host_att[h] = (s, p, sigma, delta)

    def link(self, a: int, b: int, sigma: int = 1, delta: int = 0):
        self._edits += 1
        pa, pb = len(self.sw_ports[a]), len(self.sw_ports[b])
        self.sw_ports[a].append((("s", b, pb), sigma, delta))
        self.sw_ports[b].append((("s", a, pa), sigma, delta))

    @property
    def n_switches(self) -> int:
        return len(self.sw_level)

    def arrays(self) -> dict:
        """Flat per-port and per-host tables (cached until the next edit; the
        caller must not modify them)."""
        if self._arrays is not None and self._arrays[0] == self._edits:
            return self._arrays[1]
        a = self._build_arrays()
        self._arrays = (self._edits, a)
        return a

    def _build_arrays(self) -> dict:
        base = np.zeros(self.n_switches + 1, dtype=np.int64)
        for s, ports in enumerate(self.sw_ports):
            base[s + 1] = base[s] + len(ports)
        nq = int(base[-1])
        peer = np.zeros(nq, np.int32)
        sig = np.zeros(nq, np.uint32)
        dl = np.zeros(nq, np.uint32)
        for s, ports in enumerate(self.sw_ports):
            for p, (pe, sg, d) in enumerate(ports):
                q = base[s] + p
                if pe[0] == "h":
                    peer[q] = -(pe[1] + 1)
                else:
                    peer[q] = base[pe[1]] + pe[2]
                sig[q], dl[q] = sg, d
        hp = np.zeros(self.n_hosts, np.uint32)
        hs = np.zeros(self.n_hosts, np.uint32)
        hd = np.zeros(self.n_hosts, np.uint32)
        for h, att in enumerate(self.host_att):
            assert att is not None, f"host {h} not attached"
            s, p, sg, d = att
            hp[h], hs[h], hd[h] = base[s] + p, sg, d
        return dict(sw_nports=np.diff(base).astype(np.uint32),
                    sw_level=np.array(self.sw_level, np.uint32),
                    port_peer=peer, port_sigma=sig, port_delta=dl,
                    host_port=hp, host_sigma=hs, host_delta=hd)


def single_switch(n_hosts: int, sigma: int = 1, delta: int = 0) -> Topology:
    t = Topology(f"switch{n_hosts}")
    s = t.add_switch(1)
    for h in t.add_hosts(n_hosts):
        t.attach_host(h, s, sigma, delta)
    return t


def leaf_spine(n_leaves: int, n_spines: int, hosts_per_leaf: int, delta: int = 0,
               links_per_pair: int = 1, sigma: int = 1) -> Topology:
    """Two-tier Clos: every leaf wired to every spine ``links_per_pair`` times."""
    t = Topology(f"leafspine{n_leaves}x{n_spines}")
    leaves = [t.add_switch(1) for _ in range(n_leaves)]
    spines = [t.add_switch(2) for _ in range(n_spines)]
    for l in leaves:
        for h in t.add_hosts(hosts_per_leaf):
            t.attach_host(h, l, sigma, delta)
    for l in leaves:
        for s in spines:
            for _ in range(links_per_pair):
                t.link(l, s, sigma, delta)
    return t


def fat_tree(k: int, delta: int = 0, hosts_per_edge: int | None = None,
             uplinks_per_edge: int | None = None, sigma: int = 1) -> Topology:
    """Three-tier k-ary fat-tree (k pods, k/2 edge + k/2 aggregation switches
    per pod, (k/2)^2 cores).  ``hosts_per_edge``/``uplinks_per_edge`` below
    k/2 give a partially populated or oversubscribed variant."""
    half = k // 2
    hpe = half if hosts_per_edge is None else hosts_per_edge
    upe = half if uplinks_per_edge is None else uplinks_per_edge
    t = Topology(f"fattree{k}")
    edges, aggs = [], []
    for _ in range(k):
        edges.append([t.add_switch(1) for _ in range(half)])
    for _ in range(k):
        aggs.append([t.add_switch(2) for _ in range(half)])
    cores = [t.add_switch(3) for _ in range(half * half)]
    for pod in range(k):
        for e in edges[pod]:
            for h in t.add_hosts(hpe):
                t.attach_host(h, e, sigma, delta)
    for pod in range(k):
        for e in edges[pod]:
            for a in aggs[pod][:upe]:
                t.link(e, a, sigma, delta)
    for pod in range(k):
        for j, a in enumerate(aggs[pod]):
            for u in range(half):
                t.link(a, cores[j * half + u], sigma, delta)
    return t


def rail_optimized(n_servers: int, gpus_per_server: int, servers_per_group: int,
                   n_spines: int, delta: int = 0, links_per_pair: int = 1,
                   sigma: int = 1) -> Topology:
    """Rail-optimised two tier: within a group of servers, the NICs of GPU g
    share rail leaf g; every leaf is wired to every spine.  Host numbering is
    server-major (host = server * gpus_per_server + g)."""
    t = Topology(f"rail{n_servers}")
    n_groups = n_servers // servers_per_group
    leaf = [[t.add_switch(1) for _ in range(gpus_per_server)] for _ in range(n_groups)]
    spines = [t.add_switch(2) for _ in range(n_spines)]
    hosts = t.add_hosts(n_servers * gpus_per_server)
    for srv in range(n_servers):
        for g in range(gpus_per_server):
            t.attach_host(hosts[srv * gpus_per_server + g], leaf[srv // servers_per_group][g],
                          sigma, delta)
    for grp in leaf:
        for l in grp:
            for s in spines:
                for _ in range(links_per_pair):
                    t.link(l, s, sigma, delta)
    return t


# --------------------------------------------------------------------------
# Workload DAG
# --------------------------------------------------------------------------
@dataclass
class Coll:
    kind: int
    intra: bool
    nbytes: int
    ranks: list
    nodes: list
    parts: int = 0
    alpha: int = 0
    beta_num: int = 0
    beta_den: int = 1
    a2a: dict | None = None     # (src member, dst member) -> bytes


class Workload:
    """Per-rank task graphs in the ASTRA-sim style the Multiverse page uses
    (section 3.1): nodes are compute tasks with an annotated duration, or a
    rank's membership in a collective.  Edges join nodes of the same rank."""

    def __init__(self, n_ranks: int, name: str = ""):
        self.n_ranks = n_ranks
        self.name = name
        self.nodes: list[dict] = []
        self.edges: list[tuple[int, int]] = []
        self.colls: list[Coll] = []
        self.mem = None
        self._edits, self._arrays = 0, None     # arrays() is cached until the next edit

    def compute(self, rank: int, lo_ns: int, hi_ns: int | None = None, key: int = 0) -> int:
        """A compute task lasting ``lo_ns`` (or a duration hashed from
        [lo_ns, hi_ns] with ``key`` and the experiment's duration seed)."""
        self._edits += 1
        self.nodes.append(dict(rank=rank, kind=COMPUTE, arg=0, lo=lo_ns,
                               hi=lo_ns if hi_ns is None else hi_ns, key=key))
        return len(self.nodes) - 1

    def collective(self, kind: int, ranks, nbytes: int, intra: bool = False,
                   parts: int = 0, alpha: int = 0, beta: tuple = (0, 1),
                   a2a: dict | None = None) -> list[int]:
        """One collective instance over ``ranks`` (member order = list order).
        Returns the per-member node ids, in member order."""
        self._edits += 1
        ci = len(self.colls)
        ids = []
        for r in ranks:
            self.nodes.append(dict(rank=r, kind=INTRA if intra else NET, arg=ci,
                                   lo=0, hi=0, key=0))
            ids.append(len(self.nodes) - 1)
        self.colls.append(Coll(kind, intra, int(nbytes), list(ranks), ids, parts,
                               alpha, beta[0], beta[1], a2a))
        return ids

    def edge(self, u: int, v: int):
        assert self.nodes[u]["rank"] == self.nodes[v]["rank"], "edges stay within a rank"
        self._edits += 1
        self.edges.append((u, v))

    def chain(self, *nodes):
        for u, v in zip(nodes, nodes[1:]):
            self.edge(u, v)

    def set_memory_model(self, params: int, tp: int, pp: int, layers: int,
                         micro: int, seq: int, batch: int, hidden: int, heads: int):
        self._edits += 1
        self.mem = (params, tp, pp, layers, micro, seq, batch, hidden, heads)

    def arrays(self) -> dict:
        """Flat DAG, collective and all-to-all tables (cached until the next
        edit; the caller must not modify them)."""
        if self._arrays is not None and self._arrays[0] == self._edits:
            return self._arrays[1]
        a = self._build_arrays()
        self._arrays = (self._edits, a)
        return a

    def _build_arrays(self) -> dict:
        order = sorted(range(len(self.nodes)), key=lambda i: (self.nodes[i]["rank"], i))
        loc = np.empty(len(self.nodes), np.int64)
        loc[order] = np.arange(len(order))
        rank_n = np.zeros(self.n_ranks, np.uint32)
        for n in self.nodes:
            rank_n[n["rank"]] += 1
        kind = np.array([self.nodes[i]["kind"] for i in order], np.uint32)
        arg = np.array([self.nodes[i]["arg"] for i in order], np.uint32)
        lo = np.array([self.nodes[i]["lo"] for i in order], np.uint32)
        hi = np.array([self.nodes[i]["hi"] for i in order], np.uint32)
        key = np.array([self.nodes[i]["key"] for i in order], np.uint32)
        succ = [[] for _ in order]
        npred = np.zeros(len(order), np.uint32)
        for u, v in self.edges:
            succ[loc[u]].append(int(loc[v]))
            npred[loc[v]] += 1
        nsucc = np.array([len(s) for s in succ], np.uint32)
        succ_flat = np.array([v for s in succ for v in s], np.uint32)
        ck = np.array([c.kind for c in self.colls], np.uint32)
        cin = np.array([1 if c.intra else 0 for c in self.colls], np.uint32)
        cb = np.array([c.nbytes for c in self.colls], np.uint64)
        cn = np.array([len(c.ranks) for c in self.colls], np.uint32)
        cp = np.array([c.parts for c in self.colls], np.uint32)
        ca = np.array([c.alpha for c in self.colls], np.uint32)
        cbn = np.array([c.beta_num for c in self.colls], np.uint32)
        cbd = np.array([c.beta_den for c in self.colls], np.uint32)
        mr = np.array([r for c in self.colls for r in c.ranks], np.uint32)
        mn = np.array([loc[n] for c in self.colls for n in c.nodes], np.uint32)
        # all-to-all traffic, rows (per sender, in rotation order starting at
        # the next member) and columns (per receiver, by sender index)
        row_n, row_d, row_b, col_n, col_s, col_b = [], [], [], [], [], []
        for c in self.colls:
            N = len(c.ranks)
            m = c.a2a or {}
            if m:
                src = np.array([k[0] for k in m], np.int64)
                dst = np.array([k[1] for k in m], np.int64)
                byt = np.array(list(m.values()), np.int64)
                keep = (src != dst) & (byt > 0)
                src, dst, byt = src[keep], dst[keep], byt[keep]
            else:
                src = dst = byt = np.zeros(0, np.int64)
            o = np.lexsort(((dst - src) % N, src))
            row_n += np.bincount(src, minlength=N).tolist()
            row_d += dst[o].tolist()
            row_b += byt[o].tolist()
            o = np.lexsort((src, dst))
            col_n += np.bincount(dst, minlength=N).tolist()
            col_s += src[o].tolist()
            col_b += byt[o].tolist()
        mem = np.zeros(10, np.uint64)
        if self.mem is not None:
            mem[:9] = self.mem
            mem[9] = 1
        u32 = lambda x: np.array(x, np.uint32)
        return dict(rank_nnodes=rank_n, node_kind=kind, node_arg=arg, node_npred=npred,
                    node_nsucc=nsucc, node_dur_lo=lo, node_dur_hi=hi, node_dur_key=key,
                    succ=succ_flat, coll_kind=ck, coll_intra=cin, coll_bytes=cb,
                    coll_nmembers=cn, coll_parts=cp, coll_alpha=ca, coll_beta_num=cbn,
                    coll_beta_den=cbd, member_rank=mr, member_node=mn,
                    member_a2a_n=u32(row_n), a2a_dst=u32(row_d),
                    a2a_bytes=np.array(row_b, np.uint64),
                    member_a2a_in_n=u32(col_n), a2a_in_src=u32(col_s),
                    a2a_in_bytes=np.array(col_b, np.uint64), mem=mem)


# --------------------------------------------------------------------------
# Experiments and batches
# --------------------------------------------------------------------------
@dataclass
class Experiment:
    topo: Topology
    work: Workload
    algo: int = RING
    nc: int = 1
    chunk: int = 512 * KIB
    pkt: int = 4096
    cap: int = 64
    tick_ps: int = 81920
    dur_seed: int = 0
    ecmp_seed: int = 0
    gpu_mem: int = 80 * 1024 ** 3
    rec_cap: int = 0
    voq: int = 0                 # 1: switches keep virtual output queues (no head-of-line blocking)
    cc: "DCQCN | DCTCP | None" = None   # congestion control (None: lossless credit only)
    label: dict = field(default_factory=dict)


CC_FIELDS = 16
CC_LINE = 1 << 20                # the line rate in DCQCN rate units


@dataclass
class DCQCN:
    """DCQCN parameters in the simulator's units (an experiment's `cc`).

    DCQCN (Zhu et al., SIGCOMM 2015; the Multiverse page names it in its
    implementation section without parameters): switches mark packets by
    RED on queue occupancy (kmin, kmax in packets, pmax in units of 2^-16),
    receivers send congestion notifications (at most one a flow per n
    ticks), senders cut and recover their rate (gain 2^-gshift; alpha timer
    k and rate timer t in ticks, byte counter b in packets, fast recovery
    count f, additive / hyper / minimum rates in units of 2^-20 of the line
    rate)."""
    kmin: int = 1
    kmax: int = 49
    pmax: int = 655                  # 1 %
    gshift: int = 8                  # g = 1/256
    n: int = 611
    k: int = 672
    t: int = 672
    b: int = 2560
    f: int = 5
    rai: int = 105
    rhai: int = 1049
    rmin: int = 1049

    def words(self) -> list[int]:
        w = [1, self.kmin, self.kmax, self.pmax, self.gshift, self.n, self.k, self.t, self.b,
             self.f, self.rai, self.rhai, self.rmin]
        return w + [0] * (CC_FIELDS - len(w))


@dataclass
class DCTCP:
    """DCTCP parameters (an experiment's `cc`).

    DCTCP (Alizadeh et al., SIGCOMM 2010; named by the Multiverse page):
    switches mark packets above kmark queued packets, receivers acknowledge
    every packet with its mark, senders keep a window (packets) that grows
    by one packet a window of data and shrinks by alpha / 2 when marks came
    back, alpha being the gain-weighted (2^-gshift) average marked
    fraction."""
    kmark: int = 16
    gshift: int = 4                  # g = 1/16
    w0: int = 10
    wmax: int = 256

    def words(self) -> list[int]:
        w = [0] * CC_FIELDS
        w[0], w[1], w[2], w[4], w[13], w[14] = 2, self.kmark, self.kmark, self.gshift, self.w0, \
            self.wmax
        return w


def dcqcn(tick_ps: int, pkt: int = 4096, line_gbps: float = 400.0, **over) -> DCQCN:
    """Synthetic DCQCN settings converted to ticks, packets and rate units:
    marking from 5 KB to 200 KB of queue with 1 % at the top, g = 1/256, a
    notification gap of 50 us, alpha and rate timers of 55 us, a byte
    counter of 10 MB, five fast-recovery steps, additive increase 40 Mb/s,
    hyper increase 400 Mb/s and a floor of 0.1 % of the line rate."""
    us = lambda x: -(-int(x * 1_000_000) // tick_ps)       # ceil(x us / tick)
    rate = lambda mbps: max(1, round(CC_LINE * mbps / (line_gbps * 1000)))
    c = DCQCN(kmin=max(0, 5 * 1000 // pkt), kmax=max(1, 200 * 1000 // pkt), pmax=655, gshift=8,
              n=us(50), k=us(55), t=us(55), b=max(1, 10 * 1024 * 1024 // pkt), f=5,
              rai=rate(40), rhai=rate(400), rmin=max(1, CC_LINE // 1000))
    for key, v in over.items():
        setattr(c, key, v)
    return c


TOPO_FIELDS = ["sw_nports", "sw_level", "port_peer", "port_sigma", "port_delta",
               "host_port", "host_sigma", "host_delta"]
WORK_FIELDS = ["rank_nnodes", "node_kind", "node_arg", "node_npred", "node_nsucc",
               "node_dur_lo", "node_dur_hi", "node_dur_key", "succ", "coll_kind",
               "coll_intra", "coll_bytes", "coll_nmembers", "coll_parts", "coll_alpha",
               "coll_beta_num", "coll_beta_den", "member_rank", "member_node",
               "member_a2a_n", "a2a_dst", "a2a_bytes", "member_a2a_in_n", "a2a_in_src",
               "a2a_in_bytes", "mem"]
EXP_FIELDS = [("exp_topo", np.uint32), ("exp_work", np.uint32), ("exp_algo", np.uint32),
              ("exp_nc", np.uint32), ("exp_chunk", np.uint64), ("exp_pkt", np.uint32),
              ("exp_cap", np.uint32), ("exp_tick_ps", np.uint32), ("exp_dur_seed", np.uint64),
              ("exp_ecmp_seed", np.uint64), ("exp_gpu_mem", np.uint64),
              ("exp_rec_cap", np.uint32), ("exp_voq", np.uint32)]


class Batch:
    """A list of experiments; topologies and workloads shared by identity."""

    def __init__(self, experiments: list[Experiment], name: str = ""):
        self.experiments = experiments
        self.name = name
        self.topos: list[Topology] = []
        self.works: list[Workload] = []
        for e in experiments:
            if not any(e.topo is t for t in self.topos):
                self.topos.append(e.topo)
            if not any(e.work is w for w in self.works):
                self.works.append(e.work)

    def __len__(self):
        return len(self.experiments)

    def subset(self, idx) -> "Batch":
        return Batch([self.experiments[i] for i in idx], self.name)

    def pack(self) -> dict:
        """Flat arrays.  Indices stored inside a topology's (workload's) arrays
        are local to that topology (workload); ``topo_*`` / ``work_*`` count
        arrays let a reader rebuild the per-item offsets."""
        out: dict = {"version": FORMAT_VERSION}
        ta = [t.arrays() for t in self.topos]
        out["topo_nhosts"] = np.array([t.n_hosts for t in self.topos], np.uint32)
        out["topo_nsw"] = np.array([t.n_switches for t in self.topos], np.uint32)
        out["topo_nports"] = np.array([len(a["port_peer"]) for a in ta], np.uint32)
        for f in TOPO_FIELDS:
            out[f] = np.concatenate([a[f] for a in ta])
        wa = [w.arrays() for w in self.works]
        out["work_nranks"] = np.array([w.n_ranks for w in self.works], np.uint32)
        out["work_nnodes"] = np.array([len(a["node_kind"]) for a in wa], np.uint32)
        out["work_nedges"] = np.array([len(a["succ"]) for a in wa], np.uint32)
        out["work_ncolls"] = np.array([len(a["coll_kind"]) for a in wa], np.uint32)
        out["work_nmembers"] = np.array([len(a["member_rank"]) for a in wa], np.uint32)
        out["work_na2a"] = np.array([len(a["a2a_dst"]) for a in wa], np.uint32)
        out["work_na2a_in"] = np.array([len(a["a2a_in_src"]) for a in wa], np.uint32)
        for f in WORK_FIELDS:
            out[f] = np.concatenate([a[f] for a in wa]).astype(wa[0][f].dtype)
        for f, dt in EXP_FIELDS:
            out[f] = np.zeros(len(self.experiments), dt)
        out["exp_cc"] = np.zeros(len(self.experiments) * CC_FIELDS, np.uint32)
        for i, e in enumerate(self.experiments):
            ti = next(j for j, t in enumerate(self.topos) if t is e.topo)
            wi = next(j for j, w in enumerate(self.works) if w is e.work)
            assert e.work.n_ranks <= e.topo.n_hosts
            vals = [ti, wi, e.algo, e.nc, e.chunk, e.pkt, e.cap, e.tick_ps, e.dur_seed,
                    e.ecmp_seed, e.gpu_mem, e.rec_cap, e.voq]
            for (f, _), v in zip(EXP_FIELDS, vals):
                out[f][i] = v
            if e.cc is not None:
                out["exp_cc"][i * CC_FIELDS:(i + 1) * CC_FIELDS] = e.cc.words()
        return out

    def node_counts(self) -> np.ndarray:
        """Number of DAG nodes of each experiment (size of its result rows)."""
        n = {id(w): len(w.nodes) for w in self.works}
        return np.array([n[id(e.work)] for e in self.experiments], np.int64)


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------
def single_collective(n_ranks: int, kind: int, nbytes: int, members=None,
                      parts: int = 0) -> Workload:
    """Every member rank runs one network collective and nothing else."""
    w = Workload(n_ranks, f"{KIND_NAMES[kind]}{nbytes}")
    w.collective(kind, list(range(n_ranks)) if members is None else members, nbytes,
                 parts=parts)
    return w


def relay_chain(n_hosts: int, nbytes: int, parts: int) -> Workload:
    """AlpaComm's broadcast of one slice from host 0 to hosts 1..n-1, split in
    ``parts`` partitions that each receiver forwards once it holds them."""
    return single_collective(n_hosts, RELAY, nbytes, parts=parts)


def lone_message(n_ranks: int, src: int, dst: int, nbytes: int) -> Workload:
    w = Workload(n_ranks, "p2p")
    w.collective(P2P, [src, dst], nbytes)
    return w


# --------------------------------------------------------------------------
# The five benchmark batches
# --------------------------------------------------------------------------
def config1() -> Batch:
    """Ring all-reduce of 16 MiB over 8 hosts on a 2-leaf x 2-spine fabric,
    400 Gbps, 1 us propagation, 4 KiB packets, 64-packet queues; 16
    experiments over NC in {1,2,4,8} x chunk in {128K,512K,1M,4M}."""
    tk = tick_ps(4096, 400)
    topo = leaf_spine(2, 2, 4, delta=delay_ticks(1_000_000, tk))
    work = single_collective(8, AR, 16 * MIB)
    exps = []
    for nc in (1, 2, 4, 8):
        for ch in (128 * KIB, 512 * KIB, 1 * MIB, 4 * MIB):
            exps.append(Experiment(topo, work, RING, nc, ch, 4096, 64, tk,
                                   label=dict(nc=nc, chunk=ch)))
    return Batch(exps, "ring-allreduce-16MiB-8hosts-leafspine")


def config2(seed: int = 0, n_exp: int = 256) -> Batch:
    """Pipelined broadcast over A+1 hosts on one 10 Gbps switch; (A, K) pairs
    drawn without replacement from A in 2..16, K in 1..64, slice a uniform
    whole number of MiB in [1, 64]."""
    rng = np.random.default_rng(seed)
    pairs = [(a, k) for a in range(2, 17) for k in range(1, 65)]
    pick = rng.choice(len(pairs), size=n_exp, replace=False)
    sizes = rng.integers(1, 65, size=n_exp)
    tk = tick_ps(4096, 10)
    d = delay_ticks(1_000_000, tk)
    topos: dict = {}
    exps = []
    for j, p in enumerate(pick):
        a, k = pairs[p]
        if a not in topos:
            topos[a] = single_switch(a + 1, 1, d)
        work = relay_chain(a + 1, int(sizes[j]) * MIB, k)
        exps.append(Experiment(topos[a], work, RING, 1, 0, 4096, 64, tk,
                               label=dict(A=a, K=k, mib=int(sizes[j]))))
    return Batch(exps, "pipelined-broadcast-10G")


# --------------------------------------------------------------------------
# GPT-style 1F1B training iteration (config 3 / config 5 workload)
# --------------------------------------------------------------------------
def gpt_1f1b(n_servers: int, gpus: int, pp: int, layers: int, micro: int, seq: int,
             hidden: int, heads: int, params: int, tick: int, batch: int = 1,
             dur_ns=(50_000, 500_000), tp_alpha_ns: int = 10_000,
             tp_bytes_per_tick: int = 36_864) -> Workload:
    """One training iteration, per GPU, TP = gpus (one server), PP = pp
    consecutive blocks of servers, DP = the servers of a stage, rail-aligned.

    Per layer and micro-batch, forward and backward are each compute, TP
    all-reduce, compute, TP all-reduce (the TP all-reduces are intra-server,
    analytic).  Stages pass s*b*h*2/TP bytes per GPU to the neighbouring
    stage's same GPU (pipeline p2p).  A receive sits in the GPU's chain; a
    send branches off it (posted asynchronously, as the 1F1B steady state
    posts its send and receive together), so the next op does not wait for
    the send to be delivered.  Each layer's data-parallel gradient
    all-reduce (12h^2/TP parameters, 2 bytes each) starts after that layer's
    last backward, chained in backward order on a second stream so that it
    overlaps the rest of the backward pass.  Micro-batches follow 1F1B: stage
    i runs min(pp-i-1, m) warm-up forwards, then alternates, then drains.
    Compute durations are drawn from dur_ns per (stage, micro-batch, layer,
    direction, part), the same for every GPU of a stage."""
    assert n_servers % pp == 0 and layers % pp == 0
    dp = n_servers // pp
    lps = layers // pp
    R = n_servers * gpus
    w = Workload(R, f"gpt-{n_servers}x{gpus}-pp{pp}-dp{dp}")
    act_tp = seq * batch * hidden * 2                # TP all-reduce of the activations
    act_pp = act_tp // gpus                          # pipeline p2p per GPU
    dp_bytes = 12 * hidden * hidden // gpus * 2      # gradient all-reduce per layer per GPU
    alpha = max(1, -(-tp_alpha_ns * 1000 // tick))

    def rank(srv, g):
        return srv * gpus + g

    # pipeline p2p instances: (kind, boundary, micro, dp index, gpu) -> (send, recv)
    p2p = {}
    for b in range(pp - 1):
        for j in range(micro):
            for d in range(dp):
                for g in range(gpus):
                    lo, hi = rank(b * dp + d, g), rank((b + 1) * dp + d, g)
                    p2p[("act", b, j, d, g)] = tuple(w.collective(P2P, [lo, hi], act_pp))
                    p2p[("grad", b, j, d, g)] = tuple(w.collective(P2P, [hi, lo], act_pp))
    # data-parallel all-reduces: (stage, layer, gpu) -> member nodes by dp index
    dpar = {}
    for st in range(pp):
        for l in range(lps):
            for g in range(gpus):
                dpar[(st, l, g)] = w.collective(AR, [rank(st * dp + d, g) for d in range(dp)],
                                                dp_bytes)
    for st in range(pp):
        wu = min(pp - st - 1, micro)
        prog = [("F", j) for j in range(wu)]
        for j in range(micro - wu):
            prog += [("F", wu + j), ("B", j)]
        prog += [("B", j) for j in range(micro - wu, micro)]
        for d in range(dp):
            srv = st * dp + d
            chains = [[] for _ in range(gpus)]
            sends = [[] for _ in range(gpus)]        # (chain position, send node)
            layer_end = [[None] * lps for _ in range(gpus)]

            def tp_step(fb, j, l, part):
                key = (((st * micro + j) * lps + l) * 2 + (fb == "B")) * 2 + part
                for g in range(gpus):
                    chains[g].append(w.compute(rank(srv, g), dur_ns[0], dur_ns[1], key=key))
                ids = w.collective(AR, [rank(srv, g) for g in range(gpus)], act_tp, intra=True,
                                   alpha=alpha, beta=(1, tp_bytes_per_tick))
                for g in range(gpus):
                    chains[g].append(ids[g])

            for fb, j in prog:
                if fb == "F":
                    if st > 0:
                        for g in range(gpus):
                            chains[g].append(p2p[("act", st - 1, j, d, g)][1])
                    for l in range(lps):
                        tp_step("F", j, l, 0)
                        tp_step("F", j, l, 1)
                    if st < pp - 1:
                        for g in range(gpus):
                            sends[g].append((chains[g][-1], p2p[("act", st, j, d, g)][0]))
                else:
                    if st < pp - 1:
                        for g in range(gpus):
                            chains[g].append(p2p[("grad", st, j, d, g)][1])
                    for l in reversed(range(lps)):
                        tp_step("B", j, l, 0)
                        tp_step("B", j, l, 1)
                        if j == micro - 1:
                            for g in range(gpus):
                                layer_end[g][l] = chains[g][-1]
                    if st > 0:
                        for g in range(gpus):
                            sends[g].append((chains[g][-1], p2p[("grad", st - 1, j, d, g)][0]))
            for g in range(gpus):
                w.chain(*chains[g])
                for after, node in sends[g]:
                    w.edge(after, node)
                prev = None
                for l in reversed(range(lps)):        # gradient all-reduces, backward order
                    node = dpar[(st, l, g)][d]
                    w.edge(layer_end[g][l], node)
                    if prev is not None:
                        w.edge(prev, node)
                    prev = node
    w.set_memory_model(params, gpus, pp, lps, micro, seq, batch, hidden, heads)
    return w


def config3(n_exp: int | None = None) -> Batch:
    """GPT-3 13B shape (40 layers, h 5120, 40 heads, s 2048, 8 micro-batches)
    on 128 servers x 8 GPUs: TP 8 (analytic), PP 4, DP 32, k=16 fat-tree at
    400 Gbps; 500 experiments = algorithm {ring, tree} x NC {1,2,4,8,16} x
    chunk {64K..1M} x duration seeds 0..9."""
    tk = tick_ps(4096, 400)
    topo = fat_tree(16, delta=delay_ticks(1_000_000, tk), hosts_per_edge=8)
    work = gpt_1f1b(128, 8, 4, 40, 8, 2048, 5120, 40, 13_000_000_000, tk)
    exps = []
    for algo in (RING, TREE):
        for nc in (1, 2, 4, 8, 16):
            for ch in (64 * KIB, 128 * KIB, 256 * KIB, 512 * KIB, 1 * MIB):
                for seed in range(10):
                    exps.append(Experiment(topo, work, algo, nc, ch, 4096, 64, tk, dur_seed=seed,
                                           label=dict(algo=algo, nc=nc, chunk=ch, seed=seed)))
    if n_exp is not None:
        exps = exps[:n_exp]
    return Batch(exps, "gpt13b-1f1b-128x8-fattree16")


def gpt_small(algo: int = RING, nc: int = 2, chunk: int = 64 * KIB, seeds=(0, 1),
              layers: int = 4, micro: int = 3) -> Batch:
    """The config-3 DAG shape at test size: 8 servers x 2 GPUs on a k=4
    fat-tree, PP 2, DP 4, small activations."""
    tk = tick_ps(4096, 400)
    topo = fat_tree(4, delta=3, hosts_per_edge=2)
    work = gpt_1f1b(8, 2, 2, layers, micro, 256, 512, 8, 50_000_000, tk,
                    dur_ns=(2_000, 20_000), tp_alpha_ns=2_000)
    exps = [Experiment(topo, work, algo, nc, chunk, 4096, 64, tk, dur_seed=s) for s in seeds]
    return Batch(exps, "gpt-small")


def table_limits() -> Batch:
    """Experiments at and one past each per-rank table limit (send lanes 64,
    receive counters 128, pending nodes 64, running collectives 16): the
    first of each pair must finish, the second must stop with the overflow
    status."""
    tk = 1000
    exps = []
    for nc in (64, 65):                       # ring all-reduce lanes: NC a rank
        w = single_collective(2, AR, nc * 4096)
        exps.append(Experiment(single_switch(2, 1, 0), w, RING, nc, 4096, tick_ps=tk,
                               label=dict(table="lanes", n=nc)))
    for nc in (42, 43):                       # tree receive counters: 3 NC a rank
        w = single_collective(2, AR, nc * 4096)
        exps.append(Experiment(single_switch(2, 1, 0), w, TREE, nc, 4096, tick_ps=tk,
                               label=dict(table="ports", n=3 * nc)))
    for n in (64, 65):                        # pending nodes: n roots on one rank
        w = Workload(1, "roots")
        for i in range(n):
            w.compute(0, 1000 * (1 + i % 3))
        exps.append(Experiment(single_switch(1, 1, 0), w, tick_ps=tk,
                               label=dict(table="pend", n=n)))
    for n in (16, 17):                        # running memberships: n intra collectives
        w = Workload(2, "intra")
        slow = w.compute(1, 50_000)           # rank 1 joins late: rank 0 keeps n running
        prev = slow
        for _ in range(n):
            ids = w.collective(AR, [0, 1], 4096, intra=True, alpha=3, beta=(1, 1000))
            w.edge(prev, ids[1])
            prev = ids[1]
        exps.append(Experiment(single_switch(2, 1, 0), w, tick_ps=tk,
                               label=dict(table="act", n=n)))
    return Batch(exps, "table-limits")


# --------------------------------------------------------------------------
# MoE dispatch / combine (config 4)
# --------------------------------------------------------------------------
def moe_traffic(seed: int, n_ranks: int = 512, tokens: int = 128, experts: int = 256,
                topk: int = 8, hidden: int = 7168, zipf: float = 1.2):
    """Per-(source, destination) dispatch bytes.  Expert e lives on rank 2e;
    expert popularity p_e ~ (pi(e)+1)^-zipf with pi a seeded permutation;
    each token picks topk distinct experts by Gumbel-top-k on log p."""
    rng = np.random.default_rng(seed)
    pi = rng.permutation(experts)
    logp = -zipf * np.log(pi + 1.0)
    g = rng.gumbel(size=(n_ranks, tokens, experts))
    pick = np.argpartition(-(logp[None, None, :] + g), topk, axis=2)[:, :, :topk]
    counts = np.zeros((n_ranks, experts), np.int64)
    for r in range(n_ranks):
        np.add.at(counts[r], pick[r].ravel(), 1)
    per_token = hidden * 2
    byte = np.zeros((n_ranks, n_ranks), np.int64)
    stride = max(1, n_ranks // experts)
    byte[:, np.arange(experts) * stride] = counts * per_token
    return byte


def moe_workload(byte: np.ndarray, gpus: int, alpha: int, beta=(1, 36_864)) -> Workload:
    """Dispatch then combine.  Same GPU: no traffic; same server: one analytic
    intra-server exchange per server (the largest per-GPU share); else network
    all-to-all.  A rank's combine (reverse sizes) starts once its dispatch
    parts are done (the combine-receive barrier of the MoE kernels)."""
    R = byte.shape[0]
    w = Workload(R, "moe")
    srv = np.arange(R) // gpus
    same = srv[:, None] == srv[None, :]
    net = np.where(same, 0, byte)
    intra = np.where(same & ~np.eye(R, dtype=bool), byte, 0)
    stages = []
    for M_net, M_in in ((net, intra), (net.T, intra.T)):
        m = {(i, j): int(M_net[i, j]) for i, j in zip(*np.nonzero(M_net))}
        ids_net = w.collective(A2A, list(range(R)), 0, a2a=m)
        ids_in = [None] * R
        for s in range(R // gpus):
            members = list(range(s * gpus, (s + 1) * gpus))
            b = int(M_in[members].sum(axis=1).max())
            ids = w.collective(A2A, members, b, intra=True, alpha=alpha, beta=beta)
            for r, u in zip(members, ids):
                ids_in[r] = u
        stages.append((ids_net, ids_in))
    for r in range(R):
        for a in (stages[0][0][r], stages[0][1][r]):
            for b in (stages[1][0][r], stages[1][1][r]):
                w.edge(a, b)
    return w


def config4(n_seeds: int = 256, n_exp: int | None = None) -> Batch:
    """MoE dispatch/combine, 64 servers x 8 GPUs, 128 tokens per rank, hidden
    7168 bf16, top-8 of 256 experts, Zipf(1.2); four 512-NIC fabrics x
    n_seeds router seeds; NC 4, chunk 512 KiB."""
    tk = tick_ps(4096, 400)
    dl = delay_ticks(1_000_000, tk)
    topos = [leaf_spine(16, 32, 32, dl),                      # 2-tier 1:1
             leaf_spine(16, 16, 32, dl),                      # 2-tier 2:1
             fat_tree(16, dl, hosts_per_edge=4),              # 3-tier, half populated
             rail_optimized(64, 8, 32, 32, dl)]               # rail-optimised 2-tier
    alpha = max(1, -(-10_000 * 1000 // tk))
    exps = []
    for seed in range(n_seeds):
        work = moe_workload(moe_traffic(seed), 8, alpha)
        for ti, t in enumerate(topos):
            exps.append(Experiment(t, work, RING, 4, 512 * KIB, 4096, 64, tk, dur_seed=seed,
                                   label=dict(topo=ti, seed=seed)))
            if n_exp is not None and len(exps) >= n_exp:
                return Batch(exps, "moe-dispatch-combine-512")
    return Batch(exps, "moe-dispatch-combine-512")


# --------------------------------------------------------------------------
# Topology search (config 5)
# --------------------------------------------------------------------------
def clos3(radix: int, oversub: int, n_hosts: int, rail: bool, gpus: int = 8,
          delta: int = 0, sigma: int = 1) -> Topology:
    """Three-tier Clos of radix-port switches.  Edge: u = radix // (oversub+1)
    up ports (one per aggregation switch of its pod) and d = u * oversub host
    ports.  A pod has radix/2 edges and u aggregation switches; aggregation
    switch j has radix/2 up ports to core group j (cores j*radix/2 ...), each
    core one link per pod.  Plain: consecutive hosts fill an edge; rail-
    optimised: within a pod, the NIC of GPU g sits on one of the pod's edges
    of rail g (server-major host numbering)."""
    half = radix // 2
    u = radix // (oversub + 1)
    d = u * oversub
    per_pod = half * d
    pods = -(-n_hosts // per_pod)
    assert pods <= radix, "fabric does not reach the host count"
    if rail:
        assert half % gpus == 0
    t = Topology(f"clos3-r{radix}-o{oversub}-{'rail' if rail else 'plain'}")
    edges = [[t.add_switch(1) for _ in range(half)] for _ in range(pods)]
    aggs = [[t.add_switch(2) for _ in range(u)] for _ in range(pods)]
    cores = [t.add_switch(3) for _ in range(u * half)]
    hosts = t.add_hosts(n_hosts)
    for h in hosts:
        pod, i = divmod(h, per_pod)
        if rail:
            srv, g = divmod(i, gpus)               # server within the pod, GPU
            per_rail = half // gpus                # edges per rail in a pod
            e = g * per_rail + srv // d
        else:
            e = i // d
        t.attach_host(h, edges[pod][e], sigma, delta)
    for pod in range(pods):
        for e in edges[pod]:
            for a in aggs[pod]:
                t.link(e, a, sigma, delta)
        for j, a in enumerate(aggs[pod]):
            for c in range(half):
                t.link(a, cores[j * half + c], sigma, delta)
    return t


def config5_topologies(n_hosts: int = 8192, delta: int = 12) -> list:
    """Feasible members of {2,3 tiers} x {32,48,64 ports} x {1..4:1} x
    {rail-optimised, plain} for n_hosts NICs.  A 2-tier Clos of <=64-port
    switches reaches at most 64 leaves x 64 ports, so none of the 2-tier
    members reaches 8,192 NICs: all feasible members are 3-tier."""
    out = []
    for radix in (32, 48, 64):
        for o in (1, 2, 3, 4):
            for rail in (False, True):
                out.append(clos3(radix, o, n_hosts, rail, delta=delta))
    return out


def config5(n_exp: int = 10_000, topo_idx=None, wave: tuple | None = None) -> Batch:
    """Topology search: config-3's GPT-13B DAG at DP=128 (TP 8, PP 4: 512
    servers, hosts 0..4095) on 1,024-server (8,192-NIC) fabrics, ring, NC 8,
    chunk 256 KiB; experiments cycle over the 24 fabrics, then duration seeds.
    ``wave=(start, stop)`` selects a slice of the experiment list."""
    tk = tick_ps(4096, 400)
    topos = config5_topologies(8192, delay_ticks(1_000_000, tk))
    if topo_idx is not None:
        topos = [topos[i] for i in topo_idx]
    work = gpt_1f1b(512, 8, 4, 40, 8, 2048, 5120, 40, 13_000_000_000, tk)
    idx = range(n_exp) if wave is None else range(wave[0], min(wave[1], n_exp))
    exps = [Experiment(topos[i % len(topos)], work, RING, 8, 256 * KIB, 4096, 64, tk,
                       dur_seed=i // len(topos), label=dict(topo=i % len(topos)))
            for i in idx]
    return Batch(exps, "topology-search-1024srv")
