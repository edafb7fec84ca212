"""ctypes front end of the plain-C CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this module.  It compiles ``mv_oracle.c`` with gcc on first
use, hands it the flat batch arrays from the seeded input generators, and
returns the per-experiment and per-node results as numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mv_oracle.c")
LIB = os.path.join(HERE, "libmv_oracle.so")
UNSET = 0xFFFFFFFF
ST_DONE, ST_RUNNING, ST_OOM, ST_DEADLOCK, ST_OVERFLOW, ST_ERROR = range(6)

_P32, _P64, _PI32 = C.POINTER(C.c_uint32), C.POINTER(C.c_uint64), C.POINTER(C.c_int32)

# field order of struct orc_batch in mv_oracle.c
_BATCH = [("version", C.c_uint32), ("n_topos", C.c_uint32), ("n_works", C.c_uint32),
          ("n_exps", C.c_uint32)]
_ARR = [("topo_nhosts", "u4"), ("topo_nsw", "u4"), ("topo_nports", "u4"),
        ("sw_nports", "u4"), ("sw_level", "u4"), ("port_peer", "i4"),
        ("port_sigma", "u4"), ("port_delta", "u4"), ("host_port", "u4"),
        ("host_sigma", "u4"), ("host_delta", "u4"),
        ("work_nranks", "u4"), ("work_nnodes", "u4"), ("work_nedges", "u4"),
        ("work_ncolls", "u4"), ("work_nmembers", "u4"), ("work_na2a", "u4"),
        ("work_na2a_in", "u4"),
        ("rank_nnodes", "u4"), ("node_kind", "u4"), ("node_arg", "u4"), ("node_npred", "u4"),
        ("node_nsucc", "u4"), ("node_dur_lo", "u4"), ("node_dur_hi", "u4"),
        ("node_dur_key", "u4"), ("succ", "u4"),
        ("coll_kind", "u4"), ("coll_intra", "u4"), ("coll_bytes", "u8"),
        ("coll_nmembers", "u4"), ("coll_parts", "u4"), ("coll_alpha", "u4"),
        ("coll_beta_num", "u4"), ("coll_beta_den", "u4"), ("member_rank", "u4"),
        ("member_node", "u4"), ("member_a2a_n", "u4"), ("a2a_dst", "u4"),
        ("a2a_bytes", "u8"), ("member_a2a_in_n", "u4"), ("a2a_in_src", "u4"),
        ("a2a_in_bytes", "u8"), ("mem", "u8"),
        ("exp_topo", "u4"), ("exp_work", "u4"), ("exp_algo", "u4"), ("exp_nc", "u4"),
        ("exp_chunk", "u8"), ("exp_pkt", "u4"), ("exp_cap", "u4"), ("exp_tick_ps", "u4"),
        ("exp_dur_seed", "u8"), ("exp_ecmp_seed", "u8"), ("exp_gpu_mem", "u8"),
        ("exp_rec_cap", "u4"), ("exp_voq", "u4"), ("exp_cc", "u4")]
_CT = {"u4": _P32, "u8": _P64, "i4": _PI32}
# event trace records (struct orc_event): kinds and their (a, b) fields
(EV_START, EV_END, EV_INJECT, EV_HOP, EV_DELIVER, EV_MESSAGE, EV_CNP, EV_CUT, EV_WINDOW,
 EV_ACK) = range(1, 11)
CC_FIELDS = 16                 # words of an experiment's DCQCN record (exp_cc)
EVENT = np.dtype([("tick", np.uint32), ("kind", np.uint32), ("a", np.uint32), ("b", np.uint32)])
_NP = {"u4": np.uint32, "u8": np.uint64, "i4": np.int32}


class _Batch(C.Structure):
    _fields_ = _BATCH + [(n, _CT[t]) for n, t in _ARR]


_OUT = [("status", "u4"), ("end_tick", "u4"), ("now", "u4"), ("pkts_injected", "u8"),
        ("pkt_hops", "u8"), ("pkts_delivered", "u8"), ("msgs_delivered", "u8"),
        ("digest", "u8"), ("ticks_active", "u8"), ("node_start", "u4"), ("node_end", "u4"),
        ("rec_count", "u4"), ("rec_sender", "u4"), ("rec_key", "u4"), ("rec_tick", "u4"),
        ("violations", "u8"), ("coll_start", "u4"), ("coll_end", "u4")]


class _Out(C.Structure):
    _fields_ = [(n, _CT[t]) for n, t in _OUT]


_lock = threading.Lock()
_libs = {}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C99, -O2, no target-specific flags)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC",
                               "-o", tmp, SRC])
        os.replace(tmp, LIB)
    return LIB


def _load(path: str | None = None):
    """The oracle library (built on first use), or another build of the same
    source at `path` or named by MV_ORACLE_LIB (the tests' planted-mistake
    copies)."""
    path = path or os.environ.get("MV_ORACLE_LIB") or None
    with _lock:
        key = path or LIB
        if key not in _libs:
            lib = C.CDLL(path or build())
            lib.orc_run.argtypes = [C.POINTER(_Batch), C.c_uint32, C.c_uint32, C.c_uint32,
                                    C.POINTER(_Out)]
            lib.orc_run.restype = C.c_int
            lib.orc_run_ex.argtypes = [C.POINTER(_Batch), C.c_uint32, C.c_uint32,
                                       C.c_uint32, C.POINTER(_Out), C.c_void_p,
                                       C.c_uint64, _P64, C.c_uint32]
            lib.orc_run_ex.restype = C.c_int
            lib.orc_mix64.argtypes = [C.c_uint64]
            lib.orc_mix64.restype = C.c_uint64
            lib.orc_sim_new.argtypes = [C.POINTER(_Batch), C.c_uint32]
            lib.orc_sim_new.restype = C.c_void_p
            lib.orc_sim_advance.argtypes = [C.c_void_p, C.c_uint32]
            lib.orc_sim_advance.restype = C.c_int
            lib.orc_sim_counters.argtypes = [C.c_void_p, _P64]
            lib.orc_sim_clone.argtypes = [C.c_void_p]
            lib.orc_sim_clone.restype = C.c_void_p
            lib.orc_sim_free.argtypes = [C.c_void_p]
            _libs[key] = lib
    return _libs[key]


def mix64(z: int) -> int:
    return int(_load().orc_mix64(C.c_uint64(z & (2 ** 64 - 1))))


def _batch(packed: dict):
    keep = {}
    b = _Batch()
    b.version = packed["version"]
    b.n_topos = len(packed["topo_nhosts"])
    b.n_works = len(packed["work_nranks"])
    b.n_exps = len(packed["exp_topo"])
    for n, t in _ARR:
        if n == "exp_cc" and packed.get(n) is None:
            continue                              # NULL: no congestion control
        a = np.ascontiguousarray(packed[n], dtype=_NP[t])
        if n == "exp_cc" and a.size != b.n_exps * CC_FIELDS:
            raise ValueError(f"exp_cc holds {a.size} words, not {b.n_exps} x {CC_FIELDS}")
        if a.size == 0:
            a = np.zeros(1, _NP[t])
        keep[n] = a
        setattr(b, n, a.ctypes.data_as(_CT[t]))
    return b, keep


class Paused:
    """One experiment of a packed batch, stepped in pieces: ``advance(limit)``
    simulates up to tick ``limit`` (exclusive) and can be called again with
    a larger limit; ``clone()`` copies the state, so a window of ticks can be
    timed from the same start more than once.  No per-message records."""

    def __init__(self, packed: dict, e: int, lib_path: str | None = None, _h=None, _keep=None):
        self.lib = _load(lib_path)
        if _h is None:
            self.b, self.keep = _batch(packed)
            _h = self.lib.orc_sim_new(C.byref(self.b), e)
            if not _h:
                raise RuntimeError("oracle rejected the batch")
        else:
            self.b, self.keep = _keep
        self.h = _h

    def advance(self, limit: int) -> int:
        return int(self.lib.orc_sim_advance(self.h, limit))

    def counters(self) -> dict:
        out = np.zeros(6, np.uint64)
        self.lib.orc_sim_counters(self.h, out.ctypes.data_as(_P64))
        return dict(zip(("status", "clock", "pkts_injected", "pkt_hops", "pkts_delivered",
                         "msgs_delivered"), (int(x) for x in out)))

    def clone(self) -> "Paused":
        c = Paused(None, 0, _h=self.lib.orc_sim_clone(self.h), _keep=(self.b, self.keep))
        c.lib = self.lib
        c.parent = self                       # the tables are shared with this one
        return c

    def close(self):
        if getattr(self, "h", None):
            self.lib.orc_sim_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def run(packed: dict, e0: int = 0, e1: int = 0, limit: int = UNSET - 1,
        lib_path: str | None = None, trace_cap: int = 0, no_skip: bool = False) -> dict:
    """Run experiments [e0, e1) of a packed batch (all when e1 == 0).
    Per collective instance, `coll_start` / `coll_end` hold its first
    member's start and its last member's end (UNSET while a member has not
    ended), concatenated per experiment at `coll_offset`.
    `violations` counts broken invariants (queue over capacity, a link faster
    than its serialisation time, a packet delivered to the wrong host).
    With trace_cap > 0 (one experiment: e1 = e0 + 1), `trace` holds its first
    trace_cap events (EVENT records) and `trace_total` how many happened.
    no_skip steps every tick instead of jumping over idle ones (same results
    but `ticks_active`, by the skipping rule; a brute-force check of it)."""
    lib = _load(lib_path)
    b, keep = _batch(packed)
    E = b.n_exps
    # result sizes; an out-of-range workload index is refused by the oracle
    # itself before it writes anything, so clip it here only to size arrays
    wk = np.minimum(np.asarray(packed["exp_work"], np.int64), max(0, b.n_works - 1))
    nn = packed["work_nnodes"][wk].astype(np.int64)
    rc = packed["exp_rec_cap"].astype(np.int64)
    res = {"status": np.full(E, UNSET, np.uint32), "end_tick": np.zeros(E, np.uint32),
           "now": np.zeros(E, np.uint32)}
    for k in ("pkts_injected", "pkt_hops", "pkts_delivered", "msgs_delivered", "digest",
              "ticks_active", "violations"):
        res[k] = np.zeros(E, np.uint64)
    res["node_start"] = np.full(max(1, int(nn.sum())), UNSET, np.uint32)
    res["node_end"] = np.full(max(1, int(nn.sum())), UNSET, np.uint32)
    res["rec_count"] = np.zeros(E, np.uint32)
    for k in ("rec_sender", "rec_key", "rec_tick"):
        res[k] = np.zeros(max(1, int(rc.sum())), np.uint32)
    nco = packed["work_ncolls"][wk].astype(np.int64)
    for k in ("coll_start", "coll_end"):
        res[k] = np.full(max(1, int(nco.sum())), UNSET, np.uint32)
    o = _Out()
    for n, t in _OUT:
        setattr(o, n, res[n].ctypes.data_as(_CT[t]))
    if trace_cap or no_skip:
        if trace_cap and e1 != e0 + 1:
            raise ValueError("a trace covers one experiment: e1 must be e0 + 1")
        ev = np.zeros(max(1, trace_cap), EVENT)
        n = C.c_uint64(0)
        rcode = lib.orc_run_ex(C.byref(b), e0, e1, limit, C.byref(o),
                               ev.ctypes.data_as(C.c_void_p) if trace_cap else None,
                               trace_cap, C.byref(n), 1 if no_skip else 0)
        if trace_cap:
            res["trace"] = ev[: min(trace_cap, n.value)]
            res["trace_total"] = n.value
    else:
        rcode = lib.orc_run(C.byref(b), e0, e1, limit, C.byref(o))
    if rcode != 0:
        raise RuntimeError(f"oracle rejected the batch ({rcode})")
    res["node_offset"] = np.concatenate([[0], np.cumsum(nn)])
    res["rec_offset"] = np.concatenate([[0], np.cumsum(rc)])
    res["coll_offset"] = np.concatenate([[0], np.cumsum(nco)])
    return res


def first_divergence(packed: dict, other: dict, e: int, limit: int = UNSET - 1) -> dict | None:
    """Where experiment e of `other` (results of the same packed batch from
    another implementation, in the layout mv.Simulator.results() returns)
    first departs from the oracle: the earliest tick at which a node start,
    a node end or a message completion differs, with what each side has
    there.  None when the node and message results agree.  The oracle's event
    trace around that tick (run(..., trace_cap=...)) then shows what led to
    it."""
    r = run(packed, e, e + 1, limit)
    a0, a1 = int(r["node_offset"][e]), int(r["node_offset"][e + 1])
    b0 = int(other["node_offset"][e])
    found = []
    for k in ("node_start", "node_end"):
        mine = r[k][a0:a1].astype(np.int64)
        theirs = other[k][b0:b0 + (a1 - a0)].astype(np.int64)
        bad = np.nonzero(mine != theirs)[0]
        if bad.size:
            # the earlier of the two values is where the runs have parted
            at = np.minimum(mine[bad], theirs[bad])
            j = int(np.argmin(at))
            found.append({"tick": int(at[j]), "what": k, "node": int(bad[j]),
                          "oracle": int(mine[bad[j]]), "other": int(theirs[bad[j]])})
    n_mine, n_theirs = int(r["rec_count"][e]), int(other["rec_count"][e])
    c0, c1 = int(r["rec_offset"][e]), int(other["rec_offset"][e])
    k = min(n_mine, n_theirs, int(r["rec_offset"][e + 1]) - c0)
    if k:
        keys = ("rec_tick", "rec_sender", "rec_key")
        mine = np.stack([r[x][c0:c0 + k] for x in keys], 1)
        theirs = np.stack([other[x][c1:c1 + k] for x in keys], 1)
        mine = mine[np.lexsort(mine.T[::-1])]
        theirs = theirs[np.lexsort(theirs.T[::-1])]
        bad = np.nonzero((mine != theirs).any(1))[0]
        if bad.size:
            j = int(bad[0])
            found.append({"tick": int(min(mine[j, 0], theirs[j, 0])), "what": "message",
                          "oracle": [int(x) for x in mine[j]],
                          "other": [int(x) for x in theirs[j]]})
    return min(found, key=lambda f: f["tick"]) if found else None
