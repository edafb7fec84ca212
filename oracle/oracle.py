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
        ("exp_rec_cap", "u4")]
_CT = {"u4": _P32, "u8": _P64, "i4": _PI32}
_NP = {"u4": np.uint32, "u8": np.uint64, "i4": np.int32}


class _Batch(C.Structure):
    _fields_ = _BATCH + [(n, _CT[t]) for n, t in _ARR]


_OUT = [("status", "u4"), ("end_tick", "u4"), ("now", "u4"), ("pkts_injected", "u8"),
        ("pkt_hops", "u8"), ("pkts_delivered", "u8"), ("msgs_delivered", "u8"),
        ("digest", "u8"), ("ticks_active", "u8"), ("node_start", "u4"), ("node_end", "u4"),
        ("rec_count", "u4"), ("rec_sender", "u4"), ("rec_key", "u4"), ("rec_tick", "u4"),
        ("violations", "u8")]


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
    source at `path` (the tests' planted-mistake copies)."""
    with _lock:
        key = path or LIB
        if key not in _libs:
            lib = C.CDLL(path or build())
            lib.orc_run.argtypes = [C.POINTER(_Batch), C.c_uint32, C.c_uint32, C.c_uint32,
                                    C.POINTER(_Out)]
            lib.orc_run.restype = C.c_int
            lib.orc_mix64.argtypes = [C.c_uint64]
            lib.orc_mix64.restype = C.c_uint64
            _libs[key] = lib
    return _libs[key]


def mix64(z: int) -> int:
    return int(_load().orc_mix64(C.c_uint64(z & (2 ** 64 - 1))))


def run(packed: dict, e0: int = 0, e1: int = 0, limit: int = UNSET - 1,
        lib_path: str | None = None) -> dict:
    """Run experiments [e0, e1) of a packed batch (all when e1 == 0).
    `violations` counts broken invariants (queue over capacity, a link faster
    than its serialisation time, a packet delivered to the wrong host)."""
    lib = _load(lib_path)
    keep = {}
    b = _Batch()
    b.version = packed["version"]
    b.n_topos = len(packed["topo_nhosts"])
    b.n_works = len(packed["work_nranks"])
    b.n_exps = len(packed["exp_topo"])
    for n, t in _ARR:
        a = np.ascontiguousarray(packed[n], dtype=_NP[t])
        if a.size == 0:
            a = np.zeros(1, _NP[t])
        keep[n] = a
        setattr(b, n, a.ctypes.data_as(_CT[t]))
    E = b.n_exps
    nn = packed["work_nnodes"][packed["exp_work"]].astype(np.int64)
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
    o = _Out()
    for n, t in _OUT:
        setattr(o, n, res[n].ctypes.data_as(_CT[t]))
    rcode = lib.orc_run(C.byref(b), e0, e1, limit, C.byref(o))
    if rcode != 0:
        raise RuntimeError(f"oracle rejected the batch ({rcode})")
    res["node_offset"] = np.concatenate([[0], np.cumsum(nn)])
    res["rec_offset"] = np.concatenate([[0], np.cumsum(rc)])
    return res
