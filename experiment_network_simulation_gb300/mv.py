"""Thin Python binding of the C ABI in ``include/mv.h`` (libmv.so).

Argument marshalling only: the batch arrays from :mod:`.inputs` are passed
as host pointers, PyTorch supplies the device workspace and the stream, and
every step of the simulation runs in the library's CUDA kernels.  There is
no CPU fallback: without the compiled library or a CUDA device this module
raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

UNSET = 0xFFFFFFFF
MV_OK, MV_INCOMPLETE = 0, 1
MV_EINVAL, MV_ENOMEM, MV_ECUDA, MV_ETIMEOUT, MV_EOVERFLOW = -1, -2, -3, -4, -5
EXP_DONE, EXP_RUNNING, EXP_OOM, EXP_DEADLOCK, EXP_OVERFLOW, EXP_ERROR = range(6)

_P32, _P64, _PI32 = C.POINTER(C.c_uint32), C.POINTER(C.c_uint64), C.POINTER(C.c_int32)
# (field, dtype) of mv_batch_desc after its four counts, in header order
_ARRAYS = [
    ("topo_nhosts", "u4"), ("topo_nsw", "u4"), ("topo_nports", "u4"), ("sw_nports", "u4"),
    ("sw_level", "u4"), ("port_peer", "i4"), ("port_sigma", "u4"), ("port_delta", "u4"),
    ("host_port", "u4"), ("host_sigma", "u4"), ("host_delta", "u4"), ("work_nranks", "u4"),
    ("work_nnodes", "u4"), ("work_nedges", "u4"), ("work_ncolls", "u4"),
    ("work_nmembers", "u4"), ("work_na2a", "u4"), ("work_na2a_in", "u4"),
    ("rank_nnodes", "u4"), ("node_kind", "u4"), ("node_arg", "u4"), ("node_npred", "u4"),
    ("node_nsucc", "u4"), ("node_dur_lo", "u4"), ("node_dur_hi", "u4"), ("node_dur_key", "u4"),
    ("succ", "u4"), ("coll_kind", "u4"), ("coll_intra", "u4"), ("coll_bytes", "u8"),
    ("coll_nmembers", "u4"), ("coll_parts", "u4"), ("coll_alpha", "u4"),
    ("coll_beta_num", "u4"), ("coll_beta_den", "u4"), ("member_rank", "u4"),
    ("member_node", "u4"), ("member_a2a_n", "u4"), ("a2a_dst", "u4"), ("a2a_bytes", "u8"),
    ("member_a2a_in_n", "u4"), ("a2a_in_src", "u4"), ("a2a_in_bytes", "u8"), ("mem", "u8"),
    ("exp_topo", "u4"), ("exp_work", "u4"), ("exp_algo", "u4"), ("exp_nc", "u4"),
    ("exp_chunk", "u8"), ("exp_pkt", "u4"), ("exp_cap", "u4"), ("exp_tick_ps", "u4"),
    ("exp_dur_seed", "u8"), ("exp_ecmp_seed", "u8"), ("exp_gpu_mem", "u8"),
    ("exp_rec_cap", "u4"), ("exp_voq", "u4"), ("exp_cc", "u4")]
CC_FIELDS = 16                     # words of an experiment's DCQCN record (MV_CC_FIELDS)
_CT = {"u4": _P32, "u8": _P64, "i4": _PI32}
_NP = {"u4": np.uint32, "u8": np.uint64, "i4": np.int32}


class BatchDesc(C.Structure):
    _fields_ = [("version", C.c_uint32), ("n_topos", C.c_uint32), ("n_works", C.c_uint32),
                ("n_exps", C.c_uint32)] + [(n, _CT[t]) for n, t in _ARRAYS]


_RES = [("status", "u4"), ("end_tick", "u4"), ("now", "u4"), ("pkts_injected", "u8"),
        ("pkt_hops", "u8"), ("pkts_delivered", "u8"), ("msgs_delivered", "u8"),
        ("digest", "u8"), ("rec_count", "u4"), ("node_start", "u4"), ("node_end", "u4"),
        ("rec_sender", "u4"), ("rec_key", "u4"), ("rec_tick", "u4"), ("coll_start", "u4"),
        ("coll_end", "u4")]


class ResultsView(C.Structure):
    _fields_ = [(n, _CT[t]) for n, t in _RES]


class RunOpts(C.Structure):
    _fields_ = [("watchdog_ns", C.c_uint64), ("grid_blocks", C.c_uint32),
                ("stage", C.c_uint32), ("block_warps", C.c_uint32), ("variant", C.c_uint32)]

STAGE_AUTO, STAGE_WAKE, STAGE_NONE = 0, 1, 2


_lib = None


def library(build: bool = True) -> C.CDLL:
    """Load libmv.so from the package directory (building it if asked)."""
    global _lib
    if _lib is None:
        path = _build.build() if build else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libmv.so not built ({path}); run build()")
        lib = C.CDLL(path)
        vp, u64p = C.c_void_p, C.POINTER(C.c_uint64)
        lib.mv_workspace_bytes.argtypes = [C.POINTER(BatchDesc), u64p]
        lib.mv_result_sizes.argtypes = [C.POINTER(BatchDesc), u64p, u64p, u64p]
        lib.mv_create.argtypes = [C.POINTER(BatchDesc), vp, C.c_uint64, vp, C.POINTER(vp)]
        lib.mv_run.argtypes = [vp, C.c_uint32, u64p]
        lib.mv_run_ex.argtypes = [vp, C.c_uint32, C.POINTER(RunOpts), u64p]
        lib.mv_results.argtypes = [vp, C.POINTER(ResultsView)]
        lib.mv_destroy.argtypes = [vp]
        lib.mv_reset.argtypes = [vp]
        lib.mv_last_run_ms.argtypes = [vp, C.POINTER(C.c_float)]
        lib.mv_strerror.argtypes = [C.c_int]
        lib.mv_strerror.restype = C.c_char_p
        for f in ("mv_workspace_bytes", "mv_result_sizes", "mv_create", "mv_run", "mv_run_ex",
                  "mv_results", "mv_destroy", "mv_reset", "mv_last_run_ms"):
            getattr(lib, f).restype = C.c_int
        _lib = lib
    return _lib


EXPORTED = ["mv_workspace_bytes", "mv_result_sizes", "mv_create", "mv_run", "mv_run_ex",
            "mv_results", "mv_destroy", "mv_reset", "mv_last_run_ms", "mv_strerror"]


class MVError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {library().mv_strerror(code).decode()} ({code})")


def make_desc(packed: dict):
    """ctypes descriptor pointing into (contiguous copies of) the packed arrays.
    Returns (desc, keepalive)."""
    keep = {}
    d = BatchDesc()
    d.version = int(packed["version"])
    d.n_topos = len(packed["topo_nhosts"])
    d.n_works = len(packed["work_nranks"])
    d.n_exps = len(packed["exp_topo"])
    for n, t in _ARRAYS:
        if n == "exp_cc" and packed.get(n) is None:
            continue                              # NULL: no congestion control
        a = np.ascontiguousarray(packed[n], dtype=_NP[t])
        if n == "exp_cc" and a.size != d.n_exps * CC_FIELDS:
            raise ValueError(f"exp_cc holds {a.size} words, not {d.n_exps} x {CC_FIELDS}")
        if a.size == 0:
            a = np.zeros(1, _NP[t])
        keep[n] = a
        setattr(d, n, a.ctypes.data_as(_CT[t]))
    return d, keep


def workspace_bytes(packed: dict) -> int:
    d, _ = make_desc(packed)
    n = C.c_uint64(0)
    rc = library().mv_workspace_bytes(C.byref(d), C.byref(n))
    if rc != MV_OK:
        raise MVError(rc, "mv_workspace_bytes")
    return int(n.value)


class Simulator:
    """One batch of experiments resident on a CUDA device.

    ``Simulator(packed)`` allocates the workspace as a torch uint8 tensor and
    calls ``mv_create`` on the current stream; ``run`` calls ``mv_run``;
    ``results`` calls ``mv_results``.
    """

    def __init__(self, packed: dict, device: str = "cuda", stream=None):
        import torch

        if not torch.cuda.is_available():
            raise RuntimeError("the simulator needs a CUDA device; there is no CPU fallback")
        self.lib = library()
        self.torch = torch
        self.device = torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.desc, self._keep = make_desc(packed)
        self.n_exps = int(self.desc.n_exps)
        n = C.c_uint64(0)
        rc = self.lib.mv_workspace_bytes(C.byref(self.desc), C.byref(n))
        if rc != MV_OK:
            raise MVError(rc, "mv_workspace_bytes")
        self.ws_bytes = int(n.value)
        nn, nr, nco = C.c_uint64(0), C.c_uint64(0), C.c_uint64(0)
        self.lib.mv_result_sizes(C.byref(self.desc), C.byref(nn), C.byref(nr), C.byref(nco))
        self.n_nodes, self.n_recs, self.n_colls = int(nn.value), int(nr.value), int(nco.value)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)
        self.ctx = C.c_void_p()
        with torch.cuda.device(self.device):
            rc = self.lib.mv_create(C.byref(self.desc), C.c_void_p(self.ws.data_ptr()),
                                    self.ws_bytes, C.c_void_p(self.stream.cuda_stream),
                                    C.byref(self.ctx))
        if rc != MV_OK:
            raise MVError(rc, "mv_create")
        self.steps = 0
        nn_per = packed["work_nnodes"][packed["exp_work"]].astype(np.int64)
        self.node_offset = np.concatenate([[0], np.cumsum(nn_per)])
        rc_per = packed["exp_rec_cap"].astype(np.int64)
        self.rec_offset = np.concatenate([[0], np.cumsum(rc_per)])
        nc_per = packed["work_ncolls"][packed["exp_work"]].astype(np.int64)
        self.coll_offset = np.concatenate([[0], np.cumsum(nc_per)])

    def run(self, max_ticks: int = UNSET - 1, watchdog_ns: int = 0, grid_blocks: int = 0,
            stage: int = STAGE_AUTO, block_warps: int = 0, variant: int = 0) -> int:
        steps = C.c_uint64(0)
        opts = RunOpts(watchdog_ns, grid_blocks, stage, block_warps, variant)
        with self.torch.cuda.device(self.device):
            rc = self.lib.mv_run_ex(self.ctx, int(max_ticks), C.byref(opts), C.byref(steps))
        self.steps = int(steps.value)
        if rc < 0:
            raise MVError(rc, "mv_run")
        return rc

    def reset(self):
        """Back to tick 0 on the device (enqueued, no wait)."""
        with self.torch.cuda.device(self.device):
            rc = self.lib.mv_reset(self.ctx)
        if rc != MV_OK:
            raise MVError(rc, "mv_reset")

    def last_run_ms(self) -> float:
        ms = C.c_float(0)
        rc = self.lib.mv_last_run_ms(self.ctx, C.byref(ms))
        if rc != MV_OK:
            raise MVError(rc, "mv_last_run_ms")
        return float(ms.value)

    def counters(self) -> dict:
        """Per-experiment status, clock and counters only (no per-node rows)."""
        E = self.n_exps
        r = {"status": np.zeros(E, np.uint32), "end_tick": np.zeros(E, np.uint32),
             "now": np.zeros(E, np.uint32)}
        for k in ("pkts_injected", "pkt_hops", "pkts_delivered", "msgs_delivered"):
            r[k] = np.zeros(E, np.uint64)
        v = ResultsView()
        for n, t in _RES:
            if n in r:
                setattr(v, n, r[n].ctypes.data_as(_CT[t]))
        with self.torch.cuda.device(self.device):
            rc = self.lib.mv_results(self.ctx, C.byref(v))
        if rc != MV_OK:
            raise MVError(rc, "mv_results")
        return r

    def results(self) -> dict:
        E = self.n_exps
        r = {"status": np.zeros(E, np.uint32), "end_tick": np.zeros(E, np.uint32),
             "now": np.zeros(E, np.uint32), "rec_count": np.zeros(E, np.uint32)}
        for k in ("pkts_injected", "pkt_hops", "pkts_delivered", "msgs_delivered", "digest"):
            r[k] = np.zeros(E, np.uint64)
        for k in ("node_start", "node_end"):
            r[k] = np.zeros(max(1, self.n_nodes), np.uint32)
        for k in ("rec_sender", "rec_key", "rec_tick"):
            r[k] = np.zeros(max(1, self.n_recs), np.uint32)
        for k in ("coll_start", "coll_end"):
            r[k] = np.zeros(max(1, self.n_colls), np.uint32)
        v = ResultsView()
        for n, t in _RES:
            setattr(v, n, r[n].ctypes.data_as(_CT[t]))
        with self.torch.cuda.device(self.device):
            rc = self.lib.mv_results(self.ctx, C.byref(v))
        if rc != MV_OK:
            raise MVError(rc, "mv_results")
        r["node_offset"] = self.node_offset
        r["rec_offset"] = self.rec_offset
        r["coll_offset"] = self.coll_offset
        return r

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.mv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def simulate(packed: dict, max_ticks: int = UNSET - 1, run_opts: dict | None = None,
             **kw) -> dict:
    """Create, run to completion (or the budget) and return the results."""
    sim = Simulator(packed, **kw)
    sim.run(max_ticks, **(run_opts or {}))
    out = sim.results()
    out["steps"] = sim.steps
    sim.close()
    return out
