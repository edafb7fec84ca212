"""The C-ABI library loads, exports every entry point its header declares,
and validates descriptors on the host (no GPU needed for any of this)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I
from experiment_network_simulation_gb300 import mv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "mv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mv_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = mv.library()
    names = header_functions()
    assert "mv_create" in names and "mv_run" in names and "mv_results" in names
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_bytes_and_result_sizes():
    b = I.config1()
    p = b.pack()
    n = mv.workspace_bytes(p)
    assert n > 0 and n % 256 == 0
    d, _ = mv.make_desc(p)
    nn, nr = C.c_uint64(), C.c_uint64()
    assert mv.library().mv_result_sizes(C.byref(d), C.byref(nn), C.byref(nr), None) == mv.MV_OK
    assert nn.value == 16 * 8 and nr.value == 0


def _bad(p, **changes):
    q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
    for k, f in changes.items():
        f(q[k]) if callable(f) else q.__setitem__(k, f)
    d, _ = mv.make_desc(q)
    n = C.c_uint64()
    return mv.library().mv_workspace_bytes(C.byref(d), C.byref(n))


def test_descriptor_validation():
    p = I.config1().pack()
    assert _bad(p) == mv.MV_OK
    assert _bad(p, version=2) == mv.MV_EINVAL

    def asym(a): a[0] = a[1]       # peer of a port no longer points back
    assert _bad(p, port_peer=asym) == mv.MV_EINVAL

    def zero_sigma(a): a[3] = 0
    assert _bad(p, port_sigma=zero_sigma) == mv.MV_EINVAL

    def nc0(a): a[0] = 0
    assert _bad(p, exp_nc=nc0) == mv.MV_EINVAL

    def cap1(a): a[0] = 1
    assert _bad(p, exp_cap=cap1) == mv.MV_EINVAL

    def topo_oob(a): a[0] = 7
    assert _bad(p, exp_topo=topo_oob) == mv.MV_EINVAL

    def huge(a): a[0] = 1 << 41
    assert _bad(p, coll_bytes=huge) == mv.MV_EOVERFLOW

    def pred(a): a[0] += 1         # predecessor count no longer matches the edges
    assert _bad(p, node_npred=pred) == mv.MV_EINVAL


def test_too_many_switch_ports_rejected():
    t = I.single_switch(65, 1, 0)
    w = I.lone_message(2, 0, 1, 4096)
    p = I.Batch([I.Experiment(t, w, chunk=1 << 20)]).pack()
    d, _ = mv.make_desc(p)
    n = C.c_uint64()
    assert mv.library().mv_workspace_bytes(C.byref(d), C.byref(n)) == mv.MV_EINVAL


def _both(p):
    """(library accepts, oracle accepts) for one packed batch."""
    from oracle import oracle as O
    d, _ = mv.make_desc(p)
    n = C.c_uint64()
    lib_ok = mv.library().mv_workspace_bytes(C.byref(d), C.byref(n)) == mv.MV_OK
    try:
        O.run(p, limit=1)
        orc_ok = True
    except RuntimeError:
        orc_ok = False
    return lib_ok, orc_ok


def test_library_and_oracle_refuse_the_same_batches():
    """The CUDA library and the CPU oracle take the same inputs: both refuse a
    switch of 65 ports, a link delay of 64 ticks (delay + 1 beyond the
    64-entry pop log), a serialisation time of 65,536 ticks, 1,025 queue
    slots or channels, virtual output queues over more than 64 slots, and
    the other malformed descriptors below; both accept the largest legal
    values (64 ports, delay 63, 64 slots with virtual output queues)."""
    def one(topo, **kw):
        w = I.lone_message(2, 0, 1, 4096)
        kw.setdefault("chunk", 1 << 20)
        return I.Batch([I.Experiment(topo, w, tick_ps=1000, **kw)]).pack()

    assert _both(one(I.single_switch(64, 1, 63))) == (True, True)
    assert _both(one(I.single_switch(65, 1, 0))) == (False, False)
    assert _both(one(I.single_switch(4, 1, 64))) == (False, False)
    assert _both(one(I.single_switch(4, 65536, 0))) == (False, False)
    assert _both(one(I.single_switch(4, 65535, 0))) == (True, True)
    assert _both(one(I.single_switch(4, 1, 0), cap=1025)) == (False, False)
    assert _both(one(I.single_switch(4, 1, 0), nc=1025)) == (False, False)
    assert _both(one(I.single_switch(4, 1, 0), chunk=0)) == (False, False)
    assert _both(one(I.single_switch(4, 1, 0), cap=64, voq=1)) == (True, True)
    assert _both(one(I.single_switch(4, 1, 0), cap=65, voq=1)) == (False, False)
    assert _both(one(I.single_switch(4, 1, 0), voq=2)) == (False, False)
    p = I.config1().pack()

    def changed(**changes):
        q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
        for k, f in changes.items():
            f(q[k]) if callable(f) else q.__setitem__(k, f)
        return q

    def asym(a): a[0] = a[1]
    def zero(a): a[0] = 0
    def big(a): a[0] = 1 << 41
    def inc(a): a[0] += 1
    def lev(a): a[0] = 251
    for q in (changed(version=2), changed(port_peer=asym), changed(port_sigma=zero),
              changed(exp_nc=zero), changed(coll_bytes=big), changed(node_npred=inc),
              changed(sw_level=lev), changed(host_delta=lambda a: a.__setitem__(0, 64))):
        assert _both(q) == (False, False)


def test_strerror_names_codes():
    lib = mv.library()
    for code in (0, 1, -1, -2, -3, -4, -5):
        assert lib.mv_strerror(code)


def test_binding_fails_loudly_without_a_gpu():
    """No CPU fallback: without a CUDA device the simulator refuses to start."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("checks the behaviour without a GPU")
    with pytest.raises(RuntimeError, match="CUDA"):
        mv.Simulator(I.config1().pack())


def test_binding_raises_library_errors():
    p = I.config1().pack()
    p = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
    p["exp_nc"][0] = 0
    with pytest.raises(mv.MVError) as e:
        mv.workspace_bytes(p)
    assert e.value.code == mv.MV_EINVAL and str(mv.MV_EINVAL) in str(e.value)


_FUZZ = r'''
import sys, ctypes as C
import numpy as np
sys.path.insert(0, sys.argv[1])
from experiment_network_simulation_gb300 import inputs as I, mv
rng = np.random.default_rng(int(sys.argv[2]))
bases = [I.config1().pack(), I.gpt_small(seeds=(0,)).pack(),
         I.Batch([I.Experiment(I.fat_tree(4), I.single_collective(16, I.A2A, 0), nc=2)]).pack(),
         I.config2(n_exp=4).pack()]
fixed = {k for k in bases[0] if k.startswith("topo_n") or k.startswith("work_n") or k == "version"}
lib, codes, differ = mv.library(), set(), []
check_oracle = sys.argv[4] == "1"
if check_oracle:
    from oracle import oracle as O
for it in range(int(sys.argv[3])):
    p = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in bases[it % len(bases)].items()}
    keys = [k for k, v in p.items() if isinstance(v, np.ndarray) and v.size > 0 and k not in fixed]
    for _ in range(int(rng.integers(1, 4))):
        a = p[keys[int(rng.integers(len(keys)))]]
        i = int(rng.integers(a.size))
        if a.dtype == np.int32:
            a[i] = rng.integers(-70000, 70000)
        else:
            top = int(np.iinfo(a.dtype).max)
            vals = [0, 1, int(a.flat[i]) + 1, max(int(a.flat[i]) - 1, 0),
                    int(rng.integers(0, 1 << 20)), top]
            a.flat[i] = vals[int(rng.integers(len(vals)))] % (top + 1)
    d, keep = mv.make_desc(p)
    n, nn, nr = C.c_uint64(), C.c_uint64(), C.c_uint64()
    c1 = lib.mv_workspace_bytes(C.byref(d), C.byref(n))
    codes.add(c1)
    codes.add(lib.mv_result_sizes(C.byref(d), C.byref(nn), C.byref(nr), None))
    if check_oracle:
        try:
            O.run(p, limit=1)
            ok = True
        except RuntimeError:
            ok = False
        if ok != (c1 == mv.MV_OK):
            differ.append(it)
print(sorted(codes))
print(differ)
'''


def test_descriptor_fuzz_never_crashes():
    """Validation survives corrupted descriptors: with every declared count
    left as is (so each array has its declared length), random values in the
    other arrays -- counts per rank, per node, per collective and per member
    included -- give a status code, never a crash.  (A count larger than
    the workload declared once overran a host table here.)  The run is a
    child process, so a crash fails the test instead of ending the suite."""
    import subprocess
    import sys
    p = subprocess.run([sys.executable, "-c", _FUZZ, ROOT, "7", "1500", "0"],
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    codes = eval(p.stdout.strip().splitlines()[-2])
    assert set(codes) <= {mv.MV_OK, mv.MV_EINVAL, mv.MV_EOVERFLOW} and mv.MV_EINVAL in codes


def test_descriptor_fuzz_library_and_oracle_agree():
    """On corrupted descriptors the oracle refuses exactly the batches the
    library refuses (each accepted one runs one tick in the oracle)."""
    import subprocess
    import sys
    p = subprocess.run([sys.executable, "-c", _FUZZ, ROOT, "11", "2000", "1"],
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    assert eval(p.stdout.strip().splitlines()[-1]) == []


def test_size_limits_and_empty_batches():
    """Hosts are 16-bit in a packet descriptor and member indices 16-bit in a
    send lane: 65,536 hosts or members are refused.  A batch of no
    experiments is valid and has no results."""
    p = I.config1().pack()
    q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
    q["topo_nhosts"][0] = 65536
    d, _ = mv.make_desc(q)
    n = C.c_uint64()
    assert mv.library().mv_workspace_bytes(C.byref(d), C.byref(n)) == mv.MV_EINVAL
    q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
    q["coll_nmembers"][0] = 65536
    assert _bad(q) == mv.MV_EINVAL
    e = {k: (v[:0] if k.startswith("exp_") else v) for k, v in p.items()}
    assert mv.workspace_bytes(e) > 0
    d, _ = mv.make_desc(e)
    nn, nr = C.c_uint64(), C.c_uint64()
    assert mv.library().mv_result_sizes(C.byref(d), C.byref(nn), C.byref(nr), None) == mv.MV_OK
    assert nn.value == 0 and nr.value == 0
