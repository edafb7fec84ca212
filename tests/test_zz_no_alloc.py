"""The allocation-free entry point (mv_simulate_static) against the regular
create/run/results path.

mv_simulate_static serves callers that cannot allocate device memory (a host
framework that already holds the free memory in its own pool, a plugin
policy that forbids device allocations, a loop that cannot afford
cudaMalloc's device synchronisation): its workspace is a 32 MiB array built
into the library.  Results are integers, so the two paths must agree bit for
bit, call after call, although every call reuses the same array.
"""
import ctypes as C

import numpy as np
import pytest

from experiment_network_simulation_gb300 import inputs as I

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from experiment_network_simulation_gb300 import mv  # noqa: E402

KEYS = ["status", "end_tick", "now", "pkts_injected", "pkt_hops", "pkts_delivered",
        "msgs_delivered", "digest", "rec_count", "node_start", "node_end", "coll_start",
        "coll_end"]


def simulate_static(packed):
    lib = mv.library()
    f = lib.mv_simulate_static
    f.argtypes = [C.POINTER(mv.BatchDesc), C.c_uint32, C.c_void_p, C.POINTER(mv.ResultsView),
                  C.POINTER(C.c_uint64)]
    f.restype = C.c_int
    d, keep = mv.make_desc(packed)
    nn, nr, nco = C.c_uint64(), C.c_uint64(), C.c_uint64()
    assert lib.mv_result_sizes(C.byref(d), C.byref(nn), C.byref(nr), C.byref(nco)) == mv.MV_OK
    E = int(d.n_exps)
    res = {}
    view = mv.ResultsView()
    for name, t in mv._RES:
        if name.startswith("node_"):
            n = int(nn.value)
        elif name.startswith("rec_") and name != "rec_count":
            n = int(nr.value)
        elif name.startswith("coll_"):
            n = int(nco.value)
        else:
            n = E
        res[name] = np.zeros(max(1, n), mv._NP[t])
        setattr(view, name, res[name].ctypes.data_as(mv._CT[t]))
    steps = C.c_uint64()
    stream = torch.cuda.current_stream().cuda_stream
    rc = f(C.byref(d), mv.UNSET - 1, C.c_void_p(stream), C.byref(view), C.byref(steps))
    return rc, res


def same(a, b):
    for k in KEYS:
        assert np.array_equal(a[k], b[k][: len(a[k])]), k


def test_static_matches_regular_two_calls_in_a_row():
    for packed in (I.config1().pack(), I.config2(n_exp=64, seed=5).pack()):
        want = mv.simulate(packed)
        for _ in range(2):
            rc, got = simulate_static(packed)
            assert rc == mv.MV_OK
            same(got, want)


def test_static_takes_no_device_memory():
    """Its one promise: after a first call (which loads the library's module
    and with it the array), further calls leave the device's free memory
    unchanged."""
    packed = I.config2(n_exp=32, seed=9).pack()
    rc, _ = simulate_static(packed)
    assert rc == mv.MV_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rc, _ = simulate_static(packed)
        assert rc == mv.MV_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_static_rejects_batches_beyond_its_scratch():
    exps, seed = [], 0
    while True:                          # enough broadcast experiments to exceed 32 MiB
        exps += I.config2(seed=seed).experiments
        seed += 1
        big = I.Batch(exps).pack()
        if mv.workspace_bytes(big) > 32 << 20:
            break
    rc, _ = simulate_static(big)
    assert rc == mv.MV_ENOMEM
    rc, got = simulate_static(I.config1().pack())     # still usable afterwards
    assert rc == mv.MV_OK
    same(got, mv.simulate(I.config1().pack()))
