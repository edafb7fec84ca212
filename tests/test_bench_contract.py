"""bench.py's JSON-line contract, on the CPU: the reference arm (the oracle on
the host cores) prints exactly one line with the agreed keys, and the GPU arm
fails loudly on a machine without a GPU instead of falling back."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_json_line():
    p = _bench("--impl", "reference", "--workload", "config2", "--steps", "1", "--warmup", "3")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["impl"] == "reference"
    assert r["metric"] == "simulated packet-hops/s over experiment batch"
    assert r["unit"] == "packet-hops/s" and r["higher_is_better"] is True
    assert r["value"] > 0 and r["ms_per_step"] > 0
    assert (r["n_gpus"], r["steps"], r["warmup"]) == (1, 1, 3)
    assert r["scaling"] == "weak" and r["vs_baseline"] is None and r["data"] == "synthetic"
    assert r["config"]["workload"] == "config2"
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == r["value"]
    assert cb["sample"]
    e2e = r["e2e"]
    assert e2e["value"] == r["value"] and e2e["unit"] == r["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_times_a_window():
    """A window workload: every sampled experiment runs to the window's start
    untimed, then each step times the window's ticks from a copy of that
    state; the line declares the window."""
    p = _bench("--impl", "reference", "--workload", "gpt_small", "--steps", "2", "--warmup", "3")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["config"]["window"]["start_tick"] == 3000 and r["config"]["window"]["ticks"] == 2000
    assert r["value"] > 0 and "ticks [3000, 5000)" in r["cpu_baseline"]["sample"]


def test_default_workload_is_the_config3_window():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    assert b.DEFAULT == "config3" and b.WINDOWS["config3"][0] > 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_fails_loudly_without_a_gpu():
    p = _bench("--steps", "1", "--warmup", "3")
    assert p.returncode != 0
    assert not p.stdout.strip()


def test_reference_arm_under_torchrun_prints_once():
    """Launched the way multi-GPU runs are (torchrun, 2 ranks, rendezvous on
    127.0.0.1), the reference arm runs on rank 0 alone and prints one line."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    p = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--workload", "config2", "--gpus", "2", "--steps",
                        "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["impl"] == "reference" and r["n_gpus"] == 2 and r["value"] > 0


def test_reference_arm_with_switch_and_congestion_control_variants():
    """--voq and --cc name their variant in the line's config and change the
    workload (DCTCP's windows slow config 1's ring)."""
    lines = {}
    for extra in ([], ["--voq"], ["--cc", "dctcp"]):
        p = _bench("--impl", "reference", "--workload", "config1", "--steps", "1", "--warmup", "3",
                   *extra)
        assert p.returncode == 0, p.stderr[-2000:]
        lines[tuple(extra)] = json.loads([l for l in p.stdout.splitlines() if l.strip()][-1])
    assert lines[("--voq",)]["config"]["switch"] == "virtual output queues"
    assert lines[("--cc", "dctcp")]["config"]["congestion_control"] == "dctcp"
    assert "switch" not in lines[()]["config"] and "congestion_control" not in lines[()]["config"]
