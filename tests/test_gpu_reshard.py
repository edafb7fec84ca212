"""Cross-mesh resharding schedules and 1F1B / eager-1F1B pipelines on the
CUDA path, bit-exact against the oracle: every scheduler's schedule of a
multi-host resharding run as pipelined broadcasts, and both pipeline
programs with point-to-point and partitioned transfers."""
import pytest

from experiment_network_simulation_gb300 import inputs as I
from experiment_network_simulation_gb300 import reshard as R
from oracle import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from experiment_network_simulation_gb300 import mv  # noqa: E402
from test_gpu_parity import assert_same  # noqa: E402


def reshard_batch():
    """A (64, 1024, 512) fp16 tensor from S^0 S^1 R on a 2x4 mesh (hosts 0-1,
    4 GPUs each) to R S^01 S^... layouts on a 4x2 mesh (hosts 2-3) and on a
    2x4 mesh (hosts 2-3), at 10 Gbps (AlpaComm's cluster), K = 16."""
    tk = I.tick_ps(4096, 10)
    topo = I.single_switch(4, 1, I.delay_ticks(1_000_000, tk))
    exps = []
    for dst_shape, dst_spec in (((4, 2), [None, (0, 1), None]), ((2, 4), [(1,), None, (0,)])):
        ut = R.unit_tasks((64, 1024, 512), R.Mesh((2, 4), 0), [(0,), (1,), None],
                          R.Mesh(dst_shape, 8), dst_spec, elem_bytes=2)
        hts = R.host_tasks(ut, gpus_per_host=4, parts=16)
        for sch in (R.naive(hts), R.load_balance(hts), R.dfs(hts, budget=20_000),
                    R.randomized_greedy(hts, seed=0)):
            assert R.valid(hts, sch)
            w = R.schedule_workload(hts, sch, n_hosts=4, parts=16)
            exps.append(I.Experiment(topo, w, tick_ps=tk, rec_cap=4096))
    return I.Batch(exps, "reshard")


def pipeline_batch():
    exps = []
    for eager in (False, True):
        for parts in (1, 8):
            w = R.pipeline_workload(4, 6, 40_000, 80_000, 32 * 4096, eager, parts=parts)
            exps.append(I.Experiment(I.single_switch(4, 1, 12), w, chunk=1 << 30,
                                     tick_ps=81920, rec_cap=1024))
    return I.Batch(exps, "pipelines")


@pytest.mark.parametrize("make", [reshard_batch, pipeline_batch])
def test_bit_exact(make):
    p = make().pack()
    got, want = mv.simulate(p), O.run(p)
    assert (want["status"] == O.ST_DONE).all()
    assert_same(got, want)
