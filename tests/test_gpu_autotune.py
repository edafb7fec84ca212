"""The <algorithm, NC, C> search driven by the CUDA library takes exactly the
steps the oracle-driven search takes (every profile is a bit-exact
simulation, so every decision agrees), wave by wave."""
import pytest

from experiment_network_simulation_gb300 import autotune as A
from experiment_network_simulation_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from experiment_network_simulation_gb300 import mv  # noqa: E402


def tasks():
    return [A.Task(I.leaf_spine(2, 2, 4, delta=12), 8, I.AR, 2 << 20, list(range(8)), "ar2m-ls"),
            A.Task(I.fat_tree(4, delta=3), 16, I.AR, 1 << 20, list(range(16)), "ar1m-ft4"),
            A.Task(I.fat_tree(4, delta=3), 16, I.AG, 3 << 20, list(range(0, 16, 2)), "ag3m-ft4")]


def test_gpu_driven_search_equals_oracle_driven():
    gpu = A.search(tasks(), lambda p: mv.simulate(p), starts=2, seed=11)
    cpu = A.search(tasks(), lambda p: O.run(p), starts=2, seed=11)
    assert gpu["waves"] == cpu["waves"]
    assert [c.trail for c in gpu["chains"]] == [c.trail for c in cpu["chains"]]
    assert gpu["best"] == cpu["best"]
