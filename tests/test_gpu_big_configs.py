"""Full-size batches on the CUDA path against stored CPU-oracle results.

tests/golden/big_parity.json (written by tests/golden/make_big_parity.py,
which runs only the seeded generators and the oracle) holds, for sampled
experiments of the GPT-13B 1F1B batch (config 3), the MoE dispatch/combine
batch (config 4) and the topology-search batch (config 5), the oracle's
per-experiment results and SHA-256 digests of its per-node start and end
ticks, each run to completion or to a stated tick limit.  The samples of one
batch run here together in one launch, at full size; every result must
agree bit for bit.
"""
import collections
import hashlib
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import make_big_parity as G  # noqa: E402
from experiment_network_simulation_gb300 import inputs as I  # noqa: E402
from experiment_network_simulation_gb300 import mv  # noqa: E402

ENTRIES = json.load(open(os.path.join(HERE, "golden", "big_parity.json")))["entries"]
GROUPS = collections.OrderedDict()
for e in ENTRIES:
    GROUPS.setdefault((e["batch"], e["limit"]), []).append(e)


def group_batch(name, idxs):
    if name == "config3":
        return I.config3().subset(idxs)
    if name == "config4":
        return I.config4(n_exp=max(idxs) + 1).subset(idxs)
    return I.Batch(sum((I.config5(wave=(i, i + 1)).experiments for i in idxs), []))


def sha(a):
    return hashlib.sha256(np.ascontiguousarray(a, dtype=np.uint32).tobytes()).hexdigest()


@pytest.mark.parametrize("key", list(GROUPS), ids=[f"{b}-{l or 'full'}" for b, l in GROUPS])
def test_full_size_samples_match_oracle(key):
    name, limit = key
    ents = GROUPS[key]
    p = group_batch(name, [e["index"] for e in ents]).pack()
    got = mv.simulate(p, max_ticks=limit if limit else mv.UNSET - 1)
    for j, e in enumerate(ents):
        for k in G.SCALARS:
            assert int(got[k][j]) == e[k], (name, e["index"], k, int(got[k][j]), e[k])
        a, b = got["node_offset"][j], got["node_offset"][j + 1]
        assert sha(got["node_start"][a:b]) == e["node_start_sha256"], (name, e["index"])
        assert sha(got["node_end"][a:b]) == e["node_end_sha256"], (name, e["index"])
