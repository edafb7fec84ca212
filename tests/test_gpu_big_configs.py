"""Full-size batches on the CUDA path against stored CPU-oracle results.

tests/golden/big_parity.json (written by tests/golden/make_big_parity.py,
which runs only the seeded generators and the oracle) holds, for sampled
experiments of the GPT-13B 1F1B batch (config 3: ring and tree, NC 1 and 16,
chunks of 64 KiB and 1 MiB, and two middle points), the MoE dispatch/combine
batch (config 4: one per fabric), the topology-search batch (config 5:
two fabrics) and config-3 experiments under DCQCN and under DCTCP, the oracle's per-experiment results and SHA-256 digests of its
per-node start and end ticks, its per-collective first start and last end,
and its per-message completion records sorted by (tick, sender, key), each
run through its whole iteration (the data-parallel gradient all-reduces
included; the file records how many of them started and ended).  The samples
of one batch run here together in one launch, at full size; every result
must agree bit for bit.
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


def group_batch(name, ents):
    idxs = [e["index"] for e in ents]
    if name.startswith("config3"):
        b = G.with_cc(name, I.config3().subset(idxs))
    elif name == "config4":
        b = I.config4(n_exp=max(idxs) + 1).subset(idxs)
    else:
        b = I.Batch(sum((I.config5(wave=(i, i + 1)).experiments for i in idxs), []))
    for x, e in zip(b.experiments, ents):
        x.rec_cap = e["rec_count"]          # every message the oracle delivered
    return b


def sha(a):
    return hashlib.sha256(np.ascontiguousarray(a, dtype=np.uint32).tobytes()).hexdigest()


@pytest.mark.parametrize("key", list(GROUPS), ids=[f"{b}-{l or 'full'}" for b, l in GROUPS])
def test_full_size_samples_match_oracle(key):
    name, limit = key
    ents = GROUPS[key]
    p = group_batch(name, ents).pack()
    got = mv.simulate(p, max_ticks=limit if limit else mv.UNSET - 1)
    for j, e in enumerate(ents):
        for k in G.SCALARS:
            assert int(got[k][j]) == e[k], (name, e["index"], k, int(got[k][j]), e[k])
        a, b = got["node_offset"][j], got["node_offset"][j + 1]
        assert sha(got["node_start"][a:b]) == e["node_start_sha256"], (name, e["index"])
        assert sha(got["node_end"][a:b]) == e["node_end_sha256"], (name, e["index"])
        a, b = got["coll_offset"][j], got["coll_offset"][j + 1]
        assert sha(got["coll_start"][a:b]) == e["coll_start_sha256"], (name, e["index"])
        assert sha(got["coll_end"][a:b]) == e["coll_end_sha256"], (name, e["index"])
        a, n = got["rec_offset"][j], int(got["rec_count"][j])
        assert G.records_digest(got["rec_sender"][a:a + n], got["rec_key"][a:a + n],
                                got["rec_tick"][a:a + n]) == e["records_sha256"], (name, e["index"])

