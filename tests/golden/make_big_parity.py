"""Write tests/golden/big_parity.json: CPU-oracle results for sampled
experiments of the full-size config-3, config-4 and config-5 batches.

Each entry names a batch, an experiment index in it and a tick limit (none:
run to completion).  The oracle simulates that one experiment alone (results
do not depend on the rest of the batch), and the file keeps its
per-experiment results plus SHA-256 digests of its per-node start and end
ticks.  Only the seeded input generators and oracle/ are used.

    python tests/golden/make_big_parity.py [--jobs N]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "big_parity.json")
UNSET = 0xFFFFFFFF

# (batch, experiment index, tick limit or None)
ENTRIES = [
    ("config4", 0, None), ("config4", 1, None), ("config4", 2, None), ("config4", 3, None),
    ("config3", 0, None),
    ("config3", 317, 1_500_000),
    ("config3", 499, 1_500_000),
    ("config5", 0, 300_000),
    ("config5", 13, 300_000),
]
SCALARS = ["status", "end_tick", "now", "pkts_injected", "pkt_hops", "pkts_delivered",
           "msgs_delivered", "digest", "rec_count"]


def one_batch(name: str, idx: int):
    from experiment_network_simulation_gb300 import inputs as I
    if name == "config3":
        return I.config3().subset([idx])
    if name == "config4":
        return I.config4(n_exp=idx + 1).subset([idx])
    if name == "config5":
        return I.config5(wave=(idx, idx + 1))
    raise ValueError(name)


def node_digest(a) -> str:
    import numpy as np
    return hashlib.sha256(np.ascontiguousarray(a, dtype=np.uint32).tobytes()).hexdigest()


def run_entry(entry):
    from oracle import oracle as O
    name, idx, limit = entry
    t0 = time.time()
    p = one_batch(name, idx).pack()
    r = O.run(p, 0, 1, UNSET - 1 if limit is None else limit)
    out = {"batch": name, "index": idx, "limit": limit}
    for k in SCALARS:
        out[k] = int(r[k][0])
    out["ticks_active"] = int(r["ticks_active"][0])
    out["node_start_sha256"] = node_digest(r["node_start"])
    out["node_end_sha256"] = node_digest(r["node_end"])
    out["oracle_seconds"] = round(time.time() - t0, 1)
    print(json.dumps(out), flush=True)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--jobs", type=int, default=os.cpu_count() or 1)
    args = ap.parse_args()
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(args.jobs, len(ENTRIES))) as pool:
        res = pool.map(run_entry, ENTRIES, chunksize=1)
    with open(OUT, "w") as f:
        json.dump({"generator": "tests/golden/make_big_parity.py", "entries": res}, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
