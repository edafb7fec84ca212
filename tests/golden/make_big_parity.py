"""Write tests/golden/big_parity.json: CPU-oracle results for sampled
experiments of the full-size config-3, config-4 and config-5 batches.

Each entry names a batch, an experiment index in it and a tick limit (none:
run to completion).  The oracle simulates that one experiment alone (results
do not depend on the rest of the batch) with a per-message record for every
delivered message, and the file keeps its per-experiment results plus
SHA-256 digests of
  - its per-node start and end ticks,
  - its per-collective first-start and last-end ticks (the oracle's own
    coll_start / coll_end),
  - its per-message records (sender node, connection key, delivery tick),
    sorted by (tick, sender, key), since the order in which records are
    produced is not part of the result,
and how many of its network all-reduce memberships (the data-parallel
gradient all-reduces of the GPT batches) had started and ended.  Only the
seeded input generators and oracle/ are used.

    python tests/golden/make_big_parity.py [--jobs N] [--only BATCH:INDEX ...]
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

# Config 3 experiment index = algo*250 + nc_i*50 + chunk_i*10 + seed, with
# algo ring/tree, NC (1,2,4,8,16) and chunk (64K,128K,256K,512K,1M).  The
# samples cover both algorithms x NC {1, 16} x chunk {64K, 1M}, plus two
# middle points, each through its whole iteration (data-parallel phase
# included).  Config 5: two whole iterations on two different fabrics.
# "config3-dcqcn" / "config3-dctcp": config-3 experiments with the
# generators' DCQCN or DCTCP settings.
# (batch, experiment index, tick limit or None), longest first.
ENTRIES = [
    ("config3-dctcp", 254, None), ("config3-dcqcn", 0, None),
    ("config5", 0, None), ("config5", 13, None),
    ("config3", 0, None), ("config3", 42, None), ("config3", 203, None), ("config3", 241, None),
    ("config3", 254, None), ("config3", 295, None), ("config3", 456, None),
    ("config3", 497, None), ("config3", 189, None), ("config3", 378, None),
    ("config4", 0, None), ("config4", 1, None), ("config4", 2, None), ("config4", 3, None),
]
SCALARS = ["status", "end_tick", "now", "pkts_injected", "pkt_hops", "pkts_delivered",
           "msgs_delivered", "digest", "rec_count"]
# message records kept per experiment (more than any sampled experiment delivers)
REC_CAP = {"config3": 1 << 26, "config4": 1 << 20, "config5": 1 << 27,
           "config3-dcqcn": 1 << 26, "config3-dctcp": 1 << 26}


def with_cc(name: str, b):
    """The batch's experiments with the congestion control its name asks for."""
    from experiment_network_simulation_gb300 import inputs as I
    for e in b.experiments:
        if name.endswith("-dcqcn"):
            e.cc = I.dcqcn(e.tick_ps, e.pkt)
        elif name.endswith("-dctcp"):
            e.cc = I.DCTCP()
    return b


def one_batch(name: str, idx: int, rec_cap: int = 0):
    from experiment_network_simulation_gb300 import inputs as I
    if name.startswith("config3"):
        b = with_cc(name, I.config3().subset([idx]))
    elif name == "config4":
        b = I.config4(n_exp=idx + 1).subset([idx])
    elif name == "config5":
        b = I.config5(wave=(idx, idx + 1))
    else:
        raise ValueError(name)
    for e in b.experiments:
        e.rec_cap = rec_cap
    return b


def u32_digest(a) -> str:
    import numpy as np
    return hashlib.sha256(np.ascontiguousarray(a, dtype=np.uint32).tobytes()).hexdigest()


def records_digest(sender, key, tick) -> str:
    """SHA-256 of the (tick, sender, key) triples in ascending order."""
    import numpy as np
    rec = np.stack([np.asarray(tick, np.uint32), np.asarray(sender, np.uint32),
                    np.asarray(key, np.uint32)], 1)
    rec = rec[np.lexsort(rec.T[::-1])]
    return u32_digest(rec)


def net_allreduce_counts(packed: dict, node_start, node_end) -> tuple:
    """(memberships, started, ended) of the network all-reduces of experiment 0."""
    import numpy as np
    kind = packed["node_kind"]
    nn = int(packed["work_nnodes"][0])
    ck = packed["coll_kind"][packed["node_arg"][:nn]]
    ci = packed["coll_intra"][packed["node_arg"][:nn]]
    sel = (kind[:nn] == 2) & (ck == 0) & (ci == 0)
    return (int(sel.sum()), int((node_start[:nn][sel] != UNSET).sum()),
            int((node_end[:nn][sel] != UNSET).sum()))


def run_entry(entry):
    from oracle import oracle as O
    name, idx, limit = entry
    t0 = time.time()
    p = one_batch(name, idx, REC_CAP[name]).pack()
    r = O.run(p, 0, 1, UNSET - 1 if limit is None else limit)
    out = {"batch": name, "index": idx, "limit": limit}
    for k in SCALARS:
        out[k] = int(r[k][0])
    assert out["rec_count"] <= REC_CAP[name], "records beyond the kept capacity"
    out["ticks_active"] = int(r["ticks_active"][0])
    out["violations"] = int(r["violations"][0])
    out["node_start_sha256"] = u32_digest(r["node_start"])
    out["node_end_sha256"] = u32_digest(r["node_end"])
    out["coll_start_sha256"] = u32_digest(r["coll_start"])
    out["coll_end_sha256"] = u32_digest(r["coll_end"])
    n = out["rec_count"]
    out["records_sha256"] = records_digest(r["rec_sender"][:n], r["rec_key"][:n],
                                           r["rec_tick"][:n])
    m, s, e = net_allreduce_counts(p, r["node_start"], r["node_end"])
    out["net_allreduce_members"], out["net_allreduce_started"], out["net_allreduce_ended"] = m, s, e
    out["oracle_seconds"] = round(time.time() - t0, 1)
    print(json.dumps(out), flush=True)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--jobs", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--only", nargs="*", default=None,
                    help="recompute these BATCH:INDEX entries and keep the others")
    args = ap.parse_args()
    todo = ENTRIES
    old = {}
    if args.only:
        want = {tuple(x.split(":")) for x in args.only}
        todo = [e for e in ENTRIES if (e[0], str(e[1])) in want]
        if os.path.exists(OUT):
            old = {(x["batch"], x["index"], x["limit"]): x
                   for x in json.load(open(OUT))["entries"]}
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(args.jobs, len(todo))) as pool:
        res = pool.map(run_entry, todo, chunksize=1)
    got = {(x["batch"], x["index"], x["limit"]): x for x in res}
    entries = [got.get(e) or old[e] for e in ENTRIES if e in got or e in old]
    with open(OUT, "w") as f:
        json.dump({"generator": "tests/golden/make_big_parity.py", "entries": entries}, f,
                  indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
