"""Run a window of ticks of a configured batch once: every experiment to the
start tick (one launch), then ticks [start, start + ticks) (one launch per
kernel build asked for, each from the same start state).  Prints the device
time of each window launch.  Used to profile the megakernel on one window:

    python -m experiment_network_simulation_gb300.window --workload config3 \\
        --exps 152 --start 2600000 --ticks 4000 --builds 3:16
"""
from __future__ import annotations

import argparse
import json

from . import inputs as I

BATCHES = {"config3": lambda: I.config3(), "config4": lambda: I.config4(),
           "config5": lambda: I.config5(n_exp=24), "gpt_small": lambda: I.gpt_small()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="config3", choices=sorted(BATCHES))
    ap.add_argument("--exps", type=int, default=0, help="first N experiments (0: all)")
    ap.add_argument("--start", type=int, required=True)
    ap.add_argument("--ticks", type=int, required=True)
    ap.add_argument("--builds", default="0:0", help="comma list of build:warps (0 = automatic)")
    args = ap.parse_args()

    import torch

    from . import mv

    b = BATCHES[args.workload]()
    if args.exps:
        b = b.subset(range(min(args.exps, len(b))))
    sim = mv.Simulator(b.pack())
    sim.run(max_ticks=args.start)
    c0 = sim.counters()
    builds = [tuple(int(x) for x in s.split(":")) for s in args.builds.split(",")]
    snap = sim.ws.clone() if len(builds) > 1 else None
    for i, (var, warps) in enumerate(builds):
        if i:
            sim.ws.copy_(snap)
            torch.cuda.synchronize()
        sim.run(max_ticks=args.ticks, variant=var, block_warps=warps)
        c = sim.counters()
        print(json.dumps({"build": var, "warps": warps, "ms": sim.last_run_ms(),
                          "experiments": len(b),
                          "pkt_hops": int(c["pkt_hops"].sum() - c0["pkt_hops"].sum()),
                          "pkts_injected": int(c["pkts_injected"].sum() -
                                               c0["pkts_injected"].sum())}), flush=True)
    sim.close()


if __name__ == "__main__":
    main()
