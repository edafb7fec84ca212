"""What the stored full-size oracle results cover (no GPU needed): the GPT
samples of configs 3 and 5 run through their whole iterations, so every
data-parallel gradient all-reduce membership started and ended, and the
config-3 samples span both algorithms, NC 1 and 16 and chunks of 64 KiB and
1 MiB; every sample kept all of its per-message records."""
import json
import os

from experiment_network_simulation_gb300 import inputs as I

HERE = os.path.dirname(os.path.abspath(__file__))
ENTRIES = json.load(open(os.path.join(HERE, "golden", "big_parity.json")))["entries"]


def test_gpt_samples_reach_the_data_parallel_all_reduce():
    gpt = [e for e in ENTRIES if e["batch"] in ("config3", "config5")]
    assert {e["batch"] for e in gpt} == {"config3", "config5"}
    for e in gpt:
        assert e["limit"] is None and e["status"] == 0, (e["batch"], e["index"])
        assert e["net_allreduce_members"] > 0
        assert e["net_allreduce_started"] == e["net_allreduce_members"], e["index"]
        assert e["net_allreduce_ended"] == e["net_allreduce_members"], e["index"]
    lab = {(x["algo"], x["nc"], x["chunk"]) for x in
           (I.config3().experiments[e["index"]].label for e in gpt if e["batch"] == "config3")}
    for algo in (I.RING, I.TREE):
        for nc in (1, 16):
            for ch in (64 * I.KIB, I.MIB):
                assert (algo, nc, ch) in lab


def test_every_sample_kept_all_its_records():
    for e in ENTRIES:
        assert e["rec_count"] == e["msgs_delivered"] and "records_sha256" in e
        assert e["violations"] == 0


def test_congestion_controlled_samples_run_whole_iterations():
    """A config-3 experiment under DCQCN and one under DCTCP (the generators'
    settings) are stored through their whole iterations, data-parallel
    all-reduces included, and differ from the same experiments without
    congestion control where those are stored."""
    cc = [e for e in ENTRIES if e["batch"] in ("config3-dcqcn", "config3-dctcp")]
    assert {e["batch"] for e in cc} == {"config3-dcqcn", "config3-dctcp"}
    plain = {e["index"]: e for e in ENTRIES if e["batch"] == "config3"}
    for e in cc:
        assert e["limit"] is None and e["status"] == 0, (e["batch"], e["index"])
        assert e["net_allreduce_started"] == e["net_allreduce_members"] > 0
        assert e["net_allreduce_ended"] == e["net_allreduce_members"]
        if e["index"] in plain:
            assert e["digest"] != plain[e["index"]]["digest"] or \
                e["pkt_hops"] != plain[e["index"]]["pkt_hops"]
