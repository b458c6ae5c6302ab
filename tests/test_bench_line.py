"""The decode bench's JSON line, assembled on the CPU from a stand-in run result: the keys the
bench contract names, whole-job arithmetic (bytes of all ranks over the slowest rank's time), the
roofline fraction, the ncu traffic looked up by the attention source's hash (null otherwise), the
sustained segment and the end-to-end decode loop; and the oracle arm, which builds its batch with
the oracle's block manager (identical to the C++ manager's) and never loads libpkv.so."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _args(*extra):
    return bench.parse(list(extra))


def _run(fused=True, flushed=False):
    return {"attn_bytes": 1_365_910_128, "fused": fused, "grouped": None, "num_seqs": 64, "desc": bench.WORKLOAD,
            "part_tokens": 1024, "kernels_per_step": 1, "n_pairs": 0, "num_blocks": 5235, "l2_flushed": flushed,
            "host_slot_us": 20.0, "launches": 20, "clocks": {"sm_mhz": 2070.0, "reasons": [], "samples": 12},
            "clocks_timed_region": {"sm_mhz": 2070.0, "reasons": [], "samples": 1}, "copy": None,
            "timed_launches": 200, "attn_loop": "back to back",
            "sustained": {"steps": 5200, "seconds": 1.01, "ms_per_step": 0.192, "kv_bytes": 5200 * 1.36e9,
                          "device_s": 0.9984, "clocks": {"sm_mhz": 2070.0, "samples": 10}},
            "e2e_loop": {"steps": 20, "seconds": 0.005, "kv_bytes": 20 * 1.37e9, "ms_per_step": 0.25,
                         "host_a1_us_per_step": 30.0, "copies": 0, "h2d_bytes_per_step": 2_000_000,
                         "d2h_bytes_per_step": 655_360, "staged": False},
            "e2e_replay": {"ms_per_step": 0.2, "staged_ms_per_step": 0.23, "h2d_bytes_per_step": 1_999_616,
                           "d2h_bytes_per_step": 655_360, "launch": "graph"},
            "bm": {"free_blocks": 1047, "cow_copies": 0}}


def _red(world=1):
    return {"step_ms": 0.19, "attn_ms": 0.185, "attn_ms_median": 0.2, "e2e_s": 0.005, "e2e_replay_ms": 0.2,
            "e2e_staged_ms": 0.23, "sus_s": 0.9984, "kv_total": 1.36e9 * world, "phys_total": 1.36e9 * world,
            "e2e_kv": 20 * 1.37e9 * world, "sus_kv": 5200 * 1.36e9 * world}


def test_contract_keys_and_arithmetic():
    args = _args("--steps", "20", "--warmup", "5")
    cpu = {"value": 1.6, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "all"}
    line = bench.headline_line(args, _run(), 1, cpu, _red())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks", "e2e",
                "cpu_baseline", "sustained"):
        assert key in line, key
    assert line["value"] == pytest.approx(1.36e9 / 0.19e-3 / 1e9)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert "workload" in line["config"]
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["achieved"] == pytest.approx(1_365_910_128 / 0.185e-3 / 1e9)
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert rf["timed_launches"] >= 200 and rf["launch_ms"] <= line["ms_per_step"]
    assert rf["launch_ms_median_isolated"] == 0.2
    e2e = line["e2e"]
    assert e2e["value"] == pytest.approx(20 * 1.37e9 / 0.005 / 1e9)
    assert e2e["h2d_bytes_per_step"] == 2_000_000 and e2e["d2h_bytes_per_step"] == 655_360
    assert e2e["host_a1_us_per_step"] == 30.0 and "pkv_bm_append_slots" in e2e["launch"]
    assert e2e["graph_replay"]["value"] == pytest.approx(1.36e9 / 0.2e-3 / 1e9)
    sus = line["sustained"]
    assert sus["value"] == pytest.approx(5200 * 1.36e9 / 0.9984 / 1e9)
    assert sus["ms_x_median_sm_mhz"] == pytest.approx(0.192 * 2070.0)
    assert line["clocks"]["samples"] >= 10
    assert line["cpu_baseline"] is cpu
    assert line["block_manager"]["free_blocks"] == 1047


def test_whole_job_value_over_ranks():
    args = _args()
    line = bench.headline_line(args, _run(), 4, None, _red(world=4))
    assert line["n_gpus"] == 4
    assert line["value"] == pytest.approx(4 * 1.36e9 / 0.19e-3 / 1e9)
    assert line["tokens_per_s"] == pytest.approx(4 * 64 / 0.19e-3)
    assert line["e2e"]["value"] == pytest.approx(4 * 20 * 1.37e9 / 0.005 / 1e9)
    assert "replicas" in line["parallelism"]


def test_traffic_by_source_hash(monkeypatch):
    args = _args()
    (workload, sha), recorded = next(iter(bench.NCU_TRAFFIC.items()))
    assert workload == "opt13b+append"
    monkeypatch.setattr(bench, "attention_source_sha", lambda: sha)
    assert bench.headline_line(args, _run(), 1, None, _red())["roofline"]["traffic"] == recorded
    monkeypatch.setattr(bench, "attention_source_sha", lambda: "0" * 64)
    assert bench.headline_line(args, _run(), 1, None, _red())["roofline"]["traffic"] is None   # kernel changed
    monkeypatch.setattr(bench, "attention_source_sha", lambda: sha)
    line = bench.headline_line(_args("--unfused"), _run(fused=False), 1, None, _red())
    assert line["roofline"]["traffic"] is None


def test_flushed_config():
    line = bench.headline_line(_args("--steps", "40"), _run(flushed=True), 1, None, _red())
    assert "flushed" in line["config"]["l2"]


def test_both_arms_print_the_same_config():
    # the oracle arm quotes the workload exactly as the GPU arm does
    args = _args("--steps", "20", "--warmup", "5")
    gpu_cfg = bench.headline_line(args, _run(), 1, None, _red())["config"]
    assert gpu_cfg == bench.config_block(args, bench.WORKLOAD, 64, flushed=False)


@pytest.mark.parametrize("workload", ["opt13b", "tiny", "parallel_sampling_cow", "shared_prefix"])
def test_oracle_manager_builds_the_native_batch(workload):
    # the oracle's legs build their batch with oracle/block_manager.py; it must be the batch the
    # C++ manager builds for the GPU arm: tables, lengths, this step's slots and copies, the copies
    # made while the batch grew, and the managers' summaries
    seed = bench.workload_seed(workload)
    a = bench.build_step_inputs(seed, workload, manager="native")
    b = bench.build_step_inputs(seed, workload, manager="oracle")
    assert np.array_equal(a["w"].block_tables, b["w"].block_tables)
    assert np.array_equal(a["w"].context_lens, b["w"].context_lens)
    assert np.array_equal(a["slots"], b["slots"]) and np.array_equal(a["pairs"], b["pairs"])
    assert np.array_equal(a["setup_pairs"], b["setup_pairs"])
    assert a["bm"] == b["bm"]


def test_reference_arm_stands_alone():
    # the oracle arm on the tiny batch, in a fresh process: it prints the contract line and
    # libpkv.so is never mapped into the process
    code = ("import sys, json; sys.argv = ['bench.py', '--impl', 'reference', '--workload', 'tiny', '--steps', '2', "
            "'--warmup', '1']; import bench; line = bench.run_reference(bench.parse(sys.argv[1:]), 0); "
            "maps = open('/proc/self/maps').read(); print(json.dumps({'line': line, 'pkv': 'libpkv' in maps}))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got["pkv"] is False
    line = got["line"]
    assert line["impl"] == "reference" and line["value"] > 0 and line["same_config"] is True
    assert "whole batch" in line["cpu_baseline"]["sample"] and "oracle's block manager" in line["cpu_baseline"]["sample"]
    assert line["config"] == bench.config_block(bench.parse(["--workload", "tiny"]), line["config"]["workload"], 3,
                                                flushed=True)


def test_step_form_follows_the_batch_sharing():
    # the fused step unless shared blocks make up most of the batch's K/V (L2 then serves the
    # partitions and the separate write launch is faster); --step overrides
    auto = _args()
    opt = bench.build_step_inputs(bench.workload_seed("opt13b"), "opt13b")["w"]
    shared = bench.build_step_inputs(bench.workload_seed("shared_prefix"), "shared_prefix")["w"]
    assert bench.use_fused(auto, opt) and not bench.use_fused(auto, shared)
    assert bench.use_fused(_args("--step", "fused"), shared)
    assert not bench.use_fused(_args("--step", "unfused"), opt) and not bench.use_fused(_args("--unfused"), opt)


def test_reference_sample_fits_the_wall_budget():
    # the oracle arm keeps the whole batch while the run fits its budget, else a share of the
    # batch's K/V in proportion (at least one sequence), so that a run with the default step count
    # still ends within minutes
    w = type("W", (), {"context_lens": np.array([100, 200, 300, 400])})()
    seqs = [0, 1, 2, 3]
    assert bench.fit_reference_sample(w, seqs, step_s=0.5, runs=25, budget_s=150) == seqs
    kept = bench.fit_reference_sample(w, seqs, step_s=0.5, runs=1000, budget_s=150)   # 30 % of the bytes
    assert kept == [0, 1]
    assert sum(w.context_lens[kept]) <= 0.3 * 1000 + 1e-9
    assert bench.fit_reference_sample(w, seqs, step_s=10.0, runs=1000, budget_s=150) == [0]
