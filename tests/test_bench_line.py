"""The decode bench's JSON line, assembled on the CPU from a stand-in run result: the keys the
bench contract names, whole-job arithmetic (bytes of all ranks over the slowest rank's time), the
roofline fraction, and the ncu traffic looked up by the attention source's hash (null otherwise)."""
import sys

import pytest

import bench


def _args(monkeypatch, *extra):
    monkeypatch.setattr(sys, "argv", ["bench.py", *extra])
    return bench.parse()


def _run(fused=True, flushed=False):
    return {"attn_bytes": 1_365_910_128, "fused": fused, "grouped": None, "num_seqs": 64, "desc": bench.WORKLOAD,
            "part_tokens": 1024, "n_pairs": 0, "num_blocks": 5235, "l2_flushed": flushed, "host_slot_us": 20.0,
            "launches": 4000, "clocks": {"sm_mhz": 2070.0, "reasons": []}, "copy": None,
            "e2e_step_ms": 0.2, "h2d": 1_999_616, "d2h": 655_360, "launch": "graph",
            "bm": {"free_blocks": 1047, "cow_copies": 0}}


def _line(args, r, world=1, cpu=None):
    return bench.headline_line(args, r, world, cpu, step_ms=0.19, e2e_ms=0.2, attn_ms=0.195, staged_ms=0.23,
                               attn_med=0.194, kv_total=1.36e9 * world, phys_total=1.36e9 * world)


def test_contract_keys_and_arithmetic(monkeypatch):
    args = _args(monkeypatch)
    cpu = {"value": 1.6, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "all"}
    line = _line(args, _run(), cpu=cpu)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks", "e2e",
                "cpu_baseline"):
        assert key in line, key
    assert line["value"] == pytest.approx(1.36e9 / 0.19e-3 / 1e9)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert "workload" in line["config"]
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["achieved"] == pytest.approx(1_365_910_128 / 0.195e-3 / 1e9)
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"])
    assert rf["launch_ms_median"] == 0.194
    assert rf["timed_launches"] == (args.steps + bench.EVENT_EVERY - 1) // bench.EVENT_EVERY
    e2e = line["e2e"]
    assert e2e["value"] == pytest.approx(1.36e9 / 0.2e-3 / 1e9)
    assert e2e["h2d_bytes_per_step"] == 1_999_616 and e2e["d2h_bytes_per_step"] == 655_360
    assert line["cpu_baseline"] is cpu
    assert line["block_manager"]["free_blocks"] == 1047


def test_whole_job_value_over_ranks(monkeypatch):
    args = _args(monkeypatch)
    line = _line(args, _run(), world=4)
    assert line["n_gpus"] == 4
    assert line["value"] == pytest.approx(4 * 1.36e9 / 0.19e-3 / 1e9)
    assert line["tokens_per_s"] == pytest.approx(4 * 64 / 0.19e-3)


def test_traffic_by_source_hash(monkeypatch):
    args = _args(monkeypatch)
    (workload, sha), recorded = next(iter(bench.NCU_TRAFFIC.items()))
    assert workload == "opt13b+append"
    monkeypatch.setattr(bench, "attention_source_sha", lambda: sha)
    assert _line(args, _run())["roofline"]["traffic"] == recorded
    monkeypatch.setattr(bench, "attention_source_sha", lambda: "0" * 64)
    assert _line(args, _run())["roofline"]["traffic"] is None          # the kernel changed since
    monkeypatch.setattr(bench, "attention_source_sha", lambda: sha)
    assert _line(_args(monkeypatch, "--unfused"), _run(fused=False))["roofline"]["traffic"] is None


def test_flushed_step_times_every_launch(monkeypatch):
    args = _args(monkeypatch, "--steps", "40")
    line = _line(args, _run(flushed=True))
    assert line["roofline"]["timed_launches"] == 40
    assert "flushed" in line["config"]["l2"]
