"""bench.py's reference arm (the oracle timed on the host cores) on CPU, on
the tiny workload: the line carries the contract's keys, and its figures
agree with one another (rows per step, the sample's threads, the zero-copy
end-to-end object)."""
import argparse

import pytest


@pytest.mark.parametrize("steps", [2, 7])
def test_reference_arm_line_is_consistent(monkeypatch, steps):
    import bench
    monkeypatch.setattr(bench, "REFERENCE_RUN_S", 2.0)   # a short run
    line = bench.run_reference(argparse.Namespace(workload="tiny", steps=steps, warmup=3), 0, 1)
    assert line["impl"] == "reference" and line["unit"] == bench.UNIT and line["steps"] == steps
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == bench.WORKLOADS["tiny"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and 1 <= cb["cores"]
    # a step holds whole requests: at least one request's masked rows
    assert line["sample_rows_per_step"] >= 1
    # value = rows per step / seconds per step
    per_step_s = line["ms_per_step"] / 1e3
    assert line["value"] == pytest.approx(line["sample_rows_per_step"] / per_step_s, rel=1e-9)
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_sample_wraps_around_the_batch(monkeypatch):
    """With a budget larger than the batch, a step repeats requests: its rows
    exceed one pass over the batch."""
    import bench
    cfg, inp, *_ = bench.make_workload(1000, "tiny")
    one_pass = int(inp.masked.sum())
    monkeypatch.setattr(bench, "REFERENCE_RUN_S", 5.0)
    line = bench.run_reference(argparse.Namespace(workload="tiny", steps=2, warmup=3), 0, 1)
    assert line["sample_rows_per_step"] > one_pass


def test_reference_config_equals_the_gpu_arms(monkeypatch):
    """Both arms describe the workload with the same ``config`` object; the
    GPU arm takes the box from libdllm's host-side dllm_pack_plan, the
    reference arm from the oracle."""
    import bench
    import denoise_step_token_gb300 as dllm
    monkeypatch.setattr(bench, "REFERENCE_RUN_S", 1.0)
    line = bench.run_reference(argparse.Namespace(workload="tiny", steps=2, warmup=3), 0, 1)
    cfg, inp, reqs, b, *_ = bench.make_workload(1000, "tiny")
    W, cost = dllm.pack_plan(reqs.p, b, cfg.L)
    assert line["config"] == bench.workload_config("tiny", cfg, inp, W, cost, False)
