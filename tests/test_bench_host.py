"""bench.py's host-side arithmetic on CPU: the algorithmic bytes of a step,
the launches of one pipeline step, the traffic read from the committed
capture record only while the kernel source matches, and the clock
summary."""
import types

import pytest


def test_algorithmic_bytes_dream():
    import bench
    import synth
    cfg = synth.STEP_CONFIGS["dream"]
    # masked rows x V x 2 + per-position state (ids and conf_state, read and
    # written) + per-request thr, done, accept_len, n_new, six features
    assert bench.algorithmic_bytes(cfg, 1851) == 1851 * 151936 * 2 + 128 * 32 * 16 + 128 * (4 + 1 + 4 + 4 + 24)
    assert bench.algorithmic_bytes(cfg, 1851) == 562537344


@pytest.mark.parametrize("B,L,shards,expected", [(128, 32, None, 3), (512, 64, None, 5), (128, 32, 4, 3),
                                                 (3000, 8, None, 5)])
def test_launches_per_step(B, L, shards, expected):
    import bench
    pipe = types.SimpleNamespace(B=B, shards=list(range(shards)) if shards else None,
                                 rb_arr=[L * 4, L * 4, 4, 4, 4, 4, 4])
    # pack + the step (all vocabulary shards in one launch) + commit/compaction
    # (one launch while the rows fit the fused kernel's staging, else three)
    assert bench.Pipeline.launches_per_step(pipe) == expected
    # with the commit inside the step's launch: pack + one launch
    pipe.fused = True
    assert bench.Pipeline.launches_per_step(pipe) == 2


def test_traffic_only_for_the_profiled_source(tmp_path):
    import json

    import bench
    sha = bench.step_source_sha()
    rec = tmp_path / "rec.json"
    rec.write_text(json.dumps({"source_sha256": sha, "dram_bytes_per_launch": 573530624}))
    assert bench.load_traffic(sha, path=str(rec)) == 573530624.0
    # a capture of another kernel source is not reported
    assert bench.load_traffic("0" * 16, path=str(rec)) is None
    # no record, or a malformed one: no traffic
    assert bench.load_traffic(sha, path=str(tmp_path / "missing.json")) is None
    bad = tmp_path / "bad.json"
    bad.write_text("not json")
    assert bench.load_traffic(sha, path=str(bad)) is None


def test_committed_traffic_record_is_well_formed():
    import json

    import bench
    with open(bench.TRAFFIC_JSON, encoding="utf-8") as f:
        rec = json.load(f)
    assert len(rec["source_sha256"]) == 16 and "--clock-control none" in rec["command"]
    # DRAM traffic can't be below the bytes the launch must move
    assert rec["dram_bytes_per_launch"] >= bench.algorithmic_bytes(__import__("synth").STEP_CONFIGS["dream"], 1851)


def test_clock_summary():
    import bench
    lines = ["1965, 2070, 1012.3, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "2070, 2070, 980.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "2070, 2070, 990.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "garbage line", "[N/A], 2070, 1, 0, Not Active, Not Active, Not Active, Not Active"]
    out = bench.ClockSampler.summarize(lines)
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.ClockSampler.summarize([]) is None


def test_commit_bytes_bound():
    import bench
    pipe = types.SimpleNamespace(B=128, L=32, rb_arr=[32 * 4, 32 * 4, 4, 4, 4, 4, 4])
    # block tokens 4L, b / K / rid read 12, b and evict written 5, maps 8,
    # each compacted row (276 bytes) read and written
    assert bench.Pipeline.commit_bytes_bound(pipe) == 128 * (4 * 32 + 12 + 5 + 8 + 2 * 276)


def test_roofline_kernel_label():
    import bench
    assert bench.roofline_kernel_label(False, True, False) == "step_kernel with the fused commit (dllm_step_commit)"
    assert bench.roofline_kernel_label(False, True, True) == ("step_kernel with the fused commit "
                                                              "(dllm_step_commit, fixed-steps quota)")
    assert bench.roofline_kernel_label(False, False, True) == "step_kernel (dllm_step_quota)"
    assert bench.roofline_kernel_label(True, True, False) == ("step_kernel over 4 vocabulary shards with the fused "
                                                              "commit (dllm_step_vocab_shards_commit)")
    assert bench.roofline_kernel_label(True, False, False) == "step_kernel over 4 vocabulary shards (dllm_step_vocab_shards)"
