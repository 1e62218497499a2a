"""GPU parity of dllm_step_quota (the fixed-steps rule of the BlockServe
page, section II-E) against the CPU oracle, through the C ABI.

Same bar as the threshold rule: tokens, selections, input_ids, done,
accept_len and n_new bit-exact; confidences, conf_state and features within
1e-5.  Cases carry a 1e-4 margin at every quota boundary (tests/helpers.py).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import compare_step, device_logits, device_logits_compact, device_state, enforce_margins, oracle_step

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.STEP_CONFIGS["tiny"],
    "ragged": synth.StepConfig("ragged", 8, 32, 40001, 12.0, "fraction", synth.THRESHOLD_SET, ldv=40016),
    "l64": synth.StepConfig("l64", 16, 64, 33000, 12.0, "fraction", synth.THRESHOLD_SET),
    "l100": synth.StepConfig("l100", 6, 100, 5000, 10.0, "fraction", synth.THRESHOLD_SET),
    "wide_block": synth.StepConfig("wide_block", 2, 1024, 300, 8.0, "fraction", (0.7,)),
    "all_masked": synth.StepConfig("all_masked", 6, 32, 20000, 12.0, "all", synth.THRESHOLD_SET),
}


@pytest.fixture(scope="module")
def device(dllm):
    import torch
    return torch.device("cuda", 0)


def run_quota(dllm, inp, device, quota, thr=True):
    import torch
    logits = device_logits(inp, device)
    ids, d_thr, cs = device_state(inp, device)
    q = torch.from_numpy(np.asarray(quota, dtype=np.int32)).to(device)
    out = dllm.step(logits, ids, d_thr if thr else None, cs, V=inp.cfg.V, mask_id=inp.cfg.mask_id, debug=True,
                    quota=q)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    return got, ids.cpu().numpy(), cs.cpu().numpy()


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("seed", [0, 1])
def test_quota_parity_small(dllm, device, name, seed):
    cfg = CASES[name]
    inp = synth.make_step_state(cfg, seed)
    rng = np.random.default_rng(100 + seed)
    quota = rng.integers(-1, cfg.L + 2, size=cfg.B)
    quota[0] = 1
    enforce_margins(inp, quota=quota)
    ref = oracle_step(inp, quota=quota)
    got, ids, cs = run_quota(dllm, inp, device, quota, thr=(seed == 0))
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)


@pytest.mark.parametrize("S", [32, 5, 64])
def test_quota_schedule_unmasks_a_block_in_S_steps(dllm, device, S):
    """A fully masked block under dllm_transfer_quota's schedule: step s
    unmasks exactly q(s) positions per request, each step equal to the
    oracle's, and the block is done after S steps."""
    cfg = synth.StepConfig("sched", 5, 32, 3000, 10.0, "all", synth.THRESHOLD_SET)
    inp = synth.make_step_state(cfg, 21)
    for s in range(S):
        q = np.full(cfg.B, dllm.transfer_quota(cfg.L, S, s), dtype=np.int32)
        enforce_margins(inp, quota=q)
        ref = oracle_step(inp, quota=q)
        got, ids, cs = run_quota(dllm, inp, device, q)
        compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)
        expect_new = np.minimum(q, inp.masked.sum(axis=1))
        assert np.array_equal(got["n_new"], expect_new)
        # the next step starts from the oracle's state (equal to the GPU's)
        inp = synth.StepInputs(cfg, inp.seed, ref["input_ids"].astype(np.int32),
                               inp.thr, ref["conf_state"].astype(np.float32), inp.salt)
    assert not (inp.input_ids == cfg.mask_id).any()


def test_quota_full_size(dllm, device):
    """Dream-shaped batch with per-request steps-in-block drawn at random and
    S in {32, 8}: every request against the oracle."""
    cfg = synth.STEP_CONFIGS["dream"]
    inp = synth.make_step_state(cfg, 12)
    rng = np.random.default_rng(4)
    S = rng.choice([32, 8], size=cfg.B)
    s = rng.integers(0, 40, size=cfg.B)
    quota = np.array([oracle.transfer_quota(cfg.L, int(S[b]), int(s[b])) for b in range(cfg.B)], dtype=np.int32)
    sample = list(range(cfg.B))
    enforce_margins(inp, quota=quota)
    ref = oracle_step(inp, quota=quota)
    got, ids, cs = run_quota(dllm, inp, device, quota)
    compare_step(ref, got, sample, cfg.L, ids, cs)
    m_in = inp.masked
    m_out = ids == cfg.mask_id
    assert np.array_equal(got["n_new"], np.minimum(np.maximum(quota, 0), m_in.sum(axis=1)))
    assert not (m_out & ~m_in).any()



def test_quota_with_compact_logits(dllm, device):
    import torch
    cfg = CASES["l64"]
    inp = synth.make_step_state(cfg, 3)
    quota = np.random.default_rng(7).integers(0, cfg.L + 1, size=cfg.B).astype(np.int32)
    enforce_margins(inp, quota=quota)
    ref = oracle_step(inp, quota=quota)
    logits = device_logits_compact(inp, device)
    ids, thr, cs = device_state(inp, device)
    out = dllm.step(logits, ids, None, cs, V=cfg.V, mask_id=cfg.mask_id, debug=True,
                    quota=torch.from_numpy(quota).to(device), compact=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids.cpu().numpy(), cs.cpu().numpy())
