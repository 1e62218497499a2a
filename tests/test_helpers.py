"""The test helpers' request-by-request oracle paths equal the oracle over
the whole batch (CPU): the per-request step stacked in request order, and
margins enforced request by request."""
import numpy as np
import pytest

import oracle
import synth
from helpers import enforce_margins, oracle_step, sub_batch_logits

CFG = synth.StepConfig("helpers", 13, 16, 700, 8.0, "fraction", synth.THRESHOLD_SET)


@pytest.mark.parametrize("seed", [0, 1])
def test_per_request_oracle_equals_whole_batch(seed):
    inp = synth.make_step_state(CFG, seed)
    reqs = list(range(CFG.B))
    whole = oracle.step(sub_batch_logits(inp, reqs), CFG.V, inp.input_ids, inp.thr, inp.conf_state, CFG.mask_id)
    stacked = oracle_step(inp, reqs)                 # 13 requests: the per-request path
    assert set(whole) == set(stacked)
    for k in whole:
        np.testing.assert_array_equal(stacked[k], whole[k], err_msg=k)


def test_per_request_oracle_with_quota_and_a_subset():
    inp = synth.make_step_state(CFG, 3)
    quota = np.array([(b % 4) for b in range(CFG.B)], dtype=np.int64)
    sub = [12, 0, 5, 7, 3, 9, 1, 11, 2, 4]           # any order, more than the per-request bound
    whole = oracle.step(sub_batch_logits(inp, sub), CFG.V, inp.input_ids[sub], inp.thr[sub], inp.conf_state[sub],
                        CFG.mask_id, quota=quota[sub])
    stacked = oracle_step(inp, sub, quota=quota)
    for k in whole:
        np.testing.assert_array_equal(stacked[k], whole[k], err_msg=k)


def test_margins_hold_after_enforcement():
    inp = synth.make_step_state(CFG, 4)
    enforce_margins(inp)
    ref = oracle_step(inp)
    for b in range(CFG.B):
        m = ref["masked"][b]
        if not m.any():
            continue
        t = float(np.float32(inp.thr[b]))
        c = ref["conf"][b][m]
        assert (np.abs(c - t) >= 1e-4).all()
        if not (c > t).any() and len(c) > 1:
            top = np.sort(c)[::-1]
            assert top[0] - top[1] >= 1e-4


@pytest.mark.parametrize("mode,S", [("fdfo", None), ("sync", None), ("fdfo", 8)])
def test_per_request_oracle_loop_equals_the_oracle_loop(mode, S):
    """The test-side loop that runs the oracle's step request by request
    gives, step by step, the plain oracle loop's results on the same logits
    (the whole batch's blocks stacked), and the same final tokens."""
    from helpers import per_request_oracle_loop, request_block_logits
    from oracle.loop import OracleLoop
    cfg = synth.LoopConfig("pin_loop", 12, 3, 40, 24, 8, 900, 400, 0.9, 8.0)
    reqs = synth.make_loop_requests(cfg, 21)
    prompts = [reqs.prompt_tokens[reqs.prompt_off[r]:reqs.prompt_off[r + 1]] for r in range(cfg.R)]
    args = (reqs.p, reqs.K, prompts, reqs.thr, cfg.L, cfg.V, cfg.mask_id, cfg.pad_id, cfg.budget, mode)
    a = per_request_oracle_loop(*args, S=S)
    b = OracleLoop(*args, S=S)
    salts = {}
    while not a.finished():
        assert a.admit_phase() == b.admit_phase()
        assert a.masked_rows() == b.masked_rows()
        q = a.quota()
        fn = lambda i, rows_i: request_block_logits(21, rows_i, cfg.L, cfg.V, cfg.row_stride, cfg.offset_max,
                                                    cfg.mask_id, reqs.thr[a.rid[i]], salts,
                                                    None if q is None else int(q[i]))
        ra, blocks = a.step_phase_per_request(fn)
        rb = b.step_phase(np.concatenate(blocks, axis=0))
        for k in rb:
            np.testing.assert_array_equal(ra[k], rb[k], err_msg=k)
        ea = a.finish_phase(ra["done"])
        eb = b.finish_phase(rb["done"])
        np.testing.assert_array_equal(ea[0], eb[0])
        assert a.rid == b.rid and a.b == b.b
    assert b.finished()
    for r in range(cfg.R):
        np.testing.assert_array_equal(a.gen[r], b.gen[r])
