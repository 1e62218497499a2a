"""dllm_step_noalloc: the step for callers that cannot allocate device memory.

Such callers (an engine whose pool already owns all of HBM, a plain C host
with no allocator, a loop where an allocation may not synchronise the
device) call dllm_step_noalloc, which uses a buffer built into the library
instead of a caller workspace.  This test calls it through the C ABI twice
in a row -- the second call on a larger shape, so that the buffer's reuse
across shapes is exercised -- and checks both results against dllm_step with
a caller workspace and against the CPU oracle, within the tolerances of the
other step tests.  It lives in a file of its own that pytest collects last,
and it passes both alone in a fresh process and after the rest of the
suite.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import CONF_TOL, compare_step, device_logits, device_state, enforce_margins, oracle_step

pytestmark = pytest.mark.gpu


def _outputs(torch, device, B, L):
    return {
        "done": torch.empty(B, dtype=torch.uint8, device=device),
        "accept_len": torch.empty(B, dtype=torch.int32, device=device),
        "n_new": torch.empty(B, dtype=torch.int32, device=device),
        "feats": torch.empty((B, 6), dtype=torch.float32, device=device),
        "conf": torch.empty((B, L), dtype=torch.float32, device=device),
        "lse": torch.empty((B, L), dtype=torch.float32, device=device),
        "tok": torch.empty((B, L), dtype=torch.int32, device=device),
    }


def _args(dllm, cfg, logits, ids, thr, cs, out, ws=None):
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    return dllm.StepArgs(B=cfg.B, L=cfg.L, V=cfg.V, mask_id=cfg.mask_id, ldv=logits.shape[1], logits=p(logits),
                         input_ids=p(ids), thr=p(thr), conf_state=p(cs), done=p(out["done"]),
                         accept_len=p(out["accept_len"]), n_new=p(out["n_new"]), feats=p(out["feats"]),
                         conf_out=p(out["conf"]), lse_out=p(out["lse"]), tok_out=p(out["tok"]),
                         workspace=p(ws), workspace_bytes=0 if ws is None else ws.numel())


def _host(out, ids, cs):
    h = {k: v.cpu().numpy() for k, v in out.items()}
    h["input_ids"] = ids.cpu().numpy()
    h["conf_state"] = cs.cpu().numpy()
    return h


def _same(a, b, masked):
    for k in ("done", "accept_len", "n_new", "input_ids"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(a["tok"][masked], b["tok"][masked])
    np.testing.assert_allclose(a["conf"][masked], b["conf"][masked], rtol=0, atol=CONF_TOL)
    np.testing.assert_allclose(a["lse"][masked], b["lse"][masked], rtol=0,
                               atol=CONF_TOL * max(1.0, float(np.abs(b["lse"][masked]).max())))
    np.testing.assert_allclose(a["conf_state"], b["conf_state"], rtol=0, atol=CONF_TOL, equal_nan=True)
    np.testing.assert_allclose(a["feats"], b["feats"], rtol=0, atol=CONF_TOL, equal_nan=True)


# two calls in a row: the second has more rows and chunks per row (a larger
# counter region to clear, a data region placed elsewhere in the buffer)
CALLS = [
    synth.StepConfig("noalloc_a", 24, 32, 40001, 12.0, "fraction", synth.THRESHOLD_SET, ldv=40016),
    synth.StepConfig("noalloc_b", 40, 64, 70000, 12.0, "fraction", synth.THRESHOLD_SET),
]


def test_noalloc_matches_step_and_oracle_twice(dllm):
    import torch
    device = torch.device("cuda", 0)
    lib = dllm.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    nc = lambda c: -(-c.V // 8192)
    assert CALLS[1].B * CALLS[1].L * nc(CALLS[1]) > CALLS[0].B * CALLS[0].L * nc(CALLS[0])
    for call, (cfg, seed) in enumerate(zip(CALLS, (31, 32))):
        inp = synth.make_step_state(cfg, seed)
        enforce_margins(inp)
        ref = oracle_step(inp)
        logits = device_logits(inp, device)

        ids, thr, cs = device_state(inp, device)
        out = _outputs(torch, device, cfg.B, cfg.L)
        ws = torch.zeros(lib.dllm_step_workspace_size(cfg.B, cfg.L, cfg.V), dtype=torch.uint8, device=device)
        rc = lib.dllm_step(ctypes.byref(_args(dllm, cfg, logits, ids, thr, cs, out, ws)), stream)
        assert rc == 0
        want = _host(out, ids, cs)

        ids2, thr2, cs2 = device_state(inp, device)
        out2 = _outputs(torch, device, cfg.B, cfg.L)
        rc = lib.dllm_step_noalloc(ctypes.byref(_args(dllm, cfg, logits, ids2, thr2, cs2, out2)), stream)
        assert rc == 0, f"call {call}: {lib.dllm_strerror(rc).decode()}"
        got = _host(out2, ids2, cs2)
        assert dllm.get_device_error(device) == 0
        _same(got, want, inp.masked)
        compare_step(ref, got, list(range(cfg.B)), cfg.L, got["input_ids"], got["conf_state"])


def test_noalloc_rejects_shapes_beyond_its_buffer(dllm):
    lib = dllm.load()
    cap = lib.dllm_step_noalloc_capacity()
    assert cap == 16 << 20
    # 4096 x 64 positions over a 1M vocabulary needs far more than 16 MiB
    a = dllm.StepArgs(B=4096, L=64, V=1 << 20, mask_id=0, ldv=1 << 20, logits=0x10000, input_ids=0x20000,
                      thr=0x30000, conf_state=0x40000, done=0x50000, accept_len=0x60000, n_new=0x70000)
    assert lib.dllm_step_workspace_size(4096, 64, 1 << 20) > cap
    assert lib.dllm_step_noalloc(ctypes.byref(a), None) == -7


def test_noalloc_rejected_calls_then_a_good_one(dllm):
    """Calls that fail dllm_step's own checks (alignment, stride, a missing
    pointer) return that check's code -- the library runs every check before
    it clears the buffer -- and the next valid call still matches the
    oracle."""
    import torch
    device = torch.device("cuda", 0)
    lib = dllm.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    cfg = CALLS[0]
    inp = synth.make_step_state(cfg, 33)
    enforce_margins(inp)
    ref = oracle_step(inp)
    logits = device_logits(inp, device)
    ids, thr, cs = device_state(inp, device)
    out = _outputs(torch, device, cfg.B, cfg.L)
    good = _args(dllm, cfg, logits, ids, thr, cs, out)
    # misaligned logits, a row stride that is not a multiple of 8, a missing
    # output pointer: each rejected with its code before anything is queued
    for field, value, code in (("logits", logits.data_ptr() + 2, -2), ("ldv", cfg.row_stride + 1, -2),
                               ("n_new", None, -1)):
        bad = dllm.StepArgs.from_buffer_copy(good)
        setattr(bad, field, value)
        assert lib.dllm_step_noalloc(ctypes.byref(bad), stream) == code, field
    assert lib.dllm_step_noalloc(ctypes.byref(good), stream) == 0
    got = _host(out, ids, cs)
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, got["input_ids"], got["conf_state"])
