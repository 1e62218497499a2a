"""Failure detection on the GPU, without faulting it.

- A CUDA failure injected on the host (dllm_inject_cuda_error: the call is
  reported failed and not made) reaches the caller as DllmError, launches
  nothing, and the next step is correct.
- A bounded wait that runs out: the workspace's counters are preset so that
  one request's finaliser waits for the result of a row that is never
  finished (its counter can never reach the chunk count).  The wait gives up
  after the build's limit (1 s), the device error word reads
  DLLM_DEVERR_TIMEOUT, the call returns, and after dllm_workspace_init a
  normal step matches the oracle.
- A mistake planted in the oracle loop (a wrong eviction or a wrong refill
  order) is caught by the lockstep checker of the serving loop.
"""
import time

import numpy as np
import pytest

import synth
from helpers import compare_step, device_logits, device_state, enforce_margins, oracle_step

pytestmark = pytest.mark.gpu

CFG = synth.StepConfig("fail", 2, 32, 20000, 12.0, "all", synth.THRESHOLD_SET)


@pytest.fixture(scope="module")
def device(dllm):
    import torch
    return torch.device("cuda", 0)


def _case(seed):
    inp = synth.make_step_state(CFG, seed)
    enforce_margins(inp)
    return inp, oracle_step(inp)


def _run(dllm, device, inp, workspace=None):
    logits = device_logits(inp, device)
    ids, thr, cs = device_state(inp, device)
    out = dllm.step(logits, ids, thr, cs, V=CFG.V, mask_id=CFG.mask_id, debug=True, workspace=workspace)
    return out, ids, cs


def test_injected_cuda_failure_launches_nothing(dllm, device):
    lib = dllm.load()
    inp, ref = _case(1)
    logits = device_logits(inp, device)
    ids, thr, cs = device_state(inp, device)
    assert lib.dllm_inject_cuda_error(2, 1) == 0          # cudaErrorMemoryAllocation, next call
    with pytest.raises(dllm.DllmError, match="cudaErrorMemoryAllocation"):
        dllm.step(logits, ids, thr, cs, V=CFG.V, mask_id=CFG.mask_id)
    assert np.array_equal(ids.cpu().numpy(), inp.input_ids)          # nothing ran
    assert dllm.get_device_error(device) == 0
    out, ids, cs = _run(dllm, device, inp)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare_step(ref, got, list(range(CFG.B)), CFG.L, ids.cpu().numpy(), cs.cpu().numpy())


def test_bounded_wait_times_out_and_the_workspace_recovers(dllm, device):
    import torch
    lib = dllm.load()
    inp, ref = _case(2)
    B, L = CFG.B, CFG.L
    BL = B * L
    ws = torch.zeros(lib.dllm_step_workspace_size(B, L, CFG.V), dtype=torch.uint8, device=device)
    # Workspace layout (the library's, white-box): 64 bytes of control words,
    # then int32 counters: one per row (chunks counted), one per request
    # (rows finished).  Request 0 (32 masked rows) is preset one row short
    # of complete, so its first finished row finalises it; row 1's counter is
    # preset far past the chunk count, so row 1 is never finished and its
    # result word stays zero: the finaliser's poll for it must run out.
    cnt = ws[64:64 + 4 * (BL + B)].view(torch.int32)
    assert int(inp.masked[0].sum()) == L
    cnt[BL + 0] = L - 1
    cnt[1] = 1 << 20
    t = time.perf_counter()
    _run(dllm, device, inp, workspace=ws)
    code = dllm.get_device_error(device)                # synchronises
    elapsed = time.perf_counter() - t
    assert code == 1, code                              # DLLM_DEVERR_TIMEOUT
    assert 0.9 < elapsed < 30.0
    assert dllm.get_device_error(device) == 0           # read and cleared
    assert lib.dllm_workspace_init(ws.data_ptr(), ws.numel(), dllm._stream(device)) == 0
    out, ids, cs = _run(dllm, device, inp, workspace=ws)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(B)), L, ids.cpu().numpy(), cs.cpu().numpy())


@pytest.mark.parametrize("plant", ["eviction", "refill"])
def test_lockstep_checker_catches_a_planted_mistake(dllm, device, monkeypatch, plant):
    """The mistake is planted in the oracle loop, on the CPU: at iteration 3
    it either advances the wrong rows (a flipped done flag) or admits its
    new requests in reverse order; the checker must stop at the divergence."""
    from oracle.loop import OracleLoop
    from test_gpu_loop import _lockstep_native
    if plant == "eviction":
        orig = OracleLoop.finish_phase

        def bad_finish(self, done):
            done = np.array(done, copy=True)
            if self.iteration == 3 and len(done):
                done[0] ^= 1
            return orig(self, done)

        monkeypatch.setattr(OracleLoop, "finish_phase", bad_finish)
    else:
        orig = OracleLoop.admit_phase

        def bad_admit(self):
            n_before = len(self.rid)
            new = orig(self)
            if len(new) > 1 and self.iteration >= 0:
                self.rid[n_before:] = self.rid[n_before:][::-1]
            return new

        monkeypatch.setattr(OracleLoop, "admit_phase", bad_admit)
    cfg = synth.LoopConfig("small_batch", 16, 3, 60, 24, 8, 4099, 220, 0.9, 10.0)
    with pytest.raises(AssertionError):
        _lockstep_native(dllm, device, cfg, "fdfo", seed=12)
