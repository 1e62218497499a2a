"""The mixed-state serving loop on the GPU, in lockstep with the oracle loop.

Every iteration compares admission, the packed box, the masked rows, the
step's outputs, block commits, evictions and the compacted batch; at the
end every request's generated tokens.  Each step's logits are a pure
function of (request, block, step in block, position) and carry the 1e-4
decision margins (redrawn through the oracle when needed).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import MARGIN, per_request_oracle_loop, request_block_logits
from oracle.loop import OracleLoop

pytestmark = pytest.mark.gpu


def _loop_logits(seed, rows, A, L, V, offset, mask_id, thr_of_row, salts, ldv, quota_of_row=None):
    """Logits [A*L, ldv] for the masked rows, with decision margins (at the
    threshold and fallback, or at the quota boundary)."""
    out = np.full((max(A * L, 1), ldv), synth.POISON_BITS, dtype=np.uint16)
    if not rows:
        return out
    flat = np.array([r[0] for r in rows])
    key_of = lambda r: (r[1], r[2], r[3], r[4])
    for _ in range(50):
        keys = synth.logits_row_keys(seed, [r[1] for r in rows], [r[2] for r in rows], [r[3] for r in rows],
                                     [r[4] for r in rows], [salts.get(key_of(r), 0) for r in rows])
        synth.fill_logits_rows(out, V, flat, keys, offset, mask_id)
        conf, _, _ = oracle.rows_stats(out, flat, V)
        bad = set()
        by_row = {}
        for k, r in enumerate(rows):
            t = float(np.float32(thr_of_row[r[0] // L]))
            if quota_of_row is None and abs(conf[k] - t) < MARGIN:
                bad.add(k)
            by_row.setdefault(r[0] // L, []).append(k)
        for i, ks in by_row.items():
            if quota_of_row is not None:
                q = int(quota_of_row[i])
                c = conf[ks]
                if 0 < q < len(ks):
                    order = np.argsort(-c, kind="stable")
                    if c[order[q - 1]] - c[order[q]] < MARGIN:
                        bad.add(ks[order[q]])
                continue
            t = float(np.float32(thr_of_row[i]))
            c = conf[ks]
            if not (c > t).any() and len(ks) > 1:
                order = np.argsort(-c, kind="stable")
                if c[order[0]] - c[order[1]] < MARGIN:
                    bad.add(ks[order[0]])
        if not bad:
            return out
        for k in bad:
            salts[key_of(rows[k])] = salts.get(key_of(rows[k]), 0) + 1
    raise AssertionError("no margin after 50 redraws")


def _lockstep(dllm, device, cfg, mode, seed, max_iters=10000, S=None, reloop=False, thr_fn=None):
    import torch
    from denoise_step_token_gb300.loop import DeviceLoop
    reqs = synth.make_loop_requests(cfg, seed)
    R, L, V = cfg.R, cfg.L, cfg.V
    prompts = [reqs.prompt_tokens[reqs.prompt_off[r]:reqs.prompt_off[r + 1]] for r in range(R)]
    ol = OracleLoop(reqs.p, reqs.K, prompts, reqs.thr, L, V, cfg.mask_id, cfg.pad_id, cfg.budget, mode, S=S)
    gl = DeviceLoop(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, L=L, V=V, mask_id=cfg.mask_id,
                    pad_id=cfg.pad_id, budget=cfg.budget, device=device, mode=mode, S=S, reloop=reloop)
    salts = {}
    trace = []
    while not ol.finished() and ol.iteration < max_iters:
        assert not gl.finished()
        new_o = ol.admit_phase()
        new_g = gl.admit_phase()
        assert new_o == new_g, ol.iteration
        box_o = ol.box()
        box_g = gl.pack_phase()
        assert gl.W == box_o["W"] and gl.cost == ol.cost()
        if new_o:
            # Algorithm 1 admits only while eq. (1) stays within the budget;
            # active rows widen afterwards as their blocks commit
            assert gl.cost <= cfg.budget
        for k in ("ids", "attn", "pos", "pad", "blk_start"):
            np.testing.assert_array_equal(box_g[k].cpu().numpy(), box_o[k], err_msg=k)
        rows_o = ol.masked_rows()
        assert rows_o == gl.masked_rows()
        thr_step = None if thr_fn is None else thr_fn(ol, new_o)
        thr_of_row = (np.array([reqs.thr[r] for r in ol.rid], dtype=np.float32) if thr_step is None
                      else thr_step)
        logits = _loop_logits(seed, rows_o, len(ol.rid), L, V, cfg.offset_max, cfg.mask_id, thr_of_row, salts,
                              cfg.row_stride, ol.quota())
        ref = ol.step_phase(logits[: len(ol.rid) * L], thr=thr_step)
        if thr_fn is not None:
            thr_fn.after_step(ol, ref)
        done_g, out = gl.step_phase(torch.from_numpy(logits[: len(ol.rid) * L].view(np.int16)).to(device),
                                    thr=thr_step)
        np.testing.assert_array_equal(done_g.astype(np.uint8), ref["done"])
        np.testing.assert_array_equal(out["n_new"].cpu().numpy(), ref["n_new"])
        np.testing.assert_array_equal(out["accept_len"].cpu().numpy(), ref["accept_len"])
        np.testing.assert_array_equal(gl.ids[: gl.A].cpu().numpy(), ref["input_ids"])
        np.testing.assert_allclose(out["feats"].cpu().numpy(), ref["feats"], rtol=0, atol=1e-5, equal_nan=True)
        if thr_fn is not None:
            thr_fn.before_finish(ol, ref)
        ev_o, _, _, A_o = ol.finish_phase(ref["done"])
        ev_g, A_out = gl.finish_phase(done_g)
        np.testing.assert_array_equal(ev_g, ev_o)
        if A_out is None:        # re-loop: nothing advanced, nothing ran
            assert reloop and A_o == gl.A and not ev_o.any()
        else:
            assert int(A_out.cpu().numpy()[0]) == A_o == gl.A
        assert list(gl.rid_h) == ol.rid and list(gl.b_h) == ol.b
        np.testing.assert_array_equal(gl.rid[: gl.A].cpu().numpy(), ol.rid)
        np.testing.assert_array_equal(gl.b[: gl.A].cpu().numpy(), ol.b)
        trace.append((len(rows_o), int(ref["done"].sum())))
    assert ol.finished() and gl.finished()
    gen = gl.generated()
    for r in range(R):
        np.testing.assert_array_equal(gen[r][: reqs.K[r] * L], ol.gen[r])
    assert dllm.get_device_error(device) == 0
    if reloop:
        trace.append(("reloops", gl.reloops))
    return ol, trace


@pytest.fixture(scope="module")
def device(dllm):
    import torch
    return torch.device("cuda", 0)


SMALL = synth.LoopConfig("small_loop", 24, 3, 60, 24, 8, 4099, 600, 0.9, 10.0)


@pytest.mark.parametrize("mode", ["fdfo", "sync"])
def test_loop_lockstep_small(dllm, device, mode):
    ol, trace = _lockstep(dllm, device, SMALL, mode, seed=3)
    assert ol.iteration == len(trace) > 0


def test_loop_lockstep_blockserve_shape_reduced_vocab(dllm, device):
    # the BlockServe loop's geometry (256 requests, prompts U[64, 1024], 8
    # blocks of 32, budget 2^20) with a small vocabulary so the oracle keeps up
    cfg = synth.LoopConfig("bs_small_v", 256, 64, 1024, 256, 32, 1031, 1 << 20, 0.9, 8.0)
    ol, trace = _lockstep(dllm, device, cfg, "fdfo", seed=5)
    assert sum(t[0] for t in trace) > 0


def test_fdfo_and_sync_agree_and_fdfo_wastes_nothing(dllm, device):
    f, tf = _lockstep(dllm, device, SMALL, "fdfo", seed=4)
    s, ts = _lockstep(dllm, device, SMALL, "sync", seed=4)
    for r in range(SMALL.R):
        np.testing.assert_array_equal(f.gen[r], s.gen[r])
    assert f.iteration <= s.iteration


@pytest.mark.parametrize("S", [8, 32])
def test_loop_lockstep_fixed_steps(dllm, device, S):
    """The fixed-steps rule (BlockServe page, section II-E) in the serving
    loop: every block takes exactly S steps when L >= S."""
    ol, trace = _lockstep(dllm, device, SMALL, "fdfo", seed=6, S=S)
    assert ol.iteration == len(trace) > 0


@pytest.mark.parametrize("mode", ["fdfo", "sync"])
def test_loop_in_place_reloop_matches_oracle(dllm, device, mode):
    """FDFO page, section "工程设计四" (#27877): after a step in which no
    block completed, the loop steps the same batch again (no admission,
    pack, advance or compaction; the box's block columns refreshed in
    place).  The whole trace -- admissions, boxes, steps, evictions, tokens
    -- still equals the oracle loop's, and some iterations did re-loop."""
    small_batch = synth.LoopConfig("small_batch", 16, 3, 60, 24, 8, 4099, 220, 0.9, 10.0)
    ol, trace = _lockstep(dllm, device, small_batch, mode, seed=9, reloop=True)
    reloops = trace.pop()[1]
    assert ol.iteration == len(trace) > 0
    assert 0 < reloops < ol.iteration


class OracleController:
    """The threshold controller (DiLaServe review, section 3.2) evaluated on
    the oracle loop's own features with the oracle's control functions; its
    thresholds drive both loops, so no oracle input comes from the GPU."""

    def __init__(self, cand, L, slo_s, tokens_per_s, lat_s):
        self.cand, self.L, self.slo, self.cap, self.lat = np.asarray(cand), L, slo_s, tokens_per_s * slo_s, lat_s
        self.now, self.admit, self.feats = 0.0, {}, {}
        self.log = []

    def __call__(self, ol, new):
        from oracle import control as oc
        for r in new:
            self.admit[r] = self.now
            self.feats[r] = np.full(6, np.nan, dtype=np.float32)
        L, A = self.L, len(ol.rid)
        if A == 0:
            return None
        steps = np.zeros((A, len(self.cand)))
        total = np.zeros(A)
        for i, r in enumerate(ol.rid):
            f = self.feats[r]
            m = L if np.isnan(f[0]) else int(L - np.rint(np.float32(f[5]) * L))
            left = int(ol.K_all[r]) - int(ol.b[i]) - 1
            steps[i] = [oc.predict_steps_stub(t, f, m, left, L) for t in self.cand]
            total[i] = float(ol.p_all[r] + ol.K_all[r] * L)
        caps = oc.load_control(steps * total[:, None], self.cap)
        thr = np.array([self.cand[oc.slo_threshold(steps[i], self.lat(A), self.slo - (self.now - self.admit[r]),
                                                     caps[i])] for i, r in enumerate(ol.rid)], dtype=np.float32)
        self.log.append(thr)
        return thr

    def after_step(self, ol, ref):
        for i, r in enumerate(ol.rid):
            self.feats[r] = ref["feats"][i].astype(np.float32)
        self.now += self.lat(len(ol.rid))

    def before_finish(self, ol, ref):
        done = np.asarray(ref["done"], dtype=bool)
        if ol.mode == "fdfo":
            for i, r in enumerate(ol.rid):
                if done[i]:
                    self.feats[r] = np.full(6, np.nan, dtype=np.float32)


def test_loop_lockstep_with_threshold_control(dllm, device):
    """Per-step thresholds from the DiLaServe controller (Algorithms 1 and
    2 over the stub predictor) drive the GPU loop and the oracle loop in
    lockstep; the thresholds change over the run."""
    ctl = OracleController([0.5, 0.6, 0.7, 0.8, 0.9], SMALL.L, slo_s=0.05, tokens_per_s=2.0e5,
                           lat_s=lambda A: 0.0005 + 0.00002 * A)
    ol, trace = _lockstep(dllm, device, SMALL, "fdfo", seed=7, thr_fn=ctl)
    used = np.concatenate(ctl.log)
    assert len(np.unique(used)) > 1


def test_loop_runs_under_the_library_controller(dllm, device):
    """DeviceLoop with control.ThresholdController: the queue completes,
    every threshold is a candidate, and a tight SLO lowers the thresholds."""
    from denoise_step_token_gb300.control import ThresholdController
    from denoise_step_token_gb300.loop import DeviceLoop
    import torch
    cfg = SMALL
    reqs = synth.make_loop_requests(cfg, 11)
    cand = [0.5, 0.6, 0.7, 0.8, 0.9]
    mean_thr = {}
    for slo in (10.0, 0.02):
        ctl = ThresholdController(cand, L=cfg.L, slo_s=slo, tokens_per_s=1e9, step_latency_s=lambda A: 0.001)
        gl = DeviceLoop(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, L=cfg.L, V=cfg.V,
                        mask_id=cfg.mask_id, pad_id=cfg.pad_id, budget=cfg.budget, device=device, controller=ctl)
        it = 0
        while not gl.finished() and it < 5000:
            gl.admit_phase()
            gl.pack_phase()
            rows = gl.masked_rows()
            logits = _loop_logits(11, rows, gl.A, cfg.L, cfg.V, cfg.offset_max, cfg.mask_id,
                                  np.full(max(gl.A, 1), 0.5, np.float32), {}, cfg.row_stride)
            done, _ = gl.step_phase(torch.from_numpy(logits[: gl.A * cfg.L].view(np.int16)).to(device))
            gl.finish_phase(done)
            it += 1
        assert gl.finished()
        gen = gl.generated()
        for r in range(cfg.R):
            assert not (gen[r][: reqs.K[r] * cfg.L] == cfg.mask_id).any()
        used = np.concatenate(gl.thr_log)
        assert set(np.unique(used).tolist()) <= set(np.float32(cand).tolist())
        mean_thr[slo] = float(used.mean())
    assert mean_thr[0.02] < mean_thr[10.0]


def _lockstep_native(dllm, device, cfg, mode, seed, reloop=False, S=None, max_iters=10000, per_request=False):
    """libdllm's native loop (dllm_loop_*) in lockstep with the oracle loop:
    admissions, box, masked rows, step outputs, commits, evictions and the
    final tokens.  ``per_request``: the oracle's step runs request by request
    on the host's cores and the device receives only the masked positions'
    rows (scattered into a poisoned [capacity * L, ldv] buffer), which keeps
    a full-vocabulary run within minutes."""
    import torch
    from denoise_step_token_gb300.loop import NativeLoop
    reqs = synth.make_loop_requests(cfg, seed)
    R, L, V = cfg.R, cfg.L, cfg.V
    prompts = [reqs.prompt_tokens[reqs.prompt_off[r]:reqs.prompt_off[r + 1]] for r in range(R)]
    oargs = (reqs.p, reqs.K, prompts, reqs.thr, L, V, cfg.mask_id, cfg.pad_id, cfg.budget, mode)
    ol = per_request_oracle_loop(*oargs, S=S) if per_request else OracleLoop(*oargs, S=S)
    nl = NativeLoop(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, L=L, V=V, mask_id=cfg.mask_id,
                    pad_id=cfg.pad_id, budget=cfg.budget, device=device, mode=mode, reloop=reloop, S=S)
    poison = int(np.int16(np.uint16(synth.POISON_BITS).view(np.int16)))
    dev_logits = None
    if per_request:
        dev_logits = torch.full((R * L, cfg.row_stride), poison, dtype=torch.int16, device=device)
    salts = {}
    masked_total = 0
    while not ol.finished() and ol.iteration < max_iters:
        assert not nl.finished()
        new_o = ol.admit_phase()
        inf = nl.begin()
        assert inf.admitted_last == len(new_o), ol.iteration
        rid, b, s = nl.rows()
        assert rid.tolist() == ol.rid and b.tolist() == ol.b
        box_o = ol.box()
        if ol.rid:
            assert inf.W == box_o["W"] and inf.cost == ol.cost()
            A, W = inf.A, inf.W
            for k, ptr, dt in (("ids", inf.box_ids, torch.int32), ("attn", inf.box_attn, torch.uint8),
                               ("pos", inf.box_pos, torch.int32)):
                np.testing.assert_array_equal(nl.view(ptr, (A, W), dt).cpu().numpy(), box_o[k], err_msg=k)
            np.testing.assert_array_equal(nl.view(inf.box_pad, (A,), torch.int32).cpu().numpy(), box_o["pad"])
        rows_o = ol.masked_rows()
        assert rows_o == nl.masked_rows()
        masked_total += len(rows_o)
        A = len(ol.rid)
        if per_request:
            q = ol.quota()
            fn = lambda i, rows_i: request_block_logits(seed, rows_i, L, V, cfg.row_stride, cfg.offset_max,
                                                        cfg.mask_id, reqs.thr[ol.rid[i]], salts,
                                                        None if q is None else int(q[i]))
            ref, blocks = ol.step_phase_per_request(fn)
            idx = torch.as_tensor([r[0] for r in rows_o], dtype=torch.int64, device=device)
            if len(rows_o):
                rows_h = np.stack([blocks[r[0] // L][r[4]] for r in rows_o])
                dev_logits.index_copy_(0, idx, torch.from_numpy(rows_h.view(np.int16)).to(device))
            inf = nl.end(dev_logits[: max(A, 1) * L])
            dev_logits.index_fill_(0, idx, poison)
        else:
            thr_of_row = np.array([reqs.thr[r] for r in ol.rid], dtype=np.float32)
            logits = _loop_logits(seed, rows_o, len(ol.rid), L, V, cfg.offset_max, cfg.mask_id, thr_of_row, salts,
                                  cfg.row_stride, ol.quota())
            ref = ol.step_phase(logits[: len(ol.rid) * L])
            inf = nl.end(torch.from_numpy(logits[: max(A, 1) * L].view(np.int16)).to(device))
        if A:
            np.testing.assert_array_equal(nl.view(inf.done, (A,), torch.uint8).cpu().numpy(), ref["done"])
            np.testing.assert_array_equal(nl.view(inf.n_new, (A,), torch.int32).cpu().numpy(), ref["n_new"])
            np.testing.assert_allclose(nl.view(inf.feats, (A, 6), torch.float32).cpu().numpy(), ref["feats"],
                                       rtol=0, atol=1e-5, equal_nan=True)
        ol.finish_phase(ref["done"])
        inf = nl.info()
        assert inf.A == len(ol.rid) and inf.iteration == ol.iteration
        rid, b, s = nl.rows()
        assert rid.tolist() == ol.rid and b.tolist() == ol.b
        if inf.A:
            np.testing.assert_array_equal(nl.view(inf.block_ids, (inf.A, L), torch.int32).cpu().numpy(), ol.ids)
    assert ol.finished() and nl.finished()
    gen = nl.generated()
    for r in range(R):
        np.testing.assert_array_equal(gen[r][: reqs.K[r] * L], ol.gen[r])
    assert dllm.get_device_error(device) == 0
    nl.masked_total = masked_total
    return ol, nl


@pytest.mark.parametrize("mode,reloop,S", [("fdfo", False, None), ("fdfo", True, None), ("sync", True, None),
                                           ("fdfo", True, 8)])
def test_native_loop_lockstep(dllm, device, mode, reloop, S):
    small_batch = synth.LoopConfig("small_batch", 16, 3, 60, 24, 8, 4099, 220, 0.9, 10.0)
    ol, nl = _lockstep_native(dllm, device, small_batch, mode, seed=12, reloop=reloop, S=S)
    if reloop:
        assert nl.info().reloops > 0


def test_native_loop_blockserve_shape_reduced_vocab(dllm, device):
    cfg = synth.LoopConfig("bs_small_v", 256, 64, 1024, 256, 32, 1031, 1 << 20, 0.9, 8.0)
    _lockstep_native(dllm, device, cfg, "fdfo", seed=5, reloop=True)


def test_native_loop_blockserve_full_vocabulary(dllm, device):
    """The BlockServe mixed-state loop at its own size: 256 requests with
    prompts U[64, 1024], 8 blocks of 32, V = 126464 (LLaDA-8B's vocabulary),
    token budget 2^20, FDFO with the in-place re-loop, served to completion
    in lockstep with the oracle loop (every admission, box, masked row, step
    output, commit and eviction; the final tokens)."""
    cfg = synth.LOOP_CONFIGS["blockserve"]
    assert (cfg.R, cfg.L, cfg.V, cfg.budget) == (256, 32, 126464, 1 << 20)
    ol, nl = _lockstep_native(dllm, device, cfg, "fdfo", seed=2000, reloop=True, per_request=True)
    assert ol.iteration > 0 and nl.masked_total >= cfg.R * cfg.gen


@pytest.mark.parametrize("mode,reloop", [("fdfo", False), ("fdfo", True), ("sync", False)])
def test_native_loop_threshold_control_matches_the_python_loop(dllm, device, mode, reloop):
    """The native loop's own threshold control (dllm_loop_set_control) and
    DeviceLoop with the same controller, over the same queue and logits:
    identical thresholds at every step, identical batches and generated
    tokens, and the thresholds change over the run.  (DeviceLoop under the
    controller is pinned to the oracle loop by the lockstep test above;
    both loops call the same dllm_threshold_control, pinned to the oracle's
    control functions on the CPU.)"""
    import torch
    from denoise_step_token_gb300.control import ThresholdController
    from denoise_step_token_gb300.loop import DeviceLoop, NativeLoop
    cfg = SMALL
    seed = 17
    reqs = synth.make_loop_requests(cfg, seed)

    def controller():
        return ThresholdController.affine([0.5, 0.6, 0.7, 0.8, 0.9], L=cfg.L, slo_s=0.05, tokens_per_s=2.0e5,
                                          latency_s=0.0005, latency_per_row_s=0.00002)

    common = dict(L=cfg.L, V=cfg.V, mask_id=cfg.mask_id, pad_id=cfg.pad_id, budget=cfg.budget, device=device,
                  mode=mode, reloop=reloop)
    gl = DeviceLoop(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, controller=controller(), **common)
    nl = NativeLoop(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, controller=controller(), **common)
    salts, used, it = {}, [], 0
    while not gl.finished() and it < 5000:
        assert not nl.finished()
        new = gl.admit_phase()
        inf = nl.begin()
        assert inf.admitted_last == len(new), it
        gl.pack_phase()
        rid, b, _ = nl.rows()
        assert rid.tolist() == gl.rid_h.tolist() and b.tolist() == gl.b_h.tolist(), it
        rows = gl.masked_rows()
        assert rows == nl.masked_rows(), it
        A = gl.A
        # both loops step on the GPU with the same kernel, so no decision margin is needed between them
        thr_rows = np.array([reqs.thr[r] for r in gl.rid_h], dtype=np.float32)
        logits = _loop_logits(seed, rows, A, cfg.L, cfg.V, cfg.offset_max, cfg.mask_id, thr_rows, salts,
                              cfg.row_stride)
        d = torch.from_numpy(logits[: max(A, 1) * cfg.L].view(np.int16)).to(device)
        done, _ = gl.step_phase(d)
        nl.end(d)
        if A:
            t_nat = nl.thresholds()
            t_py = np.asarray(gl.thr_log[-1], dtype=np.float32)
            assert np.array_equal(t_nat.view(np.uint32), t_py.view(np.uint32)), it
            used.append(t_nat)
        gl.finish_phase(done)
        inf = nl.info()
        assert inf.A == gl.A and inf.iteration == gl.iteration, it
        it += 1
    assert gl.finished() and nl.finished()
    g_py, g_nat = gl.generated(), nl.generated()
    for r in range(cfg.R):
        n = reqs.K[r] * cfg.L
        np.testing.assert_array_equal(g_nat[r][:n], g_py[r][:n])
        assert not (g_nat[r][:n] == cfg.mask_id).any()
    assert len(np.unique(np.concatenate(used))) > 1
    assert dllm.get_device_error(device) == 0


def test_native_loop_control_rejects_invalid_settings(dllm, device):
    """dllm_loop_set_control: candidates not strictly ascending, no
    candidates, a non-positive SLO or a negative latency term are rejected;
    NULL turns the control off (the requests' own thresholds again)."""
    import ctypes
    from denoise_step_token_gb300.loop import NativeLoop
    cfg = SMALL
    reqs = synth.make_loop_requests(cfg, 5)
    nl = NativeLoop(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, L=cfg.L, V=cfg.V,
                    mask_id=cfg.mask_id, pad_id=cfg.pad_id, budget=cfg.budget, device=device)
    lib = dllm.load()

    def ctl(cands, slo=1.0, lat=0.001, per_row=0.0):
        arr = (ctypes.c_double * max(len(cands), 1))(*cands)
        keep.append(arr)
        return dllm.LoopControl(T=len(cands), candidates=ctypes.cast(arr, ctypes.c_void_p), slo_s=slo,
                                tokens_per_s=1e5, latency_s=lat, latency_per_row_s=per_row)

    keep = []
    for bad in (ctl([0.5, 0.5]), ctl([0.9, 0.5]), ctl([]), ctl([0.5], slo=0.0), ctl([0.5], lat=-1.0),
                ctl([0.5], per_row=-1.0), ctl([float("nan")])):
        assert lib.dllm_loop_set_control(nl.handle, ctypes.byref(bad)) == -1
    assert lib.dllm_loop_set_control(nl.handle, ctypes.byref(ctl([0.5, 0.9]))) == 0
    assert lib.dllm_loop_set_control(nl.handle, None) == 0
    # off again: a step uses the requests' own thresholds
    nl.begin()
    A = nl.info().A
    rows = nl.masked_rows()
    logits = _loop_logits(5, rows, A, cfg.L, cfg.V, cfg.offset_max, cfg.mask_id,
                          np.full(max(A, 1), 0.9, np.float32), {}, cfg.row_stride)
    import torch
    rid, _, _ = nl.rows()
    nl.end(torch.from_numpy(logits[: max(A, 1) * cfg.L].view(np.int16)).to(device))
    np.testing.assert_array_equal(nl.thresholds(), np.asarray(reqs.thr, np.float32)[rid])
