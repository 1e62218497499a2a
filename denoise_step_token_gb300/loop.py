"""Mixed-state serving loop on the GPU: BlockServe Algorithm 1 with the FDFO
execution mode.

BlockServe page, section II-C (Algorithm 1): admit from the pending queue
under the token budget of eq. (1), run the active set one step, commit
finished blocks (b_i <- b_i + 1) and evict requests with b_i >= K_i.
FDFO page, sections "FDFO 的核心思想" and "工程设计一": in FDFO mode a
request whose block is done commits and leaves (or starts its next block)
at once; in sync mode (``_run_sync``) nothing commits until every active
block is done.

The host keeps only what admission needs (prompt lengths and block indices
of the active rows) and reads back one byte per row per step, the done
flags -- the pages' ``accept_length_per_req_cpu``.  Refill, packing, the
step, block commit and compaction run in libdllm's kernels.  The model
forward is outside this loop: the caller supplies each step's logits.
"""
from __future__ import annotations

import numpy as np

from . import admit, advance_compact, pack, pack_block, pack_plan, refill, step, transfer_quota


class DeviceLoop:
    """One pending queue served to completion on one device.  ``S``: None
    for the threshold rule, else the fixed-steps rule with S steps per block
    (BlockServe page, section II-E).

    ``reloop``: the in-place re-loop of the FDFO page, section "工程设计四"
    (#27877): after a step in which no row advanced, the next step runs on
    the same batch.  Nothing was committed or evicted, so admission would
    admit nothing (it stopped at the first candidate the budget rejects and
    neither the active set nor its widths changed), advance and compaction
    are no-ops, and the box differs only in its active-block columns: those
    phases are skipped and ``dllm_pack_block`` refreshes the block columns.
    The trace is identical to the loop without re-loop.

    ``controller``: a ``control.ThresholdController`` (DiLaServe review,
    section 3.2).  Before every step it picks each active request's
    threshold from the block features of the request's last step (NaN for a
    fresh block), the positions still masked, the blocks left, the request's
    total tokens and its time since admission on a modelled clock that
    advances by the controller's step latency at the current batch size."""

    def __init__(self, p, K, prompt_off, prompt_tokens, thr, *, L, V, mask_id, pad_id, budget, device,
                 mode="fdfo", capacity=None, features=True, S=None, reloop=False, controller=None):
        import torch
        assert mode in ("fdfo", "sync")
        self.S = None if S is None else int(S)
        self.reloop = bool(reloop)
        self.controller = controller
        self.now = 0.0                                  # modelled clock (controller)
        self.admit_s = np.zeros(0)                      # admission time per active row
        self.feat_h = np.zeros((0, 6), dtype=np.float32)   # last block features per active row
        self.thr_log = []                               # thresholds the controller chose, per step
        self.in_place = False        # the last step advanced no row: re-loop on the same batch
        self.reloops = 0             # iterations that ran in place
        self.torch = torch
        self.L, self.V, self.mask_id, self.pad_id = int(L), int(V), int(mask_id), int(pad_id)
        self.budget, self.mode, self.device, self.features = int(budget), mode, device, features
        self.p_all = np.asarray(p, dtype=np.int32)
        self.K_all = np.asarray(K, dtype=np.int32)
        self.thr_all = np.asarray(thr, dtype=np.float32)
        R = len(self.p_all)
        self.R = R
        # pending queue: sorted by prompt length, ties by request id
        self.pending = sorted(range(R), key=lambda r: (int(self.p_all[r]), r))
        cap = R if capacity is None else int(capacity)
        self.cap = cap
        i32, f32 = torch.int32, torch.float32
        z = lambda *shape, dtype=i32: torch.zeros(shape, dtype=dtype, device=device)
        self.rid, self.p, self.b, self.K = z(cap), z(cap), z(cap), z(cap)
        self.thr = z(cap, dtype=f32)
        self.ids = torch.full((cap, L), self.mask_id, dtype=i32, device=device)
        self.cs = torch.full((cap, L), float("nan"), dtype=f32, device=device)
        self.gen = z(R, int(self.K_all.max()) * L if R else L)
        self.prompt_off = torch.as_tensor(np.asarray(prompt_off, dtype=np.int64)).to(device)
        self.prompt_tokens = torch.as_tensor(np.asarray(prompt_tokens, dtype=np.int32)).to(device)
        # host mirrors of the active rows
        self.A = 0
        self.rid_h = np.zeros(0, dtype=np.int32)
        self.b_h = np.zeros(0, dtype=np.int32)
        self.s_h = np.zeros(0, dtype=np.int32)      # steps taken in the current block
        self.wait_h = np.zeros(0, dtype=bool)       # block done, waiting (sync mode)
        self.iteration = 0
        self.box = None
        self.W = 0
        self.cost = 0
        self.last = None

    # -- admission and refill (Algorithm 1, "admit") -------------------------
    def admit_phase(self):
        torch = self.torch
        if not self.pending or self.in_place:
            return []
        pend_p = self.p_all[self.pending]
        picked = admit(pend_p, self.p_all[self.rid_h], self.b_h, self.L, self.budget)
        if not picked:
            return []
        new = [self.pending[k] for k in picked]
        for k in sorted(picked, reverse=True):
            del self.pending[k]
        n = len(new)
        if self.A + n > self.cap:
            raise RuntimeError("active set exceeds the loop's row capacity")
        d = lambda x, dt: torch.as_tensor(np.asarray(x, dtype=dt)).to(self.device)
        refill(self.A, d(new, np.int32), d(self.p_all[new], np.int32), d(self.K_all[new], np.int32),
               d(self.thr_all[new], np.float32), self.rid, self.p, self.b, self.K, self.thr, self.ids, self.cs,
               mask_id=self.mask_id)
        self.A += n
        self.rid_h = np.concatenate([self.rid_h, np.asarray(new, dtype=np.int32)])
        self.b_h = np.concatenate([self.b_h, np.zeros(n, dtype=np.int32)])
        self.s_h = np.concatenate([self.s_h, np.zeros(n, dtype=np.int32)])
        self.wait_h = np.concatenate([self.wait_h, np.zeros(n, dtype=bool)])
        self.admit_s = np.concatenate([self.admit_s, np.full(n, self.now)])
        self.feat_h = np.concatenate([self.feat_h, np.full((n, 6), np.nan, dtype=np.float32)])
        return new

    # -- the box of eq. (1) (BlockServe section II-E) -------------------------
    def pack_phase(self):
        A = self.A
        if self.in_place and self.box is not None:
            self.reloops += 1
            pack_block(self.ids[:A], self.box["ids"], L=self.L, W=self.W)
            return self.box
        self.W, self.cost = pack_plan(self.p_all[self.rid_h], self.b_h, self.L)
        if A == 0:
            self.box = None
            return None
        self.box = pack(self.p[:A], self.b[:A], self.rid[:A], self.prompt_off, self.prompt_tokens, self.gen,
                        self.ids[:A], L=self.L, W=self.W, pad_id=self.pad_id)
        return self.box

    # -- one denoise step -------------------------------------------------------
    def control_inputs(self):
        """The controller's inputs for the active rows: features, masked
        positions, blocks left, total tokens, time since admission."""
        L = self.L
        f = self.feat_h
        frac = np.where(np.isnan(f[:, 0]), 0.0, f[:, 5])
        masked = (L - np.rint(frac * L)).astype(np.int32)
        K = self.K_all[self.rid_h]
        left = (K - self.b_h - 1).astype(np.int32)
        total = (self.p_all[self.rid_h] + K * L).astype(np.float64)
        return f, masked, left, total, self.now - self.admit_s

    def step_phase(self, logits, thr=None):
        """One step on the active rows.  ``thr``: float32 [A] thresholds for
        this step (else the controller's, else the requests' own)."""
        A = self.A
        if thr is None and self.controller is not None and A:
            thr, _, _ = self.controller.choose(*self.control_inputs())
            self.thr_log.append(thr.copy())
        if thr is not None and A:
            self.thr[:A].copy_(self.torch.from_numpy(np.ascontiguousarray(thr, dtype=np.float32)))
        quota = None
        if self.S is not None:
            q = np.array([transfer_quota(self.L, self.S, int(s)) for s in self.s_h], dtype=np.int32)
            quota = self.torch.from_numpy(q).to(self.device)
        out = step(logits, self.ids[:A], self.thr[:A], self.cs[:A], V=self.V, mask_id=self.mask_id,
                   feats=self.features, quota=quota)
        done = out["done"].cpu().numpy().astype(bool)     # the per-step readback
        self.last = out
        if self.controller is not None:
            self.feat_h = out["feats"].cpu().numpy().copy()
            self.now += float(self.controller.step_latency_s(A))
        return done, out

    # -- commit finished blocks, evict, compact ----------------------------------
    def finish_phase(self, done):
        torch = self.torch
        A = self.A
        if self.mode == "fdfo":
            adv = done
        else:
            adv = done if done.all() else np.zeros_like(done)
        # a row stepped unless its block was already done and waiting
        stepped = ~self.wait_h
        if self.reloop and not adv.any():
            # nothing commits: no advance, no compaction, same batch next step
            self.s_h = self.s_h + stepped.astype(np.int32)
            self.wait_h = done & ~adv
            self.in_place = True
            self.iteration += 1
            return np.zeros(A, dtype=bool), None
        self.in_place = False
        adv_d = torch.as_tensor(adv.astype(np.uint8)).to(self.device)
        _, _, _, A_out = advance_compact(adv_d, self.rid[:A], self.K[:A], self.b[:A], self.ids[:A], self.cs[:A],
                                         self.gen, [self.rid[:A], self.p[:A], self.b[:A], self.K[:A], self.thr[:A],
                                                    self.ids[:A], self.cs[:A]], mask_id=self.mask_id)
        b = self.b_h.copy()
        s = self.s_h + stepped.astype(np.int32)
        b[adv] += 1
        s[adv] = 0
        evict = adv & (b >= self.K_all[self.rid_h])
        keep = ~evict
        wait = done & ~adv
        self.rid_h, self.b_h, self.s_h, self.wait_h = self.rid_h[keep], b[keep], s[keep], wait[keep]
        if self.feat_h.shape[0] == A:
            self.feat_h[adv] = np.nan                     # a fresh block: nothing unmasked yet
            self.feat_h = self.feat_h[keep]
        self.admit_s = self.admit_s[keep]
        self.A = int(keep.sum())
        self.iteration += 1
        return evict, A_out

    def finished(self):
        return not self.pending and self.A == 0

    def masked_rows(self):
        """(row * L + j, rid, b, s, j) of every masked position (reads the
        block tokens back; a driver that generates logits needs this)."""
        A = self.A
        if A == 0:
            return []
        ids = self.ids[:A].cpu().numpy()
        rows, js = np.nonzero(ids == self.mask_id)
        return [(int(i) * self.L + int(j), int(self.rid_h[i]), int(self.b_h[i]), int(self.s_h[i]), int(j))
                for i, j in zip(rows, js)]

    def generated(self):
        return self.gen.cpu().numpy()


class NativeLoop:
    """The same loop driven by libdllm's native loop (dllm_loop_*): two
    calls per iteration, ``begin()`` before the model forward and
    ``end(logits)`` after it; all of the loop's device arrays live in one
    workspace tensor.  ``mode``, ``reloop`` and ``S`` as for DeviceLoop.
    ``controller``: a ``control.ThresholdController`` built with
    ``ThresholdController.affine``; the native loop then picks every step's
    thresholds itself (``dllm_loop_set_control``)."""

    def __init__(self, p, K, prompt_off, prompt_tokens, thr, *, L, V, mask_id, pad_id, budget, device,
                 mode="fdfo", reloop=False, S=None, capacity=None, controller=None):
        import ctypes
        import torch
        from . import LoopConfig, LoopInfo, _check, load
        assert mode in ("fdfo", "sync")
        self.torch, self.ctypes, self.LoopInfo, self._check = torch, ctypes, LoopInfo, _check
        self.lib = load()
        self.device = device
        self.L, self.V = int(L), int(V)
        p = np.ascontiguousarray(p, dtype=np.int32)
        K = np.ascontiguousarray(K, dtype=np.int32)
        thr = np.ascontiguousarray(thr, dtype=np.float32)
        self.R = len(p)
        cap = self.R if capacity is None else int(capacity)
        self.cfg = LoopConfig(R=self.R, L=self.L, V=self.V, mask_id=int(mask_id), pad_id=int(pad_id),
                              mode=0 if mode == "fdfo" else 1, reloop=1 if reloop else 0, S=0 if S is None else int(S),
                              capacity=max(cap, 1), budget=int(budget))
        vp = ctypes.c_void_p
        need = int(self.lib.dllm_loop_workspace_size(ctypes.byref(self.cfg), vp(p.ctypes.data), vp(K.ctypes.data)))
        if need == 0:
            raise ValueError("invalid loop configuration")
        self.ws = torch.empty(need, dtype=torch.uint8, device=device)
        self.prompt_off = torch.as_tensor(np.asarray(prompt_off, dtype=np.int64)).to(device)
        self.prompt_tokens = torch.as_tensor(np.asarray(prompt_tokens, dtype=np.int32)).to(device)
        self.handle = vp()
        self._stream = vp(torch.cuda.current_stream(device).cuda_stream)
        _check("dllm_loop_create", self.lib.dllm_loop_create(
            ctypes.byref(self.cfg), vp(p.ctypes.data), vp(K.ctypes.data), vp(thr.ctypes.data),
            vp(self.prompt_off.data_ptr()), vp(self.prompt_tokens.data_ptr()) if self.prompt_tokens.numel() else None,
            vp(self.ws.data_ptr()), need, self._stream, ctypes.byref(self.handle)))
        if controller is not None:
            if controller.latency_affine is None:
                raise ValueError("the native loop needs an affine step latency (ThresholdController.affine)")
            from . import LoopControl
            self._cand = np.ascontiguousarray(controller.cand, dtype=np.float64)
            a, b = controller.latency_affine
            lc = LoopControl(T=self._cand.size, candidates=vp(self._cand.ctypes.data), slo_s=controller.slo_s,
                             tokens_per_s=controller.tokens_per_s, latency_s=a, latency_per_row_s=b)
            _check("dllm_loop_set_control", self.lib.dllm_loop_set_control(self.handle, ctypes.byref(lc)))

    def __del__(self):
        if getattr(self, "handle", None) and self.handle.value:
            self.lib.dllm_loop_destroy(self.handle)
            self.handle = self.ctypes.c_void_p()

    def info(self):
        inf = self.LoopInfo()
        self._check("dllm_loop_info", self.lib.dllm_loop_info(self.handle, self.ctypes.byref(inf)))
        return inf

    def view(self, ptr, shape, dtype):
        """A tensor view of the workspace at device address ``ptr``."""
        torch = self.torch
        n = int(np.prod(shape))
        size = torch.empty((), dtype=dtype).element_size()
        off = int(ptr) - self.ws.data_ptr()
        return self.ws[off:off + n * size].view(dtype).view(*shape)

    def begin(self):
        self._check("dllm_loop_begin", self.lib.dllm_loop_begin(self.handle, self._stream))
        return self.info()

    def end(self, logits):
        self._check("dllm_loop_end", self.lib.dllm_loop_end(self.handle, self.ctypes.c_void_p(logits.data_ptr()),
                                                            logits.shape[-1], self._stream))
        return self.info()

    def rows(self):
        A = self.info().A
        rid, b, s = (np.zeros(max(A, 1), dtype=np.int32) for _ in range(3))
        vp = self.ctypes.c_void_p
        self._check("dllm_loop_rows", self.lib.dllm_loop_rows(self.handle, vp(rid.ctypes.data), vp(b.ctypes.data),
                                                              vp(s.ctypes.data)))
        return rid[:A], b[:A], s[:A]

    def thresholds(self):
        """The thresholds the last ``end`` gave the rows it stepped (float32,
        in their order at that step)."""
        ctypes = self.ctypes
        out = np.empty(max(self.cfg.capacity, 1), dtype=np.float32)
        n = ctypes.c_int32(0)
        self._check("dllm_loop_thresholds", self.lib.dllm_loop_thresholds(
            self.handle, ctypes.c_void_p(out.ctypes.data), ctypes.byref(n)))
        return out[: n.value].copy()
    def masked_rows(self):
        """(row * L + j, rid, b, s, j) of every masked position."""
        inf = self.info()
        if inf.A == 0:
            return []
        ids = self.view(inf.block_ids, (inf.A, self.L), self.torch.int32).cpu().numpy()
        rid, b, s = self.rows()
        rows, js = np.nonzero(ids == self.cfg.mask_id)
        return [(int(i) * self.L + int(j), int(rid[i]), int(b[i]), int(s[i]), int(j)) for i, j in zip(rows, js)]

    def generated(self):
        inf = self.info()
        return self.view(inf.gen_tokens, (self.R, inf.ld_gen), self.torch.int32).cpu().numpy()

    def finished(self):
        return bool(self.info().finished)
