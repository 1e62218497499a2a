"""Oracle of the mixed-state serving loop: admit, pack, step, advance, evict.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows BlockServe Algorithm 1 (section II-C) with the FDFO execution mode of
the FDFO page (sections "FDFO 的核心思想" and "工程设计一"): one iteration is
one denoise step; a request whose current block is done commits the block
(Algorithm 1: update its outputs, b_i <- b_i + 1) and is removed once
b_i >= K_i; the freed budget is refilled by the next admission.  In sync mode
(``_run_sync`` on the FDFO page) nothing advances until every active block is
done.  CheckEOS never fires: synthetic tokens carry no end-of-sequence.

Readings (listed in the design notes): admitted requests are appended after
the survivors in admission order; a request that finishes a block but not its
last one stays in place with a fresh all-mask block; the logits of position
``pos`` of request ``rid``'s block ``b`` at its ``s``-th denoise step of that
block are a pure function of (rid, b, s, pos), supplied by the caller.
"""
from __future__ import annotations

import numpy as np

from . import admit, box_width, compact, cost, pack, step, transfer_quota


def advance(adv, rid, b, K, ids, cs, gen, mask_id):
    """BlockServe Algorithm 1, lines "update r_i's outputs with Y[i] and set
    b_i <- b_i + 1" and "remove any request with b_i >= K_i": for every row
    whose block is committed this iteration, append the block to the
    request's output, move to the next block and flag the row for eviction
    once all K_i blocks are done; a continuing row starts its new block fully
    masked (BlockServe section II-E).  Arrays are updated in place (numpy);
    ``gen[r]`` is a list of committed tokens.  Returns the eviction flags."""
    evict = np.zeros(len(adv), dtype=bool)
    for i in range(len(adv)):
        if not adv[i]:
            continue
        r = int(rid[i])
        gen[r] = np.concatenate([gen[r], ids[i]])
        b[i] += 1
        if b[i] >= K[i]:
            evict[i] = True
        else:
            ids[i] = mask_id
            cs[i] = np.nan
    return evict


class OracleLoop:
    """``S``: None for the threshold rule, else the fixed-steps rule with S
    steps per block (``transfer_quota`` of each row's steps in its block)."""

    def __init__(self, p, K, prompts, thr, L, V, mask_id, pad_id, budget, mode="fdfo", S=None):
        assert mode in ("fdfo", "sync")
        self.S = S
        self.L, self.V, self.mask_id, self.pad_id = L, V, mask_id, pad_id
        self.budget = budget
        self.mode = mode
        self.p_all = np.asarray(p, dtype=np.int64)
        self.K_all = np.asarray(K, dtype=np.int64)
        self.thr_all = np.asarray(thr, dtype=np.float32)
        self.prompts = prompts
        R = len(self.p_all)
        # Pending queue sorted by prompt length, ties by request id.
        self.pending = sorted(range(R), key=lambda r: (int(self.p_all[r]), r))
        self.gen = [np.zeros(0, dtype=np.int64) for _ in range(R)]
        self.finish_iter = np.full(R, -1, dtype=np.int64)
        self.admit_iter = np.full(R, -1, dtype=np.int64)
        # Active set, one entry per row (SoA).
        self.rid = []
        self.b = []
        self.s = []
        self.ids = np.zeros((0, L), dtype=np.int64)
        self.cs = np.zeros((0, L))
        self.iteration = 0
        self.trace = []

    # -- Algorithm 1, line "admit" ------------------------------------------
    def admit_phase(self):
        pend_p = [int(self.p_all[r]) for r in self.pending]
        act_p = [int(self.p_all[r]) for r in self.rid]
        picked = admit(pend_p, act_p, self.b, self.L, self.budget)
        new = [self.pending[k] for k in picked]
        for k in sorted(picked, reverse=True):
            del self.pending[k]
        for r in new:
            self.admit_iter[r] = self.iteration
            self.rid.append(r)
            self.b.append(0)
            self.s.append(0)
        if new:
            self.ids = np.vstack([self.ids, np.full((len(new), self.L), self.mask_id, dtype=np.int64)])
            self.cs = np.vstack([self.cs, np.full((len(new), self.L), np.nan)])
        return new

    def box(self):
        p = [int(self.p_all[r]) for r in self.rid]
        prompts = [self.prompts[r] for r in self.rid]
        gens = [self.gen[r] for r in self.rid]
        return pack(p, self.b, self.L, prompts, gens, list(self.ids), self.pad_id)

    def cost(self):
        return cost([int(self.p_all[r]) for r in self.rid], self.b, self.L)

    def width(self):
        return box_width([int(self.p_all[r]) for r in self.rid], self.b, self.L)

    # -- rows whose logits the step reads -------------------------------------
    def masked_rows(self):
        """(row*L + j, rid, b, s, j) for every masked position of the batch."""
        out = []
        for i in range(len(self.rid)):
            for j in range(self.L):
                if self.ids[i, j] == self.mask_id:
                    out.append((i * self.L + j, self.rid[i], self.b[i], self.s[i], j))
        return out

    def quota(self):
        """Per-row counts of the fixed-steps rule this step (None under the
        threshold rule)."""
        if self.S is None:
            return None
        return np.array([transfer_quota(self.L, self.S, s) for s in self.s], dtype=np.int64)

    # -- one denoise step (FDFO page, "工程设计一") -----------------------------
    def step_phase(self, logits_bits, thr=None):
        """``thr``: float32 thresholds of the active rows for this step (else
        each request's own)."""
        if thr is None:
            thr = np.array([self.thr_all[r] for r in self.rid], dtype=np.float32)
        res = step(logits_bits, self.V, self.ids, thr, self.cs, self.mask_id, quota=self.quota())
        had_masked = res["masked"].any(axis=1)
        self.ids = res["input_ids"]
        self.cs = res["conf_state"]
        for i in range(len(self.rid)):
            if had_masked[i]:
                self.s[i] += 1
        return res

    # -- Algorithm 1: update outputs, b_i += 1, evict b_i >= K_i ---------------
    def finish_phase(self, done):
        done = np.asarray(done, dtype=bool)
        adv = done if self.mode == "fdfo" else (np.full(done.shape, done.all()) if done.size else done)
        b = np.array(self.b, dtype=np.int64)
        K = np.array([self.K_all[r] for r in self.rid], dtype=np.int64)
        evict = advance(adv, self.rid, b, K, self.ids, self.cs, self.gen, self.mask_id)
        self.b = b.tolist()
        for i in range(len(self.rid)):
            if adv[i]:
                self.s[i] = 0
                if evict[i]:
                    self.finish_iter[self.rid[i]] = self.iteration
        new_index, src_row, A2 = compact(evict)
        self.rid = [self.rid[i] for i in src_row]
        self.b = [self.b[i] for i in src_row]
        self.s = [self.s[i] for i in src_row]
        self.ids = self.ids[src_row]
        self.cs = self.cs[src_row]
        self.iteration += 1
        return evict, new_index, src_row, A2

    def finished(self):
        return not self.pending and not self.rid

    def run(self, logits_fn, max_iters=100000):
        """Drive the loop to completion; ``logits_fn(rows)`` returns uint16
        [len(rid) * L, ldv] logits for ``masked_rows()`` tuples."""
        while not self.finished() and self.iteration < max_iters:
            new = self.admit_phase()
            rows = self.masked_rows()
            logits = logits_fn(self, rows)
            res = self.step_phase(logits)
            waiting = int(((~res["masked"].any(axis=1)) & (res["done"] == 1)).sum())
            self.trace.append(dict(A=len(self.rid), W=self.width(), M=len(rows), waiting=waiting,
                                   admitted=len(new), cost=self.cost()))
            self.finish_phase(res["done"])
        return self
