"""Shared test helpers: seeded step cases with decision margins, device
upload of generated logits, comparison against the oracle.

Decision margins: wherever float arithmetic decides a discrete outcome (a
confidence against its threshold, the fallback's most confident position,
the last position a fixed-steps quota takes), the GPU computes in float32
and the oracle in float64.  Cases are drawn so that every such decision has
a margin of at least 1e-4: a masked row whose oracle confidence is within
1e-4 of its threshold, a fallback whose top two confidences are within
1e-4, or a quota boundary whose two confidences (the q-th and (q+1)-th
most confident) are within 1e-4, gets a row redrawn (salt + 1).  Only the
oracle is consulted; no expected value comes from the GPU.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle
import synth

MARGIN = 1e-4
CONF_TOL = 1e-5
PER_REQUEST_ABOVE = 8   # batches of more requests are handled request by request on a thread pool


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def _per_request(fn, reqs):
    """fn(b) for every listed request on a thread pool (the generator's C
    code and numpy's large reductions release the GIL); results in order."""
    with ThreadPoolExecutor(max_workers=_threads()) as ex:
        return list(ex.map(fn, reqs))


def _bad_rows(inp, reqs, conf_by_row, quota=None):
    """Rows of the listed requests that sit inside a decision margin."""
    cfg = inp.cfg
    L = cfg.L
    bad = []
    for b in reqs:
        rows = [b * L + j for j in range(L) if inp.input_ids[b, j] == cfg.mask_id]
        if not rows:
            continue
        confs = np.array([conf_by_row[r] for r in rows])
        if quota is not None:
            q = int(quota[b])
            if 0 < q < len(rows):
                order = np.argsort(-confs, kind="stable")
                if confs[order[q - 1]] - confs[order[q]] < MARGIN:
                    bad.append(rows[order[q]])
            continue
        t = float(np.float32(inp.thr[b]))
        near = [r for r, c in zip(rows, confs) if abs(c - t) < MARGIN]
        bad.extend(near)
        if not (confs > t).any() and len(rows) > 1:
            order = np.argsort(-confs, kind="stable")
            if confs[order[0]] - confs[order[1]] < MARGIN:
                bad.append(rows[order[0]])
    return sorted(set(bad))


def host_rows(inp, rows, nthreads=None):
    """Generated logits of the listed flat rows, compact [len(rows), ldv]."""
    cfg = inp.cfg
    rows = np.asarray(rows, dtype=np.int64)
    out = np.full((max(len(rows), 1), cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    if len(rows):
        synth.fill_logits_rows(out, cfg.V, np.arange(len(rows)), synth.step_row_keys(inp, rows),
                               cfg.offset_max, cfg.mask_id, nthreads=nthreads)
    return out[: len(rows)]


def _enforce_request(inp, b, max_iter, quota):
    """Redraw rows of request b until all its decisions have margin."""
    cfg = inp.cfg
    L = cfg.L
    flat = inp.salt.reshape(-1)
    for _ in range(max_iter):
        rows = [b * L + j for j in range(L) if inp.input_ids[b, j] == cfg.mask_id]
        if not rows:
            return
        logits = host_rows(inp, rows, nthreads=1)
        conf, _, _ = oracle.rows_stats(logits, range(len(rows)), cfg.V)
        bad = _bad_rows(inp, [b], dict(zip(rows, conf)), quota)
        if not bad:
            return
        flat[bad] += 1
    raise AssertionError(f"could not draw request {b} with decision margins")


def enforce_margins(inp, reqs=None, max_iter=50, quota=None):
    """Redraw rows of the listed requests until all decisions have margin
    (threshold rule, or the fixed-steps rule when ``quota`` [B] is given).
    Every decision lies inside one request, so requests are handled one by
    one (on a thread pool)."""
    if reqs is None:
        reqs = range(inp.input_ids.shape[0])
    assert inp.salt.reshape(-1).base is not None or inp.salt.ndim == 1   # the flat view writes through
    _per_request(lambda b: _enforce_request(inp, b, max_iter, quota), list(reqs))


def sub_batch_logits(inp, reqs, nthreads=None):
    """Oracle-side logits for a sub-batch: [len(reqs) * L, ldv], masked rows
    generated, the others poisoned."""
    cfg = inp.cfg
    L = cfg.L
    out = np.full((len(reqs) * L, cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    rows, dst = [], []
    for k, b in enumerate(reqs):
        for j in range(L):
            if inp.input_ids[b, j] == cfg.mask_id:
                rows.append(b * L + j)
                dst.append(k * L + j)
    if rows:
        synth.fill_logits_rows(out, cfg.V, np.asarray(dst), synth.step_row_keys(inp, rows), cfg.offset_max,
                               cfg.mask_id, nthreads=nthreads)
    return out


def oracle_step(inp, reqs=None, quota=None):
    """The oracle's step over the listed requests.  The step treats every
    request on its own (FDFO page, section "工程设计一": per-request
    selection, done flag and state), so a large batch is computed request by
    request on a thread pool and the per-request results are stacked."""
    cfg = inp.cfg
    if reqs is None:
        reqs = list(range(inp.input_ids.shape[0]))
    reqs = list(reqs)
    qa = None if quota is None else np.asarray(quota)

    def one(sub, nthreads=None):
        return oracle.step(sub_batch_logits(inp, sub, nthreads), cfg.V, inp.input_ids[sub], inp.thr[sub],
                           inp.conf_state[sub], cfg.mask_id, quota=None if qa is None else qa[sub])

    if len(reqs) <= PER_REQUEST_ABOVE:
        return one(reqs)
    parts = _per_request(lambda b: one([b], 1), reqs)
    return {k: np.concatenate([p[k] for p in parts], axis=0) for k in parts[0]}


def device_logits(inp, device, chunk_rows=2048):
    """Device bf16 logits [B*L, ldv] (int16 storage): poison everywhere,
    generated rows on the positions masked at entry."""
    import torch
    cfg = inp.cfg
    B, L = inp.input_ids.shape
    d = torch.empty((B * L, cfg.row_stride), dtype=torch.int16, device=device)
    d.fill_(int(np.int16(np.uint16(synth.POISON_BITS).view(np.int16))))
    rows = np.flatnonzero(inp.masked.reshape(-1))
    for s in range(0, len(rows), chunk_rows):
        part = rows[s:s + chunk_rows]
        h = host_rows(inp, part)
        d[torch.from_numpy(part).to(device)] = torch.from_numpy(h.view(np.int16)).to(device)
    return d


def device_logits_compact(inp, device, extra_rows=0, chunk_rows=2048):
    """Device bf16 logits of the masked positions only, [M + extra_rows,
    ldv]: row k is the k-th masked position in position order (extra rows
    poisoned)."""
    import torch
    cfg = inp.cfg
    rows = np.flatnonzero(inp.masked.reshape(-1))
    d = torch.empty((len(rows) + extra_rows, cfg.row_stride), dtype=torch.int16, device=device)
    d.fill_(int(np.int16(np.uint16(synth.POISON_BITS).view(np.int16))))
    for s in range(0, len(rows), chunk_rows):
        part = rows[s:s + chunk_rows]
        d[s:s + len(part)] = torch.from_numpy(host_rows(inp, part).view(np.int16)).to(device)
    return d


def device_state(inp, device):
    import torch
    return (torch.from_numpy(inp.input_ids.copy()).to(device),
            torch.from_numpy(inp.thr.copy()).to(device),
            torch.from_numpy(inp.conf_state.copy()).to(device))


def compare_step(ref, got, reqs, L, ids_after, cs_after):
    """Assert GPU results (host numpy dict) equal the oracle's for ``reqs``."""
    masked = ref["masked"]
    tok = got["tok"][reqs]
    conf = got["conf"][reqs]
    lse = got["lse"][reqs]
    np.testing.assert_array_equal(tok[masked], ref["tok"][masked])
    np.testing.assert_allclose(conf[masked], ref["conf"][masked], rtol=0, atol=CONF_TOL)
    lref = ref["lse"][masked]
    assert np.all(np.abs(lse[masked] - lref) <= CONF_TOL * np.maximum(1.0, np.abs(lref)))
    assert (tok[~masked] == -1).all() and np.isnan(conf[~masked]).all() and np.isnan(lse[~masked]).all()
    np.testing.assert_array_equal(ids_after[reqs], ref["input_ids"])
    np.testing.assert_array_equal(got["done"][reqs], ref["done"])
    np.testing.assert_array_equal(got["accept_len"][reqs], ref["accept_len"])
    np.testing.assert_array_equal(got["n_new"][reqs], ref["n_new"])
    cs = cs_after[reqs]
    both_nan = np.isnan(cs) & np.isnan(ref["conf_state"])
    assert np.array_equal(np.isnan(cs), np.isnan(ref["conf_state"]))
    np.testing.assert_allclose(cs[~both_nan], ref["conf_state"][~both_nan], rtol=0, atol=CONF_TOL)
    np.testing.assert_allclose(got["feats"][reqs], ref["feats"], rtol=0, atol=CONF_TOL, equal_nan=True)


# ---------------------------------------------------------------------------
# The serving loop at full vocabulary size: logits request by request
# ---------------------------------------------------------------------------
def _margin_bad(conf, t, q):
    """Indices (into ``conf``, one request's masked rows in position order)
    to redraw so that every decision of the step has a margin: against the
    threshold ``t`` and between the fallback's top two, or, under the
    fixed-steps rule (``q`` not None), between the q-th and (q+1)-th most
    confident."""
    bad = set()
    if q is not None:
        if 0 < q < len(conf):
            order = np.argsort(-conf, kind="stable")
            if conf[order[q - 1]] - conf[order[q]] < MARGIN:
                bad.add(int(order[q]))
        return bad
    bad.update(int(k) for k in np.flatnonzero(np.abs(conf - t) < MARGIN))
    if not (conf > t).any() and len(conf) > 1:
        order = np.argsort(-conf, kind="stable")
        if conf[order[0]] - conf[order[1]] < MARGIN:
            bad.add(int(order[0]))
    return bad


def request_block_logits(seed, rows_i, L, V, ldv, offset, mask_id, thr, salts, q=None, max_iter=50):
    """Logits [L, ldv] of one active request of the loop: its masked
    positions' rows (``rows_i``: (flat row, rid, block, step, position)
    tuples) generated from (request, block, step, position, salt), the rest
    poisoned; rows inside a decision margin are redrawn (their salt, kept in
    ``salts`` by (rid, block, step, position), goes up by one).  ``thr``:
    the request's float32 threshold; ``q``: its fixed-steps quota or None."""
    out = np.full((L, ldv), synth.POISON_BITS, dtype=np.uint16)
    if not rows_i:
        return out
    js = np.array([r[4] for r in rows_i])
    key_of = lambda r: (r[1], r[2], r[3], r[4])
    t = float(np.float32(thr))
    for _ in range(max_iter):
        keys = synth.logits_row_keys(seed, [r[1] for r in rows_i], [r[2] for r in rows_i], [r[3] for r in rows_i],
                                     js, [salts.get(key_of(r), 0) for r in rows_i])
        synth.fill_logits_rows(out, V, js, keys, offset, mask_id, nthreads=1)
        conf, _, _ = oracle.rows_stats(out, js, V)
        bad = _margin_bad(conf, t, q)
        if not bad:
            return out
        for k in bad:
            salts[key_of(rows_i[k])] = salts.get(key_of(rows_i[k]), 0) + 1
    raise AssertionError("no margin after redraws")


def _oracle_loop_class():
    from oracle.loop import OracleLoop

    class PerRequestOracleLoop(OracleLoop):
        """The oracle loop with its step computed request by request on a
        thread pool.  The step treats every request on its own (FDFO page,
        section "工程设计一"), so stacking the per-request results in row
        order gives ``step_phase``'s result; the state update after it is
        the same as ``step_phase``'s."""

        def step_phase_per_request(self, block_fn):
            """``block_fn(i, rows_i)``: the logits [L, ldv] of active row i for
            its masked rows.  Returns (the step's result, the blocks)."""
            L = self.L
            A = len(self.rid)
            by_row = [[] for _ in range(A)]
            for r in self.masked_rows():
                by_row[r[0] // L].append(r)
            thr = np.array([self.thr_all[r] for r in self.rid], dtype=np.float32)
            quota = self.quota()

            def one(i):
                blk = block_fn(i, by_row[i])
                res = oracle.step(blk, self.V, self.ids[i:i + 1], thr[i:i + 1], self.cs[i:i + 1], self.mask_id,
                                  quota=None if quota is None else quota[i:i + 1])
                return blk, res

            parts = _per_request(one, range(A))
            blocks = [p[0] for p in parts]
            res = {k: np.concatenate([p[1][k] for p in parts], axis=0) for k in parts[0][1]} if A else None
            if A:
                had_masked = res["masked"].any(axis=1)
                self.ids = res["input_ids"]
                self.cs = res["conf_state"]
                for i in range(A):
                    if had_masked[i]:
                        self.s[i] += 1
            return res, blocks

    return PerRequestOracleLoop


def per_request_oracle_loop(*args, **kw):
    """A ``PerRequestOracleLoop`` (built on ``oracle.loop.OracleLoop``)."""
    return _oracle_loop_class()(*args, **kw)
