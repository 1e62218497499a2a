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

import numpy as np

import oracle
import synth

MARGIN = 1e-4
CONF_TOL = 1e-5


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


def host_rows(inp, rows):
    """Generated logits of the listed flat rows, compact [len(rows), ldv]."""
    cfg = inp.cfg
    rows = np.asarray(rows, dtype=np.int64)
    out = np.full((max(len(rows), 1), cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    if len(rows):
        synth.fill_logits_rows(out, cfg.V, np.arange(len(rows)), synth.step_row_keys(inp, rows),
                               cfg.offset_max, cfg.mask_id)
    return out[: len(rows)]


def enforce_margins(inp, reqs=None, max_iter=50, quota=None):
    """Redraw rows of the listed requests until all decisions have margin
    (threshold rule, or the fixed-steps rule when ``quota`` [B] is given)."""
    cfg = inp.cfg
    if reqs is None:
        reqs = range(inp.input_ids.shape[0])
    reqs = list(reqs)
    L = cfg.L
    for _ in range(max_iter):
        rows = [b * L + j for b in reqs for j in range(L) if inp.input_ids[b, j] == cfg.mask_id]
        logits = host_rows(inp, rows)
        conf, _, _ = oracle.rows_stats(logits, range(len(rows)), cfg.V)
        bad = _bad_rows(inp, reqs, dict(zip(rows, conf)), quota)
        if not bad:
            return
        flat = inp.salt.reshape(-1)
        flat[bad] += 1
    raise AssertionError("could not draw a case with decision margins")


def sub_batch_logits(inp, reqs):
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
                               cfg.mask_id)
    return out


def oracle_step(inp, reqs=None, quota=None):
    cfg = inp.cfg
    if reqs is None:
        reqs = list(range(inp.input_ids.shape[0]))
    reqs = list(reqs)
    return oracle.step(sub_batch_logits(inp, reqs), cfg.V, inp.input_ids[reqs], inp.thr[reqs],
                       inp.conf_state[reqs], cfg.mask_id,
                       quota=None if quota is None else np.asarray(quota)[reqs])


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
