"""CPU oracle for the block-wise dLLM denoise step, pack and compaction.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference legs of ``bench.py`` use it.  It shares no code with the CUDA
library and never reads its outputs.

Plain numpy in float64, one function per step of the method, written for a
reader to check against the pages by eye.  Sources (cited by page title and
section):

* FDFO page -- "FDFO: 让 dLLM 推理从「整批等最慢」变成「谁先完成谁先走」"
  (SGLang PRs #27551 / #27877 write-up): sections "工程设计一" (the
  ``step(forward_batch, full_logits, states) -> done_flags`` contract and the
  LowConfidence rule), "工程设计二" (per-request state and accept_length),
  "原来的同步调度问题在哪里" / "FDFO 的核心思想" (the A/B/C example and the
  sync versus FDFO loops).
* BlockServe page -- "BlockServe: 块粒度连续批处理实现高吞吐扩散大语言模型服务":
  section II-A (p_i, g_i, K_i, b_i), Algorithm 1 (section II-C), eq. (1) and
  the sand-fill admission (section II-D), left padding, position ids and the
  gather/scatter of the active block (section II-E).
* DiLaServe review -- "DiLaServe: High SLO Attainment Serving for Diffusion
  Language Models": section 3.1 (softmax confidence, threshold, fallback),
  section 4.1 (candidate thresholds), section 4.2 item ③ (confidence
  features: min / q25 / median / avg / q75 and unmasked fraction).

Readings where the pages are silent (each one is listed in the design notes):
argmax ties go to the lowest vocabulary index; "exceeds" is a strict ``>``
against the float32 threshold; the fallback picks the most confident masked
position, ties to the lowest position; a block is done when no position holds
the mask id after the update; accept_length is L when done, else 0; features
use the confidence recorded when each position was unmasked, over the block's
unmasked positions, with linear-interpolation quantiles.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against hand-computed values, closed forms, library routines on special
cases, brute force on tiny inputs and the pages' worked examples.
"""
from __future__ import annotations

import numpy as np

FEATURE_NAMES = ("min", "q25", "median", "avg", "q75", "unmasked_frac")


# ---------------------------------------------------------------------------
# bf16 input widening (exact).
# ---------------------------------------------------------------------------
def bf16_to_f64(bits):
    """Exact value of bf16 bit patterns: the 16 bits are the top half of an
    IEEE binary32, so shifting them up gives the float32, which widens
    exactly to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# S2: the per-row reduction.
# ---------------------------------------------------------------------------
def row_stats(x):
    """Confidence, log-sum-exp and argmax token of one logits row.

    DiLaServe review, section 3.1: the confidence is the softmax probability
    of the predicted token.  At temperature 0 the predicted token is the
    argmax (FDFO page, section "工程设计三": greedy, byte-identical parity at
    temperature 0).  With m = max x and s = sum_j exp(x_j - m):
    softmax(x)_tok = exp(x_tok - m) / s = 1 / s, and log-sum-exp = m + ln s.
    ``x`` is a float64 vector of the row's V values.
    """
    m = x.max()
    tok = int(np.flatnonzero(x == m)[0])          # lowest index attaining m
    s = float(np.exp(x - m).sum())
    return 1.0 / s, m + np.log(s), tok


def rows_stats(logits_bits, rows, V):
    """row_stats over the listed rows of a [rows, ldv] uint16 bf16 matrix."""
    n = len(rows)
    conf = np.empty(n)
    lse = np.empty(n)
    tok = np.empty(n, dtype=np.int64)
    for i, r in enumerate(rows):
        conf[i], lse[i], tok[i] = row_stats(bf16_to_f64(logits_bits[r, :V]))
    return conf, lse, tok


def shard_triple(x, v0):
    """S2 over one vocabulary shard: (max m, sum_j exp(x_j - m), lowest
    global index attaining m) of the shard's values ``x`` (float64), whose
    first column is global token ``v0``.  A vocabulary-parallel LM head
    (DiLaServe review, section 2.2.2: tensor parallelism) or a chunked one
    hands the step one such shard at a time."""
    m = x.max()
    return float(m), float(np.exp(x - m).sum()), int(v0 + np.flatnonzero(x == m)[0])


def merge_triples(triples):
    """Fold per-shard (m, s, idx) triples, in shard order (ascending
    vocabulary ranges), into the row's (conf, lse, tok): M = max m_k,
    S = sum_k s_k exp(m_k - M), tok = the idx of the first shard attaining M
    (its lowest index, the shards being ordered); conf = 1/S, lse = M + ln S,
    as ``row_stats`` of the whole row."""
    M = max(t[0] for t in triples)
    S = sum(t[1] * np.exp(t[0] - M) for t in triples)
    tok = next(t[2] for t in triples if t[0] == M)
    return 1.0 / S, M + np.log(S), tok


def step_sharded(logits_bits, V, bounds, input_ids, thr, conf_state, mask_id, quota=None):
    """``step`` with S2 computed shard by shard over the vocabulary ranges
    [bounds[k], bounds[k+1]) and merged (``shard_triple``, ``merge_triples``);
    S3-S6 as ``step``."""
    input_ids = np.asarray(input_ids)
    B, L = input_ids.shape
    rows = np.flatnonzero((input_ids == mask_id).reshape(-1))
    conf = np.empty(len(rows))
    lse = np.empty(len(rows))
    tok = np.empty(len(rows), dtype=np.int64)
    for i, r in enumerate(rows):
        x = bf16_to_f64(logits_bits[r, :V])
        tr = [shard_triple(x[bounds[k]:bounds[k + 1]], bounds[k]) for k in range(len(bounds) - 1)]
        conf[i], lse[i], tok[i] = merge_triples(tr)
    return _finish_step(input_ids, thr, conf_state, mask_id, rows, conf, lse, tok, quota)


# ---------------------------------------------------------------------------
# S3: LowConfidence selection with fallback.
# ---------------------------------------------------------------------------
def select_positions(masked, conf, thr):
    """Positions of one block to unmask this step.

    FDFO page, section "工程设计一" (LowConfidence): a masked position whose
    confidence exceeds the threshold is unmasked; if no position in the round
    exceeds it, the single most confident position is unmasked so the
    process always advances (same rule: DiLaServe review, section 3.1).
    ``masked``: bool [L]; ``conf``: float [L] (read only where masked);
    ``thr``: the request's float32 threshold.  Returns bool [L].
    """
    masked = np.asarray(masked, dtype=bool)
    t = float(np.float32(thr))
    sel = np.zeros(masked.shape, dtype=bool)
    for j in range(masked.size):
        if masked[j] and conf[j] > t:
            sel[j] = True
    if not sel.any() and masked.any():
        best = -1
        for j in range(masked.size):
            if masked[j] and (best < 0 or conf[j] > conf[best]):
                best = j
        sel[best] = True
    return sel


def transfer_quota(L, S, s):
    """Tokens to unmask at step s (0-based) of a block under the fixed-steps
    rule (BlockServe page, section II-E, "向量化混合调度执行"): at the start
    of each block cycle the block's L masked tokens are spread evenly over S
    denoising steps, the same for every block since each starts fully masked.
    Reading: q(s) = floor(L / S), plus one for the first L mod S steps; a step
    past the schedule (s >= S) transfers everything still masked (returned
    as L).
    """
    if L < 1 or S < 1 or s < 0:
        raise ValueError("L, S >= 1 and s >= 0")
    if s >= S:
        return L
    return L // S + (1 if s < L % S else 0)


def select_quota(masked, conf, q):
    """The q most confident masked positions of one block (all of them when
    fewer than q are masked); ties go to the lower position.  The fixed-steps
    counterpart of ``select_positions`` (BlockServe page, section II-E).
    Plain repeated selection of the best remaining position."""
    masked = np.asarray(masked, dtype=bool)
    sel = np.zeros(masked.shape, dtype=bool)
    for _ in range(max(int(q), 0)):
        best = -1
        for j in range(masked.size):
            if masked[j] and not sel[j] and (best < 0 or conf[j] > conf[best]):
                best = j
        if best < 0:
            break
        sel[best] = True
    return sel


# ---------------------------------------------------------------------------
# S6: confidence features for a step predictor.
# ---------------------------------------------------------------------------
def quantile_linear(sorted_vals, q):
    """Linear-interpolation quantile of ascending values at rank q * (n - 1)."""
    n = len(sorted_vals)
    h = q * (n - 1)
    lo = int(np.floor(h))
    hi = min(lo + 1, n - 1)
    return sorted_vals[lo] + (h - lo) * (sorted_vals[hi] - sorted_vals[lo])


def block_features(ids_row, conf_row, mask_id):
    """DiLaServe review, section 4.2 item ③: min, q25, median, avg, q75 of
    the output tokens' confidences, plus the unmasked fraction (progress).

    The output tokens are the block's positions not holding the mask id; each
    carries the confidence recorded when it was unmasked.  With no such
    position the five statistics are NaN and the fraction is 0.
    """
    keep = np.asarray(ids_row) != mask_id
    L = keep.size
    vals = np.sort(np.asarray(conf_row, dtype=np.float64)[keep])
    n = vals.size
    if n == 0:
        return np.array([np.nan] * 5 + [0.0])
    return np.array([
        vals[0],
        quantile_linear(vals, 0.25),
        quantile_linear(vals, 0.50),
        vals.sum() / n,
        quantile_linear(vals, 0.75),
        n / L,
    ])


def features(input_ids, conf_state, mask_id):
    """block_features for every request (rows of [B, L] arrays)."""
    return np.stack([block_features(input_ids[b], conf_state[b], mask_id)
                     for b in range(input_ids.shape[0])]) if input_ids.shape[0] else np.zeros((0, 6))


# ---------------------------------------------------------------------------
# S1-S6: one denoise step.
# ---------------------------------------------------------------------------
def step(logits_bits, V, input_ids, thr, conf_state, mask_id, quota=None):
    """``step(forward_batch, full_logits, states) -> done_flags`` for one
    batch (FDFO page, section "工程设计一"): read the logits, update
    input_ids by the LowConfidence rule, report per-block completion.

    logits_bits: uint16 [B*L, ldv] (row b*L + j is position j of request b)
    input_ids:   int   [B, L]  -- current block tokens; mask_id marks masked
    thr:         float [B]     -- per-request threshold (DiLaServe review,
                                  section 4.1: chosen per request)
    conf_state:  float [B, L]  -- confidence at unmask time (per-request
                                  algorithm state carried between rounds,
                                  FDFO page, section "工程设计二")
    quota:       int [B] or None -- when given, the fixed-steps rule
                                  (``select_quota``) replaces the threshold
                                  rule and ``thr`` is not read
    Returns a dict with the updated ``input_ids`` / ``conf_state`` and the
    outputs ``done``, ``accept_len``, ``n_new``, ``feats`` and per-position
    ``conf`` / ``lse`` / ``tok`` (NaN, NaN, -1 on positions not masked at
    entry).  Inputs are not modified.
    """
    input_ids = np.array(input_ids, dtype=np.int64)
    rows = np.flatnonzero((input_ids == mask_id).reshape(-1))      # S1
    c, l, t = rows_stats(logits_bits, rows, V)                      # S2
    return _finish_step(input_ids, thr, conf_state, mask_id, rows, c, l, t, quota)


def _finish_step(input_ids, thr, conf_state, mask_id, rows, c, l, t, quota):
    """S3-S6 of ``step`` from the masked rows' (conf, lse, tok)."""
    input_ids = np.array(input_ids, dtype=np.int64)
    conf_state = np.array(conf_state, dtype=np.float64)
    B, L = input_ids.shape
    masked = input_ids == mask_id
    conf = np.full((B, L), np.nan)
    lse = np.full((B, L), np.nan)
    tok = np.full((B, L), -1, dtype=np.int64)
    conf.reshape(-1)[rows] = c
    lse.reshape(-1)[rows] = l
    tok.reshape(-1)[rows] = t
    new_ids = input_ids.copy()
    new_cs = conf_state.copy()
    n_new = np.zeros(B, dtype=np.int64)
    done = np.zeros(B, dtype=np.uint8)
    accept = np.zeros(B, dtype=np.int64)
    for b in range(B):
        if quota is None:
            sel = select_positions(masked[b], conf[b], thr[b])     # S3
        else:
            sel = select_quota(masked[b], conf[b], quota[b])
        new_ids[b, sel] = tok[b, sel]                               # S4
        new_cs[b, sel] = conf[b, sel]
        n_new[b] = int(sel.sum())                                   # S5
        done[b] = 1 if not (new_ids[b] == mask_id).any() else 0
        # FDFO page, section "工程设计二": accept_length is 0 while the block
        # continues and block_size once it can be committed.
        accept[b] = L if done[b] else 0
    feats = features(new_ids, new_cs, mask_id)                      # S6
    return dict(input_ids=new_ids, conf_state=new_cs, done=done, accept_len=accept,
                n_new=n_new, feats=feats, conf=conf, lse=lse, tok=tok, masked=masked)


# ---------------------------------------------------------------------------
# S7: the bounding box (BlockServe page, sections II-D and II-E).
# ---------------------------------------------------------------------------
def row_width(p, b, L):
    """Effective row width of a request at block index b: p + (b + 1) * L
    (BlockServe page, section II-D)."""
    return int(p) + (int(b) + 1) * int(L)


def cost(p, b, L):
    """Eq. (1): Cost(A) = |A| * max over A of (p_i + (b_i + 1) * L); 0 for
    an empty set."""
    if len(p) == 0:
        return 0
    return len(p) * max(row_width(pi, bi, L) for pi, bi in zip(p, b))


def box_width(p, b, L):
    if len(p) == 0:
        return 0
    return max(row_width(pi, bi, L) for pi, bi in zip(p, b))


def pack(p, b, L, prompts, gens, blocks, pad_id, W=None):
    """Materialise the bounding box of eq. (1) as a dense [A, W] batch.

    BlockServe page, section II-E ("逻辑位置对齐"): rows are left-padded so
    each prompt sits immediately before its generated region; position ids
    are a cumulative index over the attention mask so the first real token is
    at logical position 0.  Row i = [pad_i pads, prompt_i, the b_i completed
    blocks, the current block]; its current block therefore ends at column W.
    ``prompts[i]``: prompt tokens; ``gens[i]``: at least b_i * L generated
    tokens; ``blocks[i]``: the current block's L tokens.
    Returns ids [A, W], attn [A, W], pos [A, W], pad [A], blk_start [A]
    (logical position of the current block's first token) and W.
    """
    A = len(p)
    if W is None:
        W = box_width(p, b, L)
    ids = np.full((A, W), pad_id, dtype=np.int64)
    attn = np.zeros((A, W), dtype=np.int64)
    pad = np.zeros(A, dtype=np.int64)
    blk_start = np.zeros(A, dtype=np.int64)
    for i in range(A):
        width = row_width(p[i], b[i], L)
        pad[i] = W - width
        seq = np.concatenate([np.asarray(prompts[i][:p[i]]),
                              np.asarray(gens[i][: b[i] * L]),
                              np.asarray(blocks[i][:L])]).astype(np.int64)
        ids[i, pad[i]:] = seq
        attn[i, pad[i]:] = 1
        blk_start[i] = int(p[i]) + int(b[i]) * L
    pos = np.cumsum(attn, axis=1) - 1
    pos[attn == 0] = 0
    return dict(ids=ids, attn=attn, pos=pos, pad=pad, blk_start=blk_start, W=W)


# ---------------------------------------------------------------------------
# S8: length-aware greedy ("sand-fill") admission.
# ---------------------------------------------------------------------------
def admit(pending_p, active_p, active_b, L, budget):
    """Indices (into the pending queue, in admission order) admitted this
    iteration.

    BlockServe page, section II-D and Algorithm 1 line "admit from P while
    Cost(A ∪ {r_cand}) <= budget": the pending queue is kept sorted by prompt
    length; a candidate whose initial width p + L fits inside the current box
    without widening it is preferred ("sand-fill"); a candidate is admitted
    only if eq. (1) stays within the budget.  Reading: among fitting
    candidates take the longest prompt (earliest in the queue on ties); with
    none fitting, take the head of the queue (shortest prompt); stop at the
    first candidate the budget rejects.  ``pending_p`` must be sorted
    ascending (ties by request id).
    """
    ap = list(active_p)
    ab = list(active_b)
    remaining = list(range(len(pending_p)))
    admitted = []
    while remaining:
        w_cur = box_width(ap, ab, L)
        fit = [k for k in remaining if row_width(pending_p[k], 0, L) <= w_cur]
        if fit:
            best_p = max(pending_p[k] for k in fit)
            cand = min(k for k in fit if pending_p[k] == best_p)
        else:
            cand = remaining[0]
        if cost(ap + [pending_p[cand]], ab + [0], L) > budget:
            break
        admitted.append(cand)
        remaining.remove(cand)
        ap.append(pending_p[cand])
        ab.append(0)
    return admitted


# ---------------------------------------------------------------------------
# S9: stable compaction for FDFO eviction.
# ---------------------------------------------------------------------------
def compact(evict):
    """Survivor map of a stable compaction (FDFO page, section "FDFO 的核心
    思想": finished requests leave the batch at once; BlockServe Algorithm 1:
    remove every request with b_i >= K_i).  Survivors keep their order.
    Returns new_index [A] (-1 for evicted rows), src_row [A'] and A'."""
    evict = np.asarray(evict, dtype=bool)
    new_index = np.full(evict.size, -1, dtype=np.int64)
    src_row = []
    for i in range(evict.size):
        if not evict[i]:
            new_index[i] = len(src_row)
            src_row.append(i)
    return new_index, np.asarray(src_row, dtype=np.int64), len(src_row)
