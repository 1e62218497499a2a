"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (A/B/C example), hand computations and closed forms, library
routines on special cases (scipy's logsumexp / softmax, numpy.quantile), and
brute force or invariants over tiny inputs.  None needs a GPU.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle.loop import OracleLoop
from conftest import golden

import synth


def bf16(x):
    """Exact bf16 bit patterns of values that are representable in bf16."""
    bits = synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(bits), np.asarray(x, dtype=np.float32)), "not bf16-exact"
    return bits


# --------------------------------------------------------------------------
# bf16 widening
# --------------------------------------------------------------------------
def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC1F0, 0x4049, 0x0001, 0x8000, 0x7F7F], dtype=np.uint16)
    want = [1.0, -30.0, 3.140625, 2.0 ** -133, -0.0, (2 - 2 ** -7) * 2.0 ** 127]
    got = oracle.bf16_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert math.copysign(1.0, got[4]) == -1.0


# --------------------------------------------------------------------------
# S2: row reduction
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("c", [-3.0, 0.0, 0.5, 7.25])
def test_row_stats_all_equal(V, c):
    # Softmax of V equal logits is uniform: conf = 1/V, lse = c + ln V, and
    # the lowest index wins the tie.
    conf, lse, tok = oracle.row_stats(np.full(V, c))
    assert tok == 0
    assert conf == pytest.approx(1.0 / V, rel=1e-15)
    assert lse == pytest.approx(c + math.log(V), rel=1e-15, abs=1e-15)


def test_row_stats_v1():
    conf, lse, tok = oracle.row_stats(np.array([-2.5]))
    assert (conf, lse, tok) == (1.0, -2.5, 0)


def test_row_stats_two_logits_closed_form():
    e = math.e
    conf, lse, tok = oracle.row_stats(np.array([0.0, 1.0]))
    assert tok == 1
    assert conf == pytest.approx(e / (1 + e), rel=1e-15)
    assert lse == pytest.approx(math.log(1 + e), rel=1e-15)
    conf, lse, tok = oracle.row_stats(np.array([1.0, 0.0]))
    assert tok == 0
    assert conf == pytest.approx(e / (1 + e), rel=1e-15)


def test_row_stats_ties_lowest_index():
    x = np.array([2.0, 5.0, 5.0, 1.0])
    conf, lse, tok = oracle.row_stats(x)
    assert tok == 1
    z = math.exp(2) + 2 * math.exp(5) + math.exp(1)
    assert conf == pytest.approx(math.exp(5) / z, rel=1e-14)
    assert lse == pytest.approx(math.log(z), rel=1e-14)


def test_row_stats_mask_column_never_wins():
    x = np.array([-30.0, -29.5, -31.0])
    assert oracle.row_stats(x)[2] == 1


def test_row_stats_brute_force_tiny_grid():
    # Every row of length <= 3 over a small bf16 grid, against the textbook
    # definition softmax_k = exp(x_k) / sum_j exp(x_j) evaluated with
    # math.fsum, and an argmax by strict-greater scan.
    grid = [-1.0, 0.0, 0.5, 2.0]
    for V in (1, 2, 3):
        for row in itertools.product(grid, repeat=V):
            x = oracle.bf16_to_f64(bf16(row))
            conf, lse, tok = oracle.row_stats(x)
            best = 0
            for k in range(V):
                if x[k] > x[best]:
                    best = k
            z = math.fsum(math.exp(v) for v in x)
            assert tok == best
            assert conf == pytest.approx(math.exp(x[best]) / z, rel=1e-14)
            assert lse == pytest.approx(math.log(z), rel=1e-14, abs=1e-14)


def test_row_stats_against_scipy():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    for V in (5, 64, 1000, 4099):
        raw = rng.normal(size=V).astype(np.float32) * 3
        x = oracle.bf16_to_f64(synth.f32_to_bf16_bits(raw))
        conf, lse, tok = oracle.row_stats(x)
        assert tok == int(np.argmax(x))
        assert lse == pytest.approx(float(sp.logsumexp(x)), rel=1e-13)
        assert conf == pytest.approx(float(sp.softmax(x)[tok]), rel=1e-12)


def test_rows_stats_reads_only_first_V_columns():
    ldv = 16
    m = np.full((2, ldv), 0x7F00, dtype=np.uint16)     # 1.7e38 beyond V
    m[0, :10] = bf16(np.arange(10) * 0.25 - 1.0)
    m[1, :10] = bf16(np.zeros(10))
    conf, lse, tok = oracle.rows_stats(m, [0, 1], 10)
    assert tok[0] == 9 and tok[1] == 0
    assert conf[1] == pytest.approx(0.1)


# --------------------------------------------------------------------------
# S3: selection and fallback
# --------------------------------------------------------------------------
def test_select_hand_cases():
    masked = np.array([True, True, False, True])
    conf = np.array([0.95, 0.5, np.nan, 0.92])
    assert oracle.select_positions(masked, conf, 0.9).tolist() == [True, False, False, True]
    # nothing above 0.96: the single most confident masked position
    assert oracle.select_positions(masked, conf, 0.96).tolist() == [True, False, False, False]
    # threshold 0 unmasks every masked position
    assert oracle.select_positions(masked, conf, 0.0).tolist() == [True, True, False, True]
    # no masked position: nothing to do
    assert not oracle.select_positions(np.zeros(4, bool), conf, 0.5).any()


def test_select_strict_against_float32_threshold():
    t32 = float(np.float32(0.9))         # 0.89999997615814...
    masked = np.array([True, True])
    conf = np.array([t32, 0.1])
    # equal to the threshold does not exceed it -> fallback to position 0
    assert oracle.select_positions(masked, conf, 0.9).tolist() == [True, False]
    conf = np.array([t32 + 1e-12, 0.95])
    assert oracle.select_positions(masked, conf, 0.9).tolist() == [True, True]


def test_select_fallback_ties_lowest_position():
    masked = np.array([False, True, True, True])
    conf = np.array([0.99, 0.7, 0.7, 0.2])
    assert oracle.select_positions(masked, conf, 0.8).tolist() == [False, True, False, False]


def test_select_invariants_brute_force():
    # All mask patterns of L <= 4 and all orderings of four distinct
    # confidences, across thresholds.
    levels = [0.15, 0.45, 0.65, 0.95]
    for L in range(1, 5):
        for mpat in itertools.product([False, True], repeat=L):
            masked = np.array(mpat)
            for conf in itertools.permutations(levels, L):
                conf = np.array(conf)
                prev = None
                for thr in (-0.5, 0.0, 0.3, 0.5, 0.9, 1.0, 1.5):
                    sel = oracle.select_positions(masked, conf, thr)
                    assert not (sel & ~masked).any()
                    assert sel.any() == masked.any()
                    if masked.any():
                        passing = masked & (conf > np.float32(thr))
                        if passing.any():
                            assert np.array_equal(sel, passing)
                        else:
                            assert sel.sum() == 1
                            assert conf[sel][0] == conf[masked].max()
                    if thr < min(levels):
                        assert np.array_equal(sel, masked)
                    if thr >= 1.0 and masked.any():
                        assert sel.sum() == 1
                    if prev is not None and sel.sum() > 1:
                        assert not (sel & ~prev).any()      # raising thr only removes
                    prev = sel


# --------------------------------------------------------------------------
# S1-S6 through step()
# --------------------------------------------------------------------------
def _two_col_logits(conf_targets, V=2):
    """Rows whose softmax confidence is known in closed form: [0, a] with
    a = ln(c / (1 - c)) gives conf = 1 / (1 + e^-a) for the token 1."""
    rows = []
    for c in conf_targets:
        a = np.float32(math.log(c / (1 - c)))
        a = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(a))
        rows.append([0.0, float(a)])
    return bf16(np.array(rows, dtype=np.float32))


def test_step_closed_form_small():
    # One request, L = 4, positions 0, 1, 3 masked; mask id 7 (never a column).
    mask_id = 7
    ids = np.array([[mask_id, mask_id, 5, mask_id]])
    cs = np.array([[np.nan, np.nan, 0.97, np.nan]])
    logits = _two_col_logits([0.96, 0.55, 0.5, 0.93])
    a_vals = synth.bf16_bits_to_f32(logits[:, 1]).astype(np.float64)
    exact = 1.0 / (1.0 + np.exp(-a_vals))
    res = oracle.step(logits, 2, ids, np.array([0.9], np.float32), cs, mask_id)
    assert res["tok"][0].tolist() == [1, 1, -1, 1]
    np.testing.assert_allclose(res["conf"][0, [0, 1, 3]], exact[[0, 1, 3]], rtol=1e-14)
    assert res["input_ids"][0].tolist() == [1, mask_id, 5, 1]
    assert res["n_new"][0] == 2 and res["done"][0] == 0 and res["accept_len"][0] == 0
    np.testing.assert_allclose(res["conf_state"][0, [0, 3]], exact[[0, 3]], rtol=1e-14)
    vals = np.sort([exact[0], 0.97, exact[3]])
    f = res["feats"][0]
    assert f[0] == pytest.approx(vals[0])
    assert f[2] == pytest.approx(vals[1])
    assert f[3] == pytest.approx(vals.mean())
    assert f[5] == pytest.approx(0.75)


def _synthetic_step(seed, B=6, L=8, V=257, frac="fraction", thr=(0.9,)):
    cfg = synth.StepConfig("t", B, L, V, 8.0, frac, thr)
    return synth.make_step_inputs(cfg, seed)


@pytest.mark.parametrize("seed", range(4))
def test_step_invariants(seed):
    inp = _synthetic_step(seed)
    cfg = inp.cfg
    for thr_val, expect in ((0.0, "all"), (1.5, "one"), (None, None)):
        thr = inp.thr if thr_val is None else np.full(cfg.B, thr_val, np.float32)
        res = oracle.step(inp.logits, cfg.V, inp.input_ids, thr, inp.conf_state, cfg.mask_id)
        m_in = inp.masked
        m_out = res["input_ids"] == cfg.mask_id
        for b in range(cfg.B):
            n_sel = int((m_in[b] & ~m_out[b]).sum())
            assert res["n_new"][b] == n_sel
            assert not (m_out[b] & ~m_in[b]).any()                 # unmasked never remasked
            if m_in[b].any():
                assert n_sel >= 1                                  # progress guaranteed
            if expect == "all":
                assert not m_out[b].any()
            if expect == "one" and m_in[b].any():
                assert n_sel == 1
                j = np.flatnonzero(m_in[b] & ~m_out[b])[0]
                assert res["conf"][b, j] == np.nanmax(res["conf"][b])
            assert res["done"][b] == (0 if m_out[b].any() else 1)
            assert res["accept_len"][b] in (0, cfg.L)
            assert res["accept_len"][b] == (cfg.L if res["done"][b] else 0)
            # tokens written are the argmax tokens of their rows
            sel = m_in[b] & ~m_out[b]
            assert np.array_equal(res["input_ids"][b][sel], res["tok"][b][sel])
            assert np.array_equal(res["input_ids"][b][~m_in[b]], inp.input_ids[b][~m_in[b]])
        assert (res["tok"][~m_in] == -1).all() and np.isnan(res["conf"][~m_in]).all()


def test_step_zero_masked_request_is_done():
    inp = _synthetic_step(3)
    ids = inp.input_ids.copy()
    ids[0] = np.arange(inp.cfg.L)
    cs = inp.conf_state.copy()
    cs[0] = np.linspace(0.5, 1.0, inp.cfg.L)
    res = oracle.step(inp.logits, inp.cfg.V, ids, inp.thr, cs, inp.cfg.mask_id)
    assert res["done"][0] == 1 and res["n_new"][0] == 0 and res["accept_len"][0] == inp.cfg.L
    assert res["feats"][0][5] == 1.0


# --------------------------------------------------------------------------
# The FDFO page's A/B/C example, through the real step
# --------------------------------------------------------------------------
def _abc_batch(L=8, V=64):
    g = golden("abc_example.json")
    names = ["A", "B", "C"]
    masked_counts = [g["finish_step"][n] for n in names]
    mask_id = V - 1
    ids = np.zeros((3, L), dtype=np.int64)
    for i, mcount in enumerate(masked_counts):
        ids[i, :mcount] = mask_id
        ids[i, mcount:] = np.arange(L - mcount)
    cs = np.where(ids == mask_id, np.nan, 0.99)
    return g, names, ids, cs, mask_id


def _abc_logits(step_no, L, V):
    cfg = synth.StepConfig("abc", 3, L, V, 8.0, "half", (1.5,))
    inp = synth.make_step_state(cfg, 100 + step_no)
    inp.input_ids[:] = cfg.mask_id
    return synth.fill_step_logits(inp)


def test_abc_example_sync_and_fdfo():
    L, V = 8, 64
    g, names, ids, cs, mask_id = _abc_batch(L, V)
    thr = np.full(3, 1.5, np.float32)       # above any probability: one unmask per step
    # sync (_run_sync): every request steps until the whole batch is done
    finish = {}
    waste = 0
    step_no = 0
    cur_ids, cur_cs = ids.copy(), cs.copy()
    while True:
        step_no += 1
        res = oracle.step(_abc_logits(step_no, L, V), V, cur_ids, thr, cur_cs, mask_id)
        for i, n in enumerate(names):
            if res["done"][i] and n not in finish:
                finish[n] = step_no
            if not res["masked"][i].any():
                waste += 1             # an idle request held in the batch
        cur_ids, cur_cs = res["input_ids"], res["conf_state"]
        if res["done"].all():
            break
    assert finish == g["finish_step"]
    assert step_no == g["sync_batch_steps"]
    assert waste == g["sync_wasted_request_steps"]
    # the same total as the page's formula sum(max T - T_i)
    assert sum(step_no - t for t in finish.values()) == g["sync_wasted_request_steps"]
    # FDFO: each request leaves the batch as soon as its block is done
    live = list(range(3))
    cur_ids, cur_cs = ids.copy(), cs.copy()
    finish_f = {}
    waste_f = 0
    step_no = 0
    while live:
        step_no += 1
        res = oracle.step(_abc_logits(step_no, L, V)[: len(live) * L], V, cur_ids[live], thr[live],
                          cur_cs[live], mask_id)
        waste_f += int((~res["masked"].any(axis=1)).sum())
        keep = []
        for k, i in enumerate(live):
            cur_ids[i], cur_cs[i] = res["input_ids"][k], res["conf_state"][k]
            if res["done"][k]:
                finish_f[names[i]] = step_no
            else:
                keep.append(i)
        live = keep
    assert finish_f == g["finish_step"]
    assert waste_f == g["fdfo_wasted_request_steps"]


# --------------------------------------------------------------------------
# S6: features
# --------------------------------------------------------------------------
def test_features_hand_example():
    g = golden("quantile_example.json")
    L = g["L"]
    mask_id = -1
    ids = np.array([0, 1, mask_id, 2, 3, mask_id])
    conf = np.array([g["values"][0], g["values"][1], np.nan, g["values"][2], g["values"][3], np.nan])
    f = oracle.block_features(ids, conf, mask_id)
    want = [g["features"][k] for k in oracle.FEATURE_NAMES]
    assert len(ids) == L
    np.testing.assert_allclose(f, want, rtol=0, atol=1e-15)


def test_features_single_and_empty():
    f = oracle.block_features(np.array([9, 9, 4]), np.array([0, 0, 0.3]), mask_id=9)
    np.testing.assert_allclose(f[:5], 0.3)
    assert f[5] == pytest.approx(1 / 3)
    f = oracle.block_features(np.array([9, 9]), np.array([np.nan, np.nan]), mask_id=9)
    assert np.isnan(f[:5]).all() and f[5] == 0.0


def test_features_against_numpy_quantile():
    rng = np.random.default_rng(11)
    for n in (1, 2, 3, 5, 32, 64):
        vals = rng.random(n)
        ids = np.zeros(n, dtype=np.int64)
        f = oracle.block_features(ids, vals, mask_id=-1)
        np.testing.assert_allclose(
            f, [vals.min(), np.quantile(vals, 0.25, method="linear"), np.median(vals), vals.mean(),
                np.quantile(vals, 0.75, method="linear"), 1.0], rtol=1e-13)


# --------------------------------------------------------------------------
# S7: eq. (1) and the box
# --------------------------------------------------------------------------
def test_cost_eq1_golden():
    for case in golden("cost_eq1.json")["cases"]:
        L = case["L"]
        assert [oracle.row_width(p, b, L) for p, b in zip(case["p"], case["b"])] == case["widths"]
        assert oracle.cost(case["p"], case["b"], L) == case["cost"]


def test_pack_layout():
    L, pad_id = 4, -7
    p = [3, 6, 1]
    b = [1, 0, 2]
    prompts = [np.arange(100, 100 + n) for n in p]
    gens = [np.arange(200 + 10 * i, 200 + 10 * i + 8) for i in range(3)]
    blocks = [np.array([-1, 5, -1, 6]), np.array([-1] * 4), np.array([7, 8, 9, -1])]
    box = oracle.pack(p, b, L, prompts, gens, blocks, pad_id)
    W = box["W"]
    assert W == max(3 + 8, 6 + 4, 1 + 12) == 13
    assert box["pad"].tolist() == [2, 3, 0]
    assert box["blk_start"].tolist() == [3 + 4, 6, 1 + 8]
    for i in range(3):
        pad = box["pad"][i]
        assert (box["ids"][i, :pad] == pad_id).all() and (box["attn"][i, :pad] == 0).all()
        assert (box["pos"][i, :pad] == 0).all()
        # first real token at logical position 0, then +1 per column
        assert box["pos"][i, pad:].tolist() == list(range(W - pad))
        assert box["ids"][i, pad:pad + p[i]].tolist() == prompts[i].tolist()
        assert box["ids"][i, pad + p[i]:W - L].tolist() == gens[i][: b[i] * L].tolist()
        # the current block always sits in the last L columns
        assert box["ids"][i, W - L:].tolist() == blocks[i].tolist()
        assert box["pos"][i, W - L] == box["blk_start"][i]


def test_box_shrinks_when_widest_row_leaves():
    # BlockServe Fig. 1, example 2: evicting the row that defines the maximum
    # shrinks the box and frees budget for new admissions.
    L = 32
    p, b = [900, 100, 200], [3, 0, 1]
    before = oracle.cost(p, b, L)
    after = oracle.cost(p[1:], b[1:], L)
    assert after < before
    assert oracle.box_width(p[1:], b[1:], L) < oracle.box_width(p, b, L)
    budget = before
    picked = oracle.admit([150, 180, 230, 260], p[1:], b[1:], L, budget)
    assert len(picked) >= 2


# --------------------------------------------------------------------------
# S8: admission (hand traces)
# --------------------------------------------------------------------------
def test_admit_hand_trace_from_empty():
    # L = 4, beta = 30: widths 6, 7, 9 -> costs 6, 14, 27; the fourth (p = 9)
    # would cost 4 * 13 = 52 > 30.
    assert oracle.admit([2, 3, 5, 9], [], [], 4, 30) == [0, 1, 2]


def test_admit_hand_trace_sand_fill():
    # Active row (p = 10, b = 1) has width 18.  Fitting candidates (p + 4 <= 18)
    # are taken longest first: 14, 4, 1 (costs 36, 54, 72); then p = 20 widens
    # the box to 24: 5 * 24 = 120 > 100.
    assert oracle.admit([1, 4, 14, 20], [10], [1], 4, 100) == [2, 1, 0]


def test_admit_respects_budget_and_ties():
    assert oracle.admit([5, 5, 5], [], [], 4, 9) == [0]          # 1*9 <= 9 < 2*9
    assert oracle.admit([5, 5, 5], [], [], 4, 0) == []
    assert oracle.admit([], [3], [0], 4, 100) == []
    # equal prompt lengths that fit: the earliest in the queue first
    assert oracle.admit([3, 3], [10], [0], 4, 1000) == [0, 1]


# --------------------------------------------------------------------------
# S9: compaction
# --------------------------------------------------------------------------
def test_compact_brute_force():
    for A in range(0, 11):
        for mask in range(1 << A):
            evict = np.array([(mask >> i) & 1 for i in range(A)], dtype=bool)
            new_index, src_row, A2 = oracle.compact(evict)
            assert A2 == int((~evict).sum())
            assert np.all(np.diff(src_row) > 0) if A2 > 1 else True
            assert set(src_row.tolist()) == set(np.flatnonzero(~evict).tolist())
            assert (new_index[evict] == -1).all()
            assert all(new_index[src_row[k]] == k for k in range(A2))


# --------------------------------------------------------------------------
# The loop
# --------------------------------------------------------------------------
def _loop_logits(seed, V):
    def fn(loop, rows):
        n = len(loop.rid) * loop.L
        out = np.zeros((max(n, 1), (V + 7) // 8 * 8), dtype=np.uint16)
        if rows:
            flat = np.array([r[0] for r in rows])
            keys = synth.logits_row_keys(seed, [r[1] for r in rows], [r[2] for r in rows],
                                         [r[3] for r in rows], [r[4] for r in rows], 0)
            synth.fill_logits_rows(out, V, flat, keys, 8.0, V - 1)
        return out
    return fn


def _small_loop(mode, R=6, budget=400, thr=0.9, seed=1, S=None):
    cfg = synth.LoopConfig("small", R, 3, 40, 24, 8, 97, budget, thr, 8.0)
    reqs = synth.make_loop_requests(cfg, seed)
    prompts = [reqs.prompt_tokens[reqs.prompt_off[r]:reqs.prompt_off[r + 1]] for r in range(R)]
    lp = OracleLoop(reqs.p, reqs.K, prompts, reqs.thr, cfg.L, cfg.V, cfg.mask_id, cfg.pad_id, budget, mode, S=S)
    return lp.run(_loop_logits(seed, cfg.V)), cfg


def test_loop_completes_and_fdfo_matches_sync_tokens():
    f, cfg = _small_loop("fdfo")
    s, _ = _small_loop("sync")
    assert f.finished() and s.finished()
    for r in range(cfg.R):
        assert len(f.gen[r]) == cfg.K * cfg.L
        assert not (f.gen[r] == cfg.mask_id).any()
        # logits depend only on (request, block, step, position), so the
        # tokens cannot depend on the execution mode
        assert np.array_equal(f.gen[r], s.gen[r])
    assert f.iteration <= s.iteration
    assert sum(t["waiting"] for t in f.trace) == 0
    assert sum(t["waiting"] for t in s.trace) > 0
    for t in f.trace:
        if t["admitted"]:
            # eq. (1) within the budget right after an admission
            assert t["cost"] <= cfg.budget


def test_loop_bs1_fdfo_equals_sync():
    # FDFO page, section "工程设计三": at batch size 1 FDFO and sync see the
    # same shapes and must agree byte for byte.
    f, cfg = _small_loop("fdfo", R=1)
    s, _ = _small_loop("sync", R=1)
    assert np.array_equal(f.gen[0], s.gen[0])
    assert f.iteration == s.iteration


def test_advance_hand_case():
    # BlockServe Algorithm 1: a committed block is appended to the request's
    # output, b_i grows by one, and the request is evicted once b_i >= K_i;
    # a continuing request starts its next block fully masked.
    from oracle.loop import advance
    mask = 9
    adv = np.array([1, 0, 1], dtype=bool)
    rid = [5, 6, 7]
    b = np.array([0, 1, 1])
    K = np.array([2, 3, 2])
    ids = np.array([[1, 2], [mask, 3], [4, 5]])
    cs = np.array([[0.9, 0.8], [np.nan, 0.7], [0.6, 0.95]])
    gen = {5: np.zeros(0, dtype=np.int64), 6: np.array([7, 7]), 7: np.array([8, 8])}
    evict = advance(adv, rid, b, K, ids, cs, gen, mask)
    assert evict.tolist() == [False, False, True]
    assert b.tolist() == [1, 1, 2]
    assert gen[5].tolist() == [1, 2] and gen[6].tolist() == [7, 7] and gen[7].tolist() == [8, 8, 4, 5]
    assert ids[0].tolist() == [mask, mask] and np.isnan(cs[0]).all()      # next block starts masked
    assert ids[1].tolist() == [mask, 3] and ids[2].tolist() == [4, 5]     # untouched / evicted as is


# --------------------------------------------------------------------------
# Fixed-steps transfer rule (BlockServe page, section II-E)
# --------------------------------------------------------------------------
def test_transfer_quota_schedule_closed_form():
    # spreading L over S steps: the S quotas sum to L, take the two values
    # floor(L/S) and ceil(L/S), never increase, and the larger one occurs
    # L mod S times
    for L in range(1, 70):
        for S in range(1, 70):
            qs = [oracle.transfer_quota(L, S, s) for s in range(S)]
            assert sum(qs) == L
            assert set(qs) <= {L // S, -(-L // S)}
            assert all(a >= b for a, b in zip(qs, qs[1:]))
            assert sum(1 for q in qs if q == L // S + 1) == (L % S if L % S else 0)
    # the pages' setting L = S = 32: one token per step
    assert [oracle.transfer_quota(32, 32, s) for s in range(32)] == [1] * 32
    assert [oracle.transfer_quota(32, 5, s) for s in range(5)] == [7, 7, 6, 6, 6]
    assert [oracle.transfer_quota(4, 8, s) for s in range(8)] == [1, 1, 1, 1, 0, 0, 0, 0]
    assert oracle.transfer_quota(32, 32, 40) == 32
    with pytest.raises(ValueError):
        oracle.transfer_quota(0, 4, 0)


def test_select_quota_against_lexsort():
    # the q most confident masked positions, ties to the lower position, is
    # the first q of a lexicographic sort on (-conf, position)
    rng = np.random.default_rng(8)
    for _ in range(400):
        L = int(rng.integers(1, 13))
        masked = rng.random(L) < 0.7
        conf = np.round(rng.random(L), 1)          # many ties
        q = int(rng.integers(-1, L + 3))
        order = [j for j in np.lexsort((np.arange(L), -conf)) if masked[j]]
        want = np.zeros(L, dtype=bool)
        want[order[: max(q, 0)]] = True
        assert np.array_equal(oracle.select_quota(masked, conf, q), want)


def test_select_quota_one_is_the_threshold_fallback():
    # with every confidence in (0, 1], a threshold of 1 passes nothing, so the
    # threshold rule reduces to its fallback: the single most confident
    # masked position -- the fixed-steps rule with q = 1
    rng = np.random.default_rng(9)
    for _ in range(300):
        L = int(rng.integers(1, 10))
        masked = rng.random(L) < 0.6
        conf = np.round(rng.uniform(0.01, 1.0, L), 2)
        assert np.array_equal(oracle.select_quota(masked, conf, 1), oracle.select_positions(masked, conf, 1.0))


def test_step_quota_extremes():
    cfg = synth.StepConfig("q", 3, 8, 50, 6.0, "fraction", (0.5,))
    inp = synth.make_step_state(cfg, 4)
    rows = np.flatnonzero(inp.masked.reshape(-1))
    logits = np.full((cfg.B * cfg.L, cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    synth.fill_logits_rows(logits, cfg.V, rows, synth.step_row_keys(inp, rows), cfg.offset_max, cfg.mask_id)
    allq = oracle.step(logits, cfg.V, inp.input_ids, inp.thr, inp.conf_state, cfg.mask_id,
                       quota=np.full(cfg.B, cfg.L))
    assert (allq["done"] == 1).all() and np.array_equal(allq["n_new"], inp.masked.sum(axis=1))
    none = oracle.step(logits, cfg.V, inp.input_ids, inp.thr, inp.conf_state, cfg.mask_id,
                       quota=np.zeros(cfg.B, dtype=int))
    assert np.array_equal(none["input_ids"], inp.input_ids) and (none["n_new"] == 0).all()
    # tokens written are the argmax tokens, confidences recorded at unmask time
    one = oracle.step(logits, cfg.V, inp.input_ids, inp.thr, inp.conf_state, cfg.mask_id,
                      quota=np.ones(cfg.B, dtype=int))
    chg = one["input_ids"] != inp.input_ids
    assert np.array_equal(one["input_ids"][chg], one["tok"][chg])
    assert np.array_equal(one["conf_state"][chg], one["conf"][chg])
    assert np.array_equal(one["n_new"], inp.masked.any(axis=1).astype(int))


@pytest.mark.parametrize("S", [1, 3, 4, 8])
def test_loop_fixed_steps_blocks_take_S_steps(S):
    # BlockServe page, section II-E: with the per-step quota spreading L over
    # S steps, every block of every request is done after exactly S steps
    # (L = 8 >= S), so a request admitted at iteration a leaves at a + K S - 1
    f, cfg = _small_loop("fdfo", S=S)
    assert f.finished()
    for r in range(cfg.R):
        assert f.finish_iter[r] - f.admit_iter[r] + 1 == cfg.K * S
        assert not (f.gen[r] == cfg.mask_id).any()


# --------------------------------------------------------------------------
# DiLaServe threshold control (review, section 3.2)
# --------------------------------------------------------------------------
def test_rate_above_knots_and_limits():
    from oracle.control import rate_above
    f = [0.2, 0.4, 0.6, 0.7, 0.8, 0.5]          # min, q25, median, avg, q75, frac
    # the distribution passes through its knots
    assert rate_above(0.2, f) == 1.0
    assert rate_above(0.4, f) == 0.75
    assert rate_above(0.6, f) == 0.5
    assert rate_above(0.8, f) == 0.25
    assert rate_above(0.1, f) == 1.0 and rate_above(1.0, f) == 0.0
    # linear between knots: halfway from q25 to the median
    assert rate_above(0.5, f) == pytest.approx(0.625, abs=1e-15)
    # no unmasked position yet: uniform
    nan = [float("nan")] * 5 + [0.0]
    assert rate_above(0.7, nan) == pytest.approx(0.3, abs=1e-15)
    # never increases with the threshold
    ts = np.linspace(0, 1.2, 121)
    r = [rate_above(t, f) for t in ts]
    assert all(a >= b for a, b in zip(r, r[1:]))


def test_steps_to_clear_closed_forms():
    from oracle.control import steps_to_clear
    for m in range(0, 40):
        assert steps_to_clear(m, 0.0) == m          # the fallback alone: one per step
        assert steps_to_clear(m, 1.0) == (1 if m else 0)
    for k in range(0, 11):
        assert steps_to_clear(2 ** k, 0.5) == k + 1  # halving: 2^k, 2^(k-1), ..., 1, 0
    # by hand: 10 -3-> 7 -2-> 5 -1-> 4 -1-> 3 -1-> 2 -1-> 1 -1-> 0
    assert steps_to_clear(10, 0.3) == 7


def test_predict_steps_grows_with_the_threshold():
    from oracle.control import predict_steps_stub
    rng = np.random.default_rng(13)
    for _ in range(100):
        q = np.sort(rng.random(4))
        f = [q[0], q[1], q[2], float(q.mean()), q[3], 0.5]
        m, kb = int(rng.integers(0, 33)), int(rng.integers(0, 8))
        steps = [predict_steps_stub(t, f, m, kb, 32) for t in (0.5, 0.6, 0.7, 0.8, 0.9)]
        assert all(a <= b for a, b in zip(steps, steps[1:]))
        assert steps[0] >= (1 if m else 0) + kb


def test_predict_steps_stub_hand_values():
    """The stub's composition worked out by hand (a pin of the whole
    predictor, not of its parts alone).

    Case 1: t = 0.7, features (min .5, q25 .6, median .8, avg -, q75 .9, -),
    5 positions still masked, 2 blocks left, L = 4.
      rate_above: 0.7 lies in [q25, median) = [.6, .8):
        F = .25 + (.7 - .6) / (.8 - .6) * .25 = .375, so P = .625.
      current block, m = 5: take floor(3.125) = 3 -> 2; floor(1.25) = 1 -> 1;
        floor(.625) = 0, at least 1 -> 0: 3 steps.
      a full block, m = 4: floor(2.5) = 2 -> 2; 1 -> 1; 1 -> 0: 3 steps.
      total = 3 + 2 * 3 = 9.  (Counting the current block twice, or one
      full block too many, gives 12; leaving it out gives 6.)
    Case 2: nothing unmasked yet (NaN features) -> uniform: P = 1 - .5 = .5;
      8 masked, 3 blocks left, L = 8: 8 -> 4 -> 2 -> 1 -> 0 is 4 steps, a
      full block also 4: total = 4 + 3 * 4 = 16.
    Case 3: t above q75's segment, at .95 in [.9, 1): F = .75 + .5 * .25 =
      .875, P = .125; m = 3: floor(.375) = 0 -> 1 each step: 3 steps; no
      block left: total 3."""
    from oracle.control import predict_steps_stub
    f = [0.5, 0.6, 0.8, 0.7, 0.9, 0.25]
    assert predict_steps_stub(0.7, f, 5, 2, 4) == 9
    nan = [float("nan")] * 5 + [0.0]
    assert predict_steps_stub(0.5, nan, 8, 3, 8) == 16
    assert predict_steps_stub(0.95, f, 3, 0, 4) == 3


def test_load_control_hand_case():
    from oracle.control import load_control
    load = [[1, 2, 4], [1, 3, 5], [2, 2, 6]]
    # request 0: 0 + 4 + (1 + 2) = 7 <= 9 keeps the top; committed 4
    # request 1: 4 + 5 + 2 = 11 > 9 drops it, 4 + 3 + 2 = 9 keeps index 1; committed 7
    # request 2: 7 + 6 = 13 > 9, 7 + 2 = 9 keeps index 1
    assert load_control(load, 9.0).tolist() == [2, 1, 1]
    assert load_control(load, 1e9).tolist() == [2, 2, 2]
    assert load_control(load, 0.0).tolist() == [0, 0, 0]


def test_load_control_keeps_the_worst_case_within_capacity():
    from oracle.control import load_control
    rng = np.random.default_rng(14)
    for _ in range(200):
        R, T = int(rng.integers(1, 9)), int(rng.integers(1, 6))
        load = np.sort(rng.integers(1, 20, size=(R, T)), axis=1).astype(float)
        cap = float(rng.integers(int(load[:, 0].sum()), int(load[:, -1].sum()) + 2))
        keep = load_control(load, cap)
        # the all-lowest plan fits, so the chosen plan fits ...
        assert sum(load[i, keep[i]] for i in range(R)) <= cap
        # ... and raising the first request that is not at its top by one
        # step breaks the worst case at its turn
        for i in range(R):
            if keep[i] < T - 1:
                committed = sum(load[j, keep[j]] for j in range(i))
                assert committed + load[i, keep[i] + 1] + load[i + 1:, 0].sum() > cap
                break


def test_slo_threshold_hand_cases():
    from oracle.control import slo_threshold
    steps = [10, 20, 40]
    assert slo_threshold(steps, 0.01, 0.25) == 1          # 0.4 s > 0.25 s, 0.2 s fits
    assert slo_threshold(steps, 0.01, 1.0) == 2
    assert slo_threshold(steps, 0.01, 1.0, max_allowed=0) == 0
    assert slo_threshold(steps, 0.01, 0.05) == 0          # nothing fits: the fastest


# --------------------------------------------------------------------------
# Vocabulary-sharded S2 (triples and their merge)
# --------------------------------------------------------------------------
def test_merged_shard_triples_equal_the_whole_row():
    # exp(a - M) = exp(a - m) exp(m - M): the shards' sums rescaled to the
    # global max add up to the whole row's sum, and the first shard holding
    # the max holds its lowest index
    rng = np.random.default_rng(16)
    for _ in range(200):
        V = int(rng.integers(2, 300))
        x = oracle.bf16_to_f64(synth.f32_to_bf16_bits(rng.normal(size=V).astype(np.float32) * 2))
        if rng.random() < 0.3:                       # a tie across shards
            x[int(rng.integers(0, V))] = x.max()
        cuts = sorted(set(rng.integers(1, V, size=int(rng.integers(0, 4))).tolist()))
        bounds = [0] + cuts + [V]
        tr = [oracle.shard_triple(x[bounds[k]:bounds[k + 1]], bounds[k]) for k in range(len(bounds) - 1)]
        conf, lse, tok = oracle.merge_triples(tr)
        c0, l0, t0 = oracle.row_stats(x)
        assert tok == t0
        assert conf == pytest.approx(c0, rel=1e-12)
        assert lse == pytest.approx(l0, rel=1e-12, abs=1e-12)
    # one shard is the row itself
    x = np.array([0.5, 2.0, 2.0, -1.0])
    m, s, i = oracle.shard_triple(x, 0)
    assert (m, i) == (2.0, 1) and 1.0 / s == pytest.approx(oracle.row_stats(x)[0], rel=1e-15)


def test_step_sharded_equals_step():
    cfg = synth.StepConfig("sh", 4, 8, 200, 6.0, "fraction", (0.5, 0.7, 0.9))
    inp = synth.make_step_state(cfg, 2)
    rows = np.flatnonzero(inp.masked.reshape(-1))
    logits = np.full((cfg.B * cfg.L, cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    synth.fill_logits_rows(logits, cfg.V, rows, synth.step_row_keys(inp, rows), cfg.offset_max, cfg.mask_id)
    ref = oracle.step(logits, cfg.V, inp.input_ids, inp.thr, inp.conf_state, cfg.mask_id)
    got = oracle.step_sharded(logits, cfg.V, [0, 64, 136, 200], inp.input_ids, inp.thr, inp.conf_state, cfg.mask_id)
    for k in ("input_ids", "done", "n_new", "accept_len", "tok"):
        np.testing.assert_array_equal(got[k], ref[k])
    np.testing.assert_allclose(got["conf"], ref["conf"], rtol=1e-12, equal_nan=True)
