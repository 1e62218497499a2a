"""GPU parity of dllm_step / dllm_features against the CPU oracle, through
the C ABI (Python binding).

Bar: tokens, selections, input_ids, done, accept_len and n_new bit-exact;
confidences, conf_state and features within 1e-5 absolute, lse within
1e-5 * max(1, |lse|).  Cases carry 1e-4 decision margins (tests/helpers.py).
"""
import numpy as np
import pytest

import synth
from helpers import (CONF_TOL, compare_step, device_logits, device_logits_compact, device_state, enforce_margins,
                     oracle_step)

pytestmark = pytest.mark.gpu

SMALL_CASES = {
    "tiny": synth.STEP_CONFIGS["tiny"],
    # three reduction chunks, a partial last copy and a partial last vector;
    # row stride wider than V
    "ragged": synth.StepConfig("ragged", 8, 32, 40001, 12.0, "fraction", synth.THRESHOLD_SET, ldv=40016),
    # two positions per lane in the request finisher
    "l64": synth.StepConfig("l64", 16, 64, 33000, 12.0, "fraction", synth.THRESHOLD_SET),
    "l1": synth.StepConfig("l1", 5, 1, 9, 4.0, "half", (0.5,)),
    "wide_block": synth.StepConfig("wide_block", 2, 1024, 300, 8.0, "fraction", (0.7,)),
    "v_small": synth.StepConfig("v_small", 7, 8, 13, 6.0, "fraction", synth.THRESHOLD_SET),
    "all_masked": synth.StepConfig("all_masked", 6, 32, 20000, 12.0, "all", synth.THRESHOLD_SET),
}


def run_gpu(dllm, inp, device, **kw):
    logits = device_logits(inp, device)
    ids, thr, cs = device_state(inp, device)
    out = dllm.step(logits, ids, thr, cs, V=inp.cfg.V, mask_id=inp.cfg.mask_id, debug=True, **kw)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    return got, ids.cpu().numpy(), cs.cpu().numpy()


@pytest.fixture(scope="module")
def device(dllm):
    import torch
    return torch.device("cuda", 0)


@pytest.mark.parametrize("name", sorted(SMALL_CASES))
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_step_parity_small(dllm, device, name, seed):
    cfg = SMALL_CASES[name]
    inp = synth.make_step_state(cfg, seed)
    enforce_margins(inp)
    ref = oracle_step(inp)
    got, ids, cs = run_gpu(dllm, inp, device)
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)


@pytest.mark.parametrize("name", ["llada", "dream", "stress"])
def test_step_parity_full_size(dllm, device, name):
    """The full-size LLaDA-, Dream- and stress-shaped batches: every request's
    outputs against the oracle (computed request by request on the host's
    cores), plus the invariants of the step over the whole batch."""
    cfg = synth.STEP_CONFIGS[name]
    inp = synth.make_step_state(cfg, 7)
    enforce_margins(inp)
    ref = oracle_step(inp)
    got, ids, cs = run_gpu(dllm, inp, device)
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)
    # invariants (FDFO page, section "工程设计一"; DiLaServe review, section 3.1)
    m_in = inp.masked
    m_out = ids == cfg.mask_id
    assert not (m_out & ~m_in).any()                       # unmasked count never falls
    assert np.array_equal(got["n_new"], (m_in & ~m_out).sum(axis=1))
    assert np.array_equal(got["done"], (~m_out.any(axis=1)).astype(np.uint8))
    assert np.array_equal(got["accept_len"], np.where(got["done"] == 1, cfg.L, 0))
    has = m_in.any(axis=1)
    assert (got["n_new"][has] >= 1).all()                  # at least one per incomplete block
    chg = m_in & ~m_out
    assert np.array_equal(ids[chg], got["tok"][chg])
    assert ((got["conf"][m_in] > 0) & (got["conf"][m_in] <= 1.0 + 1e-6)).all()


def test_thresholds_zero_and_above_one(dllm, device):
    cfg = SMALL_CASES["ragged"]
    inp = synth.make_step_state(cfg, 11)
    inp.thr[:] = 0.0
    got, ids, _ = run_gpu(dllm, inp, device)
    assert not (ids == cfg.mask_id).any()
    assert (got["done"] == 1).all()
    inp.thr[:] = 1.5
    enforce_margins(inp)
    ref = oracle_step(inp)
    got, ids, cs = run_gpu(dllm, inp, device)
    assert np.array_equal(got["n_new"], inp.masked.any(axis=1).astype(np.int32))
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)


def test_batch_invariance(dllm, device):
    """A request's results are bit-identical alone or inside any batch."""
    cfg = synth.StepConfig("inv", 12, 32, 70000, 12.0, "fraction", synth.THRESHOLD_SET)
    inp = synth.make_step_state(cfg, 5)
    full, ids_full, cs_full = run_gpu(dllm, inp, device)
    for sub in ([3], [0, 7], [11, 2, 5]):
        part = synth.StepInputs(cfg, inp.seed, inp.input_ids[sub].copy(), inp.thr[sub].copy(),
                                inp.conf_state[sub].copy(), inp.salt[sub].copy())
        # the sub-batch keeps each request's own logits rows
        import torch
        L = cfg.L
        rows = np.array([b * L + j for b in sub for j in range(L)])
        logits_full = device_logits(inp, device)
        logits = logits_full[torch.from_numpy(rows).to(device)].contiguous()
        ids, thr, cs = device_state(part, device)
        out = dllm.step(logits, ids, thr, cs, V=cfg.V, mask_id=cfg.mask_id, debug=True)
        for k in ("conf", "lse", "tok", "feats", "done", "n_new", "accept_len"):
            a = out[k].cpu().numpy()
            b = full[k][sub]
            assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                  b.view(np.uint32) if b.dtype == np.float32 else b), k
        assert np.array_equal(ids.cpu().numpy(), ids_full[sub])


def test_no_masked_position_anywhere(dllm, device):
    cfg = synth.StepConfig("none", 9, 32, 5000, 8.0, "half", (0.9,))
    inp = synth.make_step_state(cfg, 2)
    inp.input_ids[inp.masked] = 5
    inp.conf_state[np.isnan(inp.conf_state)] = 0.95
    ref = oracle_step(inp)
    got, ids, cs = run_gpu(dllm, inp, device)
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)
    assert (got["done"] == 1).all() and (got["n_new"] == 0).all()


def test_ties_and_negative_infinity(dllm, device):
    """Equal logits (argmax ties to the lowest index, conf = 1/V) and rows
    with -inf entries."""
    import torch
    V, L, B = 5000, 4, 2
    rows = np.zeros((B * L, V), dtype=np.float32)
    rows[1, :] = 0.5                      # all equal: tok 0, conf 1/V
    rows[2, 100] = rows[2, 4000] = 3.0    # tie between 100 and 4000
    rows[3, :2500] = -np.inf              # half of the row at -inf
    rows[3, 3000] = 1.0
    rows[5, 7] = 2.0
    rows[6, :] = -np.inf
    rows[6, 4999] = -1.0                  # single finite value, at the end
    bits = synth.f32_to_bf16_bits(rows)
    mask_id = V + 10                     # a token id no row predicts
    ids = np.full((B, L), mask_id, dtype=np.int32)
    cs = np.full((B, L), np.nan, dtype=np.float32)
    thr = np.array([0.0, 0.0], dtype=np.float32)
    import oracle
    ref = oracle.step(bits, V, ids, thr, cs, mask_id)
    d_logits = torch.from_numpy(np.ascontiguousarray(np.pad(bits, ((0, 0), (0, 8 - V % 8 if V % 8 else 0)))
                                                     .view(np.int16))).to(device)
    d_ids = torch.from_numpy(ids).to(device)
    d_cs = torch.from_numpy(cs).to(device)
    out = dllm.step(d_logits, d_ids, torch.from_numpy(thr).to(device), d_cs, V=V, mask_id=mask_id, debug=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare_step(ref, got, [0, 1], L, d_ids.cpu().numpy(), d_cs.cpu().numpy())
    assert got["tok"][0, 1] == 0 and got["tok"][0, 2] == 100 and got["tok"][1, 2] == 4999
    assert got["conf"][0, 1] == pytest.approx(1.0 / V, abs=CONF_TOL)


def test_workspace_reuse_across_shapes(dllm, device):
    """One workspace serves calls of different shapes back to back."""
    import torch
    big = synth.StepConfig("big", 40, 32, 60000, 12.0, "fraction", synth.THRESHOLD_SET)
    nbytes = dllm.step_workspace_size(big.B, big.L, big.V)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    shapes = [big, SMALL_CASES["tiny"], SMALL_CASES["l64"], big, SMALL_CASES["ragged"]]
    for k, cfg in enumerate(shapes):
        inp = synth.make_step_state(cfg, 20 + k)
        enforce_margins(inp)
        ref = oracle_step(inp)
        got, ids, cs = run_gpu(dllm, inp, device, workspace=ws)
        compare_step(ref, got, list(range(cfg.B)), cfg.L, ids, cs)


def test_features_kernel(dllm, device):
    import torch
    import oracle
    cfg = SMALL_CASES["l64"]
    inp = synth.make_step_state(cfg, 4)
    ids = torch.from_numpy(inp.input_ids).to(device)
    cs = torch.from_numpy(inp.conf_state).to(device)
    got = dllm.features(ids, cs, mask_id=cfg.mask_id).cpu().numpy()
    ref = oracle.features(inp.input_ids, inp.conf_state, cfg.mask_id)
    np.testing.assert_allclose(got, ref, rtol=0, atol=CONF_TOL, equal_nan=True)


@pytest.mark.parametrize("L", [1, 5, 31, 32, 33, 64, 100])
def test_features_kernel_adversarial_values(dllm, device, L):
    """S6 on values chosen to break a sort: ties (values drawn from a small
    set), negatives, signed zeros and tiny magnitudes, every mask density
    from none to all.  L <= 32 takes the one-warp sort, longer blocks the
    rank count.  The minimum is one of the values, so it must match
    exactly; the interpolated quantiles and the mean within 1e-5."""
    import torch
    import oracle
    rng = np.random.default_rng(100 + L)
    B, mask_id = 96, 7
    pool = np.array([-1.5, -0.25, -0.0, 0.0, 1e-40, 1e-30, 0.125, 0.5, 0.5000001, 1.0, 1.75], dtype=np.float32)
    cs = np.where(rng.random((B, L)) < 0.5, rng.choice(pool, (B, L)),
                  rng.uniform(-2.0, 2.0, (B, L))).astype(np.float32)
    frac = np.concatenate([[0.0, 1.0], rng.random(B - 2)])
    ids = np.where(rng.random((B, L)) < frac[:, None], mask_id, 3).astype(np.int32)
    got = dllm.features(torch.from_numpy(ids).to(device), torch.from_numpy(cs).to(device),
                        mask_id=mask_id).cpu().numpy()
    ref = oracle.features(ids, cs, mask_id)
    np.testing.assert_array_equal(got[:, 0], ref[:, 0].astype(np.float32))
    np.testing.assert_allclose(got, ref, rtol=0, atol=CONF_TOL, equal_nan=True)


def test_repeated_steps_to_completion(dllm, device):
    """Step the same batch with fresh logits each step until every block is
    done; the oracle follows in lockstep."""
    import oracle
    cfg = synth.StepConfig("rep", 6, 32, 9000, 12.0, "fraction", synth.THRESHOLD_SET)
    inp = synth.make_step_state(cfg, 9)
    ids_d, thr_d, cs_d = device_state(inp, device)
    for step_no in range(40):
        inp.seed = 9 + 1000 * (step_no + 1)        # new logits per step
        inp.salt[:] = 0
        inp.input_ids = ids_d.cpu().numpy()
        inp.conf_state = cs_d.cpu().numpy()
        if not inp.masked.any():
            break
        enforce_margins(inp)
        ref = oracle_step(inp)
        logits = device_logits(inp, device)
        out = dllm.step(logits, ids_d, thr_d, cs_d, V=cfg.V, mask_id=cfg.mask_id, debug=True)
        got = {k: v.cpu().numpy() for k, v in out.items()}
        compare_step(ref, got, list(range(cfg.B)), cfg.L, ids_d.cpu().numpy(), cs_d.cpu().numpy())
    assert not (ids_d.cpu().numpy() == cfg.mask_id).any()



@pytest.mark.parametrize("name", ["tiny", "ragged", "l64", "all_masked", "v_small"])
def test_compact_logits_parity_and_identity(dllm, device, name):
    """dllm_step_compact (logits of the masked positions only, by rank)
    equals the oracle and is bit-identical to dllm_step on the full
    layout."""
    cfg = SMALL_CASES[name]
    inp = synth.make_step_state(cfg, 4)
    enforce_margins(inp)
    ref = oracle_step(inp)
    full, ids_f, cs_f = run_gpu(dllm, inp, device)
    logits = device_logits_compact(inp, device, extra_rows=3)
    ids, thr, cs = device_state(inp, device)
    out = dllm.step(logits, ids, thr, cs, V=cfg.V, mask_id=cfg.mask_id, debug=True, compact=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids.cpu().numpy(), cs.cpu().numpy())
    for k in ("conf", "lse", "tok", "feats", "done", "n_new", "accept_len"):
        a, b = got[k], full[k]
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                              b.view(np.uint32) if b.dtype == np.float32 else b), k
    assert np.array_equal(ids.cpu().numpy(), ids_f)


def test_compact_logits_full_size(dllm, device):
    cfg = synth.STEP_CONFIGS["dream"]
    inp = synth.make_step_state(cfg, 8)
    sample = list(range(cfg.B))
    enforce_margins(inp)
    ref = oracle_step(inp)
    logits = device_logits_compact(inp, device)
    ids, thr, cs = device_state(inp, device)
    out = dllm.step(logits, ids, thr, cs, V=cfg.V, mask_id=cfg.mask_id, debug=True, compact=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, sample, cfg.L, ids.cpu().numpy(), cs.cpu().numpy())


def test_compact_logits_too_few_rows_is_reported(dllm, device):
    """Fewer logits rows than masked positions: nothing is read, the device
    error word says so, and the workspace serves the next call."""
    cfg = SMALL_CASES["ragged"]
    inp = synth.make_step_state(cfg, 6)
    M = int(inp.masked.sum())
    assert M > 2
    logits = device_logits_compact(inp, device)[: M - 2].contiguous()
    ids, thr, cs = device_state(inp, device)
    dllm.step(logits, ids, thr, cs, V=cfg.V, mask_id=cfg.mask_id, compact=True)
    assert dllm.get_device_error(device) == 4          # DLLM_DEVERR_LOGITS_ROWS
    enforce_margins(inp)
    ref = oracle_step(inp)
    got, ids2, cs2 = run_gpu(dllm, inp, device)
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids2, cs2)


@pytest.mark.parametrize("name,bounds", [("ragged", [0, 16000, 40001]), ("l64", [0, 8, 4096, 20000, 33000]),
                                         ("all_masked", [0, 20000]), ("tiny", [0, 512, 1024])])
def test_vocab_sharded_step(dllm, device, name, bounds):
    """dllm_step_shard over vocabulary shards of one logits array, then
    dllm_step_merge: equal to the oracle (tokens exact, confidences within
    1e-5) and to the unsharded step's tokens."""
    cfg = SMALL_CASES[name] if name in SMALL_CASES else synth.STEP_CONFIGS[name]
    inp = synth.make_step_state(cfg, 13)
    enforce_margins(inp)
    ref = oracle_step(inp)
    full, ids_f, _ = run_gpu(dllm, inp, device)
    logits = device_logits(inp, device)
    ids, thr, cs = device_state(inp, device)
    out = dllm.step_sharded(logits, ids, thr, cs, V=cfg.V, mask_id=cfg.mask_id, bounds=bounds, debug=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids.cpu().numpy(), cs.cpu().numpy())
    assert np.array_equal(got["tok"], full["tok"]) and np.array_equal(ids.cpu().numpy(), ids_f)


def test_vocab_sharded_dream_full_size(dllm, device):
    cfg = synth.STEP_CONFIGS["dream"]
    inp = synth.make_step_state(cfg, 14)
    sample = list(range(cfg.B))
    enforce_margins(inp)
    ref = oracle_step(inp)
    logits = device_logits(inp, device)
    ids, thr, cs = device_state(inp, device)
    # four shards of a tensor-parallel LM head (V / 4 rounded to 8)
    out = dllm.step_sharded(logits, ids, thr, cs, V=cfg.V, mask_id=cfg.mask_id,
                            bounds=[0, 37984, 75968, 113952, cfg.V], debug=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, sample, cfg.L, ids.cpu().numpy(), cs.cpu().numpy())


def test_steps_on_two_streams_with_their_own_workspaces(dllm, device):
    """Two batches stepped concurrently on two streams, each with its own
    workspace, give the same results as one after the other."""
    import torch
    cases = [synth.make_step_state(SMALL_CASES["ragged"], 21), synth.make_step_state(SMALL_CASES["l64"], 22)]
    for inp in cases:
        enforce_margins(inp)
    refs = [oracle_step(inp) for inp in cases]
    streams = [torch.cuda.Stream(device=device) for _ in cases]
    state = []
    for inp, st in zip(cases, streams):
        logits = device_logits(inp, device)
        ids, thr, cs = device_state(inp, device)
        ws = torch.zeros(dllm.step_workspace_size(inp.cfg.B, inp.cfg.L, inp.cfg.V), dtype=torch.uint8, device=device)
        state.append((inp, logits, ids, thr, cs, ws, st))
    torch.cuda.synchronize()
    outs = []
    for inp, logits, ids, thr, cs, ws, st in state:
        with torch.cuda.stream(st):
            outs.append(dllm.step(logits, ids, thr, cs, V=inp.cfg.V, mask_id=inp.cfg.mask_id, debug=True,
                                  workspace=ws))
    torch.cuda.synchronize()
    assert dllm.get_device_error(device) == 0
    for (inp, logits, ids, thr, cs, ws, st), out, ref in zip(state, outs, refs):
        got = {k: v.cpu().numpy() for k, v in out.items()}
        compare_step(ref, got, list(range(inp.cfg.B)), inp.cfg.L, ids.cpu().numpy(), cs.cpu().numpy())


def test_steps_from_several_host_threads(dllm, device):
    """Four host threads call the step at once, each on its own stream with
    its own workspace and batch shape (so the library's per-device launch
    state is read and grown concurrently); every result equals the
    oracle's."""
    import threading
    import torch
    names = ["ragged", "l64", "tiny", "all_masked"]
    cases = [synth.make_step_state(SMALL_CASES[n], 40 + k) for k, n in enumerate(names)]
    for inp in cases:
        enforce_margins(inp)
    refs = [oracle_step(inp) for inp in cases]
    prepared = []
    for inp in cases:
        logits = device_logits(inp, device)
        ids, thr, cs = device_state(inp, device)
        ws = torch.zeros(dllm.step_workspace_size(inp.cfg.B, inp.cfg.L, inp.cfg.V), dtype=torch.uint8, device=device)
        prepared.append((inp, logits, ids, thr, cs, ws, torch.cuda.Stream(device=device)))
    torch.cuda.synchronize()
    start = threading.Barrier(len(prepared))
    outs, errors = [None] * len(prepared), []

    def run(k):
        inp, logits, ids, thr, cs, ws, st = prepared[k]
        try:
            start.wait()
            with torch.cuda.stream(st):
                for _ in range(3):   # the last call's outputs are checked; ids/cs move on each call
                    ids.copy_(torch.from_numpy(inp.input_ids).to(device))
                    cs.copy_(torch.from_numpy(inp.conf_state).to(device))
                    outs[k] = dllm.step(logits, ids, thr, cs, V=inp.cfg.V, mask_id=inp.cfg.mask_id, debug=True,
                                        workspace=ws)
            st.synchronize()
        except Exception as e:   # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(k,)) for k in range(len(prepared))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert dllm.get_device_error(device) == 0
    for (inp, logits, ids, thr, cs, ws, st), out, ref in zip(prepared, outs, refs):
        got = {k: v.cpu().numpy() for k, v in out.items()}
        compare_step(ref, got, list(range(inp.cfg.B)), inp.cfg.L, ids.cpu().numpy(), cs.cpu().numpy())


def test_pipeline_captured_in_a_cuda_graph(dllm, device):
    """pack, step and the fused commit/compaction (launched as programmatic
    dependents) captured in a CUDA graph: a replay equals eager execution."""
    import ctypes
    import torch
    import bench
    cfg, inp, reqs, b, gen, pending_p = bench.make_workload(31, "tiny")
    results = []
    for use_graph in (False, True):
        pipe = bench.Pipeline(cfg, inp, reqs, b, gen, pending_p, device, ring=2)
        lib = pipe.lib
        stream = torch.cuda.Stream(device=device)
        sh = ctypes.c_void_p(stream.cuda_stream)
        pa, sa, aa, ca = pipe.args[0]

        def body():
            rc = lib.dllm_pack(ctypes.byref(pa), sh)
            rc |= lib.dllm_step(ctypes.byref(sa), sh)
            rc |= lib.dllm_advance_compact(ctypes.byref(aa), ctypes.byref(ca), sh)
            assert rc == 0

        with torch.cuda.stream(stream):
            body()                        # first calls: per-device set-up outside any capture
            torch.cuda.synchronize()
            pipe.restore()
            torch.cuda.synchronize()
            if use_graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    body()
                pipe.restore()
                torch.cuda.synchronize()
                g.replay()
            else:
                body()
        torch.cuda.synchronize()
        assert dllm.get_device_error(device) == 0
        results.append((pipe.state[0].cpu().numpy(), pipe.done[0].cpu().numpy(), pipe.box_ids.cpu().numpy()))
    for a, b2 in zip(results[0], results[1]):
        np.testing.assert_array_equal(a, b2)


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


@pytest.mark.parametrize("name,bounds", [("ragged", [0, 16000, 40001]), ("l64", [0, 8, 4096, 20000, 33000]),
                                         ("all_masked", [0, 20000]), ("tiny", [0, 512, 1024])])
def test_vocab_shards_in_one_launch(dllm, device, name, bounds):
    """dllm_step_vocab_shards over views of one logits array: bit for bit the
    per-shard launches plus the merge, and the oracle within tolerance."""
    cfg = SMALL_CASES[name] if name in SMALL_CASES else synth.STEP_CONFIGS[name]
    inp = synth.make_step_state(cfg, 13)
    enforce_margins(inp)
    ref = oracle_step(inp)
    logits = device_logits(inp, device)
    ids_a, thr, cs_a = device_state(inp, device)
    multi = dllm.step_sharded(logits, ids_a, thr, cs_a, V=cfg.V, mask_id=cfg.mask_id, bounds=bounds, debug=True)
    ids_b, _, cs_b = device_state(inp, device)
    # each shard a column slice of the one array: its first column at v0, the array's row stride
    shards = [(logits[:, v0:v1], v0, v1 - v0) for v0, v1 in zip(bounds[:-1], bounds[1:])]
    out = dllm.step_vocab_shards(shards, ids_b, thr, cs_b, mask_id=cfg.mask_id, debug=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    want = {k: v.cpu().numpy() for k, v in multi.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids_b.cpu().numpy(), cs_b.cpu().numpy())
    m = inp.masked
    for k in ("tok", "conf", "lse"):
        assert np.array_equal(_bits(got[k][m]), _bits(want[k][m])), k
    for k in ("done", "accept_len", "n_new", "feats"):
        assert np.array_equal(_bits(got[k]), _bits(want[k])), k
    assert np.array_equal(ids_b.cpu().numpy(), ids_a.cpu().numpy())
    assert np.array_equal(_bits(cs_b.cpu().numpy()), _bits(cs_a.cpu().numpy()))


@pytest.mark.parametrize("widths", [[40001], [5, 40000 - 5 - 3, 3, 1], [5000] * 7 + [5001], [2047, 2049, 35905]])
@pytest.mark.parametrize("fixed_steps", [False, True])
def test_vocab_shards_in_separate_buffers(dllm, device, widths, fixed_steps):
    """Shards in buffers of their own, of any width (a shard narrower than one
    2048-element batch, one of a single token, eight shards), each with its
    own row stride: equal to the oracle under either selection rule."""
    import torch
    cfg = SMALL_CASES["ragged"]
    assert sum(widths) == cfg.V
    inp = synth.make_step_state(cfg, 21)
    quota = None
    if fixed_steps:
        quota = np.random.default_rng(22).integers(0, cfg.L + 1, size=cfg.B).astype(np.int32)
    enforce_margins(inp, quota=quota)
    ref = oracle_step(inp, quota=quota)
    full = device_logits(inp, device)
    shards, v0 = [], 0
    for w in widths:
        ldv = -(-w // 8) * 8 + 8                       # a stride of its own, wider than the shard
        t = torch.full((cfg.B * cfg.L, ldv), -1, dtype=torch.int16, device=device)
        t[:, :w] = full[:, v0:v0 + w]
        shards.append((t, v0, w))
        v0 += w
    ids, thr, cs = device_state(inp, device)
    out = dllm.step_vocab_shards(shards, ids, thr, cs, mask_id=cfg.mask_id, debug=True,
                                 quota=None if quota is None else torch.from_numpy(quota).to(device))
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids.cpu().numpy(), cs.cpu().numpy())


def test_vocab_shards_in_one_launch_dream_full_size(dllm, device):
    """The Dream-shaped batch over four shards of a tensor-parallel LM head
    in one launch: every request against the oracle."""
    cfg = synth.STEP_CONFIGS["dream"]
    inp = synth.make_step_state(cfg, 15)
    enforce_margins(inp)
    ref = oracle_step(inp)
    logits = device_logits(inp, device)
    bounds = [0, 37984, 75968, 113952, cfg.V]
    import torch
    shards = []
    for v0, v1 in zip(bounds[:-1], bounds[1:]):
        t = torch.empty((cfg.B * cfg.L, -(-(v1 - v0) // 8) * 8), dtype=torch.int16, device=device)
        t[:, :v1 - v0] = logits[:, v0:v1]
        shards.append((t, v0, v1 - v0))
    ids, thr, cs = device_state(inp, device)
    out = dllm.step_vocab_shards(shards, ids, thr, cs, mask_id=cfg.mask_id, debug=True)
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert dllm.get_device_error(device) == 0
    compare_step(ref, got, list(range(cfg.B)), cfg.L, ids.cpu().numpy(), cs.cpu().numpy())
