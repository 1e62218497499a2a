"""dllm_step_commit: the step with the FDFO block commit and the stable
compaction in the same launch.

Against the oracle (step, then oracle.loop.advance with the done flags as
the advance flags, then oracle.compact) and, element for element, against
the two-launch path it replaces (dllm_step, then dllm_advance_compact with
advance = done): every output, the eviction flags, the compaction maps, the
compacted arrays, the block indices and the committed tokens.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import compare_step, device_logits, device_logits_compact, enforce_margins, oracle_step
from oracle.loop import advance as oracle_advance

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": synth.StepConfig("ragged", 8, 32, 40001, 12.0, "fraction", synth.THRESHOLD_SET, ldv=40016),
    "dream_like": synth.StepConfig("dream_like", 48, 32, 20000, 12.0, "fraction", synth.THRESHOLD_SET),
    "l64": synth.StepConfig("l64", 16, 64, 33000, 12.0, "fraction", synth.THRESHOLD_SET),
    "all_masked": synth.StepConfig("all_masked", 6, 32, 9000, 12.0, "all", synth.THRESHOLD_SET),
    # more rows than one 480-row compaction chunk
    "many_rows": synth.StepConfig("many_rows", 600, 8, 3000, 8.0, "fraction", synth.THRESHOLD_SET),
}


# cases whose batch also carries a 5-byte row array (moved byte by byte,
# beside the 16-byte and 4-byte elements of the others)
WITH_BYTES = {"ragged", "many_rows"}


@pytest.fixture(scope="module")
def device(dllm):
    import torch
    return torch.device("cuda", 0)


def _batch(cfg, seed, quota=None):
    """Step inputs with margins (for the fixed-steps rule when ``quota`` is
    given) plus the rows' commit state: request ids (a permutation), blocks K
    in 1..4, current block b < K, and committed tokens of the earlier
    blocks."""
    inp = synth.make_step_state(cfg, seed)
    enforce_margins(inp, quota=quota)
    rng = np.random.default_rng(seed + 100)
    B, L = cfg.B, cfg.L
    K = rng.integers(1, 5, size=B).astype(np.int32)
    b = np.array([rng.integers(0, k) for k in K], dtype=np.int32)
    rid = rng.permutation(B).astype(np.int32)
    ld_gen = 4 * L
    gen = rng.integers(0, cfg.V - 2, size=(B, ld_gen)).astype(np.int32)
    return inp, rid, K, b, gen, ld_gen


def _expected(cfg, inp, rid, K, b, gen, quota=None):
    ref = oracle_step(inp, quota=quota)
    L = cfg.L
    ids = ref["input_ids"].copy()
    cs = ref["conf_state"].copy()
    bb = b.astype(np.int64).copy()
    o_gen = {int(r): gen[int(r)][: b[i] * L].astype(np.int64) for i, r in enumerate(rid)}
    evict = oracle_advance(ref["done"].astype(bool), rid, bb, K, ids, cs, o_gen, cfg.mask_id)
    new_index, src_row, A_out = oracle.compact(evict)
    return ref, dict(ids=ids, cs=cs, b=bb, gen=o_gen, evict=evict, new_index=new_index, src_row=src_row, A_out=A_out)


def _device_run(dllm, device, cfg, inp, rid, K, b, gen, ld_gen, fused, extra=None, bounds=None, quota=None,
                compact_logits=False):
    """One step with its commit and compaction on the device: in one launch
    (fused) or as the step then dllm_advance_compact; over vocabulary shards
    [bounds[k], bounds[k+1]) of the logits (column slices) when bounds is
    given; under the fixed-steps rule when ``quota`` [B] is given; reading
    the masked positions' rows only (plus three spare rows) when
    ``compact_logits``."""
    import torch
    lib = dllm.load()
    B, L = cfg.B, cfg.L
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(device)
    logits = device_logits_compact(inp, device, extra_rows=3) if compact_logits else device_logits(inp, device)
    rows = logits.shape[0] if compact_logits else -1
    d_quota = None if quota is None else t(np.asarray(quota, dtype=np.int32))
    q_ptr = None if d_quota is None else ctypes.c_void_p(d_quota.data_ptr())
    ids, thr, cs = t(inp.input_ids), t(inp.thr), t(inp.conf_state)
    d_rid, d_K, d_b, d_gen = t(rid), t(K), t(b), t(gen)
    p_arr = t(np.arange(B, dtype=np.int32) * 7)         # a row array the batch carries along
    out = {
        "done": torch.empty(B, dtype=torch.uint8, device=device),
        "accept_len": torch.empty(B, dtype=torch.int32, device=device),
        "n_new": torch.empty(B, dtype=torch.int32, device=device),
        "feats": torch.empty((B, 6), dtype=torch.float32, device=device),
        "conf": torch.empty((B, L), dtype=torch.float32, device=device),
        "lse": torch.empty((B, L), dtype=torch.float32, device=device),
        "tok": torch.empty((B, L), dtype=torch.int32, device=device),
    }
    evict = torch.full((B,), 7, dtype=torch.uint8, device=device)
    new_index = torch.full((B,), -9, dtype=torch.int32, device=device)
    src_row = torch.full((B,), -9, dtype=torch.int32, device=device)
    A_out = torch.full((1,), -9, dtype=torch.int32, device=device)
    n_sh = 1 if bounds is None else len(bounds) - 1
    ws = torch.zeros(lib.dllm_step_workspace_size(B, L, cfg.V + 8192 * (n_sh - 1)), dtype=torch.uint8,
                     device=device)
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())
    sa = dllm.StepArgs(B=B, L=L, V=cfg.V, mask_id=cfg.mask_id, ldv=logits.shape[1], logits=ptr(logits),
                       input_ids=ptr(ids), thr=ptr(thr), conf_state=ptr(cs), done=ptr(out["done"]),
                       accept_len=ptr(out["accept_len"]), n_new=ptr(out["n_new"]), feats=ptr(out["feats"]),
                       conf_out=ptr(out["conf"]), lse_out=ptr(out["lse"]), tok_out=ptr(out["tok"]),
                       workspace=ptr(ws), workspace_bytes=ws.numel())
    aa = dllm.AdvanceArgs(A=B, L=L, mask_id=cfg.mask_id, advance=ptr(out["done"]), rid=ptr(d_rid), K=ptr(d_K),
                          b=ptr(d_b), input_ids=ptr(ids), conf_state=ptr(cs), gen_tokens=ptr(d_gen), ld_gen=ld_gen,
                          evict=ptr(evict))
    arrays = [ids, cs, thr, d_b, d_K, d_rid, p_arr]
    rb = [L * 4, L * 4, 4, 4, 4, 4, 4]
    d_extra = None
    if extra is not None:
        d_extra = t(extra)
        arrays.append(d_extra)
        rb.append(extra.shape[1])
    arr = (ctypes.c_void_p * dllm.COMPACT_MAX_ARRAYS)(*[x.data_ptr() for x in arrays])
    rbs = (ctypes.c_int64 * dllm.COMPACT_MAX_ARRAYS)(*rb)
    cws = torch.empty(lib.dllm_compact_workspace_size(B, len(rb), ctypes.cast(rbs, ctypes.c_void_p)),
                      dtype=torch.uint8, device=device)
    ca = dllm.CompactArgs(A=B, n_arrays=len(arrays), evict=ptr(evict), new_index=ptr(new_index),
                          src_row=ptr(src_row), A_out=ptr(A_out), arrays=arr, row_bytes=rbs, workspace=ptr(cws),
                          workspace_bytes=cws.numel())
    stream = ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if bounds is not None:
        shards = (dllm.VocabShard * n_sh)()
        for k in range(n_sh):
            shards[k] = dllm.VocabShard(logits=ctypes.c_void_p(logits.data_ptr() + 2 * bounds[k]),
                                        ldv=logits.shape[1], v0=bounds[k], V=bounds[k + 1] - bounds[k])
        if fused:
            rc = lib.dllm_step_vocab_shards_commit(ctypes.byref(sa), n_sh, shards, q_ptr, ctypes.byref(aa),
                                                   ctypes.byref(ca), stream)
            assert rc == 0, lib.dllm_strerror(rc)
        else:
            assert lib.dllm_step_vocab_shards(ctypes.byref(sa), n_sh, shards, q_ptr, stream) == 0
            assert lib.dllm_advance_compact(ctypes.byref(aa), ctypes.byref(ca), stream) == 0
    elif fused:
        rc = lib.dllm_step_commit(ctypes.byref(sa), q_ptr, rows, ctypes.byref(aa), ctypes.byref(ca), stream)
        assert rc == 0, lib.dllm_strerror(rc)
    else:
        if compact_logits:
            assert lib.dllm_step_compact(ctypes.byref(sa), rows, q_ptr, stream) == 0
        elif quota is not None:
            assert lib.dllm_step_quota(ctypes.byref(sa), q_ptr, stream) == 0
        else:
            assert lib.dllm_step(ctypes.byref(sa), stream) == 0
        assert lib.dllm_advance_compact(ctypes.byref(aa), ctypes.byref(ca), stream) == 0
    h = {k: v.cpu().numpy() for k, v in out.items()}
    h.update(ids=ids.cpu().numpy(), cs=cs.cpu().numpy(), thr=thr.cpu().numpy(), b=d_b.cpu().numpy(),
             K=d_K.cpu().numpy(), rid=d_rid.cpu().numpy(), p=p_arr.cpu().numpy(), gen=d_gen.cpu().numpy(),
             evict=evict.cpu().numpy(), new_index=new_index.cpu().numpy(), src_row=src_row.cpu().numpy(),
             A_out=int(A_out.cpu().numpy()[0]), extra=None if d_extra is None else d_extra.cpu().numpy())
    assert dllm.get_device_error(device) == 0
    return h


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("seed", [0, 1])
def test_step_commit_matches_oracle_and_the_two_launch_path(dllm, device, name, seed):
    _check_commit(dllm, device, name, seed, None)


# vocabulary shards (multiples of 8 wide, but the last): one launch against
# the oracle and against dllm_step_vocab_shards then dllm_advance_compact
SHARD_BOUNDS = {"ragged": [0, 8, 20000, 40001], "dream_like": [0, 4096, 12000, 20000],
                "l64": [0, 33000], "all_masked": [0, 4000, 9000], "many_rows": [0, 1024, 2048, 3000]}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("quota_rule", [False, True])
def test_vocab_shards_commit_matches_oracle_and_the_two_launch_path(dllm, device, name, quota_rule):
    _check_commit(dllm, device, name, 3, SHARD_BOUNDS[name], quota_rule=quota_rule)


# the fixed-steps rule, the compact logits layout (masked rows only), and both
@pytest.mark.parametrize("name", ["ragged", "l64", "many_rows"])
@pytest.mark.parametrize("variant", ["quota", "compact", "compact_quota"])
def test_step_commit_quota_and_compact_logits(dllm, device, name, variant):
    _check_commit(dllm, device, name, 5, None, quota_rule="quota" in variant, compact_logits="compact" in variant)


def _check_commit(dllm, device, name, seed, bounds, quota_rule=False, compact_logits=False):
    cfg = CASES[name]
    quota = (np.random.default_rng(seed + 300).integers(0, cfg.L + 1, size=cfg.B).astype(np.int32)
             if quota_rule else None)
    inp, rid, K, b, gen, ld_gen = _batch(cfg, seed, quota=quota)
    ref, exp = _expected(cfg, inp, rid, K, b, gen, quota=quota)
    extra = (np.random.default_rng(seed + 200).integers(0, 255, (cfg.B, 5)).astype(np.uint8)
             if name in WITH_BYTES else None)
    kw = dict(extra=extra, bounds=bounds, quota=quota, compact_logits=compact_logits)
    got = _device_run(dllm, device, cfg, inp, rid, K, b, gen, ld_gen, fused=True, **kw)
    two = _device_run(dllm, device, cfg, inp, rid, K, b, gen, ld_gen, fused=False, **kw)
    B, L = cfg.B, cfg.L
    # the step's own outputs against the oracle (its ids / conf_state are
    # checked after the commit below)
    compare_step(ref, got, list(range(B)), L, ref["input_ids"], ref["conf_state"].astype(np.float32))
    # commit and compaction against the oracle
    A = exp["A_out"]
    assert got["A_out"] == A
    np.testing.assert_array_equal(got["evict"].astype(bool), exp["evict"])
    np.testing.assert_array_equal(got["new_index"], exp["new_index"])
    np.testing.assert_array_equal(got["src_row"][:A], exp["src_row"])
    src = exp["src_row"]
    np.testing.assert_array_equal(got["ids"][:A], exp["ids"][src])
    cs_ref = exp["cs"][src]
    assert np.array_equal(np.isnan(got["cs"][:A]), np.isnan(cs_ref))
    np.testing.assert_allclose(got["cs"][:A][~np.isnan(cs_ref)], cs_ref[~np.isnan(cs_ref)], rtol=0, atol=1e-5)
    np.testing.assert_array_equal(got["b"][:A], exp["b"][src])
    np.testing.assert_array_equal(got["K"][:A], K[src])
    np.testing.assert_array_equal(got["rid"][:A], rid[src])
    np.testing.assert_array_equal(got["p"][:A], (np.arange(B) * 7)[src])
    np.testing.assert_array_equal(got["thr"][:A], inp.thr[src])
    if extra is not None:
        np.testing.assert_array_equal(got["extra"][:A], extra[src])
        np.testing.assert_array_equal(two["extra"][:A], extra[src])
    for r, toks in exp["gen"].items():
        np.testing.assert_array_equal(got["gen"][r][: len(toks)], toks)
    # and everything element for element against the two-launch path
    for k in ("done", "accept_len", "n_new", "tok", "evict", "new_index", "gen"):
        np.testing.assert_array_equal(got[k], two[k], err_msg=k)
    for k in ("feats", "conf", "lse", "cs", "thr"):
        assert np.array_equal(got[k].view(np.uint32), two[k].view(np.uint32)), k
    assert got["A_out"] == two["A_out"]
    for k in ("ids", "b", "K", "rid", "p", "src_row"):
        np.testing.assert_array_equal(got[k][:A], two[k][:A], err_msg=k)
