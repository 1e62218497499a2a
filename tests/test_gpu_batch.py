"""GPU parity of the batch-management path (S7 pack, S9 advance / compact /
refill) against the CPU oracle, bit-exact, through the C ABI."""
import numpy as np
import pytest

import oracle
from oracle.loop import advance as oracle_advance
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def device(dllm):
    import torch
    return torch.device("cuda", 0)


def _t(x, device, dtype=None):
    import torch
    return torch.as_tensor(np.ascontiguousarray(x), dtype=dtype).to(device)


def _mixed_rows(seed, A, L, V, p_lo, p_hi, K):
    """A mixed-state batch: row i is request rid[i] at block b[i]."""
    R = A + 5
    lcfg = synth.LoopConfig("m", R, p_lo, p_hi, K * L, L, V, 1 << 30, 0.9, 8.0)
    reqs = synth.make_loop_requests(lcfg, seed)
    rng = np.random.default_rng(seed)
    rid = rng.permutation(R)[:A].astype(np.int32)
    b = rng.integers(0, K, A).astype(np.int32)
    gen = synth.committed_tokens(seed, R, K * L, V)
    blocks = rng.integers(0, V - 2, (A, L)).astype(np.int32)
    blocks[rng.random((A, L)) < 0.4] = V - 1
    return reqs, rid, b, gen, blocks


@pytest.mark.parametrize("A,L,p_lo,p_hi,K", [(1, 4, 0, 0, 1), (7, 4, 0, 9, 3), (256, 32, 64, 1024, 8), (300, 16, 1, 500, 5)])
def test_pack_parity(dllm, device, A, L, p_lo, p_hi, K):
    V = 5000
    reqs, rid, b, gen, blocks = _mixed_rows(A + L, A, L, V, p_lo, p_hi, K)
    p = reqs.p[rid].astype(np.int32)
    W, cost = dllm.pack_plan(p, b, L)
    prompts = [reqs.prompt_tokens[reqs.prompt_off[r]:reqs.prompt_off[r + 1]] for r in rid]
    ref = oracle.pack(p, b, L, prompts, [gen[r] for r in rid], list(blocks), V - 2)
    assert W == ref["W"] and cost == oracle.cost(list(p), list(b), L)
    out = dllm.pack(_t(p, device), _t(b, device), _t(rid, device), _t(reqs.prompt_off, device),
                    _t(reqs.prompt_tokens, device), _t(gen, device), _t(blocks, device), L=L, W=W, pad_id=V - 2)
    np.testing.assert_array_equal(out["ids"].cpu().numpy(), ref["ids"])
    np.testing.assert_array_equal(out["attn"].cpu().numpy(), ref["attn"])
    np.testing.assert_array_equal(out["pos"].cpu().numpy(), ref["pos"])
    np.testing.assert_array_equal(out["pad"].cpu().numpy(), ref["pad"])
    np.testing.assert_array_equal(out["blk_start"].cpu().numpy(), ref["blk_start"])
    assert dllm.get_device_error(device) == 0


def test_pack_flags_a_row_wider_than_the_box(dllm, device):
    L, V = 4, 100
    reqs, rid, b, gen, blocks = _mixed_rows(3, 5, L, V, 2, 8, 3)
    p = reqs.p[rid].astype(np.int32)
    W, _ = dllm.pack_plan(p, b, L)
    b_bad = b.copy()
    b_bad[2] += 1                      # row 2 no longer fits in W
    if p[2] + (b_bad[2] + 1) * L <= W:
        b_bad[2] += W
    out = dllm.pack(_t(p, device), _t(b_bad, device), _t(rid, device), _t(reqs.prompt_off, device),
                    _t(reqs.prompt_tokens, device), _t(gen, device), _t(blocks, device), L=L, W=W, pad_id=V - 2)
    assert dllm.get_device_error(device) == 2      # DLLM_DEVERR_ROW_WIDTH
    assert dllm.get_device_error(device) == 0      # read clears it
    prompts = [reqs.prompt_tokens[reqs.prompt_off[r]:reqs.prompt_off[r + 1]] for r in rid]
    ref = oracle.pack(p, b, L, prompts, [gen[r] for r in rid], list(blocks), V - 2)
    ok = [i for i in range(5) if i != 2]
    np.testing.assert_array_equal(out["ids"].cpu().numpy()[ok], ref["ids"][ok])


@pytest.mark.parametrize("A,L,K", [(1, 4, 1), (64, 32, 8), (257, 16, 3)])
def test_advance_parity(dllm, device, A, L, K):
    import torch
    V = 1000
    reqs, rid, b, gen, blocks = _mixed_rows(A * 3 + L, A, L, V, 0, 10, K)
    rng = np.random.default_rng(A)
    adv = (rng.random(A) < 0.6).astype(np.uint8)
    Kr = np.full(A, K, dtype=np.int32)
    cs = rng.random((A, L)).astype(np.float32)
    R = gen.shape[0]
    # oracle: committed tokens so far are the first b[i] blocks of gen
    o_gen = {int(rid[i]): np.asarray(gen[int(rid[i])][: b[i] * L]) for i in range(A)}
    o_b, o_ids, o_cs = b.astype(np.int64).copy(), blocks.astype(np.int64).copy(), cs.astype(np.float64).copy()
    o_evict = oracle_advance(adv, rid, o_b, Kr, o_ids, o_cs, o_gen, V - 1)
    d_b, d_ids, d_cs, d_gen = _t(b, device), _t(blocks, device), _t(cs, device), _t(gen, device)
    evict = dllm.advance(_t(adv, device), _t(rid, device), _t(Kr, device), d_b, d_ids, d_cs, d_gen, mask_id=V - 1)
    np.testing.assert_array_equal(evict.cpu().numpy().astype(bool), o_evict)
    np.testing.assert_array_equal(d_b.cpu().numpy(), o_b)
    np.testing.assert_array_equal(d_ids.cpu().numpy(), o_ids)
    g = d_gen.cpu().numpy()
    for i in range(A):
        r = int(rid[i])
        n = len(o_gen[r])
        np.testing.assert_array_equal(g[r][:n], o_gen[r])
    got_cs = d_cs.cpu().numpy()
    assert np.array_equal(np.isnan(got_cs), np.isnan(o_cs))
    np.testing.assert_array_equal(got_cs[~np.isnan(got_cs)], o_cs[~np.isnan(o_cs)].astype(np.float32))
    assert dllm.get_device_error(device) == 0


@pytest.mark.parametrize("A", [0, 1, 5, 255, 256, 257, 1000, 4099])
def test_compact_parity(dllm, device, A):
    rng = np.random.default_rng(A + 1)
    for trial in range(3):
        evict = (rng.random(A) < [0.0, 0.3, 1.0][trial]).astype(np.uint8)
        arrays = [rng.integers(0, 1 << 30, (A, 32)).astype(np.int32),        # word rows
                  rng.random((A, 7)).astype(np.float32),                       # 28-byte rows
                  rng.integers(0, 255, (A, 3)).astype(np.uint8),               # 3-byte rows (byte path)
                  rng.integers(0, 1 << 30, A).astype(np.int32)]                # one word per row
        d_arrays = [_t(a, device) for a in arrays]
        new_index, src_row, A_out = dllm.compact(_t(evict, device), d_arrays)
        o_new, o_src, o_A = oracle.compact(evict)
        assert int(A_out.cpu().numpy()[0]) == o_A
        np.testing.assert_array_equal(new_index.cpu().numpy()[:A], o_new)
        np.testing.assert_array_equal(src_row.cpu().numpy()[:o_A], o_src)
        for a, d in zip(arrays, d_arrays):
            np.testing.assert_array_equal(d.cpu().numpy()[:o_A], a[o_src])


def test_refill(dllm, device):
    import torch
    A0, n, L, mask_id = 3, 4, 8, 99
    rows = A0 + n + 2
    rid = _t(np.arange(rows, dtype=np.int32), device)
    p = _t(np.full(rows, 7, np.int32), device)
    b = _t(np.full(rows, 5, np.int32), device)
    K = _t(np.full(rows, 9, np.int32), device)
    thr = _t(np.full(rows, 0.3, np.float32), device)
    ids = _t(np.arange(rows * L, dtype=np.int32).reshape(rows, L), device)
    cs = _t(np.ones((rows, L), np.float32), device)
    new = [np.array(x, dtype=np.int32) for x in ([40, 41, 42, 43], [1, 2, 3, 4], [8, 8, 2, 1])]
    new_thr = np.array([0.5, 0.6, 0.7, 0.9], np.float32)
    dllm.refill(A0, _t(new[0], device), _t(new[1], device), _t(new[2], device), _t(new_thr, device),
                rid, p, b, K, thr, ids, cs, mask_id=mask_id)
    r = slice(A0, A0 + n)
    assert rid.cpu().numpy()[r].tolist() == new[0].tolist()
    assert p.cpu().numpy()[r].tolist() == new[1].tolist()
    assert K.cpu().numpy()[r].tolist() == new[2].tolist()
    assert (b.cpu().numpy()[r] == 0).all()
    np.testing.assert_array_equal(thr.cpu().numpy()[r], new_thr)
    assert (ids.cpu().numpy()[r] == mask_id).all() and np.isnan(cs.cpu().numpy()[r]).all()
    # rows outside the range untouched
    assert (ids.cpu().numpy()[A0 + n:] == np.arange((A0 + n) * L, rows * L).reshape(-1, L)).all()
    assert (b.cpu().numpy()[:A0] == 5).all()



@pytest.mark.parametrize("workspace", [True, False])
@pytest.mark.parametrize("A,L,K", [(0, 32, 4), (1, 32, 2), (77, 32, 3), (256, 32, 8), (1500, 16, 2), (300, 64, 1)])
def test_advance_compact_parity(dllm, device, A, L, K, workspace):
    """dllm_advance_compact equals the oracle's advance followed by its
    stable compaction (rows of several widths, chunked staging when the
    rows do not fit one chunk)."""
    V = 1000
    reqs, rid, b, gen, blocks = _mixed_rows(A * 5 + L + 3, A, L, V, 0, 10, K)
    rng = np.random.default_rng(A + 7)
    adv = (rng.random(A) < 0.6).astype(np.uint8)
    Kr = rng.integers(1, K + 1, size=A).astype(np.int32)
    b = np.minimum(b, Kr - 1).astype(np.int32)
    cs = rng.random((A, L)).astype(np.float32)
    extra = rng.integers(0, 255, (A, 5)).astype(np.uint8)                     # a 5-byte row array
    o_gen = {int(rid[i]): np.asarray(gen[int(rid[i])][: b[i] * L]) for i in range(A)}
    o_b, o_ids, o_cs = b.astype(np.int64).copy(), blocks.astype(np.int64).copy(), cs.astype(np.float64).copy()
    o_evict = oracle_advance(adv, rid, o_b, Kr, o_ids, o_cs, o_gen, V - 1)
    o_new, o_src, o_A = oracle.compact(o_evict)
    d = {k: _t(v, device) for k, v in dict(rid=rid, K=Kr, b=b, ids=blocks, cs=cs, extra=extra).items()}
    d_gen = _t(gen, device)
    # an odd A adds a 5-byte row array, which takes the byte-copy path
    arrays = [d["rid"], d["K"], d["b"], d["ids"], d["cs"]] + ([d["extra"]] if A % 2 else [])
    evict, new_index, src_row, A_out = dllm.advance_compact(
        _t(adv, device), d["rid"], d["K"], d["b"], d["ids"], d["cs"], d_gen, arrays, mask_id=V - 1,
        workspace=workspace)
    assert int(A_out.cpu().numpy()[0]) == o_A
    if A:
        np.testing.assert_array_equal(evict.cpu().numpy()[:A].astype(bool), o_evict)
        np.testing.assert_array_equal(new_index.cpu().numpy()[:A], o_new)
        np.testing.assert_array_equal(src_row.cpu().numpy()[:o_A], o_src)
    np.testing.assert_array_equal(d["rid"].cpu().numpy()[:o_A], rid[o_src])
    np.testing.assert_array_equal(d["K"].cpu().numpy()[:o_A], Kr[o_src])
    np.testing.assert_array_equal(d["b"].cpu().numpy()[:o_A], o_b[o_src])
    np.testing.assert_array_equal(d["ids"].cpu().numpy()[:o_A], o_ids[o_src])
    if A % 2:
        np.testing.assert_array_equal(d["extra"].cpu().numpy()[:o_A], extra[o_src])
    got_cs = d["cs"].cpu().numpy()[:o_A]
    want_cs = o_cs[o_src]
    assert np.array_equal(np.isnan(got_cs), np.isnan(want_cs))
    np.testing.assert_array_equal(got_cs[~np.isnan(got_cs)], want_cs[~np.isnan(want_cs)].astype(np.float32))
    g = d_gen.cpu().numpy()
    for i in range(A):
        r = int(rid[i])
        n = len(o_gen[r])
        np.testing.assert_array_equal(g[r][:n], o_gen[r])
    assert dllm.get_device_error(device) == 0
