"""The C ABI without a GPU: the library loads, exports every function the
header declares, the binding's structs match, host-side validation rejects
bad arguments before any CUDA call, and the native host planners
(eq. (1), sand-fill admission) agree with the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import denoise_step_token_gb300 as dllm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(dllm_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function():
    lib = dllm.load()
    names = declared_functions()
    assert "dllm_step" in names and "dllm_pack" in names and "dllm_compact" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(dllm.exported_symbols()) <= set(names)
    assert lib.dllm_abi_version() == dllm.ABI_VERSION


def test_struct_sizes_match_binding():
    lib = dllm.load()
    for which, cls in enumerate((dllm.StepArgs, dllm.PackArgs, dllm.CompactArgs, dllm.AdvanceArgs, dllm.RefillArgs,
                                 dllm.LoopConfig, dllm.LoopInfo, dllm.VocabShard)):
        assert lib.dllm_struct_size(which) == ctypes.sizeof(cls)
    assert lib.dllm_struct_size(99) == 0


def test_strerror():
    lib = dllm.load()
    for code in (0, -1, -2, -3, -4, -5, -6, 17):
        assert lib.dllm_strerror(code)


def _args(**kw):
    base = dict(B=2, L=4, V=16, mask_id=15, ldv=16, logits=0x10000, input_ids=0x20000, thr=0x30000,
                conf_state=0x40000, done=0x50000, accept_len=0x60000, n_new=0x70000, workspace=0x100000,
                workspace_bytes=1 << 20)
    base.update(kw)
    return dllm.StepArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(L=0), -1), (dict(L=1025), -1), (dict(V=0), -1), (dict(ldv=8), -1), (dict(B=-1), -1),
    (dict(logits=None), -1), (dict(thr=None), -1), (dict(done=None), -1),
    (dict(ldv=20), -2), (dict(logits=0x10002), -2),
    (dict(workspace=None), -5), (dict(workspace=0x100010), -5), (dict(workspace_bytes=64), -5),
])
def test_step_host_validation(kw, code):
    lib = dllm.load()
    assert lib.dllm_step(ctypes.byref(_args(**kw)), None) == code


def test_step_empty_batch_is_a_no_op():
    lib = dllm.load()
    assert lib.dllm_step(ctypes.byref(_args(B=0, logits=None, input_ids=None)), None) == 0


def test_workspace_size_shape_rules():
    lib = dllm.load()
    assert lib.dllm_step_workspace_size(0, 0, 10) == 0
    a = lib.dllm_step_workspace_size(128, 32, 151936)
    b = lib.dllm_step_workspace_size(512, 64, 151936)
    assert 0 < a < b and a % 256 == 0


def test_pack_plan_matches_eq1():
    rng = np.random.default_rng(1)
    for _ in range(50):
        A = int(rng.integers(0, 20))
        p = rng.integers(0, 2000, A)
        b = rng.integers(0, 9, A)
        L = int(rng.integers(1, 64))
        W, cost = dllm.pack_plan(p, b, L)
        assert W == oracle.box_width(list(p), list(b), L)
        assert cost == oracle.cost(list(p), list(b), L)


def test_admit_matches_oracle_random():
    rng = np.random.default_rng(2)
    for trial in range(300):
        n = int(rng.integers(0, 40))
        pend = np.sort(rng.integers(0, 300, n))
        if trial % 3 == 0:
            pend = np.sort(rng.integers(0, 8, n) * 16)     # many equal lengths
        A = int(rng.integers(0, 6))
        ap = rng.integers(0, 300, A)
        ab = rng.integers(0, 4, A)
        L = int(rng.choice([4, 8, 32]))
        budget = int(rng.integers(0, 6000))
        got = dllm.admit(pend, ap, ab, L, budget)
        want = oracle.admit(list(pend), list(ap), list(ab), L, budget)
        assert got == want, (trial, pend, ap, ab, L, budget)


def test_admit_rejects_unsorted_queue():
    lib = dllm.load()
    pend = np.array([5, 3], dtype=np.int32)
    idx = np.zeros(2, dtype=np.int32)
    n = ctypes.c_int32(0)
    rc = lib.dllm_admit(2, pend.ctypes.data, 0, None, None, 4, 100, idx.ctypes.data, ctypes.byref(n))
    assert rc == -1


def test_transfer_quota_matches_oracle():
    lib = dllm.load()
    for L in (1, 2, 7, 32, 33, 64, 1024):
        for S in (1, 3, 5, 8, 32, 100):
            for s in range(0, S + 2):
                assert lib.dllm_transfer_quota(L, S, s) == oracle.transfer_quota(L, S, s), (L, S, s)
    assert lib.dllm_transfer_quota(0, 4, 0) == -1
    assert lib.dllm_transfer_quota(4, 0, 0) == -1
    assert lib.dllm_transfer_quota(4, 4, -1) == -1


def test_step_quota_validation():
    lib = dllm.load()
    assert lib.dllm_step_quota(ctypes.byref(_args()), None, None) == -1
    assert lib.dllm_step_quota(ctypes.byref(_args(L=0)), ctypes.c_void_p(0x20000), None) == -1
    assert lib.dllm_step_quota(ctypes.byref(_args(ldv=20)), ctypes.c_void_p(0x20000), None) == -2
    assert lib.dllm_step_quota(ctypes.byref(_args(B=0)), ctypes.c_void_p(0x20000), None) == 0


def _dptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def test_threshold_control_matches_oracle():
    """dllm_predict_steps_stub, dllm_load_control and dllm_slo_thresholds
    (host functions) equal the oracle exactly on random inputs."""
    from oracle import control as oc
    lib = dllm.load()
    rng = np.random.default_rng(15)
    cand = np.array([0.5, 0.6, 0.7, 0.8, 0.9])
    T, L = len(cand), 32
    for trial in range(20):
        R = int(rng.integers(1, 40))
        q = np.sort(rng.random((R, 4)).astype(np.float32), axis=1)
        feats = np.stack([q[:, 0], q[:, 1], q[:, 2], q.mean(axis=1), q[:, 3], rng.random(R)], axis=1).astype(np.float32)
        feats[rng.random(R) < 0.2, :5] = np.nan
        masked = rng.integers(0, L + 1, size=R).astype(np.int32)
        left = rng.integers(0, 8, size=R).astype(np.int32)
        steps = np.empty((R, T))
        assert lib.dllm_predict_steps_stub(R, T, _dptr(cand), L, _dptr(feats), _dptr(masked), _dptr(left),
                                           _dptr(steps)) == 0
        want = np.array([[oc.predict_steps_stub(t, feats[i], masked[i], left[i], L) for t in cand]
                         for i in range(R)])
        np.testing.assert_array_equal(steps, want)
        load = steps * rng.integers(100, 1300, size=(R, 1))
        cap = float(rng.uniform(load[:, 0].sum() * 0.8, load[:, -1].sum() * 1.1))
        keep = np.empty(R, dtype=np.int32)
        assert lib.dllm_load_control(R, T, _dptr(np.ascontiguousarray(load)), cap, _dptr(keep)) == 0
        np.testing.assert_array_equal(keep, oc.load_control(load, cap))
        lat = rng.uniform(0.005, 0.05, size=R)
        slo = rng.uniform(0.0, 5.0, size=R)
        choice = np.empty(R, dtype=np.int32)
        assert lib.dllm_slo_thresholds(R, T, _dptr(steps), _dptr(lat), _dptr(slo), _dptr(keep), _dptr(choice)) == 0
        np.testing.assert_array_equal(choice, [oc.slo_threshold(steps[i], lat[i], slo[i], keep[i]) for i in range(R)])
    bad = np.array([7], dtype=np.int32)
    one = np.ones(T)
    # the same rejection when an entry is out of range after a valid one
    two = np.array([0, 7], dtype=np.int32)
    assert lib.dllm_slo_thresholds(2, T, _dptr(np.ones(2 * T)), _dptr(np.ones(2)), _dptr(np.ones(2)), _dptr(two),
                                   _dptr(np.empty(2, dtype=np.int32))) == -1
    assert lib.dllm_slo_thresholds(1, T, _dptr(one), _dptr(one[:1]), _dptr(one[:1]), _dptr(bad),
                                   _dptr(np.empty(1, dtype=np.int32))) == -1
    assert lib.dllm_load_control(1, 0, None, 1.0, None) == -1


def test_threshold_control_decision_matches_oracle():
    """dllm_threshold_control (the whole decision: predicted steps, load =
    steps x total tokens, Algorithm 2 at capacity = tokens/s x SLO, Algorithm
    1 against the SLO left since arrival) equals the oracle's functions
    composed in that order, exactly, on random inputs."""
    from oracle import control as oc
    lib = dllm.load()
    rng = np.random.default_rng(16)
    cand = np.array([0.5, 0.6, 0.7, 0.8, 0.9])
    T, L = len(cand), 32
    for trial in range(20):
        R = int(rng.integers(1, 60))
        q = np.sort(rng.random((R, 4)).astype(np.float32), axis=1)
        feats = np.stack([q[:, 0], q[:, 1], q[:, 2], q.mean(axis=1), q[:, 3], rng.random(R)], axis=1).astype(np.float32)
        feats[rng.random(R) < 0.2, :5] = np.nan
        masked = rng.integers(0, L + 1, size=R).astype(np.int32)
        left = rng.integers(0, 8, size=R).astype(np.int32)
        total = rng.integers(64 + 256, 1024 + 256, size=R).astype(np.int64)
        elapsed = rng.uniform(0.0, 2.0, size=R)
        slo, tps, lat = float(rng.uniform(0.5, 3.0)), float(rng.uniform(1e4, 2e5)), float(rng.uniform(1e-3, 2e-2))
        steps = np.empty((R, T))
        cap = np.empty(R, dtype=np.int32)
        choice = np.empty(R, dtype=np.int32)
        assert lib.dllm_threshold_control(R, T, _dptr(cand), L, _dptr(feats), _dptr(masked), _dptr(left),
                                          _dptr(total), _dptr(elapsed), slo, tps, lat, _dptr(steps), _dptr(cap),
                                          _dptr(choice)) == 0
        want_steps = np.array([[oc.predict_steps_stub(t, feats[i], masked[i], left[i], L) for t in cand]
                               for i in range(R)])
        np.testing.assert_array_equal(steps, want_steps)
        want_cap = oc.load_control(want_steps * total[:, None].astype(np.float64), tps * slo)
        np.testing.assert_array_equal(cap, want_cap)
        want_choice = [oc.slo_threshold(want_steps[i], lat, slo - elapsed[i], want_cap[i]) for i in range(R)]
        np.testing.assert_array_equal(choice, want_choice)
    z = np.zeros(1)
    assert lib.dllm_threshold_control(1, T, _dptr(cand), L, _dptr(np.zeros(6, np.float32)), _dptr(np.zeros(1, np.int32)),
                                      _dptr(np.zeros(1, np.int32)), _dptr(np.array([-1], np.int64)), _dptr(z), 1.0,
                                      1.0, 1.0, _dptr(np.empty(T)), _dptr(np.empty(1, np.int32)),
                                      _dptr(np.empty(1, np.int32))) == -1
    assert lib.dllm_threshold_control(0, T, None, L, None, None, None, None, None, 1.0, 1.0, 1.0, None, None,
                                      None) == 0


def test_injected_cuda_error_reaches_the_caller():
    """The status plumbing from a failing CUDA call to the caller, with the
    failure injected on the host (the call is not made, so the fake pointer
    below is never touched): the entry point returns DLLM_ERR_CUDA,
    dllm_last_cuda_error names the injected status and the binding raises
    DllmError with that name."""
    lib = dllm.load()
    OOM = 2                                     # cudaErrorMemoryAllocation
    assert lib.dllm_inject_cuda_error(OOM, -1) == -1
    assert lib.dllm_inject_cuda_error(0, 1) == -1
    assert lib.dllm_inject_cuda_error(OOM, 1) == 0
    assert lib.dllm_workspace_init(ctypes.c_void_p(0x100000), 256, None) == -3
    name = ctypes.c_char_p()
    assert lib.dllm_last_cuda_error(ctypes.byref(name)) == OOM
    assert name.value == b"cudaErrorMemoryAllocation"
    with pytest.raises(dllm.DllmError, match="cudaErrorMemoryAllocation"):
        dllm._check("dllm_workspace_init", -3)
    assert lib.dllm_inject_cuda_error(0, 0) == 0


def test_injection_countdown_without_a_gpu():
    """Countdown 2: the first CUDA call is made (and, with no GPU, fails with
    its own status); the second reports the injected one."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("the first call would really run")
    lib = dllm.load()
    OOM = 2
    assert lib.dllm_inject_cuda_error(OOM, 2) == 0
    assert lib.dllm_workspace_init(ctypes.c_void_p(0x100000), 256, None) == -3
    assert lib.dllm_last_cuda_error(None) not in (0, OOM)
    assert lib.dllm_workspace_init(ctypes.c_void_p(0x100000), 256, None) == -3
    assert lib.dllm_last_cuda_error(None) == OOM


def test_step_commit_argument_checks():
    """dllm_step_commit rejects an advance or compaction that is not the
    step's own batch before any CUDA call."""
    lib = dllm.load()
    sa = dllm.StepArgs(B=4, L=8, V=64, mask_id=63, ldv=64, logits=0x10000, input_ids=0x20000, thr=0x30000,
                       conf_state=0x40000, done=0x50000, accept_len=0x60000, n_new=0x70000, workspace=0x100000,
                       workspace_bytes=1 << 20)
    ok = dict(A=4, L=8, mask_id=63, advance=0x50000, rid=0x80000, K=0x90000, b=0xa0000, input_ids=0x20000,
              conf_state=0x40000, gen_tokens=0xb0000, ld_gen=32, evict=0xc0000)
    ca = dllm.CompactArgs(A=4, n_arrays=0, A_out=0xd0000)
    for k, v in (("A", 5), ("L", 4), ("mask_id", 1), ("input_ids", 0x20004), ("conf_state", 0x40004),
                 ("advance", 0x50004), ("rid", None), ("ld_gen", -1)):
        bad = dict(ok)
        bad[k] = v
        aa = dllm.AdvanceArgs(**bad)
        assert lib.dllm_step_commit(ctypes.byref(sa), None, -1, ctypes.byref(aa), ctypes.byref(ca), None) == -1, k
    ca_bad = dllm.CompactArgs(A=3, n_arrays=0, A_out=0xd0000)
    assert lib.dllm_step_commit(ctypes.byref(sa), None, -1, ctypes.byref(dllm.AdvanceArgs(**ok)), ctypes.byref(ca_bad),
                                None) == -1


def test_vocab_shards_argument_checks():
    """dllm_step_vocab_shards rejects a shard list that does not tile [0, V)
    in order, NULL or misaligned shards, before any CUDA call."""
    lib = dllm.load()
    a = _args(V=40, ldv=0, logits=None)

    def call(specs, n=None):
        arr = (dllm.VocabShard * max(len(specs), 1))()
        for k, (ptr, ldv, v0, V) in enumerate(specs):
            arr[k] = dllm.VocabShard(logits=ptr, ldv=ldv, v0=v0, V=V)
        return lib.dllm_step_vocab_shards(ctypes.byref(a), len(specs) if n is None else n, arr, None, None)

    ok = [(0x10000, 16, 0, 16), (0x20000, 24, 16, 24)]
    assert call(ok[:1] + [(0x20000, 24, 17, 24)]) == -1          # gap between shards
    assert call([(0x10000, 16, 0, 16), (0x20000, 24, 16, 20)]) == -1   # widths do not add up to V
    assert call([(None, 16, 0, 16), ok[1]]) == -1                 # NULL shard
    assert call([(0x10000, 8, 0, 16), ok[1]]) == -1               # row stride below the width
    assert call([(0x10000, 16, 0, 0), (0x20000, 40, 0, 40)]) == -1   # empty shard
    assert call(ok, n=0) == -1 and call(ok, n=9) == -1
    assert call([(0x10008, 16, 0, 16), ok[1]]) == -2              # misaligned shard
    assert call([(0x10000, 20, 0, 16), ok[1]]) == -2              # stride not a multiple of 8


def test_vocab_shards_commit_argument_checks():
    """dllm_step_vocab_shards_commit applies both sets of checks -- the shard
    table's and the commit's -- before any CUDA call."""
    lib = dllm.load()
    sa = dllm.StepArgs(B=4, L=8, V=64, mask_id=63, ldv=0, logits=None, input_ids=0x20000, thr=0x30000,
                       conf_state=0x40000, done=0x50000, accept_len=0x60000, n_new=0x70000, workspace=0x100000,
                       workspace_bytes=1 << 20)
    ok = dict(A=4, L=8, mask_id=63, advance=0x50000, rid=0x80000, K=0x90000, b=0xa0000, input_ids=0x20000,
              conf_state=0x40000, gen_tokens=0xb0000, ld_gen=32, evict=0xc0000)
    ca = dllm.CompactArgs(A=4, n_arrays=0, A_out=0xd0000)

    def call(specs, adv=ok, cmp=ca):
        arr = (dllm.VocabShard * len(specs))()
        for k, (ptr, ldv, v0, V) in enumerate(specs):
            arr[k] = dllm.VocabShard(logits=ptr, ldv=ldv, v0=v0, V=V)
        return lib.dllm_step_vocab_shards_commit(ctypes.byref(sa), len(specs), arr, None,
                                                 ctypes.byref(dllm.AdvanceArgs(**adv)), ctypes.byref(cmp), None)

    good = [(0x10000, 32, 0, 32), (0x20000, 32, 32, 32)]
    assert call([(0x10000, 32, 0, 32), (0x20000, 32, 33, 31)]) == -1           # shards do not tile [0, V)
    assert call([(0x10008, 32, 0, 32), (0x20000, 32, 32, 32)]) == -2           # misaligned shard
    assert call(good, adv=dict(ok, A=5)) == -1                                 # not the step's batch
    assert call(good, adv=dict(ok, input_ids=0x20004)) == -1
    assert call(good, cmp=dllm.CompactArgs(A=3, n_arrays=0, A_out=0xd0000)) == -1


def test_native_loop_control_argument_checks():
    """dllm_loop_set_control / dllm_loop_thresholds reject a NULL loop (the
    host checks; a loop itself needs a device)."""
    lib = dllm.load()
    cand = (ctypes.c_double * 3)(0.5, 0.7, 0.9)
    lc = dllm.LoopControl(T=3, candidates=ctypes.cast(cand, ctypes.c_void_p), slo_s=1.0, tokens_per_s=1e5,
                          latency_s=0.001, latency_per_row_s=0.0)
    assert lib.dllm_loop_set_control(None, ctypes.byref(lc)) == -1
    n = ctypes.c_int32(0)
    assert lib.dllm_loop_thresholds(None, None, ctypes.byref(n)) == -1
    assert ctypes.sizeof(dllm.LoopControl) == lib.dllm_struct_size(8)


def test_vocab_shards_workspace_holds_the_extra_chunks():
    """Each shard is cut into chunks from its own start, so a sharded step
    needs dllm_step_workspace_size(B, L, V + 8192 * (n_shards - 1)) bytes:
    one sized for V alone is rejected (DLLM_ERR_WORKSPACE) before any CUDA
    call, by both sharded entry points."""
    lib = dllm.load()
    ERR_WORKSPACE = -5
    B, L, V = 64, 32, 126464
    # shards of 30000 tokens: 4 + 4 + 4 + 5 = 17 chunks per row, against 16 unsharded
    bounds = [0, 30000, 60000, 90000, V]
    arr = (dllm.VocabShard * 4)()
    for k in range(4):
        arr[k] = dllm.VocabShard(logits=0x100000 * (k + 1), ldv=36464, v0=bounds[k], V=bounds[k + 1] - bounds[k])
    small = lib.dllm_step_workspace_size(B, L, V)
    need = lib.dllm_step_workspace_size(B, L, V + 8192 * 3)
    assert need > small
    a = dllm.StepArgs(B=B, L=L, V=V, mask_id=0, ldv=0, logits=None, input_ids=0x20000, thr=0x30000,
                      conf_state=0x40000, done=0x50000, accept_len=0x60000, n_new=0x70000, workspace=0x1000000,
                      workspace_bytes=small)
    assert lib.dllm_step_vocab_shards(ctypes.byref(a), 4, arr, None, None) == ERR_WORKSPACE
    adv = dllm.AdvanceArgs(A=B, L=L, mask_id=0, advance=0x50000, rid=0x80000, K=0x90000, b=0xa0000,
                           input_ids=0x20000, conf_state=0x40000, gen_tokens=0xb0000, ld_gen=256, evict=0xc0000)
    ca = dllm.CompactArgs(A=B, n_arrays=0, A_out=0xd0000)
    assert lib.dllm_step_vocab_shards_commit(ctypes.byref(a), 4, arr, None, ctypes.byref(adv), ctypes.byref(ca),
                                             None) == ERR_WORKSPACE
    # the size the header asks for passes the workspace check (and stops at the first CUDA call: no device here)
    a.workspace_bytes = need
    assert lib.dllm_step_vocab_shards(ctypes.byref(a), 4, arr, None, None) != ERR_WORKSPACE
