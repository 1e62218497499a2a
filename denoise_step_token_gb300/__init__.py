"""Python binding of libdllm.so (ctypes): argument marshalling only.

Every step of the path runs in the library's CUDA kernels or its native host
functions.  PyTorch supplies device memory and the current stream.  There is
no fallback: if the library cannot be built or loaded, or no CUDA device is
present, the calls raise.

Names follow the C ABI in ``include/dllm.h``:

* ``step``      -- one denoise step (FDFO page, section "工程设计一").
* ``features``  -- confidence features (DiLaServe review, section 4.2 ③).
* ``pack_plan`` / ``admit`` -- eq. (1) and sand-fill admission (BlockServe
  page, section II-D), host functions of the library.
* ``pack``      -- the left-padded box (BlockServe page, section II-E).
* ``advance``   -- block commit and eviction flags (BlockServe Algorithm 1).
* ``compact``   -- stable in-place compaction (FDFO eviction).
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import threading

import numpy as np

from . import _build

__all__ = ["load", "step", "step_host", "features", "pack_plan", "admit", "pack", "advance", "compact", "refill",
           "get_device_error", "DllmError", "NUM_FEATURES", "LIB_PATH"]

LIB_PATH = _build.LIB_PATH
NUM_FEATURES = 6
ABI_VERSION = 2        # include/dllm.h DLLM_ABI_VERSION this binding was written for
COMPACT_MAX_ARRAYS = 16

DLLM_OK = 0


class DllmError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {code} ({msg})")
        self.code = code


_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class StepArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("L", _i32), ("V", _i32), ("mask_id", _i32), ("ldv", _i64),
                ("logits", _p), ("input_ids", _p), ("thr", _p), ("conf_state", _p),
                ("done", _p), ("accept_len", _p), ("n_new", _p), ("feats", _p),
                ("conf_out", _p), ("lse_out", _p), ("tok_out", _p),
                ("workspace", _p), ("workspace_bytes", _sz)]


class PackArgs(ctypes.Structure):
    _fields_ = [("A", _i32), ("L", _i32), ("W", _i32), ("pad_id", _i32),
                ("p", _p), ("b", _p), ("rid", _p), ("prompt_off", _p), ("prompt_tokens", _p),
                ("gen_tokens", _p), ("ld_gen", _i64), ("block_ids", _p),
                ("ids", _p), ("attn", _p), ("pos", _p), ("pad", _p), ("blk_start", _p)]


class CompactArgs(ctypes.Structure):
    _fields_ = [("A", _i32), ("n_arrays", _i32), ("evict", _p), ("new_index", _p), ("src_row", _p),
                ("A_out", _p), ("arrays", _p * COMPACT_MAX_ARRAYS), ("row_bytes", _i64 * COMPACT_MAX_ARRAYS),
                ("workspace", _p), ("workspace_bytes", _sz)]


class AdvanceArgs(ctypes.Structure):
    _fields_ = [("A", _i32), ("L", _i32), ("mask_id", _i32), ("pad0", _i32),
                ("advance", _p), ("rid", _p), ("K", _p), ("b", _p), ("input_ids", _p), ("conf_state", _p),
                ("gen_tokens", _p), ("ld_gen", _i64), ("evict", _p)]


class VocabShard(ctypes.Structure):
    _fields_ = [("logits", _p), ("ldv", _i64), ("v0", _i32), ("V", _i32)]


MAX_VOCAB_SHARDS = 8


class LoopConfig(ctypes.Structure):
    _fields_ = [("R", _i32), ("L", _i32), ("V", _i32), ("mask_id", _i32), ("pad_id", _i32), ("mode", _i32),
                ("reloop", _i32), ("S", _i32), ("capacity", _i32), ("pad0", _i32), ("budget", _i64)]


class LoopInfo(ctypes.Structure):
    _fields_ = [("A", _i32), ("W", _i32), ("cost", _i64), ("iteration", _i32), ("reloops", _i32),
                ("pending", _i32), ("admitted_last", _i32), ("finished", _i32), ("in_place", _i32),
                ("ld_gen", _i64), ("block_ids", _p), ("conf_state", _p), ("box_ids", _p), ("box_attn", _p),
                ("box_pos", _p), ("box_pad", _p), ("box_blk_start", _p), ("gen_tokens", _p), ("done", _p),
                ("n_new", _p), ("accept_len", _p), ("feats", _p)]


class LoopControl(ctypes.Structure):
    _fields_ = [("T", _i32), ("pad0", _i32), ("candidates", _p), ("slo_s", ctypes.c_double),
                ("tokens_per_s", ctypes.c_double), ("latency_s", ctypes.c_double),
                ("latency_per_row_s", ctypes.c_double)]


class RefillArgs(ctypes.Structure):
    _fields_ = [("A0", _i32), ("n", _i32), ("L", _i32), ("mask_id", _i32),
                ("new_rid", _p), ("new_p", _p), ("new_K", _p), ("new_thr", _p),
                ("rid", _p), ("p", _p), ("b", _p), ("K", _p), ("thr", _p), ("input_ids", _p), ("conf_state", _p)]


_lib = None
_lock = threading.Lock()

# name -> (restype, argtypes)
_SIGNATURES = {
    "dllm_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "dllm_abi_version": (ctypes.c_int, []),
    "dllm_inject_cuda_error": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32]),
    "dllm_last_cuda_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_char_p)]),
    "dllm_struct_size": (_sz, [ctypes.c_int]),
    "dllm_get_device_error": (ctypes.c_int, [_p, ctypes.POINTER(_i32)]),
    "dllm_step_workspace_size": (_sz, [_i32, _i32, _i32]),
    "dllm_workspace_init": (ctypes.c_int, [_p, _sz, _p]),
    "dllm_step": (ctypes.c_int, [ctypes.POINTER(StepArgs), _p]),
    "dllm_step_quota": (ctypes.c_int, [ctypes.POINTER(StepArgs), _p, _p]),
    "dllm_step_compact": (ctypes.c_int, [ctypes.POINTER(StepArgs), ctypes.c_int64, _p, _p]),
    "dllm_step_shard": (ctypes.c_int, [ctypes.POINTER(StepArgs), ctypes.c_int32, _p, _p, _p, _p]),
    "dllm_step_merge": (ctypes.c_int, [ctypes.POINTER(StepArgs), ctypes.c_int32, _p, _p, _p, ctypes.c_int64, _p,
                                       _p]),
    "dllm_step_vocab_shards": (ctypes.c_int, [ctypes.POINTER(StepArgs), ctypes.c_int32, ctypes.POINTER(VocabShard),
                                              _p, _p]),
    "dllm_predict_steps_stub": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _p, ctypes.c_int32, _p, _p, _p, _p]),
    "dllm_load_control": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _p, ctypes.c_double, _p]),
    "dllm_slo_thresholds": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _p, _p, _p, _p, _p]),
    "dllm_threshold_control": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, _p, ctypes.c_int32, _p, _p, _p, _p, _p,
                                              ctypes.c_double, ctypes.c_double, ctypes.c_double, _p, _p, _p]),
    "dllm_transfer_quota": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "dllm_step_noalloc": (ctypes.c_int, [ctypes.POINTER(StepArgs), _p]),
    "dllm_step_noalloc_capacity": (_sz, []),
    "dllm_features": (ctypes.c_int, [_i32, _i32, _i32, _p, _p, _p, _p]),
    "dllm_pack_plan": (ctypes.c_int, [_i32, _p, _p, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i64)]),
    "dllm_admit": (ctypes.c_int, [_i32, _p, _i32, _p, _p, _i32, _i64, _p, ctypes.POINTER(_i32)]),
    "dllm_pack": (ctypes.c_int, [ctypes.POINTER(PackArgs), _p]),
    "dllm_pack_block": (ctypes.c_int, [ctypes.POINTER(PackArgs), _p]),
    "dllm_loop_workspace_size": (_sz, [ctypes.POINTER(LoopConfig), _p, _p]),
    "dllm_loop_create": (ctypes.c_int, [ctypes.POINTER(LoopConfig), _p, _p, _p, _p, _p, _p, _sz, _p,
                                        ctypes.POINTER(_p)]),
    "dllm_loop_destroy": (None, [_p]),
    "dllm_loop_begin": (ctypes.c_int, [_p, _p]),
    "dllm_loop_end": (ctypes.c_int, [_p, _p, _i64, _p]),
    "dllm_loop_info": (ctypes.c_int, [_p, ctypes.POINTER(LoopInfo)]),
    "dllm_loop_rows": (ctypes.c_int, [_p, _p, _p, _p]),
    "dllm_loop_set_control": (ctypes.c_int, [_p, ctypes.POINTER(LoopControl)]),
    "dllm_loop_thresholds": (ctypes.c_int, [_p, _p, _p]),
    "dllm_advance_compact": (ctypes.c_int, [ctypes.POINTER(AdvanceArgs), ctypes.POINTER(CompactArgs), _p]),
    "dllm_step_commit": (ctypes.c_int, [ctypes.POINTER(StepArgs), _p, ctypes.c_int64, ctypes.POINTER(AdvanceArgs),
                                        ctypes.POINTER(CompactArgs), _p]),
    "dllm_step_vocab_shards_commit": (ctypes.c_int, [ctypes.POINTER(StepArgs), ctypes.c_int32,
                                                     ctypes.POINTER(VocabShard), _p, ctypes.POINTER(AdvanceArgs),
                                                     ctypes.POINTER(CompactArgs), _p]),
    "dllm_advance": (ctypes.c_int, [ctypes.POINTER(AdvanceArgs), _p]),
    "dllm_compact_workspace_size": (_sz, [_i32, _i32, _p]),
    "dllm_compact": (ctypes.c_int, [ctypes.POINTER(CompactArgs), _p]),
    "dllm_refill": (ctypes.c_int, [ctypes.POINTER(RefillArgs), _p]),
}


def exported_symbols():
    """The C-ABI entry points this binding expects in libdllm.so."""
    return sorted(_SIGNATURES)


def _build_locked():
    os.makedirs(_build.BUILD_DIR, exist_ok=True)
    with open(os.path.join(_build.BUILD_DIR, ".lock"), "w") as fh:
        fcntl.flock(fh, fcntl.LOCK_EX)
        try:
            _build.build()
        finally:
            fcntl.flock(fh, fcntl.LOCK_UN)


def load(build=True):
    """Load libdllm.so (building it first when stale).  Raises on failure."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build:
            _build_locked()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdllm.so is missing at {LIB_PATH}; run __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.dllm_abi_version() != ABI_VERSION:
            raise RuntimeError(f"libdllm ABI version {lib.dllm_abi_version()}, binding expects {ABI_VERSION}")
        for which, cls in enumerate((StepArgs, PackArgs, CompactArgs, AdvanceArgs, RefillArgs, LoopConfig, LoopInfo,
                                     VocabShard, LoopControl)):
            if lib.dllm_struct_size(which) != ctypes.sizeof(cls):
                raise RuntimeError(f"ABI mismatch for {cls.__name__}: library {lib.dllm_struct_size(which)} "
                                   f"bytes, binding {ctypes.sizeof(cls)}")
        _lib = lib
        return lib


def _check(fn, rc):
    if rc != DLLM_OK:
        lib = load()
        msg = lib.dllm_strerror(rc).decode()
        if rc == -3:
            name = ctypes.c_char_p()
            code = lib.dllm_last_cuda_error(ctypes.byref(name))
            msg += f": cudaError {code} {name.value.decode() if name.value else ''}"
        raise DllmError(fn, rc, msg)


# ---------------------------------------------------------------------------
# torch plumbing
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _require_cuda(*tensors):
    torch = _torch()
    if not torch.cuda.is_available():
        raise RuntimeError("libdllm needs a CUDA device; none is available")
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors live on different devices")
    return dev


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class _Workspaces:
    """Per-device zero-initialised workspaces, grown on demand."""

    def __init__(self):
        self.buf = {}

    def get(self, device, nbytes):
        torch = _torch()
        key = (device.type, device.index)
        cur = self.buf.get(key)
        if cur is None or cur.numel() < nbytes:
            # torch.zeros: the step's counter region must start at zero
            cur = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            self.buf[key] = cur
        return cur

    def reset(self):
        self.buf.clear()


_step_ws = _Workspaces()
_compact_ws = _Workspaces()


def step_workspace_size(B, L, V):
    return int(load().dllm_step_workspace_size(B, L, V))


def step(logits, input_ids, thr, conf_state, *, V, mask_id, feats=True, debug=False, out=None, workspace=None,
         quota=None, compact=False):
    """One denoise step (dllm_step, or dllm_step_quota when ``quota`` is
    given) on the current stream.

    logits:     bf16 (or 16-bit) CUDA tensor of B*L rows with V <= row stride
                (shape [B, L, ldv] or [B*L, ldv]); ldv % 8 == 0
    input_ids:  int32 [B, L] (updated in place)
    thr:        float32 [B] (threshold rule; may be None with ``quota``)
    conf_state: float32 [B, L] (updated in place)
    quota:      int32 [B] CUDA tensor or None: positions to unmask per
                request under the fixed-steps rule
    compact:    logits hold only the masked positions' rows, in position
                order (dllm_step_compact); any number of rows >= the masked
                count
    workspace:  uint8 CUDA tensor of at least dllm_step_workspace_size
                bytes, zeroed once before first use; without one, a
                workspace cached per device is used, so steps that may run
                at the same time (on different streams) must each pass their
                own
    Returns a dict of output tensors: done (uint8 [B]), accept_len, n_new
    (int32 [B]), feats (float32 [B, 6]) and, with debug, conf / lse / tok [B, L].
    """
    torch = _torch()
    if quota is None:
        dev = _require_cuda(logits, input_ids, thr, conf_state)
        if thr.dtype != torch.float32:
            raise TypeError("thr float32 expected")
    else:
        dev = _require_cuda(logits, input_ids, conf_state, quota, *(() if thr is None else (thr,)))
        if quota.dtype != torch.int32 or quota.numel() != input_ids.shape[0]:
            raise TypeError("quota must be int32 [B]")
    B, L = input_ids.shape
    if input_ids.dtype != torch.int32 or conf_state.dtype != torch.float32:
        raise TypeError("input_ids int32, conf_state float32 expected")
    if logits.element_size() != 2:
        raise TypeError("logits must be a 16-bit (bf16) tensor")
    ldv = logits.shape[-1]
    if not compact and logits.numel() != B * L * ldv:
        raise ValueError("logits must hold B*L rows of the row stride")
    if out is None:
        out = {
            "done": torch.empty(B, dtype=torch.uint8, device=dev),
            "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
            "n_new": torch.empty(B, dtype=torch.int32, device=dev),
        }
        if feats:
            out["feats"] = torch.empty((B, NUM_FEATURES), dtype=torch.float32, device=dev)
        if debug:
            out["conf"] = torch.empty((B, L), dtype=torch.float32, device=dev)
            out["lse"] = torch.empty((B, L), dtype=torch.float32, device=dev)
            out["tok"] = torch.empty((B, L), dtype=torch.int32, device=dev)
    lib = load()
    need = int(lib.dllm_step_workspace_size(B, L, V))
    ws = workspace if workspace is not None else _step_ws.get(dev, need)
    a = StepArgs(B=B, L=L, V=V, mask_id=mask_id, ldv=ldv,
                 logits=_ptr(logits), input_ids=_ptr(input_ids), thr=_ptr(thr), conf_state=_ptr(conf_state),
                 done=_ptr(out["done"]), accept_len=_ptr(out["accept_len"]), n_new=_ptr(out["n_new"]),
                 feats=_ptr(out.get("feats")), conf_out=_ptr(out.get("conf")), lse_out=_ptr(out.get("lse")),
                 tok_out=_ptr(out.get("tok")), workspace=_ptr(ws), workspace_bytes=ws.numel())
    if compact:
        rows = logits.numel() // ldv
        _check("dllm_step_compact", lib.dllm_step_compact(ctypes.byref(a), rows, _ptr(quota), _stream(dev)))
    elif quota is None:
        _check("dllm_step", lib.dllm_step(ctypes.byref(a), _stream(dev)))
    else:
        _check("dllm_step_quota", lib.dllm_step_quota(ctypes.byref(a), _ptr(quota), _stream(dev)))
    return out


def step_sharded(logits, input_ids, thr, conf_state, *, V, mask_id, bounds, feats=True, debug=False, quota=None):
    """The step with S2 split over vocabulary shards [bounds[k], bounds[k+1])
    of one logits array (dllm_step_shard per shard, then dllm_step_merge):
    the single-GPU form of a vocabulary-parallel or chunked LM head.  Each
    bound must be a multiple of 8.  Returns the outputs of ``step``."""
    torch = _torch()
    dev = _require_cuda(logits, input_ids, conf_state, thr, quota)
    B, L = input_ids.shape
    ldv = logits.shape[-1]
    BL = B * L
    n = len(bounds) - 1
    if n < 1 or bounds[0] != 0 or bounds[-1] != V or any(b % 8 for b in bounds[:-1]):
        raise ValueError("bounds must run from 0 to V in multiples of 8")
    tm = torch.empty((n, BL), dtype=torch.float32, device=dev)
    ts = torch.empty((n, BL), dtype=torch.float32, device=dev)
    ti = torch.empty((n, BL), dtype=torch.int32, device=dev)
    lib = load()
    base = logits.data_ptr()
    for k in range(n):
        v0, v1 = bounds[k], bounds[k + 1]
        need = int(lib.dllm_step_workspace_size(B, L, v1 - v0))
        ws = _step_ws.get(dev, need)
        a = StepArgs(B=B, L=L, V=v1 - v0, mask_id=mask_id, ldv=ldv, logits=ctypes.c_void_p(base + v0 * 2),
                     input_ids=_ptr(input_ids), workspace=_ptr(ws), workspace_bytes=ws.numel())
        _check("dllm_step_shard", lib.dllm_step_shard(ctypes.byref(a), v0, _ptr(tm[k]), _ptr(ts[k]), _ptr(ti[k]),
                                                      _stream(dev)))
    out = {"done": torch.empty(B, dtype=torch.uint8, device=dev),
           "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "n_new": torch.empty(B, dtype=torch.int32, device=dev)}
    if feats:
        out["feats"] = torch.empty((B, NUM_FEATURES), dtype=torch.float32, device=dev)
    if debug:
        out["conf"] = torch.full((B, L), float("nan"), dtype=torch.float32, device=dev)
        out["lse"] = torch.full((B, L), float("nan"), dtype=torch.float32, device=dev)
        out["tok"] = torch.full((B, L), -1, dtype=torch.int32, device=dev)
    ws = _step_ws.get(dev, int(lib.dllm_step_workspace_size(B, L, 1)))
    a = StepArgs(B=B, L=L, V=V, mask_id=mask_id, ldv=ldv, logits=None, input_ids=_ptr(input_ids), thr=_ptr(thr),
                 conf_state=_ptr(conf_state), done=_ptr(out["done"]), accept_len=_ptr(out["accept_len"]),
                 n_new=_ptr(out["n_new"]), feats=_ptr(out.get("feats")), conf_out=_ptr(out.get("conf")),
                 lse_out=_ptr(out.get("lse")), tok_out=_ptr(out.get("tok")), workspace=_ptr(ws),
                 workspace_bytes=ws.numel())
    _check("dllm_step_merge", lib.dllm_step_merge(ctypes.byref(a), n, _ptr(tm), _ptr(ts), _ptr(ti), BL, _ptr(quota),
                                                  _stream(dev)))
    return out


def step_vocab_shards(shards, input_ids, thr, conf_state, *, mask_id, feats=True, debug=False, quota=None,
                      workspace=None):
    """The step over logits held as vocabulary shards on this device, in one
    launch (dllm_step_vocab_shards): ``shards`` is a list of (logits, v0, V)
    with logits a 16-bit CUDA tensor of B*L rows holding global tokens
    [v0, v0 + V) in its first V columns (a column slice of a wider array is
    fine: its row stride is taken from the tensor), shards in vocabulary
    order from 0.  Returns the outputs of ``step`` (equal, bit for bit, to
    ``step_sharded`` over the same shards)."""
    torch = _torch()
    dev = _require_cuda(input_ids, conf_state, thr, quota)
    B, L = input_ids.shape
    n = len(shards)
    if not 1 <= n <= MAX_VOCAB_SHARDS:
        raise ValueError(f"1 to {MAX_VOCAB_SHARDS} shards")
    V = sum(w for _, _, w in shards)
    arr = (VocabShard * n)()
    for k, (t, v0, w) in enumerate(shards):
        if not t.is_cuda or t.device != dev:
            raise ValueError("each shard is a CUDA tensor on the device of input_ids")
        if t.element_size() != 2 or t.dim() != 2 or t.shape[0] != B * L or t.stride(1) != 1 or t.shape[1] < w:
            raise ValueError("each shard holds B*L rows of 16-bit logits, at least V columns, unit column stride")
        arr[k] = VocabShard(logits=_ptr(t), ldv=t.stride(0), v0=v0, V=w)
    out = {"done": torch.empty(B, dtype=torch.uint8, device=dev),
           "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "n_new": torch.empty(B, dtype=torch.int32, device=dev)}
    if feats:
        out["feats"] = torch.empty((B, NUM_FEATURES), dtype=torch.float32, device=dev)
    if debug:
        out["conf"] = torch.empty((B, L), dtype=torch.float32, device=dev)
        out["lse"] = torch.empty((B, L), dtype=torch.float32, device=dev)
        out["tok"] = torch.empty((B, L), dtype=torch.int32, device=dev)
    lib = load()
    need = int(lib.dllm_step_workspace_size(B, L, V + 8192 * (n - 1)))
    ws = workspace if workspace is not None else _step_ws.get(dev, need)
    a = StepArgs(B=B, L=L, V=V, mask_id=mask_id, ldv=0, logits=None, input_ids=_ptr(input_ids), thr=_ptr(thr),
                 conf_state=_ptr(conf_state), done=_ptr(out["done"]), accept_len=_ptr(out["accept_len"]),
                 n_new=_ptr(out["n_new"]), feats=_ptr(out.get("feats")), conf_out=_ptr(out.get("conf")),
                 lse_out=_ptr(out.get("lse")), tok_out=_ptr(out.get("tok")), workspace=_ptr(ws),
                 workspace_bytes=ws.numel())
    _check("dllm_step_vocab_shards", lib.dllm_step_vocab_shards(ctypes.byref(a), n, arr, _ptr(quota), _stream(dev)))
    return out


def transfer_quota(L, S, s):
    """dllm_transfer_quota: positions to unmask at step s of a block under
    the fixed-steps rule (L over S steps, the remainder to the first steps;
    L once s >= S)."""
    q = int(load().dllm_transfer_quota(int(L), int(S), int(s)))
    if q < 0:
        raise ValueError("transfer_quota needs L >= 1, S >= 1, s >= 0")
    return q


def step_host(logits_host, input_ids, thr, conf_state, *, V, mask_id, device=None):
    """End-to-end step from host buffers: copy inputs to the device, run
    dllm_step, read the results back.  Host tensors should be pinned for
    asynchronous copies.  Returns host tensors (input_ids / conf_state
    updated, done, accept_len, n_new, feats)."""
    torch = _torch()
    device = device or torch.device("cuda", torch.cuda.current_device())
    d_logits = logits_host.to(device, non_blocking=True)
    d_ids = input_ids.to(device, non_blocking=True)
    d_thr = thr.to(device, non_blocking=True)
    d_cs = conf_state.to(device, non_blocking=True)
    out = step(d_logits, d_ids, d_thr, d_cs, V=V, mask_id=mask_id)
    res = {k: v.to("cpu", non_blocking=True) for k, v in out.items()}
    res["input_ids"] = d_ids.to("cpu", non_blocking=True)
    res["conf_state"] = d_cs.to("cpu", non_blocking=True)
    torch.cuda.current_stream(device).synchronize()
    return res


def features(input_ids, conf_state, *, mask_id, out=None):
    torch = _torch()
    dev = _require_cuda(input_ids, conf_state)
    B, L = input_ids.shape
    if out is None:
        out = torch.empty((B, NUM_FEATURES), dtype=torch.float32, device=dev)
    _check("dllm_features", load().dllm_features(B, L, mask_id, _ptr(input_ids), _ptr(conf_state), _ptr(out),
                                                 _stream(dev)))
    return out


def get_device_error(device=None):
    torch = _torch()
    device = device or torch.device("cuda", torch.cuda.current_device())
    code = _i32(0)
    _check("dllm_get_device_error", load().dllm_get_device_error(_stream(device), ctypes.byref(code)))
    return int(code.value)


# ---------------------------------------------------------------------------
# host planning
# ---------------------------------------------------------------------------
def _host_i32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def pack_plan(p, b, L):
    """(W, cost) of eq. (1) for the active rows (host arrays)."""
    p = _host_i32(p)
    b = _host_i32(b)
    W = _i32(0)
    cost = _i64(0)
    _check("dllm_pack_plan", load().dllm_pack_plan(p.size, p.ctypes.data if p.size else None,
                                                   b.ctypes.data if b.size else None, L,
                                                   ctypes.byref(W), ctypes.byref(cost)))
    return int(W.value), int(cost.value)


def admit(pending_p, active_p, active_b, L, budget):
    """Indices into the sorted pending queue admitted this iteration."""
    pp = _host_i32(pending_p)
    ap = _host_i32(active_p)
    ab = _host_i32(active_b)
    idx = np.zeros(max(pp.size, 1), dtype=np.int32)
    n = _i32(0)
    _check("dllm_admit", load().dllm_admit(pp.size, pp.ctypes.data if pp.size else None, ap.size,
                                           ap.ctypes.data if ap.size else None, ab.ctypes.data if ab.size else None,
                                           L, int(budget), idx.ctypes.data, ctypes.byref(n)))
    return idx[: n.value].tolist()


# ---------------------------------------------------------------------------
# device batch management
# ---------------------------------------------------------------------------
def pack(p, b, rid, prompt_off, prompt_tokens, gen_tokens, block_ids, *, L, W, pad_id, out=None):
    """The [A, W] box (ids, attn, pos) plus pad and blk_start per row."""
    torch = _torch()
    dev = _require_cuda(p, b, rid, prompt_off, prompt_tokens, gen_tokens, block_ids)
    A = p.numel()
    if out is None:
        out = {
            "ids": torch.empty((A, W), dtype=torch.int32, device=dev),
            "attn": torch.empty((A, W), dtype=torch.uint8, device=dev),
            "pos": torch.empty((A, W), dtype=torch.int32, device=dev),
            "pad": torch.empty(A, dtype=torch.int32, device=dev),
            "blk_start": torch.empty(A, dtype=torch.int32, device=dev),
        }
    a = PackArgs(A=A, L=L, W=W, pad_id=pad_id, p=_ptr(p), b=_ptr(b), rid=_ptr(rid), prompt_off=_ptr(prompt_off),
                 prompt_tokens=_ptr(prompt_tokens), gen_tokens=_ptr(gen_tokens), ld_gen=gen_tokens.shape[-1],
                 block_ids=_ptr(block_ids), ids=_ptr(out["ids"]), attn=_ptr(out.get("attn")),
                 pos=_ptr(out.get("pos")), pad=_ptr(out.get("pad")), blk_start=_ptr(out.get("blk_start")))
    _check("dllm_pack", load().dllm_pack(ctypes.byref(a), _stream(dev)))
    return out


def pack_block(block_ids, box_ids, *, L, W):
    """dllm_pack_block: rewrite the active-block columns [W - L, W) of a
    packed box ``box_ids`` [A, W] from ``block_ids`` [A, L] (the in-place
    re-loop's update: nothing else in the box changed)."""
    dev = _require_cuda(block_ids, box_ids)
    A = block_ids.shape[0]
    a = PackArgs(A=A, L=L, W=W, block_ids=_ptr(block_ids), ids=_ptr(box_ids))
    _check("dllm_pack_block", load().dllm_pack_block(ctypes.byref(a), _stream(dev)))
    return box_ids


def advance(adv, rid, K, b, input_ids, conf_state, gen_tokens, *, mask_id, evict=None):
    torch = _torch()
    dev = _require_cuda(adv, rid, K, b, input_ids, conf_state, gen_tokens)
    A, L = input_ids.shape
    if evict is None:
        evict = torch.empty(A, dtype=torch.uint8, device=dev)
    a = AdvanceArgs(A=A, L=L, mask_id=mask_id, advance=_ptr(adv), rid=_ptr(rid), K=_ptr(K), b=_ptr(b),
                    input_ids=_ptr(input_ids), conf_state=_ptr(conf_state), gen_tokens=_ptr(gen_tokens),
                    ld_gen=gen_tokens.shape[-1], evict=_ptr(evict))
    _check("dllm_advance", load().dllm_advance(ctypes.byref(a), _stream(dev)))
    return evict


def compact(evict, arrays, *, new_index=None, src_row=None, A_out=None):
    """Stable in-place compaction of the row arrays by ``evict``."""
    torch = _torch()
    dev = _require_cuda(evict, *arrays)
    A = evict.numel()
    if len(arrays) > COMPACT_MAX_ARRAYS:
        raise ValueError("too many arrays")
    if new_index is None:
        new_index = torch.empty(A, dtype=torch.int32, device=dev)
    if src_row is None:
        src_row = torch.empty(max(A, 1), dtype=torch.int32, device=dev)
    if A_out is None:
        A_out = torch.empty(1, dtype=torch.int32, device=dev)
    rb = [(t.numel() // A) * t.element_size() if A else 1 for t in arrays]
    for t in arrays:
        if A and t.shape[0] != A:
            raise ValueError("every array needs A rows")
    lib = load()
    rb_arr = (_i64 * COMPACT_MAX_ARRAYS)(*rb)
    need = int(lib.dllm_compact_workspace_size(A, len(arrays), ctypes.cast(rb_arr, ctypes.c_void_p)))
    ws = _compact_ws.get(dev, need)
    arr_ptrs = (_p * COMPACT_MAX_ARRAYS)(*[t.data_ptr() for t in arrays])
    a = CompactArgs(A=A, n_arrays=len(arrays), evict=_ptr(evict), new_index=_ptr(new_index), src_row=_ptr(src_row),
                    A_out=_ptr(A_out), arrays=arr_ptrs, row_bytes=rb_arr, workspace=_ptr(ws),
                    workspace_bytes=ws.numel())
    _check("dllm_compact", lib.dllm_compact(ctypes.byref(a), _stream(dev)))
    return new_index, src_row, A_out


def advance_compact(adv, rid, K, b, input_ids, conf_state, gen_tokens, arrays, *, mask_id, evict=None,
                    new_index=None, src_row=None, A_out=None, workspace=True):
    """dllm_advance_compact: commit the advanced rows' blocks, then compact
    ``arrays`` (which may include b / input_ids / conf_state) by the evict
    flags.  With ``workspace`` a compaction workspace is passed, which lets
    large batches take the multi-CTA path.  Returns (evict, new_index,
    src_row, A_out)."""
    torch = _torch()
    dev = _require_cuda(adv, rid, K, b, input_ids, conf_state, gen_tokens, *arrays)
    A, L = input_ids.shape
    if len(arrays) > COMPACT_MAX_ARRAYS:
        raise ValueError("too many arrays")
    for t in arrays:
        if A and t.shape[0] != A:
            raise ValueError("every array needs A rows")
    if evict is None:
        evict = torch.empty(max(A, 1), dtype=torch.uint8, device=dev)
    if new_index is None:
        new_index = torch.empty(max(A, 1), dtype=torch.int32, device=dev)
    if src_row is None:
        src_row = torch.empty(max(A, 1), dtype=torch.int32, device=dev)
    if A_out is None:
        A_out = torch.empty(1, dtype=torch.int32, device=dev)
    aa = AdvanceArgs(A=A, L=L, mask_id=mask_id, advance=_ptr(adv), rid=_ptr(rid), K=_ptr(K), b=_ptr(b),
                     input_ids=_ptr(input_ids), conf_state=_ptr(conf_state), gen_tokens=_ptr(gen_tokens),
                     ld_gen=gen_tokens.shape[-1], evict=_ptr(evict))
    rb = [(t.numel() // A) * t.element_size() if A else 1 for t in arrays]
    rb_arr = (_i64 * COMPACT_MAX_ARRAYS)(*rb)
    arr_ptrs = (_p * COMPACT_MAX_ARRAYS)(*[t.data_ptr() for t in arrays])
    ws = None
    if workspace:
        need = int(load().dllm_compact_workspace_size(A, len(arrays), ctypes.cast(rb_arr, ctypes.c_void_p)))
        ws = _compact_ws.get(dev, need)
    ca = CompactArgs(A=A, n_arrays=len(arrays), evict=_ptr(evict), new_index=_ptr(new_index),
                     src_row=_ptr(src_row), A_out=_ptr(A_out), arrays=arr_ptrs, row_bytes=rb_arr,
                     workspace=_ptr(ws), workspace_bytes=0 if ws is None else ws.numel())
    _check("dllm_advance_compact", load().dllm_advance_compact(ctypes.byref(aa), ctypes.byref(ca), _stream(dev)))
    return evict, new_index, src_row, A_out


def refill(A0, new_rid, new_p, new_K, new_thr, rid, p, b, K, thr, input_ids, conf_state, *, mask_id):
    """Initialise rows [A0, A0 + n) for admitted requests (dllm_refill)."""
    dev = _require_cuda(new_rid, new_p, new_K, new_thr, rid, p, b, K, thr, input_ids, conf_state)
    n = new_rid.numel()
    a = RefillArgs(A0=A0, n=n, L=input_ids.shape[1], mask_id=mask_id, new_rid=_ptr(new_rid), new_p=_ptr(new_p),
                   new_K=_ptr(new_K), new_thr=_ptr(new_thr), rid=_ptr(rid), p=_ptr(p), b=_ptr(b), K=_ptr(K),
                   thr=_ptr(thr), input_ids=_ptr(input_ids), conf_state=_ptr(conf_state))
    _check("dllm_refill", load().dllm_refill(ctypes.byref(a), _stream(dev)))
