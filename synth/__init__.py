"""Seeded synthetic inputs for the denoise step, the pack and the compaction.

Test and benchmark infrastructure.  This module holds none of the method's
arithmetic: it only draws inputs.  Both the CUDA path and the CPU oracle take
their inputs from here, so neither has to trust the other's input handling.

Every random number comes from one counter-based generator, the SplitMix64
output function (Steele, Lea & Flood, OOPSLA 2014), addressed by a key chain
``out(key, k) = mix(key + (k + 1) * 0x9e3779b97f4a7c15)``.  Small per-request
and per-position arrays are drawn here in numpy; whole logits rows are drawn
by the C half (``synth.c``) from per-row keys computed here.

Workload shapes follow the pages:

* Block length L = 32 and the LLaDA-8B / Dream-7B vocabularies (BlockServe
  page, section III-A; DiLaServe review, section 6.1).
* Per-request thresholds from the administrator's candidate set
  {0.5, 0.6, 0.7, 0.8, 0.9} (DiLaServe review, section 4.1).
* Prompt lengths and gen length 256 in blocks of 32 for the mixed-state loop
  (BlockServe page, sections II-A and II-D).

Logits model (one reading; the pages give no logits distribution): each
element is a bf16 draw of N(0, 1) through a 2^16-entry inverse-normal table;
each row has one planted peak token whose value is the table maximum plus an
offset U[0, O]; the mask column holds -30 so it is never the argmax.
"""
from __future__ import annotations

import ctypes
import os
import statistics
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lib_lock = threading.Lock()

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Sub-stream tags (first link of every key chain after the seed).
TAG_MASK_FRACTION = 1
TAG_MASK_DRAW = 2
TAG_THRESHOLD = 3
TAG_TOKEN = 4
TAG_CONF_STATE = 5
TAG_PROMPT_LEN = 6
TAG_LOGITS = 7
TAG_PROMPT_TOKEN = 8
TAG_BLOCK_INDEX = 9
TAG_GEN_TOKEN = 10

THRESHOLD_SET = (0.5, 0.6, 0.7, 0.8, 0.9)


# --------------------------------------------------------------------------
# SplitMix64, vectorised over uint64 arrays (wrapping arithmetic).
# --------------------------------------------------------------------------
def mix(z):
    z = np.asarray(z, dtype=np.uint64).copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def out(key, k):
    """k-th SplitMix64 output of the stream seeded with ``key`` (broadcasts)."""
    key = np.asarray(key, dtype=np.uint64)
    k = np.asarray(k, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix(key + (k + np.uint64(1)) * GAMMA)


def chain(seed, *ids):
    """Key chain: out(out(out(seed, id0), id1), ...), broadcasting over ids."""
    key = np.asarray(np.uint64(seed & 0xFFFFFFFFFFFFFFFF), dtype=np.uint64)
    for i in ids:
        key = out(key, np.asarray(i, dtype=np.int64).astype(np.uint64))
    return key


def uniform01(key, k):
    """Uniform double in [0, 1) with 53 random bits."""
    return (out(key, k) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform_int(key, k, lo, hi):
    """Uniform integer in [lo, hi] (inclusive); modulo bias below 2^-40."""
    span = np.uint64(hi - lo + 1)
    return (out(key, k) % span).astype(np.int64) + lo


# --------------------------------------------------------------------------
# bf16 tables.
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (round to nearest even); returns uint16."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_bg_cache = None
_peak_cache: dict = {}


def bg_table():
    """bf16 of the N(0,1) quantile at (k + 0.5) / 2^16, k = 0..65535."""
    global _bg_cache
    if _bg_cache is None:
        nd = statistics.NormalDist()
        q = np.array([nd.inv_cdf((k + 0.5) / 65536.0) for k in range(65536)], dtype=np.float64)
        _bg_cache = f32_to_bf16_bits(q.astype(np.float32))
    return _bg_cache


def bg_max():
    return float(bf16_bits_to_f32(bg_table()).max())


def peak_table(offset_max):
    """bf16 of bg_max + offset_max * (k + 0.5) / 2^16: the planted peak value."""
    key = float(offset_max)
    if key not in _peak_cache:
        k = np.arange(65536, dtype=np.float64)
        v = np.float32(bg_max()) + (offset_max * (k + 0.5) / 65536.0).astype(np.float32)
        _peak_cache[key] = f32_to_bf16_bits(v.astype(np.float32))
    return _peak_cache[key]


# --------------------------------------------------------------------------
# C bulk generator.
# --------------------------------------------------------------------------
def build(force=False, cc="gcc"):
    """Compile synth.c into libsynth.so next to it."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([cc, "-O2", "-std=c99", "-shared", "-fPIC", "-pthread", src, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.synth_logits_rows.restype = ctypes.c_int
            lib.synth_logits_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int]
            lib.synth_splitmix_out.restype = ctypes.c_uint64
            lib.synth_splitmix_out.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            _lib = lib
    return _lib


def default_threads():
    return max(1, min(32, os.cpu_count() or 1))


def fill_logits_rows(out_u16, V, dst_rows, row_keys, offset_max, mask_col, nthreads=None):
    """Write generated rows into ``out_u16`` (2-D uint16 array [rows, ldv]).

    ``out_u16`` may be a numpy array or any object exposing a host pointer via
    ``__array_interface__`` (pinned torch tensors go through ``.numpy()``).
    """
    lib = _load()
    arr = out_u16
    assert arr.dtype == np.uint16 and arr.ndim == 2 and arr.flags["C_CONTIGUOUS"]
    dst = np.ascontiguousarray(dst_rows, dtype=np.int64)
    keys = np.ascontiguousarray(row_keys, dtype=np.uint64)
    assert dst.shape == keys.shape
    if dst.size and (dst.min() < 0 or dst.max() >= arr.shape[0]):
        raise ValueError("destination row out of range")
    bg = bg_table()
    pk = peak_table(offset_max)
    rc = lib.synth_logits_rows(arr.ctypes.data, arr.shape[1], V, dst.size,
                               dst.ctypes.data, keys.ctypes.data, bg.ctypes.data, pk.ctypes.data,
                               int(mask_col), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("synth_logits_rows rejected its arguments")


def logits_row_keys(seed, rid, block, step, pos, salt):
    """Per-row keys for the logits of position ``pos`` of request ``rid``'s
    block ``block`` at denoise step ``step`` (all broadcast)."""
    return chain(seed, TAG_LOGITS, rid, block, step, pos, salt)


# --------------------------------------------------------------------------
# Workload recipes.
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class StepConfig:
    """One denoise-step workload over a mixed-state batch."""
    name: str
    B: int
    L: int
    V: int
    offset_max: float
    mask_mode: str                    # "half" or "fraction"
    thresholds: tuple                 # candidate set; one value = fixed
    features: bool = True
    ldv: int = 0                      # 0: V rounded up to a multiple of 8

    @property
    def row_stride(self):
        return self.ldv if self.ldv else (self.V + 7) // 8 * 8

    @property
    def mask_id(self):
        return self.V - 1


@dataclass(frozen=True)
class LoopConfig:
    """BlockServe-style mixed-state loop: FDFO step, evict, refill."""
    name: str
    R: int                 # requests in the pending queue
    p_lo: int
    p_hi: int
    gen: int               # g_i for every request
    L: int
    V: int
    budget: int            # token budget of eq. (1)
    threshold: float
    offset_max: float

    @property
    def K(self):
        return -(-self.gen // self.L)

    @property
    def mask_id(self):
        return self.V - 1

    @property
    def pad_id(self):
        return self.V - 2

    @property
    def row_stride(self):
        return (self.V + 7) // 8 * 8


STEP_CONFIGS = {
    "tiny": StepConfig("tiny", 4, 32, 1024, 8.0, "half", (0.9,)),
    "llada": StepConfig("llada", 64, 32, 126464, 12.0, "fraction", (0.9,)),
    "dream": StepConfig("dream", 128, 32, 151936, 12.0, "fraction", THRESHOLD_SET),
    "stress": StepConfig("stress", 512, 64, 151936, 12.0, "fraction", THRESHOLD_SET),
}

LOOP_CONFIGS = {
    "blockserve": LoopConfig("blockserve", 256, 64, 1024, 256, 32, 126464, 1 << 20, 0.9, 12.0),
    # the same queue shape served at a small batch: the budget of eq. (1)
    # holds about four widest rows
    "blockserve_small": LoopConfig("blockserve_small", 64, 64, 1024, 256, 32, 126464, 5120, 0.9, 12.0),
}


@dataclass
class StepInputs:
    """Host arrays of one step workload.  ``logits`` is filled only on the
    masked rows; unmasked rows hold ``fill_bits`` (never read by the step)."""
    cfg: StepConfig
    seed: int
    input_ids: np.ndarray        # int32 [B, L]
    thr: np.ndarray              # float32 [B]
    conf_state: np.ndarray       # float32 [B, L]; NaN on masked positions
    salt: np.ndarray             # int64 [B, L]; per-position redraw counter
    logits: np.ndarray = field(default=None)   # uint16 [B*L, ldv]

    @property
    def masked(self):
        return self.input_ids == self.cfg.mask_id


def make_step_state(cfg: StepConfig, seed: int, B=None):
    """Draw input_ids / thresholds / conf_state for a step workload."""
    B = cfg.B if B is None else B
    L, V = cfg.L, cfg.V
    b = np.arange(B, dtype=np.int64)
    pos = (b[:, None] * L + np.arange(L, dtype=np.int64)[None, :])
    if cfg.mask_mode == "half":
        frac = np.full(B, 0.5)
    elif cfg.mask_mode == "fraction":
        frac = uniform01(chain(seed, TAG_MASK_FRACTION), b)
    elif cfg.mask_mode == "all":
        frac = np.ones(B)
    else:
        raise ValueError(cfg.mask_mode)
    masked = uniform01(chain(seed, TAG_MASK_DRAW), pos) < frac[:, None]
    if len(cfg.thresholds) == 1:
        thr = np.full(B, cfg.thresholds[0], dtype=np.float32)
    else:
        pick = uniform_int(chain(seed, TAG_THRESHOLD), b, 0, len(cfg.thresholds) - 1)
        thr = np.asarray(cfg.thresholds, dtype=np.float32)[pick]
    tokens = uniform_int(chain(seed, TAG_TOKEN), pos, 0, V - 2)
    input_ids = np.where(masked, cfg.mask_id, tokens).astype(np.int32)
    u = uniform01(chain(seed, TAG_CONF_STATE), pos)
    cs = (thr.astype(np.float64)[:, None] + u * (1.0 - thr.astype(np.float64)[:, None])).astype(np.float32)
    conf_state = np.where(masked, np.float32(np.nan), cs).astype(np.float32)
    return StepInputs(cfg, seed, input_ids, thr, conf_state, np.zeros((B, L), dtype=np.int64))


def step_row_keys(inp: StepInputs, flat_rows):
    L = inp.cfg.L
    flat_rows = np.asarray(flat_rows, dtype=np.int64)
    rid = flat_rows // L
    pos = flat_rows % L
    return logits_row_keys(inp.seed, rid, 0, 0, pos, inp.salt.reshape(-1)[flat_rows])


POISON_BITS = np.uint16(0x7F00)   # bf16 1.7e38: overflows any softmax that reads it


def fill_step_logits(inp: StepInputs, out=None, rows=None, fill_bits=POISON_BITS, nthreads=None):
    """Generate the logits of the masked rows (or of ``rows``) into ``out``."""
    cfg = inp.cfg
    B, L = inp.input_ids.shape
    if out is None:
        out = np.empty((B * L, cfg.row_stride), dtype=np.uint16)
        if fill_bits is not None:
            out.fill(fill_bits)
    if rows is None:
        rows = np.flatnonzero(inp.masked.reshape(-1))
    rows = np.asarray(rows, dtype=np.int64)
    fill_logits_rows(out, cfg.V, rows, step_row_keys(inp, rows), cfg.offset_max, cfg.mask_id, nthreads)
    inp.logits = out
    return out


def make_step_inputs(cfg: StepConfig, seed: int, fill_bits=POISON_BITS, nthreads=None):
    inp = make_step_state(cfg, seed)
    fill_step_logits(inp, fill_bits=fill_bits, nthreads=nthreads)
    return inp


# --------------------------------------------------------------------------
# Loop workload: the pending queue.
# --------------------------------------------------------------------------
@dataclass
class LoopRequests:
    cfg: LoopConfig
    seed: int
    p: np.ndarray             # int32 [R] prompt length
    K: np.ndarray             # int32 [R] blocks to generate
    prompt_off: np.ndarray    # int64 [R + 1]
    prompt_tokens: np.ndarray  # int32 [sum p]
    thr: np.ndarray           # float32 [R]


def make_loop_requests(cfg: LoopConfig, seed: int, R=None):
    R = cfg.R if R is None else R
    rid = np.arange(R, dtype=np.int64)
    p = uniform_int(chain(seed, TAG_PROMPT_LEN), rid, cfg.p_lo, cfg.p_hi).astype(np.int32)
    off = np.zeros(R + 1, dtype=np.int64)
    off[1:] = np.cumsum(p)
    owner = np.repeat(rid, p)
    within = np.arange(off[-1], dtype=np.int64) - off[owner]
    toks = uniform_int(chain(seed, TAG_PROMPT_TOKEN), owner * 65536 + within, 0, cfg.V - 3).astype(np.int32)
    K = np.full(R, cfg.K, dtype=np.int32)
    thr = np.full(R, cfg.threshold, dtype=np.float32)
    return LoopRequests(cfg, seed, p, K, off, toks, thr)


def mixed_block_index(seed, R, K):
    """Block index b_i ~ U{0..K-1} per request: a mixed-state batch in which
    requests sit at different blocks (BlockServe page, section II-A)."""
    return uniform_int(chain(seed, TAG_BLOCK_INDEX), np.arange(R, dtype=np.int64), 0, K - 1).astype(np.int32)


def committed_tokens(seed, R, n, V):
    """Tokens of already committed blocks, [R, n] (never the mask or pad id)."""
    idx = np.arange(R * n, dtype=np.int64)
    return uniform_int(chain(seed, TAG_GEN_TOKEN), idx, 0, V - 3).astype(np.int32).reshape(R, n)
