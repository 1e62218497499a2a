#!/usr/bin/env python3
"""Benchmark of the denoise-step hot path on the Dream-7B-shaped batch.

One step = one FDFO iteration of the whole hot path over a mixed-state batch
of 128 requests (L = 32, V = 151936, per-request thresholds from
{0.5, ..., 0.9}, per-request mask fraction U[0, 1], prompt lengths
U[64, 1024] and block indices U{0..7}):

  S8      dllm_admit    host sand-fill admission plan under the 2^20 budget
  S7      dllm_pack     the left-padded [128, W] box
  S1-S6   dllm_step     confidence / argmax / select / update / done / features
  S9      dllm_advance + dllm_compact   commit finished blocks, evict, compact

Every step starts from the same state: the mutable state of R steps is staged
in a ring in HBM and restored with one device copy per pass over the ring
(inside the timed region).  The logits (0.62 GB of masked rows, 1.24 GB
allocated) exceed the 129 MB L2, so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "masked positions/sec and logits GB/s per denoise step (% of GB300 HBM peak), 1 GPU"
UNIT = "masked positions/s"
WORKLOADS = {
    "dream": "dream7b_shaped_mixed_state_step",
    "dream_fixed_steps": "dream7b_shaped_mixed_state_step_fixed_steps_S32",
    "dream_vocab4": "dream7b_shaped_mixed_state_step_4_vocab_shards",
    "llada": "llada8b_shaped_mixed_state_step",
    "stress": "large_batch_stress_step",
    "tiny": "tiny_step",
    "blockserve": "blockserve_mixed_state_loop",
    "blockserve_small": "blockserve_mixed_state_loop_small_batch",
}
LOOP_K = 8                     # blocks per request (gen 256 / L 32)
BUDGET = 1 << 20               # token budget of eq. (1)
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0       # GB300 HBM3e nominal, for context beside the measured peak
RING = 64


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: one independent batch per rank)
# ---------------------------------------------------------------------------
def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(units_local, seconds_local, dist=None):
    """Whole-job units and the max elapsed time over ranks."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(units_local), float(seconds_local)
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    u = torch.tensor([float(units_local)], dtype=torch.float64, device=dev)
    t = torch.tensor([float(seconds_local)], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(u.item()), float(t.item())


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
FIXED_STEPS_S = 32   # the pages' S = 32 denoising steps per block of L = 32


def step_config_name(name):
    """Step configuration behind a workload name (the fixed-steps workload
    runs the Dream-shaped batch under the fixed-steps rule)."""
    return "dream" if name in synth.LOOP_CONFIGS or name in ("dream_fixed_steps", "dream_vocab4") else name


def make_workload(seed, name="dream"):
    cfg = synth.STEP_CONFIGS[step_config_name(name)]
    inp = synth.make_step_state(cfg, seed)
    lcfg = synth.LoopConfig("mixed", cfg.B, 64, 1024, LOOP_K * cfg.L, cfg.L, cfg.V, BUDGET, 0.9, cfg.offset_max)
    reqs = synth.make_loop_requests(lcfg, seed)
    b = synth.mixed_block_index(seed, cfg.B, LOOP_K)
    gen = synth.committed_tokens(seed, cfg.B, LOOP_K * cfg.L, cfg.V)
    pend = synth.make_loop_requests(lcfg, seed + 77)
    pending_p = np.sort(pend.p).astype(np.int32)
    return cfg, inp, reqs, b, gen, pending_p


def workload_config(name, cfg, inp, W, cost, fixed):
    """The ``config`` object of the JSON line: what the workload is, the
    same for the GPU arm and the reference arm."""
    return {"workload": WORKLOADS[name], "B": cfg.B, "L": cfg.L, "V": cfg.V, "masked_rows": int(inp.masked.sum()),
            "rule": (f"fixed steps, S = {FIXED_STEPS_S} per block" if fixed else
                     "threshold per request from {0.5,0.6,0.7,0.8,0.9}"),
            "mask_fraction": "U[0,1] per request", "box_W": int(W), "box_cost": int(cost), "token_budget": BUDGET}


def algorithmic_bytes(cfg, M):
    """Bytes one dllm_step launch must move: the masked logits rows plus the
    per-position state (input_ids and conf_state read and written) and the
    per-request inputs / outputs (thr, done, accept_len, n_new, features)."""
    B, L, V = cfg.B, cfg.L, cfg.V
    return M * V * 2 + B * L * 16 + B * (4 + 1 + 4 + 4 + 24)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "step_kernel_dream.json")


def load_traffic(step_src_sha, path=TRAFFIC_JSON):
    """ncu DRAM bytes per launch of the step kernel on the Dream-shaped
    batch, from the committed capture record, if that capture was taken on
    the current kernel source; else None."""
    try:
        with open(path, encoding="utf-8") as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != step_src_sha:
        return None
    v = rec.get("dram_bytes_per_launch")
    return float(v) if v is not None else None


def step_source_sha():
    import hashlib
    h = hashlib.sha256()
    for fn in ("step.cu", "common.cuh", "compact.cuh"):
        with open(os.path.join(ROOT, "denoise_step_token_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_id:
            cmd[1:1] = ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock, the maximum clock and every throttle reason seen
        active, from `nvidia-smi --query-gpu=<FIELDS> --format=csv,noheader,
        nounits` lines (malformed lines are skipped); None without a sample."""
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU pipeline
# ---------------------------------------------------------------------------
class Pipeline:
    """Device buffers and prebuilt C-ABI argument structs for one batch."""

    def __init__(self, cfg, inp, reqs, b, gen, pending_p, device, ring=RING, fixed_steps=None, vocab_shards=None,
                 fused=True):
        import torch
        import denoise_step_token_gb300 as dllm
        self.torch, self.dllm, self.lib = torch, dllm, dllm.load()
        self.cfg, self.device, self.ring = cfg, device, ring
        B, L, V = cfg.B, cfg.L, cfg.V
        KL = LOOP_K * L
        self.B, self.L = B, L
        self.M = int(inp.masked.sum())
        # logits: poison everywhere, generated rows where masked
        ldv = cfg.row_stride
        self.logits = torch.empty((B * L, ldv), dtype=torch.int16, device=device)
        self.logits.fill_(int(np.uint16(synth.POISON_BITS).view(np.int16)))
        rows = np.flatnonzero(inp.masked.reshape(-1))
        self.masked_rows = rows
        for s0 in range(0, len(rows), 1024):
            part = rows[s0:s0 + 1024]
            h = np.empty((len(part), ldv), dtype=np.uint16)
            synth.fill_logits_rows(h, V, np.arange(len(part)), synth.step_row_keys(inp, part), cfg.offset_max,
                                   cfg.mask_id)
            self.logits[torch.from_numpy(part).to(device)] = torch.from_numpy(h.view(np.int16)).to(device)
        # static pack inputs
        self.prompt_off = torch.from_numpy(reqs.prompt_off).to(device)
        self.prompt_tokens = torch.from_numpy(reqs.prompt_tokens).to(device)
        # slot layout (int32 words): ids | cs | thr | p | b | K | rid | gen
        self.words = {"ids": B * L, "cs": B * L, "thr": B, "p": B, "b": B, "K": B, "rid": B, "gen": B * KL}
        off, self.off = 0, {}
        for k, n in self.words.items():
            self.off[k] = off
            off += n
        self.slot_words = off
        host = np.zeros(off, dtype=np.int32)
        host[self.off["ids"]:self.off["ids"] + B * L] = inp.input_ids.reshape(-1)
        host[self.off["cs"]:self.off["cs"] + B * L] = inp.conf_state.reshape(-1).view(np.int32)
        host[self.off["thr"]:self.off["thr"] + B] = inp.thr.view(np.int32)
        host[self.off["p"]:self.off["p"] + B] = reqs.p
        host[self.off["b"]:self.off["b"] + B] = b
        host[self.off["K"]:self.off["K"] + B] = LOOP_K
        host[self.off["rid"]:self.off["rid"] + B] = np.arange(B, dtype=np.int32)
        host[self.off["gen"]:self.off["gen"] + B * KL] = gen.reshape(-1)
        self.slot_host = host
        pristine = torch.from_numpy(np.tile(host, (ring, 1))).to(device)
        self.pristine = pristine
        self.state = pristine.clone()
        # outputs (per slot, not restored): one contiguous block per slot --
        # feats | accept_len | n_new | A_out | done -- so that a reader
        # fetches a step's results with one copy
        o_acc, o_new, o_A = B * 24, B * 28, B * 32
        o_done = o_A + 16
        self.out_bytes = (o_done + B + 255) // 256 * 256
        self.out = torch.zeros((ring, self.out_bytes), dtype=torch.uint8, device=device)
        self.feats = self.out[:, :o_acc].view(torch.float32).unflatten(1, (B, 6))
        self.accept = self.out[:, o_acc:o_new].view(torch.int32)
        self.n_new = self.out[:, o_new:o_A].view(torch.int32)
        self.A_out = self.out[:, o_A:o_A + 4].view(torch.int32)
        self.done = self.out[:, o_done:o_done + B]
        self.evict = torch.empty((ring, B), dtype=torch.uint8, device=device)
        self.new_index = torch.empty((ring, B), dtype=torch.int32, device=device)
        self.src_row = torch.empty((ring, B), dtype=torch.int32, device=device)
        # box (shared by every slot)
        self.W, self.cost = dllm.pack_plan(reqs.p, b, L)
        self.box_ids = torch.empty((B, self.W), dtype=torch.int32, device=device)
        self.box_attn = torch.empty((B, self.W), dtype=torch.uint8, device=device)
        self.box_pos = torch.empty((B, self.W), dtype=torch.int32, device=device)
        self.box_pad = torch.empty(B, dtype=torch.int32, device=device)
        self.box_start = torch.empty(B, dtype=torch.int32, device=device)
        # workspaces
        # a vocabulary-sharded step has one more partial chunk per shard boundary
        ws_bytes = self.lib.dllm_step_workspace_size(B, L, V + 8192 * (int(vocab_shards or 1) - 1))
        self.step_ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
        rb = [L * 4, L * 4, 4, 4, 4, 4, 4]
        self.rb_arr = (ctypes.c_int64 * dllm.COMPACT_MAX_ARRAYS)(*rb)
        cws = self.lib.dllm_compact_workspace_size(B, len(rb), ctypes.cast(self.rb_arr, ctypes.c_void_p))
        self.compact_ws = torch.empty(cws, dtype=torch.uint8, device=device)
        # host admission inputs (S8)
        self.pending_p = np.ascontiguousarray(pending_p, dtype=np.int32)
        self.active_p = np.ascontiguousarray(reqs.p, dtype=np.int32)
        self.active_b = np.ascontiguousarray(b, dtype=np.int32)
        self.admit_idx = np.zeros(max(len(pending_p), 1), dtype=np.int32)
        self.n_admit = ctypes.c_int32(0)
        self.args = [self._build_args(s) for s in range(ring)]
        # fixed-steps rule: request b has taken L - (its masked count) steps
        # of its block (one token per step at S = L), so its quota is
        # transfer_quota(L, S, that step)
        # vocabulary shards: column slices of the logits array, all stepped in
        # one launch (dllm_step_vocab_shards)
        self.shards = None
        if vocab_shards:
            n = int(vocab_shards)
            width = -(-(cfg.V // n) // 8) * 8
            bounds = [min(k * width, cfg.V) for k in range(n)] + [cfg.V]
            self.shards = (dllm.VocabShard * n)()
            for k in range(n):
                self.shards[k] = dllm.VocabShard(logits=ctypes.c_void_p(self.logits.data_ptr() + bounds[k] * 2),
                                                 ldv=self.logits.shape[1], v0=bounds[k], V=bounds[k + 1] - bounds[k])
        # the step, block commit and compaction in one launch; else the step,
        # then dllm_advance_compact (the comparison pipeline)
        self.fused = bool(fused)
        self.quota = None
        if fixed_steps is not None:
            steps = L - inp.masked.sum(axis=1)
            q = np.array([dllm.transfer_quota(L, fixed_steps, int(t)) for t in steps], dtype=np.int32)
            self.quota = torch.from_numpy(q).to(device)
            self.quota_ptr = ctypes.c_void_p(self.quota.data_ptr())

    def view(self, slot, name, dtype=None, shape=None):
        t = self.state[slot, self.off[name]:self.off[name] + self.words[name]]
        if dtype is not None:
            t = t.view(dtype)
        return t.view(*shape) if shape else t

    def _build_args(self, s):
        torch, dllm = self.torch, self.dllm
        B, L, cfg = self.B, self.L, self.cfg
        ptr = lambda t: ctypes.c_void_p(t.data_ptr())
        ids = self.view(s, "ids")
        cs = self.view(s, "cs", torch.float32)
        thr = self.view(s, "thr", torch.float32)
        p, b, K, rid, gen = (self.view(s, n) for n in ("p", "b", "K", "rid", "gen"))
        pa = dllm.PackArgs(A=B, L=L, W=self.W, pad_id=cfg.V - 2, p=ptr(p), b=ptr(b), rid=ptr(rid),
                           prompt_off=ptr(self.prompt_off), prompt_tokens=ptr(self.prompt_tokens), gen_tokens=ptr(gen),
                           ld_gen=LOOP_K * L, block_ids=ptr(ids), ids=ptr(self.box_ids), attn=ptr(self.box_attn),
                           pos=ptr(self.box_pos), pad=ptr(self.box_pad), blk_start=ptr(self.box_start))
        sa = dllm.StepArgs(B=B, L=L, V=cfg.V, mask_id=cfg.mask_id, ldv=self.logits.shape[1], logits=ptr(self.logits),
                           input_ids=ptr(ids), thr=ptr(thr), conf_state=ptr(cs), done=ptr(self.done[s]),
                           accept_len=ptr(self.accept[s]), n_new=ptr(self.n_new[s]), feats=ptr(self.feats[s]),
                           conf_out=None, lse_out=None, tok_out=None, workspace=ptr(self.step_ws),
                           workspace_bytes=self.step_ws.numel())
        aa = dllm.AdvanceArgs(A=B, L=L, mask_id=cfg.mask_id, advance=ptr(self.done[s]), rid=ptr(rid), K=ptr(K),
                              b=ptr(b), input_ids=ptr(ids), conf_state=ptr(cs), gen_tokens=ptr(gen),
                              ld_gen=LOOP_K * L, evict=ptr(self.evict[s]))
        arrays = [ids, cs, thr, p, b, K, rid]
        arr = (ctypes.c_void_p * dllm.COMPACT_MAX_ARRAYS)(*[t.data_ptr() for t in arrays])
        ca = dllm.CompactArgs(A=B, n_arrays=len(arrays), evict=ptr(self.evict[s]), new_index=ptr(self.new_index[s]),
                              src_row=ptr(self.src_row[s]), A_out=ptr(self.A_out[s]), arrays=arr,
                              row_bytes=self.rb_arr, workspace=ptr(self.compact_ws),
                              workspace_bytes=self.compact_ws.numel())
        return pa, sa, aa, ca

    def admit_host(self):
        lib = self.lib
        rc = lib.dllm_admit(len(self.pending_p), self.pending_p.ctypes.data, len(self.active_p),
                            self.active_p.ctypes.data, self.active_b.ctypes.data, self.L, BUDGET,
                            self.admit_idx.ctypes.data, ctypes.byref(self.n_admit))
        if rc:
            raise RuntimeError(f"dllm_admit failed: {rc}")

    def run(self, slot, stream, ev_before=None, ev_after=None, compact=None):
        """One pipeline step on state slot ``slot``.  ``compact``: (device
        logits of the masked rows only, their count) to read those through
        the compact layout instead of the full logits array.  With the fused
        commit the step, block commit and compaction are one launch
        (dllm_step_commit); otherwise the step, then dllm_advance_compact."""
        lib = self.lib
        pa, sa, aa, ca = self.args[slot]
        self.admit_host()
        rc = lib.dllm_pack(ctypes.byref(pa), stream)
        if ev_before is not None:
            ev_before.record()
        if self.fused:
            rc |= self.launch_step_commit(slot, stream, compact)
        else:
            rc |= self.launch_step(slot, stream, compact)
        if ev_after is not None:
            ev_after.record()
        if not self.fused:
            rc |= lib.dllm_advance_compact(ctypes.byref(aa), ctypes.byref(ca), stream)
        if rc:
            raise RuntimeError("a dllm call failed inside the timed loop")

    def launch_step_commit(self, slot, stream, compact=None):
        """The step with its block commit and compaction (dllm_step_commit,
        or dllm_step_vocab_shards_commit over vocabulary shards) on state
        slot ``slot``; returns the status code."""
        pa, sa, aa, ca = self.args[slot]
        quota = self.quota_ptr if self.quota is not None else None
        if self.shards is not None and compact is None:
            saved = sa.logits
            sa.logits = None
            rc = self.lib.dllm_step_vocab_shards_commit(ctypes.byref(sa), len(self.shards), self.shards, quota,
                                                        ctypes.byref(aa), ctypes.byref(ca), stream)
            sa.logits = saved
            return rc
        if compact is None:
            return self.lib.dllm_step_commit(ctypes.byref(sa), quota, -1, ctypes.byref(aa), ctypes.byref(ca), stream)
        buf, rows = compact
        saved = sa.logits
        sa.logits = ctypes.c_void_p(buf.data_ptr())
        rc = self.lib.dllm_step_commit(ctypes.byref(sa), quota, rows, ctypes.byref(aa), ctypes.byref(ca), stream)
        sa.logits = saved
        return rc

    def launch_step(self, slot, stream, compact=None):
        """The step of one pipeline step on state slot ``slot`` (dllm_step,
        dllm_step_quota, dllm_step_vocab_shards or dllm_step_compact);
        returns the OR of the status codes."""
        lib = self.lib
        sa = self.args[slot][1]
        rc = 0
        if self.shards is not None and compact is None:
            saved = sa.logits
            sa.logits = None
            rc |= lib.dllm_step_vocab_shards(ctypes.byref(sa), len(self.shards), self.shards, None, stream)
            sa.logits = saved
        elif compact is not None:
            buf, rows = compact
            saved = sa.logits
            sa.logits = ctypes.c_void_p(buf.data_ptr())
            rc |= lib.dllm_step_compact(ctypes.byref(sa), rows, self.quota_ptr if self.quota is not None else None,
                                        stream)
            sa.logits = saved
        elif self.quota is None:
            rc |= lib.dllm_step(ctypes.byref(sa), stream)
        else:
            rc |= lib.dllm_step_quota(ctypes.byref(sa), self.quota_ptr, stream)
        return rc

    def restore(self):
        self.state.copy_(self.pristine)

    def launches_per_step(self):
        """Kernels one ``run`` launches: pack, then either the step with the
        fused commit (one launch), or the step over the vocabulary shards
        (one launch) and advance + compaction (one launch while the state
        rows fit its staging buffer, else advance, scatter and copy-back)."""
        if getattr(self, "fused", False):
            return 2
        step = 1
        row_total = sum(self.rb_arr[k] for k in range(7))
        commit = 1 if self.B * row_total <= FUSED_STAGE_BYTES else 3
        return 1 + step + commit

    def commit_bytes_bound(self):
        """Bytes the fused commit moves at most (every row committed and
        moved): block tokens into the committed tokens, the row's b / K /
        rid read, b and evict written, the compaction maps, and each row of
        the compacted arrays read and written once."""
        row_total = sum(self.rb_arr[k] for k in range(7))
        return self.B * (4 * self.L + 12 + 5 + 8 + 2 * row_total)


def roofline_kernel_label(sharded, fused, fixed):
    """Which launch the roofline times: the step kernel over one logits
    array or over vocabulary shards, with the commit inside it or not."""
    if sharded:
        entry = "dllm_step_vocab_shards_commit" if fused else "dllm_step_vocab_shards"
        return f"step_kernel over 4 vocabulary shards{' with the fused commit' if fused else ''} ({entry})"
    entry = ("dllm_step_commit" if fused else ("dllm_step_quota" if fixed else "dllm_step"))
    quota = ", fixed-steps quota" if fixed and fused else ""
    return f"step_kernel{' with the fused commit' if fused else ''} ({entry}{quota})"


FUSED_STAGE_BYTES = 96 * 1024   # state rows dllm_advance_compact stages in one CTA (one launch)
KERNEL_TIMING_LAUNCHES = 48   # step launches timed alone for the roofline (fixed, whatever --steps is)
ORACLE_SAMPLE_CPU_S = 12.0   # CPU time the oracle baseline runs for (whole passes)
E2E_ROUNDS = 3              # timed rounds of the end-to-end leg (the median is reported)
REFERENCE_RUN_S = 90.0      # the reference arm's whole run (warm-up and timed steps), about


def time_step_kernel(pipe, stream, launch, n=KERNEL_TIMING_LAUNCHES):
    """Launch duration of the step kernel as ``launch(slot, stream)`` issues
    it (the pipeline's step, with or without its fused commit), measured two
    ways on fresh state slots (the ring is restored first, outside every
    event):

    * per launch: ``n`` step launches, each between its own pair of CUDA
      events on the launching stream, after one untimed launch (so the first
      timed launch does not follow a host synchronisation); mean, median
      and minimum over the n;
    * back to back: ``n`` step launches in a row, each a programmatic
      dependent of the previous one as in the pipeline, between one pair
      of events; their mean.

    The count is fixed (independent of the pipeline's step count)."""
    torch = pipe.torch
    n = min(n, pipe.ring - 1)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    pipe.restore()
    torch.cuda.synchronize()
    rc = launch(0, stream)
    for k in range(n):
        ev[k][0].record()
        rc |= launch(k + 1, stream)
        ev[k][1].record()
    torch.cuda.synchronize()
    per_launch = [a.elapsed_time(b) for a, b in ev]
    pipe.restore()
    b0 = torch.cuda.Event(enable_timing=True)
    b1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    rc |= launch(0, stream)
    b0.record()
    for k in range(n):
        rc |= launch(k + 1, stream)
    b1.record()
    torch.cuda.synchronize()
    if rc:
        raise RuntimeError("a dllm call failed in the step-kernel timing pass")
    pipe.restore()
    return {"n": n, "mean_ms": statistics.fmean(per_launch), "median_ms": statistics.median(per_launch),
            "min_ms": min(per_launch), "max_ms": max(per_launch),
            "back_to_back_mean_ms": b0.elapsed_time(b1) / n}


def run_gpu(args, rank, world, local_rank, dist):
    import torch
    import denoise_step_token_gb300 as dllm
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dllm.load()
    cfg, inp, reqs, b, gen, pending_p = make_workload(1000 + rank, args.workload)
    pipe = Pipeline(cfg, inp, reqs, b, gen, pending_p, device,
                    fixed_steps=FIXED_STEPS_S if args.workload == "dream_fixed_steps" else None,
                    vocab_shards=4 if args.workload == "dream_vocab4" else None,
                    fused=not args.separate_commit)
    stream = torch.cuda.current_stream(device)
    sh = ctypes.c_void_p(stream.cuda_stream)
    K, W = args.steps, args.warmup
    # warm-up
    for k in range(W):
        if k % pipe.ring == 0:
            pipe.restore()
        pipe.run(k % pipe.ring, sh)
    torch.cuda.synchronize()
    if dllm.get_device_error(device):
        raise RuntimeError("device error during warm-up")
    pipe.restore()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(device).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = None
    sampler = ClockSampler(gpu_uuid)
    sampler.start()
    time.sleep(0.3)
    if dist is not None and dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    t0.record()
    for k in range(K):
        slot = k % pipe.ring
        if slot == 0 and k > 0:
            pipe.restore()
        pipe.run(slot, sh)
    t1.record()
    torch.cuda.synchronize()
    if dist is not None and dist.is_initialized():
        dist.barrier()
    # the step kernel as the pipeline launches it, for the roofline, and the
    # step without the commit beside it (outside the timed pipeline region,
    # so that their events do not slow the pipeline down)
    kernel = time_step_kernel(pipe, sh, pipe.launch_step_commit if pipe.fused else pipe.launch_step)
    step_only = time_step_kernel(pipe, sh, pipe.launch_step) if pipe.fused else None
    clocks = sampler.stop()
    err = dllm.get_device_error(device)
    if err:
        raise RuntimeError(f"device error {err} during the timed region")
    total_ms = t0.elapsed_time(t1)
    units, seconds = aggregate(pipe.M * K, total_ms / 1e3, dist)
    res = {
        "pipe": pipe, "units": units, "seconds": seconds, "total_ms": total_ms, "kernel": kernel, "step_only": step_only,
        "clocks": clocks, "cfg": cfg, "inp": inp, "device": device,
    }
    return res


def measure_h2d_gbs(dst, src, reps=5):
    """Plain host-to-device bandwidth of this box's link: ``src`` (pinned
    host) copied into ``dst`` with one cudaMemcpyAsync, timed with CUDA
    events on the current stream; the median of ``reps`` copies, in GB/s."""
    torch = __import__("torch")
    stream = torch.cuda.current_stream(dst.device)
    vals = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(src, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        vals.append(src.numel() * src.element_size() / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return statistics.median(vals)


def run_e2e(pipe, steps, rounds=E2E_ROUNDS):
    """Same step through the public API from pinned host buffers: every step
    copies its inputs host->device (the masked positions' logits rows, which
    are all the step reads, through dllm_step_compact; the batch state) and
    reads its results back (the slot's output block and the updated
    input_ids | conf_state).  The uploads are double-buffered: step k + 1's
    inputs cross the link on a copy stream while step k runs and its results
    come back (two logits buffers, two state slots, events between the
    streams).  ``rounds`` rounds of ``steps`` steps are timed; the value is
    the median round (a host stall of tens of ms in one round moves the mean
    of a 10-step round by half).  The link's own bandwidth (a plain pinned
    copy of the same logits bytes) and the rate it allows are reported
    beside it."""
    torch = pipe.torch
    dev = pipe.device
    rows_d = torch.from_numpy(pipe.masked_rows).to(dev)
    bufs = [pipe.logits[rows_d].contiguous()]
    bufs.append(torch.empty_like(bufs[0]))
    logits_h = torch.empty(bufs[0].shape, dtype=bufs[0].dtype, pin_memory=True)
    logits_h.copy_(bufs[0])
    state_h = torch.from_numpy(pipe.slot_host.copy()).pin_memory()
    n_state = pipe.words["ids"] + pipe.words["cs"]   # adjacent in the slot: ids | cs
    assert pipe.off["cs"] == pipe.off["ids"] + pipe.words["ids"]
    out_h = torch.empty(pipe.out_bytes, dtype=torch.uint8, pin_memory=True)
    state_out_h = torch.empty(n_state, dtype=torch.int32, pin_memory=True)
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)
    rows = bufs[0].shape[0]
    up_done = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]   # the last step on slot i no longer reads its inputs

    def upload(i):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(used[i])
            bufs[i].copy_(logits_h, non_blocking=True)
            pipe.state[i].copy_(state_h, non_blocking=True)
            up_done[i].record(copy_stream)

    def run_round(n):
        for i in (0, 1):
            used[i].record(stream)
        upload(0)
        for k in range(n):
            i = k % 2
            stream.wait_event(up_done[i])
            pipe.run(i, sh, compact=(bufs[i], rows))
            used[i].record(stream)
            if k + 1 < n:
                upload((k + 1) % 2)            # crosses the link while step k runs
            out_h.copy_(pipe.out[i], non_blocking=True)
            state_out_h.copy_(pipe.state[i, pipe.off["ids"]:pipe.off["ids"] + n_state], non_blocking=True)
            stream.synchronize()

    run_round(2)
    torch.cuda.synchronize()
    vals = []
    for _ in range(rounds):
        t = time.perf_counter()
        run_round(steps)
        vals.append(pipe.M * steps / (time.perf_counter() - t))
    torch.cuda.synchronize()
    h2d = bufs[0].numel() * 2 + pipe.slot_words * 4
    d2h = pipe.out_bytes + n_state * 4
    link = measure_h2d_gbs(bufs[1], logits_h)
    bound = pipe.M / (h2d / (link * 1e9))
    value = statistics.median(vals)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "rounds": [round(v, 1) for v in vals], "statistic": "median round",
            "uploads": "double-buffered on a copy stream",
            "link_h2d_gbs": link, "link_bound_value": bound, "frac_of_link_bound": value / bound}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_request_logits(inp, b):
    cfg = inp.cfg
    L = cfg.L
    out = np.full((L, cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    js = [j for j in range(L) if inp.input_ids[b, j] == cfg.mask_id]
    if js:
        rows = np.array([b * L + j for j in js])
        synth.fill_logits_rows(out, cfg.V, np.array(js), synth.step_row_keys(inp, rows), cfg.offset_max,
                               cfg.mask_id, nthreads=1)
    return out


def fixed_steps_quota(inp, S):
    """Per-request counts of the fixed-steps rule for a mixed-state batch:
    request b has taken L - (its masked count) steps of its block."""
    import oracle
    L = inp.cfg.L
    return np.array([oracle.transfer_quota(L, S, int(L - m)) for m in inp.masked.sum(axis=1)], dtype=np.int64)


def oracle_over_requests(inp, reqs, threads, quota=None, min_cpu_s=0.0, max_wall_s=30.0, cache=None):
    """Run the oracle's step on each listed request (one sub-batch each) on a
    thread pool; returns (masked rows processed, wall seconds of the oracle
    calls alone, passes).  Whole passes over ``reqs`` repeat until the
    process has used ``min_cpu_s`` seconds of CPU time or ``max_wall_s`` of
    wall time.  ``quota``: per-request counts of the fixed-steps rule, or
    None for the threshold rule.  ``cache``: a dict of requests' logits kept
    across calls (built outside the timed part either way)."""
    import oracle
    cfg = inp.cfg
    logits = cache if cache is not None else {}
    for b in dict.fromkeys(reqs):
        if b not in logits:
            logits[b] = oracle_request_logits(inp, b)
    rows = int(sum(inp.masked[b].sum() for b in reqs))

    def one(b):
        oracle.step(logits[b], cfg.V, inp.input_ids[b:b + 1], inp.thr[b:b + 1], inp.conf_state[b:b + 1],
                    cfg.mask_id, quota=None if quota is None else quota[b:b + 1])

    passes = 0
    c0, t = time.process_time(), time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            list(ex.map(one, reqs))
            passes += 1
            if time.process_time() - c0 >= min_cpu_s or time.perf_counter() - t >= max_wall_s:
                break
    return rows * passes, time.perf_counter() - t, passes


def cpu_baseline(inp, quota=None):
    threads = os.cpu_count() or 1
    reqs = list(range(inp.cfg.B))
    c0 = time.process_time()
    rows, secs, passes = oracle_over_requests(inp, reqs, threads, quota, min_cpu_s=ORACLE_SAMPLE_CPU_S)
    cpu_s = time.process_time() - c0
    return {"value": rows / secs, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{passes} full passes of the oracle over the {inp.cfg.B}-request batch "
                      f"({rows} masked rows, {secs:.2f} s wall and {cpu_s:.1f} s of CPU time on {threads} threads, "
                      f"one request per task)"}


def run_reference(args, rank, world):
    """The oracle, as it stands, timed on the host cores (reference arm)."""
    import oracle
    cfg, inp, lreqs, blk, *_ = make_workload(1000, args.workload)
    fixed = args.workload == "dream_fixed_steps"
    quota = fixed_steps_quota(inp, FIXED_STEPS_S) if fixed else None
    threads = os.cpu_count() or 1
    order = [b for b in range(cfg.B) if inp.masked[b].any()]
    # probe: one pass over the batch on every thread, to size each step's
    # sample so that the whole run takes about REFERENCE_RUN_S
    cache = {}
    probe_rows, probe_s, _ = oracle_over_requests(inp, order, threads, quota, cache=cache)
    rate = probe_rows / max(probe_s, 1e-9)
    total_steps = args.steps + args.warmup
    target_rows = max(1, int(REFERENCE_RUN_S * rate / total_steps))
    cursor = 0

    def sample():
        # whole requests in batch order, wrapping around (a request may
        # repeat) until the step holds target_rows masked rows
        nonlocal cursor
        picked, rows = [], 0
        while rows < target_rows:
            b = order[cursor % len(order)]
            cursor += 1
            picked.append(b)
            rows += int(inp.masked[b].sum())
        return picked

    for _ in range(args.warmup):
        oracle_over_requests(inp, sample(), threads, quota, cache=cache)
    units = 0
    secs = 0.0
    busy = 1   # threads with work: one request per task
    for _ in range(args.steps):
        reqs = sample()
        busy = max(busy, min(threads, len(reqs)))
        r, s, _ = oracle_over_requests(inp, reqs, threads, quota, cache=cache)
        units += r
        secs += s
    value = units / secs
    rows_per_step = units / args.steps
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": workload_config(args.workload, cfg, inp, oracle.box_width(list(lreqs.p), list(blk), cfg.L),
                                  oracle.cost(list(lreqs.p), list(blk), cfg.L), fixed),
        "sample_rows_per_step": rows_per_step,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": busy, "kind": "oracle",
                         "sample": f"each step: {rows_per_step:.0f} masked rows on average, whole requests of the "
                                   f"{cfg.B}-request batch taken in order (wrapping around), one request per task "
                                   f"on up to {busy} of {threads} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# BlockServe mixed-state loop: 256 requests served to completion
# ---------------------------------------------------------------------------
def run_loop_bench(args, rank, world, local_rank):
    """FDFO serving loop over a BlockServe-shaped queue, with the in-place
    re-loop, and the same queue again without it for comparison.  The timed
    part of each iteration is the hot path (admission, refill, pack, step,
    done readback, advance, compaction); producing the step's logits (the
    model forward's job) is not timed: each masked position's row is
    gathered on the device from a pool of generated rows, chosen by a hash
    of (request, block, step, position)."""
    import torch
    import denoise_step_token_gb300 as dllm
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dllm.load()
    lcfg = synth.LOOP_CONFIGS[args.workload]
    # untimed warm-up of every driver on a short queue of the same shape:
    # the first launch of each kernel loads its module and the library
    # sets up per-device attributes on first use
    warm = dataclasses.replace(lcfg, R=16)
    for reloop, native in ((True, True), (False, True), (True, False)):
        serve_queue(warm, 1900 + rank, device, reloop=reloop, native=native, pool_rows=256)
    on = serve_queue(lcfg, 2000 + rank, device, reloop=True, native=True)
    off = serve_queue(lcfg, 2000 + rank, device, reloop=False, native=True)
    py = serve_queue(lcfg, 2000 + rank, device, reloop=True, native=False)
    secs = on["secs"]
    out = {
        "metric": METRIC, "value": on["masked"] / secs, "unit": UNIT, "n_gpus": world, "steps": on["iters"],
        "warmup": 0, "ms_per_step": secs * 1e3 / on["iters"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "input_dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "requests": lcfg.R, "prompt_len": [lcfg.p_lo, lcfg.p_hi],
                   "gen": lcfg.gen, "L": lcfg.L, "V": lcfg.V, "token_budget": lcfg.budget,
                   "threshold": lcfg.threshold, "mode": "fdfo", "in_place_reloop": True, "driver": "native (dllm_loop_*)",
                   "timed": "admit+refill+pack+step+done readback+advance+compact per iteration"},
        "loop": {"iterations": on["iters"], "timed_s": secs, "masked_positions": on["masked"],
                 "mean_active_rows": on["mean_A"],
                 "logits_gbs": on["masked"] * lcfg.V * 2 / secs / 1e9,
                 "reloop_iterations": on["reloops"]},
        "without_reloop": {"value": off["masked"] / off["secs"], "timed_s": off["secs"],
                           "iterations": off["iters"], "ms_per_step": off["secs"] * 1e3 / off["iters"]},
        "python_driver": {"value": py["masked"] / py["secs"], "timed_s": py["secs"],
                          "iterations": py["iters"], "ms_per_step": py["secs"] * 1e3 / py["iters"]},
    }
    assert on["iters"] == off["iters"] == py["iters"] and on["masked"] == off["masked"] == py["masked"]
    out["threshold_control"] = time_threshold_control(lcfg, seed=3000 + rank)
    # the native loop choosing every step's thresholds itself (DiLaServe
    # controller, an affine step-latency model near the measured iteration)
    from denoise_step_token_gb300.control import ThresholdController
    ctl = ThresholdController.affine([0.5, 0.6, 0.7, 0.8, 0.9], L=lcfg.L, slo_s=2.0, tokens_per_s=1.0e7,
                                     latency_s=2.0e-4, latency_per_row_s=8.0e-7)
    cc = serve_queue(lcfg, 2000 + rank, device, reloop=True, native=True, controller=ctl)
    out["native_threshold_control"] = {
        "value": cc["masked"] / cc["secs"], "timed_s": cc["secs"], "iterations": cc["iters"],
        "ms_per_step": cc["secs"] * 1e3 / cc["iters"], "masked_positions": cc["masked"],
        "mean_threshold": cc["mean_threshold"],
        "controller": "candidates 0.5..0.9, SLO 2 s, 1e7 tokens/s, step latency 0.2 ms + 0.8 us per row"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


def time_threshold_control(lcfg, seed, A=256, reps=200):
    """Host cost of one DiLaServe threshold decision (stub step prediction,
    Algorithm 2, Algorithm 1) for a batch of A active requests over the five
    candidate thresholds, on this machine's host CPU."""
    from denoise_step_token_gb300.control import ThresholdController
    rng = np.random.default_rng(seed)
    L, K = lcfg.L, lcfg.K
    q = np.sort(rng.uniform(0.3, 1.0, size=(A, 4)).astype(np.float32), axis=1)
    feats = np.stack([q[:, 0], q[:, 1], q[:, 2], q.mean(axis=1), q[:, 3], rng.random(A)], axis=1).astype(np.float32)
    feats[rng.random(A) < 0.1, :5] = np.nan
    masked = rng.integers(0, L + 1, size=A)
    left = rng.integers(0, K, size=A)
    total = rng.integers(lcfg.p_lo, lcfg.p_hi + 1, size=A) + lcfg.gen
    elapsed = rng.uniform(0.0, 1.0, size=A)
    ctl = ThresholdController([0.5, 0.6, 0.7, 0.8, 0.9], L=L, slo_s=2.0, tokens_per_s=1.0e7,
                              step_latency_s=lambda n: 0.0006)
    ctl.choose(feats, masked, left, total, elapsed)
    t = time.perf_counter()
    for _ in range(reps):
        thr, choice, cap = ctl.choose(feats, masked, left, total, elapsed)
    us = (time.perf_counter() - t) / reps * 1e6
    return {"requests": A, "candidates": 5, "us_per_decision": us,
            "mean_threshold": float(thr.mean()), "capped_requests": int((cap < 4).sum())}


def serve_queue(lcfg, seed, device, reloop, native=True, pool_rows=4096, controller=None):
    """Serve one generated queue to completion, with libdllm's native loop
    (two calls per iteration) or the Python DeviceLoop, optionally under a
    threshold controller; returns the timed seconds, iterations, masked
    positions and re-loops."""
    import torch
    from denoise_step_token_gb300.loop import DeviceLoop, NativeLoop
    reqs = synth.make_loop_requests(lcfg, seed)
    L, V, ldv = lcfg.L, lcfg.V, lcfg.row_stride
    pool_h = np.empty((pool_rows, ldv), dtype=np.uint16)
    keys = synth.logits_row_keys(seed, np.arange(pool_rows), 0, 0, 0, 0)
    synth.fill_logits_rows(pool_h, V, np.arange(pool_rows), keys, lcfg.offset_max, lcfg.mask_id)
    pool = torch.from_numpy(pool_h.view(np.int16)).to(device)
    cls = NativeLoop if native else DeviceLoop
    loop = cls(reqs.p, reqs.K, reqs.prompt_off, reqs.prompt_tokens, reqs.thr, L=L, V=V,
               mask_id=lcfg.mask_id, pad_id=lcfg.pad_id, budget=lcfg.budget, device=device, mode="fdfo",
               reloop=reloop, controller=controller)
    logits = torch.empty((lcfg.R * L, ldv), dtype=torch.int16, device=device)
    ev = []
    active = []
    masked_total = 0
    iters = 0
    thr_sum, thr_n = 0.0, 0
    if native:
        while not loop.finished():
            # timed: admission, refill, pack (dllm_loop_begin)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            inf = loop.begin()
            torch.cuda.synchronize()
            t_begin = time.perf_counter() - t0
            # untimed: the model forward's stand-in
            rows = loop.masked_rows()
            _fill_loop_logits(logits, pool, rows, seed, pool_rows, device)
            # timed: step, done readback, advance + compaction (dllm_loop_end)
            torch.cuda.synchronize()
            t1 = time.perf_counter()
            active.append(inf.A)
            loop.end(logits[: max(inf.A, 1) * L])
            torch.cuda.synchronize()
            ev.append(t_begin + time.perf_counter() - t1)
            iters += 1
            masked_total += len(rows)
            if controller is not None and inf.A:
                thr_sum += float(loop.thresholds().sum())
                thr_n += inf.A
        return {"secs": sum(ev), "iters": iters, "masked": masked_total, "reloops": loop.info().reloops,
                "mean_A": float(np.mean(active)) if active else 0.0,
                "mean_threshold": thr_sum / thr_n if thr_n else None}
    while not loop.finished():
        # timed: admission (host) and refill
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        loop.admit_phase()
        torch.cuda.synchronize()
        t_admit = time.perf_counter() - t0
        # untimed: the model forward's stand-in -- pool rows for the masked positions
        rows = loop.masked_rows()
        _fill_loop_logits(logits, pool, rows, seed, pool_rows, device)
        # timed: pack, step, done readback, advance, compaction
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        loop.pack_phase()
        active.append(loop.A)
        done, _ = loop.step_phase(logits[: loop.A * L])
        loop.finish_phase(done)
        torch.cuda.synchronize()
        ev.append(t_admit + time.perf_counter() - t1)
        iters += 1
        masked_total += len(rows)
    return {"secs": sum(ev), "iters": iters, "masked": masked_total, "reloops": loop.reloops,
            "mean_A": float(np.mean(active)) if active else 0.0}


def _fill_loop_logits(logits, pool, rows, seed, pool_rows, device):
    """The model forward's stand-in (not timed): each masked position's
    logits row is a pool row chosen by a hash of (request, block, step,
    position)."""
    import torch
    if not rows:
        return
    flat = torch.as_tensor([r[0] for r in rows], device=device)
    h = synth.out(np.uint64(seed), np.asarray([((r[1] * 64 + r[2]) * 4096 + r[3]) * 64 + r[4] for r in rows],
                                              dtype=np.uint64))
    pick = torch.as_tensor((h % np.uint64(pool_rows)).astype(np.int64), device=device)
    logits[flat] = pool[pick]


READ_CEILING_SHAPES = [(14, 3, 4096), (16, 3, 4096), (8, 3, 8192), (12, 2, 8192), (4, 3, 16384), (8, 2, 4096),
                       (24, 2, 4096)]   # (warps per CTA, ring slots, bytes per bulk copy)


def run_read_ceiling(local_rank, gib=2, reps=5):
    """The GPU's read-bandwidth ceiling, for the roofline of the step
    kernel: a ``gib`` GiB device buffer read once per launch with no
    arithmetic, by bulk copies into per-warp shared-memory rings (the step
    kernel's way of reading logits; several ring shapes) and by plain 16-byte
    loads; the best of ``reps`` launches each, CUDA events."""
    import torch
    from denoise_step_token_gb300 import _build
    import denoise_step_token_gb300 as dllm
    dllm.load()
    lib = ctypes.CDLL(_build.PROBE_LIB_PATH)
    p = ctypes.c_void_p
    lib.dllm_probe_bulk_read.argtypes = [p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p]
    lib.dllm_probe_load_read.argtypes = [p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, p, p]
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    nbytes = gib << 30
    buf = torch.ones(nbytes, dtype=torch.uint8, device=device)
    sink = torch.zeros(2, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    sh = p(stream.cuda_stream)
    sms = torch.cuda.get_device_properties(device).multi_processor_count

    def best(launch):
        out = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = launch()
            e1.record(stream)
            e1.synchronize()
            if rc:
                raise RuntimeError(f"probe launch failed: {rc}")
            out.append(nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
        return max(out)

    rows = []
    for w, st, cb in READ_CEILING_SHAPES:
        gbs = best(lambda: lib.dllm_probe_bulk_read(p(buf.data_ptr()), nbytes, sms, w, st, cb, p(sink.data_ptr()), sh))
        rows.append({"kind": "bulk copies", "warps": w, "slots": st, "copy_bytes": cb,
                     "in_flight_per_sm": w * st * cb, "gbs": gbs})
    for threads, per_sm in ((1024, 2), (512, 8)):
        gbs = best(lambda: lib.dllm_probe_load_read(p(buf.data_ptr()), nbytes, sms * per_sm, threads,
                                                    p(sink.data_ptr()), sh))
        rows.append({"kind": "16-byte loads", "threads": threads, "ctas_per_sm": per_sm, "gbs": gbs})
    if int(sink[1].item()) != 0:
        raise RuntimeError("a probe wait ran out")
    peak, src = load_peaks()
    return {"read_ceiling": rows, "max_gbs": max(r["gbs"] for r in rows), "buffer_bytes": nbytes,
            "measured_copy_peak_gbs": peak, "peak_source": src}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--separate-commit", action="store_true",
                    help="commit and compact in a launch of their own after the step (the comparison pipeline)")
    ap.add_argument("--read-ceiling", action="store_true",
                    help="measure the GPU's read-bandwidth ceiling (bulk copies and plain loads) instead")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dream",
                    help="dream (default, the headline), dream_fixed_steps, llada, stress, tiny, or the blockserve loop")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_info()

    if args.read_ceiling:
        if rank == 0:
            print(json.dumps(run_read_ceiling(local_rank)), flush=True)
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0

    if args.workload in synth.LOOP_CONFIGS:
        return run_loop_bench(args, rank, world, local_rank)

    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_gpu(args, rank, world, local_rank, dist)
    pipe, cfg = res["pipe"], res["cfg"]
    K = args.steps
    kern, step_only = res["kernel"], res["step_only"]
    step_ms = kern["mean_ms"]
    alg = algorithmic_bytes(cfg, pipe.M) + (pipe.commit_bytes_bound() if pipe.fused else 0)
    achieved = alg / (step_ms / 1e3) / 1e9
    peak, peak_src = load_peaks()
    # the committed capture is of the Dream-shaped step launch only
    traffic = load_traffic(step_source_sha()) if args.workload == "dream" else None
    value = res["units"] / res["seconds"]
    e2e = run_e2e(pipe, args.e2e_steps)
    cpu = None
    fixed = args.workload == "dream_fixed_steps"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(res["inp"], fixed_steps_quota(res["inp"], FIXED_STEPS_S) if fixed else None)
    if dist is not None:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": res["seconds"] * 1e3 / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "input_dtype": "bf16", "data": "synthetic",
            "config": workload_config(args.workload, cfg, res["inp"], pipe.W, pipe.cost, fixed),
            "timing": {"step": (f"admit (host) + pack + step + block commit + compaction: "
                                f"{pipe.launches_per_step()} kernel launches"
                                + (" (the commit and compaction inside the step's launch)" if pipe.fused else "")),
                       "l2": "inputs larger than L2: 0.62 GB of masked logits rows per step, no flush",
                       "state_ring": RING,
                       "roofline": (f"{kern['n']} step launches after the timed region, each between "
                                    f"its own CUDA events on fresh state; frac from their mean")},
            "logits_gbs": pipe.M * cfg.V * 2 * K / res["seconds"] / 1e9 / world,
            "step_kernel_ms": step_ms,
            "step_kernel_ms_median": kern["median_ms"],
            "step_kernel_ms_min": kern["min_ms"],
            "step_kernel_ms_max": kern["max_ms"],
            "step_kernel_samples": kern["n"],
            "step_kernel_back_to_back_ms": kern["back_to_back_mean_ms"],
            "step_only_kernel_ms": None if step_only is None else step_only["mean_ms"],
            "step_only_kernel_back_to_back_ms": None if step_only is None else step_only["back_to_back_mean_ms"],
            "step_only_frac": (None if step_only is None else
                               algorithmic_bytes(cfg, pipe.M) / (step_only["mean_ms"] / 1e3) / 1e9 / peak),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                         "frac_of_nominal_8000_gbs": achieved / NOMINAL_HBM_GBS,
                         "all_rows_logits_bytes_per_launch": cfg.B * cfg.L * cfg.V * 2,
                         "kernel": roofline_kernel_label(pipe.shards is not None, pipe.fused, fixed),
                         "algorithmic_bytes_per_launch": alg,
                         "algorithmic_bytes_note": ("masked logits rows + per-position state + per-request I/O"
                                                    + (" + the commit at its bound (every row committed and moved)"
                                                       if pipe.fused else ""))},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": pipe.launches_per_step() * K,
            "clocks": res["clocks"],
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
