"""DiLaServe's confidence-threshold controller for one serving instance.

DiLaServe review, section 3.2 ("Confidence Threshold Controller"): before a
step, every active request gets a threshold from an ascending candidate list
(section 4.1, e.g. {0.5, ..., 0.9}).  Algorithm 2 (adaptive load control,
``dllm_load_control``) caps each request's threshold so that the worst-case
aggregate load stays within the instance's capacity; Algorithm 1 (SLO-aware
adjustment, ``dllm_slo_thresholds``) then takes the highest allowed threshold
whose predicted remaining latency fits the request's remaining SLO budget.
Remaining steps come from ``dllm_predict_steps_stub`` over the block
features the step emits -- a stand-in for the review's trained step
predictor.  All of it is host arithmetic in libdllm; this class marshals
arrays.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import NUM_FEATURES, _check, load


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


class ThresholdController:
    """``candidates``: ascending thresholds; ``L``: block length; ``slo_s``:
    each request's latency SLO; ``tokens_per_s``: the instance's processing
    rate (capacity = tokens_per_s * slo_s); ``step_latency_s``: a callable
    giving the latency of one step at a batch of ``A`` rows (the review's
    one-off profile)."""

    def __init__(self, candidates, *, L, slo_s, tokens_per_s, step_latency_s):
        self.cand = np.ascontiguousarray(candidates, dtype=np.float64)
        if self.cand.ndim != 1 or self.cand.size < 1 or np.any(np.diff(self.cand) <= 0):
            raise ValueError("candidates must be a non-empty ascending list")
        self.L = int(L)
        self.slo_s = float(slo_s)
        self.capacity = float(tokens_per_s) * self.slo_s
        self.step_latency_s = step_latency_s

    def choose(self, feats, masked, blocks_left, total_tokens, elapsed_s):
        """Thresholds (float32 [A]) for the active rows, in arrival order.

        feats: float32 [A, 6] block features of the last step (NaN rows for
        blocks with nothing unmasked); masked: positions still masked in the
        current block; blocks_left: blocks after the current one;
        total_tokens: prompt + output tokens; elapsed_s: time since arrival.
        Also returns the chosen candidate indices and the load caps."""
        lib = load()
        A = len(masked)
        T = self.cand.size
        if A == 0:
            return np.zeros(0, np.float32), np.zeros(0, np.int32), np.zeros(0, np.int32)
        feats = np.ascontiguousarray(feats, dtype=np.float32).reshape(A, NUM_FEATURES)
        masked = np.ascontiguousarray(masked, dtype=np.int32)
        left = np.ascontiguousarray(blocks_left, dtype=np.int32)
        steps = np.empty((A, T), dtype=np.float64)
        _check("dllm_predict_steps_stub",
               lib.dllm_predict_steps_stub(A, T, _p(self.cand), self.L, _p(feats), _p(masked), _p(left), _p(steps)))
        load_ = np.ascontiguousarray(steps * np.asarray(total_tokens, dtype=np.float64)[:, None])
        cap = np.empty(A, dtype=np.int32)
        _check("dllm_load_control", lib.dllm_load_control(A, T, _p(load_), self.capacity, _p(cap)))
        lat = np.full(A, float(self.step_latency_s(A)), dtype=np.float64)
        slo_left = np.ascontiguousarray(self.slo_s - np.asarray(elapsed_s, dtype=np.float64))
        choice = np.empty(A, dtype=np.int32)
        _check("dllm_slo_thresholds",
               lib.dllm_slo_thresholds(A, T, _p(steps), _p(lat), _p(slo_left), _p(cap), _p(choice)))
        return self.cand[choice].astype(np.float32), choice, cap
