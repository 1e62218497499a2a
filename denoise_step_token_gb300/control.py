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
predictor.  All of it, loads and SLO budgets included, is host arithmetic
in libdllm (``dllm_threshold_control``); this class marshals arrays and
evaluates the caller's step-latency model at the batch size.
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
        self.tokens_per_s = float(tokens_per_s)
        self.step_latency_s = step_latency_s
        self.latency_affine = None   # (a, b) when step_latency_s is a + b * A

    @classmethod
    def affine(cls, candidates, *, L, slo_s, tokens_per_s, latency_s, latency_per_row_s):
        """A controller whose step latency at A rows is latency_s +
        latency_per_row_s * A -- the form the native loop evaluates itself
        (``dllm_loop_set_control``)."""
        a, b = float(latency_s), float(latency_per_row_s)
        ctl = cls(candidates, L=L, slo_s=slo_s, tokens_per_s=tokens_per_s, step_latency_s=lambda A: a + b * A)
        ctl.latency_affine = (a, b)
        return ctl

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
        total = np.ascontiguousarray(total_tokens, dtype=np.int64)
        elapsed = np.ascontiguousarray(elapsed_s, dtype=np.float64)
        steps = np.empty((A, T), dtype=np.float64)
        cap = np.empty(A, dtype=np.int32)
        choice = np.empty(A, dtype=np.int32)
        _check("dllm_threshold_control",
               lib.dllm_threshold_control(A, T, _p(self.cand), self.L, _p(feats), _p(masked), _p(left), _p(total),
                                          _p(elapsed), self.slo_s, self.tokens_per_s,
                                          float(self.step_latency_s(A)), _p(steps), _p(cap), _p(choice)))
        return self.cand[choice].astype(np.float32), choice, cap
