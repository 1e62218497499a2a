"""Oracle of DiLaServe's per-request confidence-threshold control.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

DiLaServe review, section 3.2 ("Confidence Threshold Controller"):

* item ① (Algorithm 1, SLO-aware threshold adjustment): the remaining latency
  of a request at a threshold is its predicted remaining steps times the
  step latency; take the highest threshold whose remaining latency fits the
  remaining SLO budget.
* item ② (Algorithm 2, adaptive load control): a request's load is its total
  token count times its predicted remaining steps; an instance's capacity is
  the tokens it processes per second times the SLO.  Requests are visited in
  arrival order; for each, thresholds are tried from the highest down, and a
  threshold is dropped from the request's allowed set while the worst-case
  aggregate load -- the load already committed, plus this request at that
  threshold, plus every later request at the lowest threshold -- exceeds the
  capacity.  This leaves each request the widest feasible threshold range.
* item ③ (step prediction): the review's predictor is a gradient-boosted
  model over 11 features, trained offline; it needs trained weights and is
  out of scope.  ``predict_steps_stub`` stands in for it (a reading: it uses
  only the block features the step emits and is not the review's model).

Readings (listed in the design notes): a request whose every threshold
breaks the budget keeps the lowest; Algorithm 1 with no threshold meeting
the SLO takes the lowest allowed one; "committed load" adds each visited
request's load at its highest allowed threshold.
"""
from __future__ import annotations

import math

import numpy as np


def rate_above(t, feats):
    """Stub predictor, step 1: the probability that a masked position's
    confidence will exceed ``t``, read off the block's confidence features
    (min, q25, median, avg, q75, unmasked fraction) as a piecewise-linear
    distribution through (min, 0), (q25, .25), (median, .5), (q75, .75),
    (1, 1).  With no unmasked position yet (NaN features) confidences are
    taken as uniform on [0, 1]: 1 - t."""
    mn, q25, med, _avg, q75, _frac = (float(x) for x in feats)
    if math.isnan(mn):
        return min(1.0, max(0.0, 1.0 - t))
    xs = [mn, q25, med, q75, 1.0]
    ps = [0.0, 0.25, 0.5, 0.75, 1.0]
    if t < xs[0]:
        return 1.0
    if t >= xs[-1]:
        return 0.0
    F = 1.0
    for k in range(4):
        if xs[k] <= t < xs[k + 1]:
            F = ps[k] + (t - xs[k]) / (xs[k + 1] - xs[k]) * (ps[k + 1] - ps[k])
            break
    return 1.0 - F


def steps_to_clear(m, P):
    """Stub predictor, step 2: steps to unmask ``m`` positions when a step
    unmasks a fraction ``P`` of those still masked, at least one (the
    threshold rule's fallback): m <- m - max(1, floor(P m))."""
    n = 0
    while m > 0:
        m -= max(1, math.floor(P * m))
        n += 1
    return n


def predict_steps_stub(t, feats, masked, blocks_left, L):
    """Predicted remaining denoising steps of a request at threshold ``t``:
    its current block's ``masked`` positions, then ``blocks_left`` more
    blocks of L (a stand-in for the review's step predictor)."""
    P = rate_above(t, feats)
    return steps_to_clear(int(masked), P) + int(blocks_left) * steps_to_clear(int(L), P)


def load_control(load, capacity):
    """Algorithm 2.  ``load``: [R][T] (requests in arrival order, thresholds
    ascending).  Returns, per request, the index of its highest allowed
    threshold (every lower one stays allowed)."""
    load = np.asarray(load, dtype=np.float64)
    R, T = load.shape
    out = np.zeros(R, dtype=np.int64)
    # rest[i] = the later requests at the lowest threshold, summed from the
    # back: rest[R-1] = 0, rest[i] = load[i+1][0] + rest[i+1]
    rest_of = [0.0] * R
    for i in range(R - 2, -1, -1):
        rest_of[i] = float(load[i + 1, 0]) + rest_of[i + 1]
    committed = 0.0
    for i in range(R):
        rest = rest_of[i]
        keep = 0
        for k in range(T - 1, -1, -1):
            worst = committed + float(load[i, k]) + rest
            if worst <= capacity:
                keep = k
                break
        out[i] = keep
        committed += float(load[i, keep])
    return out


def slo_threshold(rem_steps, step_latency, slo_left, max_allowed=None):
    """Algorithm 1 for one request.  ``rem_steps``: [T] predicted remaining
    steps per threshold (ascending thresholds); returns the index of the
    highest allowed threshold whose remaining latency fits ``slo_left``,
    else the lowest threshold."""
    T = len(rem_steps)
    top = T - 1 if max_allowed is None else int(max_allowed)
    for k in range(top, -1, -1):
        if float(rem_steps[k]) * float(step_latency) <= float(slo_left):
            return k
    return 0
