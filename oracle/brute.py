"""Brute-force sampler for tiny vocabularies (pure Python, no numpy).

TEST INFRASTRUCTURE ONLY (same import rule as oracle/sampler.py).

An independent second statement of the same definition, used to pin the
oracle: a full Python sort for top-k, an explicit descending walk for top-p
(Arc PR #222, section 3(b): "zero-rest", "top-p walk", "min-p scan"), and an
explicit running sum over ascending token ids for the draw.  It uses plain
Python floats (IEEE fp64) and math.exp; sums run left to right in the same
orders as the oracle's cumulative sums, so the two must agree exactly.
"""
from __future__ import annotations

import math
import struct


def _f32(x: float) -> float:
    """Round a Python float to the nearest fp32 value."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def penalize(z, hist, rep, freq, pres):
    counts = {}
    for t in hist:
        counts[t] = counts.get(t, 0) + 1
    out = list(z)
    for i, c in counts.items():
        v = out[i]
        v = _f32(v / rep) if v > 0 else _f32(v * rep)
        v = _f32(v - _f32(c * freq))
        v = _f32(v - pres)
        out[i] = v
    return out


def sample(z, T, top_k, top_p, min_p, u, hist=(), rep=1.0, freq=0.0, pres=0.0):
    """Token for one row of fp32-valued logits `z` (list of floats) and uniform u."""
    V = len(z)
    z = [(-math.inf if x != x else x) for x in z]
    rep, freq, pres = _f32(rep), _f32(freq), _f32(pres)
    z = penalize(z, hist, rep, freq, pres)
    m = max(z)
    if m == -math.inf:
        return 0
    if T == 0.0 or top_k == 1:
        for i in range(V):
            if z[i] == m:
                return i
    if m == math.inf:
        w = [1.0 if x == m else 0.0 for x in z]
    else:
        w = [math.exp((x - m) / T) for x in z]

    # top-k: full sort by (value desc, index asc), keep the first k
    if 1 <= top_k < V:
        ranked = sorted(range(V), key=lambda i: (-z[i], i))
        keep = set(ranked[:top_k])
    else:
        keep = set(range(V))

    # top-p: walk the kept entries by (w desc, index asc) until the mass reaches p * S
    if top_p < 1.0:
        walk = sorted(keep, key=lambda i: (-w[i], i))
        total = 0.0
        for i in walk:
            total += w[i]
        target = top_p * total
        run = 0.0
        cut = w[walk[-1]]
        for i in walk:
            run += w[i]
            if run >= target:
                cut = w[i]
                break
        keep = {i for i in keep if w[i] >= cut}

    # min-p scan
    if min_p > 0.0:
        keep = {i for i in keep if w[i] >= min_p}

    # inverse CDF over ascending token ids
    total = 0.0
    for i in range(V):
        if i in keep:
            total += w[i]
    t = u * total
    run = 0.0
    last = None
    for i in range(V):
        if i in keep:
            run += w[i]
            last = i
            if run > t:
                return i
    return last
