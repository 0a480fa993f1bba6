"""fp64 CPU oracle for on-device logits sampling.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only `tests/`, `__graft_entry__.smoke()` and the
`cpu_baseline` / `--impl reference` legs of `bench.py` use it.  It shares no
code with the CUDA library (no kernels, headers, helpers or constants).

What it computes, per row r of a [B, V] logits batch (plain definition, slow
on purpose: a full sort and an explicit CDF):

 1. z_i = float32(logit_i).  NaN counts as -inf and raises ERR_NAN.
 2. Penalties for ids in the row's history (count c_i > 0): repetition, then
    frequency, then presence, each an fp32 round-to-nearest operation:
        z <- z / rep  if z > 0 else z * rep
        z <- z - fl32(c * freq)
        z <- z - pres
    The Arc pages name penalties only as parameters; this is the CTRL-style
    repetition rule with OpenAI-style frequency/presence terms.  A disabled
    penalty must leave every logit untouched (Arc PR #222, section 3(a): a
    disabled DRY at multiplier 0.0 is a proven no-op).
 3. Greedy when T == 0 or top_k == 1: the smallest index attaining max z.
 4. w_i = exp((z_i - m) / T) in fp64 with m = max z (w = [z == m] when m = +inf).
 5. top-k (1 <= k < V): the first k indices ordered by (z desc, index asc).
 6. top-p (p < 1) over the top-k survivors K: walk K by (w desc, index asc),
    accumulating mass; tau* is the w at which the running mass first reaches
    p * S_K; survivors are every entry of K with w >= tau* (ties kept).
 7. min-p (min_p > 0): survivors need w >= min_p * max w = min_p.
    Items 5-7 follow the filter order of Arc PR #222, section 3(b): top-k
    "zero-rest", then the top-p walk, then the min-p scan.
 8. u = (splitmix64(seed ^ (row << 32) ^ step) >> 11) * 2^-53, where
    splitmix64(x) is one output of the generator whose state is x (add the
    golden-ratio increment, then the two xor-shift-multiply rounds and the
    final xor-shift; Steele, Lea and Flood, OOPSLA 2014).  Arc PR #217 and the
    hybrid-nucleus commit of PR #194 name Splitmix64 as the device generator.
 9. Inverse CDF in ascending token-id order over the survivors R: the smallest
    i in R whose running mass exceeds u * S_R (the last survivor if rounding
    leaves none).

Degenerate rows: all -inf (or NaN) -> token 0 with ERR_DEGENERATE.
Invalid parameters -> token -1 with ERR_PARAM; history id outside [0, V) ->
token -1 with ERR_HIST_ID.

Every function here is pinned by tests/test_oracle_pins.py against brute force,
closed forms, published generator outputs and a chi-square test.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15

ERR_PARAM = 1 << 0
ERR_HIST_ID = 1 << 1
ERR_NAN = 1 << 2
ERR_DEGENERATE = 1 << 3

MODE_INVALID = -1
MODE_GREEDY = 0
MODE_INERT = 1
MODE_FILTERED = 2


# ---------------------------------------------------------------- generator
def splitmix64(x: int) -> int:
    """One splitmix64 output for state x (Steele, Lea, Flood 2014)."""
    z = (x + GOLDEN_GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def draw_bits(seed: int, row: int, step: int) -> int:
    """53 random bits for (seed, row, step): splitmix64(seed ^ row<<32 ^ step) >> 11."""
    x = (int(seed) ^ ((int(row) << 32) & MASK64) ^ int(step)) & MASK64
    return splitmix64(x) >> 11


def uniform(seed: int, row: int, step: int) -> float:
    """u in [0, 1), an exact multiple of 2^-53."""
    return draw_bits(seed, row, step) * 2.0 ** -53


# ---------------------------------------------------------------- penalties
def apply_penalties(z: np.ndarray, hist: np.ndarray, rep: float, freq: float,
                    pres: float) -> np.ndarray:
    """Penalised logits, each step an fp32 round-to-nearest operation.

    Each fp32 operation is evaluated in fp64 and rounded to fp32 once; for
    +, -, *, / that equals the correctly rounded fp32 result because fp64 has
    more than 2 * 24 + 2 significand bits.
    """
    z = np.asarray(z, dtype=np.float32).copy()
    if hist.size == 0:
        return z
    counts = np.bincount(np.asarray(hist, dtype=np.int64), minlength=z.size)
    rep32, freq32, pres32 = np.float32(rep), np.float32(freq), np.float32(pres)
    for i in np.nonzero(counts)[0]:
        v = np.float64(z[i])
        if v > 0:
            v = np.float64(np.float32(v / np.float64(rep32)))
        else:
            v = np.float64(np.float32(v * np.float64(rep32)))
        cf = np.float32(np.float64(counts[i]) * np.float64(freq32))
        v = np.float64(np.float32(v - np.float64(cf)))
        v = np.float64(np.float32(v - np.float64(pres32)))
        z[i] = np.float32(v)
    return z


# ---------------------------------------------------------------- row sampler
@dataclass
class RowResult:
    token: int
    mode: int
    err: int
    z: np.ndarray                    # penalised logits, fp32 values
    w: np.ndarray | None = None      # fp64 weights exp((z - m)/T)
    K: np.ndarray | None = None      # bool mask, top-k survivors
    R: np.ndarray | None = None      # bool mask, final survivors
    tau: float | None = None         # top-p cutoff value (w units), None if inactive
    S_K: float | None = None
    S_R: float | None = None
    u: float | None = None
    rbits: int | None = None
    cdf: np.ndarray | None = None    # running mass over R in index order


def params_valid(prm, V: int) -> bool:
    T = float(prm["temperature"])
    ok = math.isfinite(T) and T >= 0.0
    p = float(prm["top_p"])
    ok &= (not math.isnan(p)) and 0.0 < p <= 1.0
    mp = float(prm["min_p"])
    ok &= (not math.isnan(mp)) and 0.0 <= mp <= 1.0
    rep = float(prm["repetition_penalty"])
    ok &= math.isfinite(rep) and rep > 0.0
    ok &= math.isfinite(float(prm["frequency_penalty"]))
    ok &= math.isfinite(float(prm["presence_penalty"]))
    ok &= int(prm["flags"]) == 0
    return bool(ok)


def row_mode(prm, V: int) -> int:
    T = float(prm["temperature"])
    k = int(prm["top_k"])
    if T == 0.0 or k == 1:
        return MODE_GREEDY
    topk_on = 1 <= k < V
    if not topk_on and float(prm["top_p"]) >= 1.0 and float(prm["min_p"]) == 0.0:
        return MODE_INERT
    return MODE_FILTERED


def top_k_mask(z: np.ndarray, k: int) -> np.ndarray:
    """First k indices ordered by (z desc, index asc)."""
    V = z.size
    order = np.lexsort((np.arange(V), -z.astype(np.float64)))
    mask = np.zeros(V, dtype=bool)
    mask[order[:k]] = True
    return mask


def top_p_cutoff(w: np.ndarray, K: np.ndarray, p: float) -> tuple[float, float]:
    """(tau*, S_K): walk K by (w desc, index asc) until the running mass reaches p * S_K."""
    idx = np.nonzero(K)[0]
    order = idx[np.lexsort((idx, -w[idx]))]
    run = np.cumsum(w[order])
    S_K = float(run[-1])
    target = float(p) * S_K
    j = int(np.argmax(run >= target)) if bool((run >= target).any()) else order.size - 1
    return float(w[order[j]]), S_K


def inverse_cdf(w: np.ndarray, R: np.ndarray, u: float) -> tuple[int, np.ndarray, float]:
    """Smallest i in R (ascending id) whose running mass over R exceeds u * S_R."""
    run = np.cumsum(np.where(R, w, 0.0))
    S_R = float(run[-1])
    t = u * S_R
    hit = (run > t) & R
    if hit.any():
        tok = int(np.argmax(hit))
    else:
        tok = int(np.nonzero(R)[0][-1])
    return tok, run, S_R


def sample_row_u(logits_f32: np.ndarray, prm, u: float,
                 hist: np.ndarray | None = None) -> RowResult:
    """Sample one row by the plain definition with a given uniform u."""
    V = int(logits_f32.size)
    hist = np.zeros(0, dtype=np.int32) if hist is None else np.asarray(hist)
    z0 = np.asarray(logits_f32, dtype=np.float32)
    err = 0
    if not params_valid(prm, V):
        return RowResult(-1, MODE_INVALID, ERR_PARAM, z0)
    if hist.size and (hist.min() < 0 or hist.max() >= V):
        return RowResult(-1, MODE_INVALID, ERR_HIST_ID, z0)
    nan = np.isnan(z0)
    if nan.any():
        err |= ERR_NAN
        z0 = np.where(nan, np.float32(-np.inf), z0).astype(np.float32)
    z = apply_penalties(z0, hist, float(prm["repetition_penalty"]),
                        float(prm["frequency_penalty"]), float(prm["presence_penalty"]))
    mode = row_mode(prm, V)
    m = float(np.max(z))
    if m == -math.inf:
        return RowResult(0, mode, err | ERR_DEGENERATE, z)
    if mode == MODE_GREEDY:
        return RowResult(int(np.argmax(z == np.float32(m))), mode, err, z)

    T = float(np.float32(prm["temperature"]))
    zd = z.astype(np.float64)
    if m == math.inf:
        w = (zd == m).astype(np.float64)
    else:
        with np.errstate(under="ignore"):
            w = np.exp((zd - m) / T)

    k = int(prm["top_k"])
    K = top_k_mask(z, k) if 1 <= k < V else np.ones(V, dtype=bool)
    R = K.copy()
    tau = None
    S_K = None
    p = float(np.float32(prm["top_p"]))
    if p < 1.0:
        tau, S_K = top_p_cutoff(w, K, p)
        R &= w >= tau
    mp = float(np.float32(prm["min_p"]))
    if mp > 0.0:
        R &= w >= mp
    tok, run, S_R = inverse_cdf(w, R, u)
    if S_K is None:
        S_K = float(np.sum(np.where(K, w, 0.0)))
    return RowResult(tok, mode, err, z, w=w, K=K, R=R, tau=tau, S_K=S_K, S_R=S_R,
                     u=u, cdf=run)


def sample_row(logits_f32: np.ndarray, prm, row: int,
               hist: np.ndarray | None = None) -> RowResult:
    """Sample row `row` of a batch: u comes from (seed, row, step) of its parameters."""
    rbits = draw_bits(int(prm["seed"]), row, int(prm["step"]))
    res = sample_row_u(logits_f32, prm, rbits * 2.0 ** -53, hist)
    res.rbits = rbits
    return res


def sample_batch(logits_f32: np.ndarray, params: np.ndarray,
                 hist_offsets: np.ndarray | None = None,
                 hist_ids: np.ndarray | None = None,
                 rows=None) -> list[RowResult]:
    """sample_row over the rows of a batch (all rows unless `rows` is given)."""
    B = logits_f32.shape[0]
    out = []
    for r in (range(B) if rows is None else rows):
        h = None
        if hist_offsets is not None:
            h = hist_ids[int(hist_offsets[r]):int(hist_offsets[r + 1])]
        out.append(sample_row(logits_f32[r], params[r], r, h))
    return out


def top_logprobs(z: np.ndarray, temperature: float, n: int) -> tuple[np.ndarray, np.ndarray]:
    """The n most likely ids of a row and their log-probabilities.

    Arc PR #222, section 3(b), names the top-n log-probability output as a
    reader of the sampler's sort; the pages give no formula.  The reading here:
      * order: (z desc, id asc) over the penalised logits z -- the order of the
        top-k filter (temperature does not change it);
      * value: log-softmax over every id at the row's sampling temperature,
        before the top-k / top-p / min-p filters:
            lp_i = (z_i - m) / T - ln(sum_j exp((z_j - m) / T)),  m = max z,
        in fp64, with T = 1 for a greedy row (T == 0);
      * -inf logits have lp = -inf; when the max is +inf, the +inf entries
        share the mass (lp = -ln(count)) and the rest are -inf; a row with no
        finite or +inf logit lists ids in ascending order with lp = -inf;
      * n > V: the entries past V are (id -1, lp -inf).
    Returns (ids int64[n], lp float64[n]).
    """
    z = np.asarray(z, dtype=np.float32)
    V = int(z.size)
    T = float(np.float32(temperature))
    if not T > 0.0:
        T = 1.0
    zd = z.astype(np.float64)
    order = np.lexsort((np.arange(V), -zd))
    ids = np.full(n, -1, dtype=np.int64)
    lp = np.full(n, -math.inf)
    take = order[:min(n, V)]
    ids[:take.size] = take
    m = float(zd.max())
    if m == -math.inf:
        return ids, lp
    if m == math.inf:
        top = zd == math.inf
        lse = math.log(float(top.sum()))
        vals = np.where(top, -lse, -math.inf)
    else:
        with np.errstate(under="ignore"):
            lse = math.log(float(np.sum(np.exp((zd - m) / T))))
            vals = (zd - m) / T - lse
    lp[:take.size] = vals[take]
    return ids, lp


def draw_many(w: np.ndarray, R: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Inverse-CDF tokens for many uniforms over one fixed (w, R) (distribution tests)."""
    run = np.cumsum(np.where(R, w, 0.0))
    t = np.asarray(u, dtype=np.float64) * run[-1]
    tok = np.searchsorted(run, t, side="right")
    last = int(np.nonzero(R)[0][-1])
    return np.minimum(tok, last)
