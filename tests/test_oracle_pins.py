"""Pins for the fp64 oracle: brute force, closed forms, known answers, statistics.

These run on CPU (not marked gpu).  Each pin is chosen so that a plausible
mistake in the oracle (a dropped term, a wrong comparison, an off-by-one, a
wrong shift or index in the generator) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute
from conftest import read_golden
from device_logits_sampling_gb300 import workloads as wl


def prm(T=1.0, top_k=-1, top_p=1.0, min_p=0.0, rep=1.0, freq=0.0, pres=0.0, seed=0, step=0):
    p = wl.make_params(1)[0]
    p["temperature"] = T
    p["top_k"] = top_k
    p["top_p"] = top_p
    p["min_p"] = min_p
    p["repetition_penalty"] = rep
    p["frequency_penalty"] = freq
    p["presence_penalty"] = pres
    p["seed"] = seed
    p["step"] = step
    return p


# ------------------------------------------------------------ generator pins
def test_splitmix64_known_answers():
    rows = read_golden("splitmix64_state0.txt")
    assert len(rows) == 3
    for state, expect in rows:
        assert oracle.splitmix64(int(state, 16)) == int(expect, 16)


def test_uniform_is_53_bit_exact_and_mixes_row_seed_step():
    # u is an exact multiple of 2^-53 in [0, 1)
    for s in range(50):
        u = oracle.uniform(s, 3, 7)
        assert 0.0 <= u < 1.0
        assert float(u * 2**53).is_integer()
    # x = seed ^ (row << 32) ^ step, so these triples share one state
    x = 0x0123456789ABCDEF
    a = oracle.draw_bits(x, 0, 0)
    assert oracle.draw_bits(x ^ (5 << 32), 5, 0) == a
    assert oracle.draw_bits(x ^ 9, 0, 9) == a
    assert oracle.draw_bits(0, 0, 0) == 0xE220A8397B1DCDAF >> 11
    # row enters shifted by 32 bits, not as-is
    assert oracle.draw_bits(0, 1, 0) == oracle.splitmix64(1 << 32) >> 11
    assert oracle.draw_bits(0, 1, 0) != oracle.draw_bits(0, 0, 1)


# ------------------------------------------------------------ worked examples
def test_worked_example_v4():
    z = np.array([2.0, 0.0, 1.0, 2.0], dtype=np.float32)
    for k, p, mp, u, tok in read_golden("worked_example_v4.txt"):
        pr = prm(T=1.0, top_k=int(k), top_p=float(p), min_p=float(mp))
        r = oracle.sample_row_u(z, pr, float(u))
        assert r.token == int(tok), (k, p, mp, u)
        b = brute.sample(list(map(float, z)), 1.0, int(k), float(np.float32(p)),
                         float(np.float32(mp)), float(u))
        assert b == int(tok)


def test_penalty_example():
    z = np.array([2.0, -1.0, 0.5, 3.0], dtype=np.float32)
    hist = np.array([0, 0, 1, 3], dtype=np.int32)
    for rep, freq, pres, z0, z1, z2, z3, g in read_golden("penalty_example.txt"):
        zp = oracle.apply_penalties(z, hist, float(rep), float(freq), float(pres))
        assert zp.tolist() == [float(z0), float(z1), float(z2), float(z3)]
        r = oracle.sample_row_u(z, prm(T=0.0, rep=float(rep), freq=float(freq), pres=float(pres)),
                                0.5, hist)
        assert r.token == int(g)


def test_d2h_bytes_figure():
    (B, V, eb, nbytes, mb), = read_golden("d2h_bytes.txt")
    assert int(B) * int(V) * int(eb) == int(nbytes)
    assert round(int(nbytes) / 1e6, 1) == float(mb)
    assert wl.VOCAB_V4 == int(V)


# ------------------------------------------------------------ brute force
def _rand_row(rng, V, ties):
    x = rng.standard_normal(V) * rng.uniform(0.3, 3.0)
    if ties:
        x = np.round(x)
    return x.astype(np.float32)


@pytest.mark.parametrize("ties", [False, True])
def test_oracle_matches_brute_force_tiny(ties):
    rng = np.random.default_rng(1234 + ties)
    u_grid = [0.0, 0.013, 0.25, 0.4999, 0.5, 0.77, 0.999999]
    checked = 0
    for trial in range(60):
        V = int(rng.integers(1, 17))
        z = _rand_row(rng, V, ties)
        hist = rng.integers(0, V, size=int(rng.integers(0, 6))).astype(np.int32)
        T = float(np.float32(rng.choice([0.0, 0.25, 0.7, 1.0, 2.5])))
        k = int(rng.choice([-1, 0, 1, 2, 3, V - 1, V, V + 3]))
        p = float(np.float32(rng.choice([1.0, 0.9, 0.5, 0.1, 1e-6])))
        mp = float(np.float32(rng.choice([0.0, 0.05, 0.3, 1.0])))
        rep = float(np.float32(rng.choice([1.0, 1.3, 0.7])))
        fr = float(np.float32(rng.choice([0.0, 0.4, -0.2])))
        pr_ = float(np.float32(rng.choice([0.0, 0.5, -0.1])))
        pr = prm(T=T, top_k=k, top_p=p, min_p=mp, rep=rep, freq=fr, pres=pr_)
        for u in u_grid:
            a = oracle.sample_row_u(z, pr, u, hist).token
            b = brute.sample(list(map(float, z)), T, k, p, mp, u, hist.tolist(), rep, fr, pr_)
            assert a == b, (trial, V, z.tolist(), hist.tolist(), T, k, p, mp, u)
            checked += 1
    assert checked == 60 * len(u_grid)


# ------------------------------------------------------------ closed forms
def test_one_hot_returns_hot_index_in_every_mode():
    V = 37
    for hot in (0, 11, V - 1):
        z = np.full(V, -1e4, dtype=np.float32)
        z[hot] = 0.0
        for kw in (dict(T=0.0), dict(T=1.0), dict(T=0.7, top_k=5), dict(T=1.0, top_p=0.9),
                   dict(T=1.0, min_p=0.05), dict(T=1.3, top_k=V - 1, top_p=0.5, min_p=0.01)):
            for u in (0.0, 0.3, 0.999999999):
                assert oracle.sample_row_u(z, prm(**kw), u).token == hot
        # an exact -inf background gives the same answer
        z2 = np.full(V, -np.inf, dtype=np.float32)
        z2[hot] = 3.0
        assert oracle.sample_row_u(z2, prm(T=1.0), 0.99).token == hot


def test_tiny_temperature_is_argmax():
    rng = np.random.default_rng(7)
    for _ in range(20):
        z = rng.standard_normal(200).astype(np.float32)
        am = int(np.argmax(z))
        for u in (0.0, 0.5, 0.999999):
            assert oracle.sample_row_u(z, prm(T=1e-6), u).token == am


def test_top_k_one_is_greedy_under_ties():
    z = np.array([1.0, 5.0, 3.0, 5.0, 5.0], dtype=np.float32)
    for u in (0.0, 0.5, 0.99):
        assert oracle.sample_row_u(z, prm(T=1.0, top_k=1), u).token == 1
        assert oracle.sample_row_u(z, prm(T=0.0), u).token == 1


def test_all_equal_row_closed_forms():
    V = 1024
    z = np.zeros(V, dtype=np.float32)
    assert oracle.sample_row_u(z, prm(T=0.0), 0.7).token == 0
    for seed in range(200):
        bits = oracle.draw_bits(seed, 2, 5)
        u = bits * 2.0 ** -53
        # uniform CDF over a power-of-two V: token = floor(u * V) exactly
        assert oracle.sample_row_u(z, prm(T=1.0, seed=seed), u).token == bits >> (53 - 10)


def test_top_k_equal_V_is_inert():
    rng = np.random.default_rng(3)
    z = rng.standard_normal(300).astype(np.float32)
    for u in np.linspace(0, 0.999, 25):
        a = oracle.sample_row_u(z, prm(T=0.9, top_k=300), u).token
        b = oracle.sample_row_u(z, prm(T=0.9), u).token
        assert a == b
    assert oracle.row_mode(prm(T=0.9, top_k=300), 300) == oracle.MODE_INERT
    assert oracle.row_mode(prm(T=0.9, top_k=299), 300) == oracle.MODE_FILTERED


def test_neutral_penalties_are_bit_exact_no_op():
    rng = np.random.default_rng(11)
    z = (rng.standard_normal(500) * 4).astype(np.float32)
    hist = rng.integers(0, 500, size=300).astype(np.int32)
    zp = oracle.apply_penalties(z, hist, 1.0, 0.0, 0.0)
    assert zp.tobytes() == z.tobytes()


def test_penalty_direction_and_count():
    z = np.array([4.0, -4.0, 4.0], dtype=np.float32)
    zp = oracle.apply_penalties(z, np.array([0, 1, 2, 2, 2], dtype=np.int32), 2.0, 1.0, 0.5)
    # positive logit divided, negative multiplied; count 3 for id 2
    assert zp.tolist() == [4 / 2 - 1 - 0.5, -4 * 2 - 1 - 0.5, 4 / 2 - 3 - 0.5]


def test_min_p_one_keeps_only_max_ties():
    z = np.array([0.0, 2.0, 1.0, 2.0, -3.0], dtype=np.float32)
    got = {oracle.sample_row_u(z, prm(T=1.0, min_p=1.0), u).token for u in np.linspace(0, 0.9999, 40)}
    assert got == {1, 3}


def test_tiny_top_p_keeps_only_max_ties():
    z = np.array([0.0, 2.0, 1.0, 2.0, -3.0], dtype=np.float32)
    r = oracle.sample_row_u(z, prm(T=1.0, top_p=1e-6), 0.3)
    assert np.nonzero(r.R)[0].tolist() == [1, 3]


def test_top_p_boundary_keeps_every_tie():
    # four tied top entries (w = 1) and four at w = e^-1: the walk reaches
    # 0.1 * S after the first tied entry, and every entry tied with it stays
    z = np.array([1.0, 0, 0, 1.0, 1.0, 0, 1.0, 0], dtype=np.float32)
    r = oracle.sample_row_u(z, prm(T=1.0, top_p=0.1), 0.0)
    assert np.nonzero(r.R)[0].tolist() == [0, 3, 4, 6]
    assert r.tau == 1.0


def test_top_k_matches_stable_sort_and_partition():
    rng = np.random.default_rng(5)
    for _ in range(30):
        V = int(rng.integers(2, 3000))
        z = np.round(rng.standard_normal(V) * 3, 1).astype(np.float32)
        k = int(rng.integers(1, V))
        K = oracle.top_k_mask(z, k)
        assert K.sum() == k
        order = np.argsort(-z.astype(np.float64), kind="stable")
        assert set(np.nonzero(K)[0]) == set(order[:k].tolist())
        kth = np.partition(z, V - k)[V - k]
        assert z[K].min() == kth
        assert (z[~K] <= kth).all()


def test_filters_compose_in_page_order():
    # top-p is computed over the top-k survivors, not over the whole row
    z = np.array([3.0, 2.9, 2.8] + [0.0] * 50, dtype=np.float32)
    r = oracle.sample_row_u(z, prm(T=1.0, top_k=2, top_p=0.6), 0.1)
    # over K = {0, 1}: w = [1, e^-0.1], S_K = 1.9048; 0.6 * S_K = 1.143 -> both kept
    assert np.nonzero(r.R)[0].tolist() == [0, 1]
    # over the whole row S = 1 + e^-0.1 + e^-0.2 + 50 e^-3 = 5.213; 0.6 * S = 3.128
    # is reached inside the 50 tied zeros, so every one of them is kept
    r2 = oracle.sample_row_u(z, prm(T=1.0, top_p=0.6), 0.1)
    assert r2.R.all()
    # 0.5 * S = 2.606 is reached at the third entry
    r3 = oracle.sample_row_u(z, prm(T=1.0, top_p=0.5), 0.1)
    assert np.nonzero(r3.R)[0].tolist() == [0, 1, 2]
    # min-p after top-p: e^-0.2 = 0.8187 < 0.85 drops id 2
    r4 = oracle.sample_row_u(z, prm(T=1.0, top_p=0.5, min_p=0.85), 0.1)
    assert np.nonzero(r4.R)[0].tolist() == [0, 1]


def test_degenerate_and_invalid_rows():
    z = np.full(8, -np.inf, dtype=np.float32)
    r = oracle.sample_row_u(z, prm(T=1.0), 0.4)
    assert r.token == 0 and r.err & oracle.ERR_DEGENERATE
    zn = np.array([np.nan, 1.0, np.nan, 0.5], dtype=np.float32)
    r = oracle.sample_row_u(zn, prm(T=0.0), 0.4)
    assert r.token == 1 and r.err & oracle.ERR_NAN
    for bad in (dict(T=-1.0), dict(T=float("nan")), dict(top_p=0.0), dict(top_p=1.5),
                dict(min_p=-0.1), dict(min_p=1.01), dict(rep=0.0), dict(freq=float("inf"))):
        r = oracle.sample_row_u(np.zeros(4, np.float32), prm(**bad), 0.2)
        assert r.token == -1 and r.err == oracle.ERR_PARAM
    r = oracle.sample_row_u(np.zeros(4, np.float32), prm(), 0.2, np.array([4], np.int32))
    assert r.token == -1 and r.err == oracle.ERR_HIST_ID
    zi = np.array([1.0, np.inf, 0.0, np.inf], dtype=np.float32)
    assert oracle.sample_row_u(zi, prm(T=1.0), 0.2).token == 1
    assert oracle.sample_row_u(zi, prm(T=1.0), 0.7).token == 3


# ------------------------------------------------------------ statistics
def _chi2(counts, probs, n):
    from scipy.stats import chi2

    exp = probs * n
    order = np.argsort(exp)
    obs_m, exp_m = [], []
    acc_o = acc_e = 0.0
    for i in order:  # merge small bins so every bin expects >= 5
        acc_o += counts[i]
        acc_e += exp[i]
        if acc_e >= 5:
            obs_m.append(acc_o)
            exp_m.append(acc_e)
            acc_o = acc_e = 0.0
    if acc_e > 0:
        obs_m[-1] += acc_o
        exp_m[-1] += acc_e
    obs_m, exp_m = np.array(obs_m), np.array(exp_m)
    stat = float(((obs_m - exp_m) ** 2 / exp_m).sum())
    return float(chi2.sf(stat, len(obs_m) - 1))


def _softmax(z, T):
    m = max(z)
    e = [math.exp((x - m) / T) for x in z]
    s = sum(e)
    return np.array([x / s for x in e])


@pytest.mark.parametrize("case", ["plain", "top_k", "top_p"])
def test_frequencies_match_softmax_chi_square(case):
    pytest.importorskip("scipy")
    z = np.array([1.5, -0.5, 0.2, 2.0, 1.9, -2.0, 0.0, 0.7], dtype=np.float32)
    T = 0.8
    n = 100_000
    u = np.array([oracle.uniform(s, 0, 0) for s in range(n)])
    kw = dict(T=T)
    target = _softmax(z.tolist(), T)
    if case == "top_k":
        kw["top_k"] = 3
        keep = np.argsort(-z, kind="stable")[:3]
        t = np.zeros(8)
        t[keep] = target[keep]
        target = t / t.sum()
    elif case == "top_p":
        kw["top_p"] = 0.7
        order = np.argsort(-target, kind="stable")
        c = np.cumsum(target[order])
        n_keep = int(np.argmax(c >= float(np.float32(0.7)))) + 1
        t = np.zeros(8)
        t[order[:n_keep]] = target[order[:n_keep]]
        target = t / t.sum()
    r = oracle.sample_row_u(z, prm(**kw), 0.0)
    toks = oracle.draw_many(r.w, r.R, u)
    counts = np.bincount(toks, minlength=8)
    # spot-check the vectorised draw against the row sampler
    for s in range(0, n, 9973):
        assert oracle.sample_row_u(z, prm(**kw), float(u[s])).token == toks[s]
    pval = _chi2(counts, target, n)
    tv = 0.5 * np.abs(counts / n - target).sum()
    assert pval > 1e-3, (pval, counts, target * n)
    assert tv < 0.01
    # negative control: a narrowed distribution must be rejected
    narrow = _softmax(z.tolist(), T * 0.7)
    if case != "plain":
        narrow = np.where(target > 0, narrow, 0)
        narrow /= narrow.sum()
    assert _chi2(counts, narrow, n) < 1e-6


def test_mixed_workload_rows_use_the_stated_quarters():
    w = wl.mixed_batch(B=8, V=4096)
    modes = [oracle.row_mode(w.params[r], w.V) for r in range(8)]
    assert modes == [0, 1, 2, 2] * 2
    res = oracle.sample_batch(w.logits_f32(), w.params)
    for r in range(0, 8, 4):
        assert res[r].token == int(np.argmax(w.logits_f32()[r]))


# ---------------------------------------------------------------- top-n log-probabilities
def _brute_top_logprobs(z, T, n):
    """Explicit sort of (id, value) pairs and probabilities summed with math.fsum."""
    T = float(np.float32(T)) if float(np.float32(T)) > 0 else 1.0
    pairs = sorted(range(len(z)), key=lambda i: (-float(z[i]), i))
    m = max(float(v) for v in z)
    e = [math.exp((float(v) - m) / T) if v != -math.inf else 0.0 for v in z]
    tot = math.fsum(e)
    out = []
    for i in pairs[:n]:
        out.append((i, math.log(e[i] / tot) if e[i] > 0 else -math.inf))
    return out


@pytest.mark.parametrize("ties", [False, True])
def test_top_logprobs_brute_force_tiny(ties):
    rng = np.random.default_rng(123 + ties)
    for _ in range(200):
        V = int(rng.integers(1, 13))
        z = (rng.integers(-3, 4, size=V) if ties else rng.standard_normal(V) * 2).astype(np.float32)
        if V > 2 and rng.random() < 0.2:
            z[int(rng.integers(0, V))] = -np.inf
        if not np.isfinite(z).any():
            continue
        T = float(rng.choice([0.0, 0.5, 1.0, 1.7]))
        n = int(rng.integers(1, V + 3))
        ids, lp = oracle.top_logprobs(z, T, n)
        want = _brute_top_logprobs(z, T, n)
        assert ids[:len(want)].tolist() == [i for i, _ in want]
        for (i, v), g in zip(want, lp):
            assert (v == -math.inf and g == -math.inf) or abs(g - v) <= 1e-12 * max(1.0, abs(v)), (v, g)
        assert (ids[len(want):] == -1).all() and (lp[len(want):] == -math.inf).all()


def test_top_logprobs_closed_forms():
    # a flat row: every id has probability 1/V, listed in id order
    ids, lp = oracle.top_logprobs(np.zeros(1000, dtype=np.float32), 0.7, 5)
    assert ids.tolist() == [0, 1, 2, 3, 4] and np.allclose(lp, -math.log(1000), rtol=0, atol=1e-12)
    # two levels: k ids at a, V - k at b
    V, k, a, b = 500, 3, 2.0, -1.0
    T = float(np.float32(0.8))  # the row parameter is an fp32 value
    z = np.full(V, b, dtype=np.float32)
    z[[7, 100, 42]] = a
    ids, lp = oracle.top_logprobs(z, T, 5)
    top = -math.log(k + (V - k) * math.exp((b - a) / T))
    assert ids.tolist() == [7, 42, 100, 0, 1]
    assert np.allclose(lp[:3], top, rtol=0, atol=1e-12)
    assert np.allclose(lp[3:], (b - a) / T + top, rtol=0, atol=1e-12)
    # a greedy row (T = 0) reports the distribution at T = 1
    z = np.random.default_rng(3).standard_normal(64).astype(np.float32)
    assert np.array_equal(oracle.top_logprobs(z, 0.0, 8)[1], oracle.top_logprobs(z, 1.0, 8)[1])
    # +inf entries share all the mass
    z[[5, 9]] = np.inf
    ids, lp = oracle.top_logprobs(z, 1.0, 3)
    assert ids[:2].tolist() == [5, 9] and np.allclose(lp[:2], -math.log(2)) and lp[2] == -math.inf


def test_top_logprobs_are_a_distribution_in_sorted_order():
    rng = np.random.default_rng(9)
    z = (rng.standard_normal(3000) * 3).astype(np.float32)
    ids, lp = oracle.top_logprobs(z, 0.9, 3000)
    assert sorted(ids.tolist()) == list(range(3000))
    assert np.all(np.diff(lp) <= 0)
    assert abs(math.fsum(np.exp(lp)) - 1.0) <= 1e-12
    # the ids are the top-k filter's set for every k
    for k in (1, 17, 500):
        assert set(ids[:k].tolist()) == set(np.nonzero(oracle.top_k_mask(z, k))[0].tolist())
