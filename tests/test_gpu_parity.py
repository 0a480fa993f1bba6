"""Parity of the CUDA sampler with the fp64 oracle (needs a GB300 and the built library).

Every call goes through the C ABI (ctypes binding).  Rules: greedy tokens and
top-k survivor sets bit-exact; top-p / min-p survivors and sampled tokens
equal up to the 1e-6 boundary exemptions of tests/parity.py, which are counted.
"""
import functools

import numpy as np
import pytest

import oracle
import parity
from device_logits_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run(S, w, ld=None, ctas_per_row=0, max_hist_len=0, autoinc=False, params=None, force_bisection=False):
    import torch

    logits = S.logits_tensor(w, ld=ld)
    prm = params if params is not None else S.params_tensor(w.params)
    hoff, hids = S.history_tensors(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dbg = S.debug_tensor(w.B)
    S.sample_batch(logits, prm, out, hoff, hids, err_word=err, debug=dbg, ctas_per_row=ctas_per_row,
                   max_hist_len=max_hist_len, autoinc=autoinc, force_bisection=force_bisection)
    torch.cuda.synchronize()
    return out.cpu().numpy(), S.debug_records(dbg), int(err.item()) & 0xFFFFFFFF


@functools.lru_cache(maxsize=None)
def named(name):
    w = wl.NAMED[name]()
    res = oracle.sample_batch(w.logits_f32(), w.params, w.hist_offsets, w.hist_ids)
    return w, res


@pytest.mark.parametrize("name", ["small_fp32", "mixed_quarters", "penalized", "adversarial_ties"])
def test_named_workload_parity(cuda_lib, name):
    w, res = named(name)
    tokens, dbg, err = run(cuda_lib, w, max_hist_len=256 if w.hist_offsets is not None else 0)
    rep = parity.check_batch(w, tokens, dbg, results=res)
    print(f"{name}: rows={rep.rows} greedy={rep.greedy} sampled={rep.sampled} "
          f"set_exempt={rep.set_exempt} token_exempt={rep.token_exempt}")
    assert rep.rows == w.B
    assert err & ~parity.GPU_ERR_NAN == 0, hex(err)
    # boundary exemptions stay rare
    assert rep.set_exempt + rep.token_exempt <= max(2, w.B // 50)
    # the modes the workload intends are the ones the kernel took
    modes = np.array([oracle.row_mode(w.params[r], w.V) for r in range(w.B)])
    assert np.array_equal(dbg["mode"], modes)


def test_single_row_decode_loop_1000_steps(cuda_lib):
    """B=1 peaked row, the server defaults, step advanced on device for 1,000 calls."""
    import torch

    S = cuda_lib
    w = wl.single_row_peaked()
    logits = S.logits_tensor(w)
    prm = S.params_tensor(w.params)
    out = torch.zeros(1000, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = S.workspace_tensor(1, w.V, w.dtype)
    for step in range(1000):
        S.sample_batch(logits, prm, out[step:step + 1], err_word=err, workspace=ws, autoinc=True)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert int(err.item()) == 0
    assert S.debug_records  # binding loaded
    # the step counter advanced on device
    p = prm.cpu().numpy().view(wl.ROW_PARAMS_DTYPE)[0]
    assert int(p["step"]) == 1000
    r0 = oracle.sample_row_u(w.logits_f32()[0], w.params[0], 0.0)
    u = np.array([oracle.uniform(0, 0, s) for s in range(1000)])
    want = oracle.draw_many(r0.w, r0.R, u)
    mism = np.nonzero(got != want)[0]
    run_ = np.cumsum(np.where(r0.R, r0.w, 0.0))
    S_ = float(run_[-1])
    # draws whose u lies within 1e-6 of the oracle's CDF at a boundary of the
    # drawn token (counted and reported); a differing token's own CDF interval
    # must come within 1e-6 of u
    near = np.array([min(abs(run_[want[s]] / S_ - u[s]), abs(run_[want[s] - 1] / S_ - u[s]) if want[s] > 0 else 1.0)
                     for s in range(1000)])
    boundary = np.nonzero(near <= 1e-6)[0]
    print(f"decode loop: {mism.size} of 1000 tokens differ, {boundary.size} draws lie within 1e-6 of a boundary")
    for s in mism.tolist():
        assert s in set(boundary.tolist()), s
        assert parity.token_within(r0.R, run_, S_, int(got[s]), float(u[s])), s
    assert mism.size <= 10
    # the draws follow the softmax: spikes carry most of the mass
    spikes = set(w.notes["spikes"].tolist())
    frac = np.mean([t in spikes for t in got])
    mass = r0.w[list(spikes)].sum() / r0.w.sum()
    assert abs(frac - mass) < 0.06
    # greedy version: every step returns the argmax
    wg = wl.single_row_peaked(greedy=True)
    tok, dbg, err = run(S, wg)
    assert tok[0] == int(np.argmax(wg.logits_f32()[0]))


@pytest.mark.parametrize("name", ["small_fp32", "single_row_peaked", "mixed_quarters", "penalized",
                                  "adversarial_ties"])
def test_greedy_kernel_is_exact_argmax(cuda_lib, name):
    import torch

    w = wl.NAMED[name]()
    logits = cuda_lib.logits_tensor(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    cuda_lib.sample_greedy(logits, out)
    torch.cuda.synchronize()
    z = w.logits_f32()
    assert out.cpu().numpy().tolist() == np.argmax(z, axis=1).tolist()


@pytest.mark.parametrize("V,dtype,ld_pad,B", [
    (1, 1, 0, 3), (5, 0, 0, 4), (8, 1, 0, 5), (9, 1, 0, 6), (1000, 0, 0, 12), (4097, 1, 0, 12),
    (12345, 1, 0, 12), (12345, 0, 3, 12), (4097, 1, 8, 12), (33333, 1, 1, 12), (200_000, 1, 0, 6),
    (129_280, 0, 4, 6),
    # fp16 logits
    (7, 2, 0, 4), (4097, 2, 3, 12), (33333, 2, 0, 12), (129_280, 2, 0, 40), (200_000, 2, 8, 6),
])
def test_ragged_and_strided_rows(cuda_lib, V, dtype, ld_pad, B):
    w = wl.random_case(seed=V * 7 + dtype + ld_pad, B=B, V=V, dtype=dtype, ties=(V % 2 == 1))
    tokens, dbg, err = run(cuda_lib, w, ld=V + ld_pad if ld_pad else None)
    rep = parity.check_batch(w, tokens, dbg)
    assert rep.rows == B


@pytest.mark.parametrize("name", ["small_fp32", "mixed_quarters", "penalized", "adversarial_ties"])
def test_fp16_logits_parity(cuda_lib, name):
    """The named workloads as fp16 logits: the oracle on the fp16 values, the
    same rules; greedy rows also through arc_sample_greedy."""
    import torch

    w = wl.as_f16(wl.NAMED[name]())
    res = oracle.sample_batch(w.logits_f32(), w.params, w.hist_offsets, w.hist_ids)
    tokens, dbg, err = run(cuda_lib, w, max_hist_len=256 if w.hist_offsets is not None else 0)
    rep = parity.check_batch(w, tokens, dbg, results=res)
    assert rep.rows == w.B
    assert err & ~parity.GPU_ERR_NAN == 0, hex(err)
    assert rep.set_exempt + rep.token_exempt <= max(2, w.B // 50)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    cuda_lib.sample_greedy(cuda_lib.logits_tensor(w), out)
    torch.cuda.synchronize()
    assert out.cpu().numpy().tolist() == np.argmax(w.logits_f32(), axis=1).tolist()


@pytest.mark.parametrize("hist_len", [1, 64, 700])
def test_penalties_random(cuda_lib, hist_len):
    w = wl.random_case(seed=100 + hist_len, B=24, V=30011, dtype=1, hist_len=hist_len)
    tokens, dbg, err = run(cuda_lib, w, max_hist_len=hist_len)
    rep = parity.check_batch(w, tokens, dbg)
    assert rep.rows == w.B and err == 0


def test_ctas_per_row_does_not_change_results(cuda_lib):
    """Survivor sets are exact for every split of the row; tokens agree up to the
    chunk-level rounding of the default-row masses (boundary cases only)."""
    w = wl.random_case(seed=9, B=30, V=20000, dtype=1, ties=True)
    base = None
    for s in (3, 5, 8, 16, 32):
        tok, dbg, err = run(cuda_lib, w, ctas_per_row=s)
        parity.check_batch(w, tok, dbg)
        fields = dbg[["kappa_k", "iota_k"]]
        if base is None:
            base = (tok, fields)
        else:
            assert np.array_equal(fields, base[1]), s
            assert np.mean(tok == base[0]) >= 0.9, s


def test_mixed_batch_geometries_agree(cuda_lib):
    w, res = named("mixed_quarters")
    t8, d8, _ = run(cuda_lib, w, ctas_per_row=32)
    t16, d16, _ = run(cuda_lib, w, ctas_per_row=16)
    parity.check_batch(w, t16, d16, results=res)
    assert np.mean(t8 == t16) >= 0.99
    assert np.array_equal(d8[["kappa_k", "iota_k"]], d16[["kappa_k", "iota_k"]])


def test_top_k_ties_break_to_lowest_ids(cuda_lib):
    V = 50_000
    z = np.zeros((4, V), dtype=np.float32)
    z[:, ::7] = 3.0  # 7143 tied entries at the top
    p = wl.make_params(4)
    p["top_k"] = [5, 100, 7142, 7144]
    p["temperature"] = 1.0
    p["seed"] = [1, 2, 3, 4]
    w = wl.Workload("ties", wl.DTYPE_F32, z, p)
    tokens, dbg, err = run(cuda_lib, w)
    parity.check_batch(w, tokens, dbg)
    assert dbg["iota_k"][0] == 7 * 4 + 1
    assert dbg["iota_k"][1] == 7 * 99 + 1


@pytest.mark.parametrize("dtype", [wl.DTYPE_F32, wl.DTYPE_BF16])
def test_top_k_cut_inside_small_tie_group(cuda_lib, dtype):
    """The k-th logit falls in a run of 30 equal values above 20 distinct ones and
    a N(0, 1) background: few candidates, so the direct selection ranks them.
    Rows alternate pure top-k (the survivors are K), top-k with top-p (the cut
    can land inside K) and top-k with min-p."""
    B, V = 12, 40_000
    rng = np.random.default_rng(11)
    z = rng.standard_normal((B, V)).astype(np.float32)
    p = wl.make_params(B)
    ks = [25, 20, 21, 50, 49, 3]
    tied_ids = []
    for r in range(B):
        ids = rng.choice(V, size=50, replace=False)
        z[r, ids[:20]] = 8.0 + 0.125 * np.arange(20, dtype=np.float32)  # exact in bf16 too
        z[r, ids[20:]] = 6.0
        tied_ids.append(np.sort(ids[20:]))
        p[r]["top_k"] = ks[r % len(ks)]
        p[r]["temperature"] = 1.0 if r % 2 == 0 else 0.7
        if r % 3 == 1:
            p[r]["top_p"] = 0.6
        elif r % 3 == 2:
            p[r]["min_p"] = 0.02
        p[r]["seed"] = 100 + r
    logits = wl.f32_to_bf16_bits(z) if dtype == wl.DTYPE_BF16 else z
    w = wl.Workload("tie_group", dtype, logits, p)
    tokens, dbg, err = run(cuda_lib, w)
    rep = parity.check_batch(w, tokens, dbg)
    assert rep.rows == B
    assert err == 0, hex(err)
    for r in range(B):
        k = int(p[r]["top_k"])
        if 20 < k < 50:  # the cut inside the run: the first k - 20 tied ids survive
            assert dbg["iota_k"][r] == tied_ids[r][k - 21] + 1, r
        else:  # the cut between distinct values, or after the run: every id of the key survives
            assert dbg["iota_k"][r] == V, r


def test_row_errors_and_degenerate_rows(cuda_lib):
    V = 3000
    rng = np.random.default_rng(0)
    z = rng.standard_normal((8, V)).astype(np.float32)
    z[4, :] = -np.inf
    z[5, 10] = np.nan
    z[6, [3, 77]] = np.inf
    z[7, :] = np.nan
    p = wl.make_params(8)
    p["seed"] = np.arange(8)
    p[0]["temperature"] = -1.0
    p[1]["top_p"] = 0.0
    p[2]["min_p"] = 2.0
    p[3]["flags"] = 1
    w = wl.Workload("errors", wl.DTYPE_F32, z, p)
    tokens, dbg, err = run(cuda_lib, w)
    assert tokens[:4].tolist() == [-1, -1, -1, -1]
    assert all(dbg["err"][:4] & parity.GPU_ERR_PARAM)
    assert tokens[4] == 0 and dbg["err"][4] & parity.GPU_ERR_DEGENERATE
    assert tokens[5] != 10 and dbg["err"][5] & parity.GPU_ERR_NAN
    assert tokens[6] in (3, 77)
    assert tokens[7] == 0 and dbg["err"][7] & parity.GPU_ERR_DEGENERATE
    assert err & parity.GPU_ERR_PARAM and err & parity.GPU_ERR_NAN
    parity.check_batch(w, tokens, dbg, rows=[5, 6])
    # history id out of range
    w2 = wl.random_case(seed=3, B=4, V=500, dtype=0, hist_len=4)
    w2.hist_offsets = np.array([0, 1, 2, 3, 4], dtype=np.int32)
    w2.hist_ids = np.array([1, 500, 2, -1], dtype=np.int32)
    tokens, dbg, err = run(cuda_lib, w2)
    assert tokens[1] == -1 and tokens[3] == -1
    assert dbg["err"][1] & parity.GPU_ERR_HIST_ID and dbg["err"][3] & parity.GPU_ERR_HIST_ID
    assert tokens[0] >= 0 and tokens[2] >= 0
    # a history longer than the declared bound
    w3 = wl.random_case(seed=4, B=2, V=500, dtype=1, hist_len=40)
    w3.hist_offsets = np.array([0, 40, 40], dtype=np.int32)
    w3.hist_ids = np.arange(40, dtype=np.int32)
    tokens, dbg, err = run(cuda_lib, w3, max_hist_len=16)
    assert tokens[0] == -1 and dbg["err"][0] & 0x10
    assert tokens[1] >= 0


@pytest.mark.parametrize("kind", ["plain", "top_k", "top_p_min_p"])
def test_distribution_matches_softmax(cuda_lib, kind):
    """10^5 draws of one row (one per seed) against the oracle's exact probabilities."""
    from scipy.stats import chi2

    V, B = 64, 100_000
    rng = np.random.default_rng(42)
    row = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = wl.make_params(B)
    p["temperature"] = 0.9
    if kind == "top_k":
        p["top_k"] = 10
    elif kind == "top_p_min_p":
        p["top_p"] = 0.8
        p["min_p"] = 0.02
    p["seed"] = np.arange(B, dtype=np.uint64) * 7919 + 13
    w = wl.Workload("dist", wl.DTYPE_F32, np.tile(row, (B, 1)), p)
    tokens, dbg, err = run(cuda_lib, w)
    r0 = oracle.sample_row_u(row, p[0], 0.0)
    probs = np.where(r0.R, r0.w, 0.0) / np.where(r0.R, r0.w, 0.0).sum()
    counts = np.bincount(tokens, minlength=V)
    assert counts[~r0.R].sum() == 0
    keep = probs > 0
    exp = probs[keep] * B
    stat = float(((counts[keep] - exp) ** 2 / exp).sum())
    pval = chi2.sf(stat, keep.sum() - 1)
    tv = 0.5 * np.abs(counts / B - probs).sum()
    assert pval > 1e-4, (pval, tv)
    assert tv < 0.01
    # narrowed control: the same counts must reject a sharper distribution
    sharp = np.where(r0.R, np.exp((row - row.max()) / 0.6), 0.0)
    sharp /= sharp.sum()
    exp2 = sharp[keep] * B
    assert chi2.sf(float(((counts[keep] - exp2) ** 2 / exp2).sum()), keep.sum() - 1) < 1e-6
    # and the individual tokens follow the oracle
    rows = list(range(0, B, 997))
    parity.check_batch(w, tokens, dbg, rows=rows)
    # the threshold bisection draws the same token for (nearly) every seed: the
    # two selections are at total-variation distance <= 5e-5
    tokens_b, dbg_b, _ = run(cuda_lib, w, force_bisection=True)
    assert int((tokens_b != tokens).sum()) <= 5  # masses agree to ~1e-7 (see the test below)
    if kind != "plain":
        assert (dbg_b["passes"] >= 2).all()


@pytest.mark.parametrize("name", ["mixed_quarters", "adversarial_ties", "penalized"])
def test_enumeration_and_bisection_agree(cuda_lib, name):
    """Exact enumeration of the few ids above the floor and threshold bisection
    over the whole row select the same survivors and draw the same tokens;
    the debug pass counts tell which path each filtered row took."""
    w, res = named(name)
    mhl = 256 if w.hist_offsets is not None else 0
    t1, d1, e1 = run(cuda_lib, w, max_hist_len=mhl)
    t2, d2, e2 = run(cuda_lib, w, max_hist_len=mhl, force_bisection=True)
    assert e1 == e2
    assert np.array_equal(d1["mode"], d2["mode"])
    # the bisection rounds each 16-byte vector's fp32 weight sum to fixed point,
    # the enumeration each id's weight: masses agree to ~1e-7, so a token may
    # differ only where u lies that close to a boundary
    m1, m2 = d1["mass_r"].astype(np.float64), d2["mass_r"].astype(np.float64)
    assert np.allclose(m1, m2, rtol=1e-6, atol=2.0)
    assert int((t1 != t2).sum()) <= max(1, w.B // 100)
    # a survivor threshold may sit anywhere between two distinct keys: each
    # path's survivor sets and tokens go to the oracle
    for t, d in ((t1, d1), (t2, d2)):
        rep = parity.check_batch(w, t, d, results=res)
        assert rep.set_exempt + rep.token_exempt <= max(2, w.B // 50)
    filtered = d1["mode"] == 2
    assert (d2["passes"][filtered] >= 2).all()
    assert (d2["passes"][~filtered] == d1["passes"][~filtered]).all()
    direct = int((d1["passes"][filtered] == 1).sum())
    print(f"{name}: filtered rows {int(filtered.sum())}, direct selection {direct}, "
          f"bisection {int(filtered.sum()) - direct}")
    if name != "adversarial_ties":  # (whose tied nucleus holds tens of thousands of ids)
        assert direct >= 0.9 * int(filtered.sum())


def _rows(w, B, reps=1):
    """A workload of w's first B rows, repeated reps times (history included)."""
    import dataclasses

    idx = np.tile(np.arange(B), reps)
    ho, hi = None, None
    if w.hist_offsets is not None:
        lens = np.diff(w.hist_offsets)[idx]
        ho = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        hi = np.concatenate([w.hist_ids[w.hist_offsets[r]:w.hist_offsets[r + 1]] for r in idx]).astype(np.int32)
    return dataclasses.replace(w, logits=w.logits[idx].copy(), params=w.params[idx].copy(), hist_offsets=ho,
                               hist_ids=hi)


@pytest.mark.parametrize("name,B,force", [("adversarial_ties", 64, False), ("mixed_quarters", 16, True),
                                          ("penalized", 24, True), ("adversarial_ties", 8, False)])
def test_split_finish_matches_one_cta_per_row(cuda_lib, name, B, force):
    """A small batch finishes each row on a cluster of CTAs that splits the
    threshold bisection; the same rows at the head of a batch too large for
    that (one finish CTA per row, same slices) give identical tokens and
    debug records, and the split rows match the oracle."""
    S = cuda_lib
    w, _ = named(name)
    small, big = _rows(w, B), _rows(w, B, reps=(320 + B - 1) // B)
    mhl = 256 if w.hist_offsets is not None else 0
    s = 16 if w.dtype == wl.DTYPE_BF16 else 32  # the fewest slices a 129,280-id row allows
    assert S.plan(small.B, w.V, w.dtype, ctas_per_row=s).finish_ctas > 1
    assert S.plan(big.B, w.V, w.dtype, ctas_per_row=s).finish_ctas == 1
    t1, d1, e1 = run(S, small, ctas_per_row=s, max_hist_len=mhl, force_bisection=force)
    t2, d2, e2 = run(S, big, ctas_per_row=s, max_hist_len=mhl, force_bisection=force)
    assert np.array_equal(t1, t2[:B])
    assert np.array_equal(d1, d2[:B])
    filtered = d1["mode"] == 2
    assert (d1["passes"][filtered] >= 2).any()  # the bisection ran on split rows
    res = oracle.sample_batch(small.logits_f32(), small.params, small.hist_offsets, small.hist_ids)
    rep = parity.check_batch(small, t1, d1, results=res)
    assert rep.set_exempt + rep.token_exempt <= max(2, B // 50)


def test_graph_replay_reads_step_from_device(cuda_lib):
    """A captured launch replayed 64 times draws 64 different steps (generator state on device)."""
    import torch

    S = cuda_lib
    V = 4096
    z = np.zeros((1, V), dtype=np.float32)
    p = wl.make_params(1)
    p["seed"] = 5
    w = wl.Workload("flat", wl.DTYPE_F32, z, p)
    logits = S.logits_tensor(w)
    prm = S.params_tensor(w.params)
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = S.workspace_tensor(1, V, w.dtype)
    S.sample_batch(logits, prm, out, workspace=ws)  # first call sets kernel attributes
    torch.cuda.synchronize()
    prm.copy_(S.params_tensor(w.params))
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            S.sample_batch(logits, prm, out, workspace=ws, autoinc=True, stream=stream)
    got = []
    for _ in range(64):
        g.replay()
        torch.cuda.synchronize()
        got.append(int(out.item()))
    want = [oracle.draw_bits(5, 0, s) >> (53 - 12) for s in range(64)]  # uniform over 4096
    assert got == want
    assert len(set(got)) > 60


@pytest.mark.parametrize("B,V,dtype,hist_len", [(1, 129_280, 1, 0), (4, 1024, 0, 0), (8, 30_011, 1, 64),
                                                 (8, 129_280, 1, 0), (3, 131_072, 1, 0), (7, 4097, 0, 0)])
def test_cluster_path_matches_two_kernels(cuda_lib, B, V, dtype, hist_len):
    """Small batches take one launch: a cluster of CTAs per row, their slice
    summaries combined through distributed shared memory.  With the same slices
    the two-kernel path (scan, workspace, finish) gives the same tokens and the
    same debug records, bit for bit; both match the oracle."""
    S = cuda_lib
    w = wl.random_case(seed=900 + B + V, B=B, V=V, dtype=dtype, ties=(V % 2 == 1), hist_len=hist_len)
    g = S.plan(B, V, dtype, has_history=hist_len > 0, max_hist_len=hist_len)
    assert g.launches == 1
    t1, d1, e1 = run(S, w, max_hist_len=hist_len)
    t2, d2, e2 = run(S, w, max_hist_len=hist_len, ctas_per_row=g.ctas_per_row)
    assert S.plan(B, V, dtype, has_history=hist_len > 0, max_hist_len=hist_len,
                  ctas_per_row=g.ctas_per_row).launches == 2
    assert np.array_equal(t1, t2) and e1 == e2
    assert np.array_equal(d1, d2)
    rep = parity.check_batch(w, t1, d1)
    assert rep.rows == B


def _check_top_logprobs(w, res, got, n):
    """ids exact; log-probabilities within 2e-6 + 1e-6 |lp| of the fp64 oracle
    (the fp32 chunk masses carry ~1e-7 relative error into ln S)."""
    bad = 0
    for r, rr in enumerate(res):
        g = got[r]
        if rr.mode == oracle.MODE_INVALID:
            assert (g["id"] == -1).all() and np.isneginf(g["logprob"]).all(), r
            continue
        ids, lp = oracle.top_logprobs(rr.z, float(w.params[r]["temperature"]), n)
        assert g["id"].tolist() == ids.tolist(), (r, g["id"][:8].tolist(), ids[:8].tolist())
        fin = np.isfinite(lp)
        assert np.array_equal(np.isfinite(g["logprob"]), fin), r
        err = np.abs(g["logprob"][fin].astype(np.float64) - lp[fin])
        bad += int((err > 2e-6 + 1e-6 * np.abs(lp[fin])).sum())
    assert bad == 0, bad


@pytest.mark.parametrize("name,n", [("small_fp32", 8), ("mixed_quarters", 5), ("penalized", 20),
                                    ("adversarial_ties", 64)])
def test_top_logprobs_match_the_oracle(cuda_lib, name, n):
    """Top-n (id, log-probability) per row through the C ABI, next to the
    sampled tokens, which the option leaves unchanged."""
    import torch

    S = cuda_lib
    w, res = named(name)
    mhl = 256 if w.hist_offsets is not None else 0
    logits = S.logits_tensor(w)
    prm = S.params_tensor(w.params)
    hoff, hids = S.history_tensors(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    tl = S.top_logprobs_tensor(w.B, n)
    S.sample_batch(logits, prm, out, hoff, hids, max_hist_len=mhl, top_n=n, top_logprobs=tl)
    torch.cuda.synchronize()
    _check_top_logprobs(w, res, S.top_logprobs_records(tl, n), n)
    base, _, _ = run(S, w, max_hist_len=mhl)
    assert np.array_equal(out.cpu().numpy(), base)


def test_top_logprobs_edge_rows(cuda_lib):
    """Ragged V below n (padding), NaN, -inf, +inf and invalid rows, ties; one
    launch (cluster) and two launches give the same records."""
    import torch

    S = cuda_lib
    V, n = 3000, 16
    rng = np.random.default_rng(5)
    z = rng.standard_normal((8, V)).astype(np.float32)
    z[1, :] = -np.inf
    z[2, 17] = np.nan
    z[3, [3, 77]] = np.inf
    z[4, :] = np.round(z[4, :])  # heavy ties
    z[5, :] = 0.0
    p = wl.make_params(8)
    p["seed"] = np.arange(8)
    p[6]["temperature"] = -1.0  # invalid
    p[7]["temperature"] = 0.0   # greedy: log-probabilities at T = 1
    p[0]["top_k"] = 10
    p[0]["temperature"] = 0.5
    w = wl.Workload("edges", wl.DTYPE_F32, z, p)
    res = oracle.sample_batch(w.logits_f32(), w.params)
    for cpr in (0, 5):
        logits = S.logits_tensor(w)
        prm = S.params_tensor(w.params)
        out = torch.zeros(8, dtype=torch.int32, device="cuda")
        tl = S.top_logprobs_tensor(8, n)
        S.sample_batch(logits, prm, out, ctas_per_row=cpr, top_n=n, top_logprobs=tl)
        torch.cuda.synchronize()
        _check_top_logprobs(w, res, S.top_logprobs_records(tl, n), n)
    # fewer ids than n: the rest is (-1, -inf)
    w2 = wl.random_case(seed=8, B=3, V=5, dtype=1)
    res2 = oracle.sample_batch(w2.logits_f32(), w2.params)
    logits = S.logits_tensor(w2)
    prm = S.params_tensor(w2.params)
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    tl = S.top_logprobs_tensor(3, 8)
    S.sample_batch(logits, prm, out, top_n=8, top_logprobs=tl)
    torch.cuda.synchronize()
    got = S.top_logprobs_records(tl, 8)
    _check_top_logprobs(w2, res2, got, 8)
    assert (got["id"][:, 5:] == -1).all()
