"""The decode-loop commit (include/arc_decode.h) against its oracle.

CPU: the oracle pinned to hand-worked cases, the host-only ring drain over a
ring in ordinary host memory, and the commit's host argument checks.  GPU:
the commit after the sampler record for record against the oracle, refused
rows, and a sample + commit step captured in a CUDA graph and replayed with
the host draining the ring without any CUDA call.
"""
import ctypes

import numpy as np
import pytest

from oracle import decode_commit as oc
from device_logits_sampling_gb300 import decode, sampler


# ---------------------------------------------------------------- oracle pins
def test_oracle_commit_hand_worked():
    # V = 10, max_position = 6, ring of 4 records, head 3 (the ring wraps)
    ring = oc.empty_ring(4)
    ids, pos, ring, head, fault = oc.commit(tokens=[4, 10, 2, -1], V=10, next_ids=[0, 0, 0, 0],
                                            positions=[0, 1, 6, 5], max_position=6,
                                            owners=[7, 8, 9, 10], head=3, capacity=4, ring=ring)
    assert ids == [4, 0, 0, 0]          # only row 0 commits
    assert pos == [1, 1, 6, 5]
    assert head == 7
    assert fault == oc.BAD_TOKEN | oc.BAD_POSITION
    # record i at slot i % 4, stamp i + 1; refused rows publish token -1
    assert ring[3] == (4, 0, 7, 4)      # record 3
    assert ring[0] == (-1, 1, 8, 5)     # record 4: token 10 is outside [0, 10)
    assert ring[1] == (-1, 6, 9, 6)     # record 5: position 6 is not below 6
    assert ring[2] == (-1, 5, 10, 7)    # record 6: token -1


def test_oracle_commit_is_sticky_and_leaves_inputs_alone():
    ids0, pos0 = [1, 1], [3, 3]
    ids, pos, ring, head, fault = oc.commit([5, 5], 8, ids0, pos0, 4, None, 0, 2, oc.empty_ring(2),
                                            fault=oc.BAD_POSITION)
    assert fault == oc.BAD_POSITION and ids == [5, 5] and pos == [4, 4]
    assert ids0 == [1, 1] and pos0 == [3, 3]
    assert [r[2] for r in ring] == [0, 0]  # no owners: tag 0
    assert oc.commit([5], 8, [0], [0], 4, None, (1 << 32) - 1, 2, oc.empty_ring(2))[2][1][3] == 0  # stamp wraps


# ---------------------------------------------------------------- host-only drain
@pytest.fixture(scope="module")
def lib():
    return sampler.load()


def host_ring(records):
    arr = oc.as_records(records)
    return arr, arr.ctypes.data


def test_drain_reads_complete_records_in_order(lib):
    _, _, ring, head, _ = oc.commit([1, 2, 3], 5, [0] * 3, [0] * 3, 9, [4, 5, 6], 0, 8, oc.empty_ring(8))
    arr, addr = host_ring(ring)
    got = decode.ring_drain(addr, 8, 0, 3, max_spins=10)
    assert got["token"].tolist() == [1, 2, 3] and got["owner"].tolist() == [4, 5, 6]
    assert got["stamp"].tolist() == [1, 2, 3]


def test_drain_stops_short_at_a_missing_record(lib):
    _, _, ring, _, _ = oc.commit([1, 2], 5, [0] * 2, [0] * 2, 9, None, 0, 8, oc.empty_ring(8))
    arr, addr = host_ring(ring)
    got = decode.ring_drain(addr, 8, 0, 5, max_spins=1000)
    assert len(got) == 2  # records 2..4 never landed


def test_drain_detects_an_overwritten_slot(lib):
    ring = oc.empty_ring(4)
    head = 0
    for _ in range(3):  # 6 records through a ring of 4: records 0 and 1 are gone
        _, _, ring, head, _ = oc.commit([1, 2], 5, [0, 0], [0, 0], 9, None, head, 4, ring)
    arr, addr = host_ring(ring)
    with pytest.raises(sampler.ArcError) as e:
        decode.ring_drain(addr, 4, 0, 1, max_spins=10)
    assert e.value.rc == decode.ARC_E_RING_OVERRUN
    assert decode.ring_drain(addr, 4, 2, 4, max_spins=10)["stamp"].tolist() == [3, 4, 5, 6]


def test_drain_across_the_stamp_wrap(lib):
    first = (1 << 32) - 2
    _, _, ring, _, _ = oc.commit([1, 2, 3], 5, [0] * 3, [0] * 3, 9, None, first, 4, oc.empty_ring(4))
    arr, addr = host_ring(ring)
    got = decode.ring_drain(addr, 4, first, 3, max_spins=10)
    assert got["stamp"].tolist() == [(1 << 32) - 1, 0, 1] and got["token"].tolist() == [1, 2, 3]


def _words(ring):
    """The ring's 8-byte words, [capacity, 3]: (value, stamp) each."""
    return ring.view(np.uint64).reshape(len(ring), 3)


def _put(ring, slot, values, stamp, words=(0, 1, 2)):
    """Store words of one slot the way the device does: one 8-byte store per
    word, the stamp in the high half."""
    w = _words(ring)
    for k in words:
        w[slot, k] = np.uint64((int(stamp) << 32) | (int(values[k]) & 0xFFFFFFFF))


def test_record_layout_is_three_stamped_words():
    assert decode.RECORD_DTYPE.itemsize == 24
    ring = np.zeros(1, dtype=decode.RECORD_DTYPE)
    _put(ring, 0, (-1, 7, 9), 5)
    r = ring[0]
    assert (int(r["token"]), int(r["position"]), int(r["owner"])) == (-1, 7, 9)
    assert int(r["stamp"]) == int(r["stamp_pos"]) == int(r["stamp_owner"]) == 5


def test_drain_never_confirms_a_slot_that_is_being_rewritten(lib):
    """A slot in the middle of a rewrite (some words of the new lap stored,
    the others still of the old one) is not a record of either lap: the old
    record reads as overrun, the new one as not yet published."""
    cap = 4
    ring = np.zeros(cap, dtype=decode.RECORD_DTYPE)
    for i in range(cap):  # lap 0 published
        _put(ring, i, (10 + i, i, 7), i + 1)
    new = cap + 1  # record 5 is being written into slot 1: its token word first
    _put(ring, 1, (99, 5, 8), new + 1, words=(0,))
    assert decode.ring_drain(ring.ctypes.data, cap, 0, 1, max_spins=50)["token"].tolist() == [10]
    with pytest.raises(sampler.ArcError) as e:
        decode.ring_drain(ring.ctypes.data, cap, 1, 1, max_spins=50)
    assert e.value.rc == decode.ARC_E_RING_OVERRUN
    assert len(decode.ring_drain(ring.ctypes.data, cap, new, 1, max_spins=50)) == 0
    _put(ring, 1, (99, 5, 8), new + 1, words=(2,))  # the owner word: still not whole
    assert len(decode.ring_drain(ring.ctypes.data, cap, new, 1, max_spins=50)) == 0
    _put(ring, 1, (99, 5, 8), new + 1, words=(1,))  # the rewrite completes
    got = decode.ring_drain(ring.ctypes.data, cap, new, 1)
    assert (int(got[0]["token"]), int(got[0]["position"]), int(got[0]["owner"]), int(got[0]["stamp"])) == \
        (99, 5, 8, new + 1)


def test_drain_against_a_writer_that_laps_it(lib):
    """A writer thread rewrites slots word by word as the commit does (one
    8-byte store per word, in a varying order) and laps the reader at will:
    every record the drain returns is whole (its fields agree with its
    stamp); a lapped read is an overrun, never a mixed record."""
    import threading

    cap, n = 8, 4000
    ring = np.zeros(cap, dtype=decode.RECORD_DTYPE)
    done = []
    orders = [(0, 1, 2), (2, 1, 0), (1, 0, 2)]

    def writer():
        for i in range(n):
            for k in orders[i % 3]:
                _put(ring, i % cap, (3 * i, i, i % 1000), i + 1, words=(k,))
        done.append(True)

    t = threading.Thread(target=writer)
    t.start()
    seen = 0
    first = 0
    while not done or first < n:
        try:
            got = decode.ring_drain(ring.ctypes.data, cap, first, 4, max_spins=200)
        except sampler.ArcError as e:
            assert e.rc == decode.ARC_E_RING_OVERRUN
            first = max(first + 1, int(ring["stamp"].max()) - cap)  # skip ahead of the writer
            continue
        for r in got:
            i = int(r["stamp"]) - 1
            assert (int(r["token"]), int(r["position"]), int(r["owner"])) == (3 * i, i, i % 1000)
            assert int(r["stamp_pos"]) == int(r["stamp_owner"]) == i + 1
        seen += len(got)
        first += len(got)
        if done and len(got) == 0:
            break
    t.join()
    assert seen > 0


def test_drain_waits_for_records_published_concurrently(lib):
    """A writer thread publishes records word by word while the C drain,
    which runs without the interpreter lock, polls for them."""
    import threading
    import time

    cap, n = 16, 200
    ring = np.zeros(cap, dtype=decode.RECORD_DTYPE)
    drained = []

    def writer():
        for i in range(n):
            while len(drained) + cap <= i:  # never lap the reader
                time.sleep(0)
            for k in (2, 0, 1):
                _put(ring, i % cap, (i * 3, i, 5), i + 1, words=(k,))
                if i % 7 == 0:
                    time.sleep(0.0002)

    t = threading.Thread(target=writer)
    t.start()
    first = 0
    while first < n:
        got = decode.ring_drain(ring.ctypes.data, cap, first, min(4, n - first), max_spins=1 << 30)
        drained.extend(got["token"].tolist())
        first += len(got)
    t.join()
    assert drained == [3 * i for i in range(n)]


def test_commit_rejects_bad_arguments_before_any_cuda_call(lib):
    F = 0x1000  # never dereferenced: every check below fails first
    c = lib.arc_decode_commit
    assert c(None, 2, 10, F, F, 5, None, F, 8, F, None, None) == -1  # tokens NULL
    assert c(F, 0, 10, F, F, 5, None, F, 8, F, None, None) == -2     # B <= 0
    assert c(F, 2, 0, F, F, 5, None, F, 8, F, None, None) == -2      # V <= 0
    assert c(F, 2, 10, F, F, 0, None, F, 8, F, None, None) == -2     # max_position <= 0
    assert c(F, 9, 10, F, F, 5, None, F, 8, F, None, None) == -2     # capacity < B
    assert c(F, 2, 10, F, F, 5, None, None, 8, F, None, None) == -1  # ring NULL
    assert c(F, 2, 10, F, F, 5, None, F, 8, None, None, None) == -1  # head NULL
    assert c(F, 2, 10, F, F, 5, None, F + 4, 8, F, None, None) == -4  # ring not 8-byte aligned
    assert c(F, 2, 10, F, F, 5, None, F, 8, F + 4, None, None) == -4  # head not 8-byte aligned
    assert lib.arc_ring_drain(None, 4, 0, 1, None, 1) == -1


def _commit_call(lib, tgt, B=2, logits=0x1000):
    F = 0x1000
    opts = sampler.make_options()
    t = ctypes.byref(tgt) if tgt is not None else None
    return lib.arc_sample_batch_commit(logits, B, 8, 8, 1, F, None, None, F, None, F, 1 << 20, ctypes.byref(opts),
                                       t, None)


def test_sample_and_commit_rejects_bad_arguments_before_any_cuda_call(lib):
    F = 0x1000
    T = sampler.CommitTarget
    assert _commit_call(lib, None) == -1                                   # no commit target
    assert _commit_call(lib, T(None, F, None, F, F, None, 5, 8)) == -1     # next_ids NULL
    assert _commit_call(lib, T(F, None, None, F, F, None, 5, 8)) == -1     # positions NULL
    assert _commit_call(lib, T(F, F, None, None, F, None, 5, 8)) == -1     # ring NULL
    assert _commit_call(lib, T(F, F, None, F, None, None, 5, 8)) == -1     # head NULL
    assert _commit_call(lib, T(F, F, None, F, F + 4, None, 5, 8)) == -4    # head not 8-byte aligned
    assert _commit_call(lib, T(F, F, None, F + 4, F, None, 5, 8)) == -4    # ring not 8-byte aligned
    assert _commit_call(lib, T(F, F, None, F, F, None, 0, 8)) == -2        # max_position <= 0
    assert _commit_call(lib, T(F, F, None, F, F, None, 5, 1)) == -2        # capacity < B
    assert _commit_call(lib, T(F, F, None, F, F, None, 5, (1 << 30) + 1)) == -2  # capacity too large
    # then the sampler's own checks
    assert _commit_call(lib, T(F, F, None, F, F, None, 5, 8), logits=None) == -1
    assert _commit_call(lib, T(F, F, None, F, F, None, 5, 8), B=0) == -2
    assert "overwritten" in sampler.strerror(decode.ARC_E_RING_OVERRUN)


# ---------------------------------------------------------------- GPU
def _run_oracle(tokens, V, ids, pos, maxp, owners, head, cap, ring_recs, fault):
    # the library's records as the oracle's (token, position, owner, stamp)
    ring = [(int(r["token"]), int(r["position"]), int(r["owner"]), int(r["stamp"])) for r in ring_recs]
    return oc.commit(tokens, V, ids, pos, maxp, owners, head, cap, ring, fault)


@pytest.mark.gpu
def test_commit_after_sampling_matches_the_oracle(cuda_lib):
    import torch
    from device_logits_sampling_gb300 import workloads as wl

    w = wl.NAMED["small_fp32"]()
    logits = sampler.logits_tensor(w)
    prm = sampler.params_tensor(w.params)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    sampler.sample_batch(logits, prm, out)
    ring = decode.Ring(16)
    ids = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    pos = torch.tensor([0, 3, 9, 100], dtype=torch.int32, device="cuda")
    owners = torch.tensor([11, 12, 13, 14], dtype=torch.int32, device="cuda")
    head = torch.tensor([14], dtype=torch.int64, device="cuda")  # the step's records wrap around slot 0
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = ring.records().copy()
    decode.decode_commit(out, ids, pos, 10, w.V, ring, head, owners=owners, fault_word=fault)
    torch.cuda.synchronize()
    tokens = out.cpu().tolist()
    e_ids, e_pos, e_ring, e_head, e_fault = _run_oracle(tokens, w.V, [0] * 4, [0, 3, 9, 100], 10,
                                                        [11, 12, 13, 14], 14, 16, before, 0)
    assert ids.cpu().tolist() == e_ids and pos.cpu().tolist() == e_pos
    assert int(head.item()) == e_head and int(fault.item()) == e_fault == oc.BAD_POSITION
    assert np.array_equal(ring.records(), oc.as_records(e_ring))
    ring.next = 14
    got = ring.drain(4, max_spins=10)
    assert got["token"].tolist()[:3] == tokens[:3] and got["token"][3] == -1
    ring.close()


@pytest.mark.gpu
def test_commit_refuses_out_of_range_rows(cuda_lib):
    import torch

    V, maxp = 1000, 50
    tokens = torch.tensor([0, 999, 1000, -5, 7, 8], dtype=torch.int32, device="cuda")
    pos0 = [0, 49, 1, 2, 50, -1]
    ids = torch.full((6,), 77, dtype=torch.int32, device="cuda")
    pos = torch.tensor(pos0, dtype=torch.int32, device="cuda")
    head = torch.zeros(1, dtype=torch.int64, device="cuda")
    fault = torch.zeros(1, dtype=torch.int32, device="cuda")
    ring = decode.Ring(8)
    decode.decode_commit(tokens, ids, pos, maxp, V, ring, head, fault_word=fault)
    torch.cuda.synchronize()
    e_ids, e_pos, e_ring, e_head, e_fault = oc.commit(tokens.cpu().tolist(), V, [77] * 6, pos0, maxp, None, 0, 8,
                                                      oc.empty_ring(8))
    assert ids.cpu().tolist() == e_ids == [0, 999, 77, 77, 77, 77]
    assert pos.cpu().tolist() == e_pos == [1, 50, 1, 2, 50, -1]
    assert int(fault.item()) == e_fault == oc.BAD_TOKEN | oc.BAD_POSITION
    assert np.array_equal(ring.records(), oc.as_records(e_ring))
    ring.close()


@pytest.mark.gpu
def test_captured_sample_and_commit_replay_drained_from_the_host(cuda_lib):
    """N replays of a graph holding arc_sample_batch (step advanced on device)
    and arc_decode_commit: the host drains N*B records with no CUDA call, they
    equal N eager steps, and an idle stream with fewer records than asked is
    a definite short read."""
    import torch
    from device_logits_sampling_gb300 import workloads as wl

    w = wl.NAMED["mixed_quarters"]()
    B, V, N = 32, w.V, 8
    logits = sampler.logits_tensor(w)[:B]
    params = w.params[:B].copy()

    def fresh():
        prm = sampler.params_tensor(params)
        out = torch.zeros(B, dtype=torch.int32, device="cuda")
        ws = sampler.workspace_tensor(B, V, w.dtype)
        ids = torch.zeros(B, dtype=torch.int32, device="cuda")
        pos = torch.zeros(B, dtype=torch.int32, device="cuda")
        owners = torch.arange(100, 100 + B, dtype=torch.int32, device="cuda")
        head = torch.zeros(1, dtype=torch.int64, device="cuda")
        fault = torch.zeros(1, dtype=torch.int32, device="cuda")
        return prm, out, ws, ids, pos, owners, head, fault

    # eager reference
    prm, out, ws, ids, pos, owners, head, fault = fresh()
    ring_e = decode.Ring(N * B)
    eager = []
    for _ in range(N):
        sampler.sample_batch(logits, prm, out, workspace=ws, autoinc=True)
        decode.decode_commit(out, ids, pos, 1 << 20, V, ring_e, head, owners=owners, fault_word=fault)
        torch.cuda.synchronize()
        eager.append(out.cpu().numpy().copy())
    eager = np.stack(eager)
    assert np.array_equal(ring_e.drain(N * B, max_spins=10)["token"], eager.reshape(-1))

    # captured
    prm, out, ws, ids, pos, owners, head, fault = fresh()
    ring = decode.Ring(4 * N * B)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sampler.sample_batch(logits, prm, out, workspace=ws, stream=s)  # first call sets kernel attributes
        s.synchronize()
        prm.copy_(sampler.params_tensor(params))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            sampler.sample_batch(logits, prm, out, workspace=ws, autoinc=True, stream=s)
            decode.decode_commit(out, ids, pos, 1 << 20, V, ring, head, owners=owners, fault_word=fault, stream=s)
        head.zero_()
        pos.zero_()
        prm.copy_(sampler.params_tensor(params))
        s.synchronize()
        for _ in range(N):
            g.replay()
    got = ring.drain(N * B, max_spins=1 << 26)  # host polls only
    s.synchronize()
    assert len(got) == N * B
    assert np.array_equal(got["token"], eager.reshape(-1))
    assert np.array_equal(got["owner"], np.tile(np.arange(100, 100 + B), N))
    assert np.array_equal(got["position"], np.repeat(np.arange(N), B))
    assert int(fault.item()) == 0 and int(head.item()) == N * B
    # idle but short: every step retired, and no record beyond them will come
    assert decode.stream_idle(s) == 1
    assert len(ring.drain(1, max_spins=1000)) == 0
    ring.close()
    ring_e.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name,B", [("mixed_quarters", 256), ("small_fp32", 4), ("single_row_peaked", 1),
                                    ("adversarial_ties", 8)])
def test_commit_folded_into_the_sampler_matches_sample_then_commit(cuda_lib, name, B):
    """arc_sample_batch_commit over several steps (step advanced on device, some
    rows running out of positions, one row with invalid parameters) leaves the
    same tokens, next ids, positions, ring, head and fault word as
    arc_sample_batch followed by arc_decode_commit, and both match the oracle
    commit of the sampled tokens.  The single-row and small fp32 batches take
    the one-launch cluster path, the others the two-kernel path (the tied
    batch of 8 rows with a cluster of 8 finish CTAs per row, CTA 0 committing)."""
    import torch
    from device_logits_sampling_gb300 import workloads as wl

    w = wl.NAMED[name]()
    B = min(B, w.B)
    V, N, maxp = w.V, 5, 3
    logits = sampler.logits_tensor(w)[:B]
    params = w.params[:B].copy()
    if B > 2:
        params["temperature"][2] = -1.0  # invalid: token -1, refused as BAD_TOKEN
    pos0 = (np.arange(B) % 4).astype(np.int32)  # rows at 3 are refused from the first step on
    owners0 = (1000 + np.arange(B)).astype(np.int32)
    cap = 3 * B + 5

    def run(fused):
        prm = sampler.params_tensor(params)
        out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        ws = sampler.workspace_tensor(B, V, w.dtype)
        ids = torch.full((B,), 5, dtype=torch.int32, device="cuda")
        pos = torch.tensor(pos0, device="cuda")
        owners = torch.tensor(owners0, device="cuda")
        head = torch.tensor([7, 0], dtype=torch.int64, device="cuda")  # records wrap the ring
        fault = torch.zeros(1, dtype=torch.int32, device="cuda")
        ring = decode.Ring(cap)
        toks, states = [], []
        for _ in range(N):
            if fused:
                decode.sample_and_commit(logits, prm, out, ids, pos, maxp, ring, head, owners=owners,
                                         fault_word=fault, workspace=ws, autoinc=True)
            else:
                sampler.sample_batch(logits, prm, out, workspace=ws, autoinc=True)
                decode.decode_commit(out, ids, pos, maxp, V, ring, head[:1], owners=owners, fault_word=fault)
            torch.cuda.synchronize()
            toks.append(out.cpu().numpy().copy())
            states.append((ids.cpu().numpy().copy(), pos.cpu().numpy().copy(), ring.records().copy(),
                           head.cpu().numpy().copy(), int(fault.item())))
        ring.close()
        return toks, states

    t_sep, s_sep = run(False)
    t_fus, s_fus = run(True)
    ring_o = oc.empty_ring(cap)
    ids_o, pos_o, head_o, fault_o = [5] * B, pos0.tolist(), 7, 0
    for step in range(N):
        assert np.array_equal(t_fus[step], t_sep[step])
        ids_o, pos_o, ring_o, head_o, fault_o = oc.commit(t_sep[step].tolist(), V, ids_o, pos_o, maxp,
                                                          owners0.tolist(), head_o, cap, ring_o, fault_o)
        for st in (s_sep[step], s_fus[step]):
            ids, pos, recs, head, fault = st
            assert ids.tolist() == ids_o and pos.tolist() == pos_o
            assert np.array_equal(recs, oc.as_records(ring_o))
            assert int(head[0]) == head_o and fault == fault_o
        assert int(s_fus[step][3][1]) == 0  # the arrival count is back at 0 after every call
    if B > 2:
        assert fault_o == oc.BAD_TOKEN | oc.BAD_POSITION
