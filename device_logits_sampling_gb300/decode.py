"""Binding of arc_decode.h: the decode-loop commit after on-device sampling.

Argument marshalling only: the commit is a kernel of libarcsample.so, the
ring drain its host function.  Record layout (24 bytes, three 8-byte words):
(token, stamp), (position, stamp), (owner, stamp).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import sampler

RECORD_DTYPE = np.dtype([("token", "<i4"), ("stamp", "<u4"), ("position", "<i4"), ("stamp_pos", "<u4"),
                         ("owner", "<u4"), ("stamp_owner", "<u4")])
ARC_COMMIT_BAD_TOKEN = 0x1
ARC_COMMIT_BAD_POSITION = 0x2
ARC_E_RING_OVERRUN = -9


def decode_commit(tokens, next_ids, positions, max_position: int, V: int, ring: "Ring", head,
                  owners=None, fault_word=None, stream=None, check: bool = True) -> int:
    """arc_decode_commit on CUDA tensors: tokens / next_ids / positions int32 [B],
    owners uint32-as-int32 [B] or None, head int64 [1], fault_word int32 [1] or None."""
    B = int(tokens.numel())
    ptr = sampler._ptr
    rc = sampler.load().arc_decode_commit(ptr(tokens), B, int(V), ptr(next_ids), ptr(positions),
                                          int(max_position), ptr(owners), ring.device, ring.capacity,
                                          ptr(head), ptr(fault_word), sampler._stream(stream))
    if check and rc != sampler.ARC_OK:
        raise sampler.ArcError(rc)
    return rc


def sample_and_commit(logits, params, out, next_ids, positions, max_position: int, ring: "Ring", head,
                      owners=None, fault_word=None, hist_offsets=None, hist_ids=None, err_word=None, debug=None,
                      workspace=None, ctas_per_row=0, max_hist_len=0, autoinc=False, stream=None,
                      check: bool = True) -> int:
    """arc_sample_batch_commit: sample_batch's arguments plus the commit's;
    head is int64 [2] (records published; rows committed in the running call,
    0 between calls)."""
    B, V = int(logits.shape[0]), int(logits.shape[1])
    ld = int(logits.stride(0)) if B > 1 else V
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    if workspace is None:
        workspace = sampler.workspace_tensor(B, V, sampler._dtype_code(logits), hist_offsets is not None,
                                             ctas_per_row, max_hist_len, device=logits.device)
    ptr = sampler._ptr
    opts = sampler.make_options(ctas_per_row, max_hist_len, autoinc, debug)
    tgt = sampler.CommitTarget(ptr(next_ids), ptr(positions), ptr(owners), ring.device, ptr(head),
                               ptr(fault_word), int(max_position), ring.capacity)
    rc = sampler.load().arc_sample_batch_commit(ptr(logits), B, V, ld, sampler._dtype_code(logits), ptr(params),
                                                ptr(hist_offsets), ptr(hist_ids), ptr(out), ptr(err_word),
                                                ptr(workspace), int(workspace.numel()), ctypes.byref(opts),
                                                ctypes.byref(tgt), sampler._stream(stream))
    if check and rc != sampler.ARC_OK:
        raise sampler.ArcError(rc)
    return rc


def stream_idle(stream=None) -> int:
    """1 when every piece of work on the stream has retired, 0 while some has
    not, < 0 on a (possibly asynchronous) CUDA error.  Never blocks."""
    return sampler.load().arc_stream_idle(sampler._stream(stream))


def ring_drain(ring_host: int, capacity: int, first: int, count: int, max_spins: int = 1 << 20) -> np.ndarray:
    """Records first .. first + count - 1 of a ring at host address ring_host
    (fewer when one has not landed within max_spins polls).  Raises on overrun."""
    out = np.zeros(count, dtype=RECORD_DTYPE)
    n = sampler.load().arc_ring_drain(ring_host, capacity, first, count,
                                      out.ctypes.data if count else None, max_spins)
    if n < 0:
        raise sampler.ArcError(int(n))
    return out[:n]


class Ring:
    """A pinned, device-mapped host ring of `capacity` records (arc_ring_alloc)."""

    def __init__(self, capacity: int):
        self.capacity = int(capacity)
        h, d = ctypes.c_void_p(), ctypes.c_void_p()
        rc = sampler.load().arc_ring_alloc(self.capacity * RECORD_DTYPE.itemsize, ctypes.byref(h), ctypes.byref(d))
        if rc != sampler.ARC_OK:
            raise sampler.ArcError(rc)
        self.host, self.device = h.value, d.value
        self.next = 0  # the host's read cursor: records drained so far

    def records(self) -> np.ndarray:
        """A numpy view of the ring's host memory (for inspection)."""
        buf = (ctypes.c_uint8 * (self.capacity * RECORD_DTYPE.itemsize)).from_address(self.host)
        return np.frombuffer(buf, dtype=RECORD_DTYPE)

    def drain(self, count: int, max_spins: int = 1 << 20) -> np.ndarray:
        recs = ring_drain(self.host, self.capacity, self.next, count, max_spins)
        self.next += len(recs)
        return recs

    def close(self):
        if self.host:
            sampler.load().arc_ring_free(self.host)
            self.host = self.device = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
