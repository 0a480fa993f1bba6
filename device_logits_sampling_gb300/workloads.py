"""Seeded synthetic inputs for the on-device sampler and its oracle.

This module only *generates inputs*: logits, per-row parameter records and
token histories.  It holds none of the sampling arithmetic, so both the CUDA
path and the fp64 oracle can consume its output without sharing any of the
method's code.

Workloads follow the shapes of the Arc sampling pages: a V4-class vocabulary
of 129,280 entries (Arc PR #222, "ARC_SAMPLE_ON_DEVICE", section 2: the
[B, 1, vocab] logits copy of 256 x 129,280 x 2 B), bf16 or fp32 logits, and
the mixed sampling parameters a serving engine sends (server defaults
top_k=-1, top_p=1.0, min_p=0.0 from the same page, section 3(b)).

All randomness comes from numpy's PCG64, which gives the same bytes on x86
and Arm hosts.  bf16 logits are produced by round-to-nearest-even from fp32
and are returned as their raw uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

VOCAB_V4 = 129_280

DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_F16 = 2

# Layout of one per-row parameter record, identical to `arc_row_params` in
# include/arc_sample.h (48 bytes, little endian).
ROW_PARAMS_DTYPE = np.dtype(
    [
        ("temperature", "<f4"),
        ("top_k", "<i4"),
        ("top_p", "<f4"),
        ("min_p", "<f4"),
        ("repetition_penalty", "<f4"),
        ("frequency_penalty", "<f4"),
        ("presence_penalty", "<f4"),
        ("flags", "<u4"),
        ("seed", "<u8"),
        ("step", "<u8"),
    ],
    align=True,
)
assert ROW_PARAMS_DTYPE.itemsize == 48


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to IEEE half (numpy's round to nearest, ties to even);
    return uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen IEEE half bit patterns to fp32 values (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def as_f16(w: "Workload") -> "Workload":
    """The same rows as fp16 logits, rounded to nearest (exact for every value
    in fp16's normal range, 2^-14 .. 65,504 in magnitude, with at most 11
    significant bits: bf16 values there included)."""
    import dataclasses

    return dataclasses.replace(w, name=w.name + "_as_f16", dtype=DTYPE_F16, logits=f32_to_f16_bits(w.logits_f32()))


def make_params(B: int) -> np.ndarray:
    """B parameter records with every filter disabled and T = 1."""
    p = np.zeros(B, dtype=ROW_PARAMS_DTYPE)
    p["temperature"] = 1.0
    p["top_k"] = -1
    p["top_p"] = 1.0
    p["min_p"] = 0.0
    p["repetition_penalty"] = 1.0
    return p


@dataclass
class Workload:
    """One batch of sampler inputs.

    logits: [B, V] array.  For dtype == DTYPE_BF16 (DTYPE_F16) it holds uint16
    bf16 (IEEE half) bit patterns, for DTYPE_F32 float32 values.
    hist_offsets / hist_ids: CSR token history (None when no row has one).
    """

    name: str
    dtype: int
    logits: np.ndarray
    params: np.ndarray
    hist_offsets: np.ndarray | None = None
    hist_ids: np.ndarray | None = None
    notes: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.logits.shape[0])

    @property
    def V(self) -> int:
        return int(self.logits.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == DTYPE_F32 else 2

    def logits_f32(self) -> np.ndarray:
        """The logits as fp32 values (exact widening for bf16)."""
        if self.dtype == DTYPE_BF16:
            return bf16_bits_to_f32(self.logits)
        if self.dtype == DTYPE_F16:
            return f16_bits_to_f32(self.logits)
        return np.asarray(self.logits, dtype=np.float32)

    def history(self, row: int) -> np.ndarray:
        if self.hist_offsets is None:
            return np.zeros(0, dtype=np.int32)
        a, b = int(self.hist_offsets[row]), int(self.hist_offsets[row + 1])
        return self.hist_ids[a:b]


def _spiked_rows(rng: np.random.Generator, B: int, V: int, sigma: float,
                 n_spikes: int, lo: float, hi: float) -> np.ndarray:
    """N(0, sigma^2) logits with `n_spikes` distinct indices per row raised by U(lo, hi)."""
    x = rng.standard_normal((B, V), dtype=np.float64) * sigma
    for r in range(B):
        idx = rng.choice(V, size=n_spikes, replace=False)
        x[r, idx] += rng.uniform(lo, hi, size=n_spikes)
    return x.astype(np.float32)


# Parameter quarters of the mixed batch: row % 4 selects the row type.
MIXED_QUARTERS = (
    dict(temperature=0.0),                                  # greedy
    dict(temperature=1.0),                                  # server defaults
    dict(temperature=0.7, top_k=50),                        # top-k
    dict(temperature=0.8, top_p=0.9, min_p=0.05),           # top-p + min-p
)


def small_fp32(seed: int = 1, B: int = 4, V: int = 1024) -> Workload:
    """B=4, V=1024 fp32 logits iid N(0, 2^2): greedy, defaults, top-k 8, top-p/min-p rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = (rng.standard_normal((B, V), dtype=np.float64) * 2.0).astype(np.float32)
    p = make_params(B)
    kinds = (
        dict(temperature=0.0),
        dict(temperature=1.0),
        dict(temperature=0.7, top_k=8),
        dict(temperature=1.0, top_p=0.9, min_p=0.05),
    )
    for r in range(B):
        for k, v in kinds[r % 4].items():
            p[r][k] = v
        p[r]["seed"] = r
        p[r]["step"] = 0
    return Workload("small_fp32_B4_V1024", DTYPE_F32, logits, p)


def single_row_peaked(seed: int = 2, V: int = VOCAB_V4, greedy: bool = False) -> Workload:
    """B=1 bf16 row N(0, 3^2) with 20 distinct indices raised by +10 (peaked, LM-like).

    The decode loop drives `step` from 0 upwards with the logits fixed;
    `greedy` selects T=0, otherwise the server defaults (T=1, no filters).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((1, V), dtype=np.float64) * 3.0
    idx = rng.choice(V, size=20, replace=False)
    x[0, idx] += 10.0
    logits = f32_to_bf16_bits(x.astype(np.float32))
    p = make_params(1)
    p[0]["temperature"] = 0.0 if greedy else 1.0
    p[0]["seed"] = 0
    p[0]["step"] = 0
    return Workload("single_row_peaked_B1_V129280_bf16" + ("_greedy" if greedy else "_defaults"),
                    DTYPE_BF16, logits, p, notes=dict(spikes=idx))


def mixed_batch(seed: int = 3, B: int = 256, V: int = VOCAB_V4) -> Workload:
    """B=256 bf16 rows N(0, 3^2) + 20 spikes of U(6, 12) per row; parameters cycle by row % 4."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = f32_to_bf16_bits(_spiked_rows(rng, B, V, 3.0, 20, 6.0, 12.0))
    p = make_params(B)
    for r in range(B):
        for k, v in MIXED_QUARTERS[r % 4].items():
            p[r][k] = v
        p[r]["seed"] = r
        p[r]["step"] = 0
    return Workload(f"mixed_quarters_B{B}_V{V}_bf16", DTYPE_BF16, logits, p)


def penalized_batch(seed: int = 4, B: int = 512, V: int = VOCAB_V4, hist_len: int = 256) -> Workload:
    """B=512 spiked bf16 rows, each with a 256-token uniform history (duplicates allowed).

    repetition 1.1, frequency 0.3, presence 0.2; top_k=1000, top_p=0.95, T=0.9.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = f32_to_bf16_bits(_spiked_rows(rng, B, V, 3.0, 20, 6.0, 12.0))
    ids = rng.integers(0, V, size=(B, hist_len), dtype=np.int64).astype(np.int32)
    offsets = (np.arange(B + 1, dtype=np.int64) * hist_len).astype(np.int32)
    p = make_params(B)
    p["temperature"] = 0.9
    p["top_k"] = 1000
    p["top_p"] = 0.95
    p["repetition_penalty"] = 1.1
    p["frequency_penalty"] = 0.3
    p["presence_penalty"] = 0.2
    p["seed"] = np.arange(B, dtype=np.uint64)
    p["step"] = 0
    return Workload(f"penalized_B{B}_V{V}_bf16_hist{hist_len}", DTYPE_BF16, logits, p,
                    hist_offsets=offsets, hist_ids=ids.reshape(-1))


LEVELS16 = np.arange(-7.5, 8.0, 1.0, dtype=np.float32)  # {-7.5, -6.5, ..., 7.5}


def adversarial_ties(seed: int = 5, B: int = 64, V: int = VOCAB_V4) -> Workload:
    """B=64 fp32 rows quantised to 16 levels (massive ties); row 0 all equal, row 1 one-hot.

    top_k=V, top_p=0.999, min_p=1e-4, T=1, seed = row.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((B, V), dtype=np.float64) * 3.0
    q = np.clip(np.floor(x) + 0.5, -7.5, 7.5).astype(np.float32)
    q[0, :] = 0.0
    hot = int(rng.integers(0, V))
    q[1, :] = -1e4
    q[1, hot] = 0.0
    p = make_params(B)
    p["temperature"] = 1.0
    p["top_k"] = V
    p["top_p"] = 0.999
    p["min_p"] = 1e-4
    p["seed"] = np.arange(B, dtype=np.uint64)
    p["step"] = 0
    return Workload(f"adversarial_ties_B{B}_V{V}_fp32", DTYPE_F32, q, p, notes=dict(hot=hot))


def random_case(seed: int, B: int, V: int, dtype: int, *, ties: bool = False,
                hist_len: int = 0, param_mix: str = "all") -> Workload:
    """Generic seeded case for parity sweeps: ragged V, mixed parameters, optional history."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((B, V), dtype=np.float64) * rng.uniform(0.5, 4.0)
    if ties:
        x = np.round(x * 2.0) / 2.0
    x = x.astype(np.float32)
    logits = f32_to_bf16_bits(x) if dtype == DTYPE_BF16 else (f32_to_f16_bits(x) if dtype == DTYPE_F16 else x)
    p = make_params(B)
    for r in range(B):
        kind = r % 6 if param_mix == "all" else int(param_mix)
        if kind == 0:
            p[r]["temperature"] = 0.0
        elif kind == 1:
            p[r]["temperature"] = float(rng.uniform(0.3, 1.5))
        elif kind == 2:
            p[r]["temperature"] = float(rng.uniform(0.3, 1.5))
            p[r]["top_k"] = int(rng.integers(2, max(3, V)))
        elif kind == 3:
            p[r]["temperature"] = float(rng.uniform(0.3, 1.5))
            p[r]["top_p"] = float(rng.uniform(0.05, 0.99))
        elif kind == 4:
            p[r]["temperature"] = float(rng.uniform(0.3, 1.5))
            p[r]["min_p"] = float(rng.uniform(0.001, 0.5))
        else:
            p[r]["temperature"] = float(rng.uniform(0.3, 1.5))
            p[r]["top_k"] = int(rng.integers(2, max(3, V)))
            p[r]["top_p"] = float(rng.uniform(0.05, 0.99))
            p[r]["min_p"] = float(rng.uniform(0.0, 0.2))
        p[r]["seed"] = int(rng.integers(0, 2**63))
        p[r]["step"] = int(rng.integers(0, 2**20))
    offs = ids = None
    if hist_len > 0:
        lens = rng.integers(0, hist_len + 1, size=B)
        offs = np.zeros(B + 1, dtype=np.int32)
        offs[1:] = np.cumsum(lens)
        ids = rng.integers(0, V, size=int(offs[-1]), dtype=np.int64).astype(np.int32)
        p["repetition_penalty"] = rng.uniform(0.8, 1.5, size=B).astype(np.float32)
        p["frequency_penalty"] = rng.uniform(-0.5, 0.5, size=B).astype(np.float32)
        p["presence_penalty"] = rng.uniform(-0.5, 0.5, size=B).astype(np.float32)
    return Workload(f"random_s{seed}_B{B}_V{V}_{'bf16' if dtype else 'f32'}", dtype, logits, p,
                    hist_offsets=offs, hist_ids=ids)


# The five named workloads, smallest first.
NAMED = {
    "small_fp32": small_fp32,
    "single_row_peaked": single_row_peaked,
    "mixed_quarters": mixed_batch,
    "penalized": penalized_batch,
    "adversarial_ties": adversarial_ties,
}
