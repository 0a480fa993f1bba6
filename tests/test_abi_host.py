"""Host-side checks of the C ABI: the library loads, exports what the header
declares, and rejects bad arguments before touching CUDA (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from conftest import ROOT
from device_logits_sampling_gb300 import sampler, workloads

HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sampler.LIB_PATH):
        from device_logits_sampling_gb300 import build

        build.build()
    return sampler.load()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"^\s*(?:int|int64_t|size_t|const char\s*\*)\s*(arc_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(["arc_sample_batch", "arc_sample_batch_static", "arc_sample_batch_commit",
                            "arc_sample_greedy",
                            "arc_sample_plan", "arc_sample_workspace_bytes", "arc_sample_strerror",
                            "arc_sample_abi_version",
                            "arc_decode_commit", "arc_ring_drain", "arc_stream_idle", "arc_ring_alloc",
                            "arc_ring_free"]), names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sampler.LIB_PATH], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (arc_\w+)", out.stdout))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else with the public prefix leaks out
    assert exported == set(declared_functions())


def test_abi_version_and_strerror(lib):
    assert lib.arc_sample_abi_version() == 3
    assert sampler.strerror(0) == "ok"
    for rc in range(-1, -9, -1):
        assert len(sampler.strerror(rc)) > 10 and "unknown" not in sampler.strerror(rc)
    assert "unknown" in sampler.strerror(-99)


def test_struct_layouts_match_header():
    assert workloads.ROW_PARAMS_DTYPE.itemsize == 48
    assert sampler.ROW_DEBUG_DTYPE.itemsize == 72
    assert ctypes.sizeof(sampler.Options) == 32
    assert sampler.TOP_LOGPROB_DTYPE.itemsize == 8
    assert ctypes.sizeof(sampler.Geometry) == 48
    assert ctypes.sizeof(sampler.CommitTarget) == 56
    # field offsets of arc_row_params as laid out in the header
    off = {n: workloads.ROW_PARAMS_DTYPE.fields[n][1] for n in workloads.ROW_PARAMS_DTYPE.names}
    assert off["temperature"] == 0 and off["top_k"] == 4 and off["flags"] == 28
    assert off["seed"] == 32 and off["step"] == 40


FAKE = 0x1000  # a non-NULL, aligned pointer that is never dereferenced


def call_batch(lib, logits=FAKE, B=2, V=8, ld=8, dtype=1, params=FAKE, hoff=None, hids=None, out=FAKE,
               opts=None, ws=FAKE, ws_bytes=1 << 20):
    o = ctypes.byref(opts) if opts is not None else None
    return lib.arc_sample_batch(logits, B, V, ld, dtype, params, hoff, hids, out, None, ws, ws_bytes, o, None)


def test_bad_arguments_fail_before_any_cuda_call(lib):
    assert call_batch(lib, logits=None) == sampler.ARC_E_NULL
    assert call_batch(lib, out=None) == sampler.ARC_E_NULL
    assert call_batch(lib, params=None) == sampler.ARC_E_NULL
    assert call_batch(lib, hoff=FAKE, hids=None) == sampler.ARC_E_NULL
    assert call_batch(lib, B=0) == sampler.ARC_E_SHAPE
    assert call_batch(lib, B=-3) == sampler.ARC_E_SHAPE
    assert call_batch(lib, V=0) == sampler.ARC_E_SHAPE
    assert call_batch(lib, V=2**31) == sampler.ARC_E_SHAPE
    assert call_batch(lib, ld=7) == sampler.ARC_E_SHAPE
    assert call_batch(lib, dtype=3) == sampler.ARC_E_DTYPE
    assert call_batch(lib, dtype=-1) == sampler.ARC_E_DTYPE
    assert call_batch(lib, logits=FAKE + 1) == sampler.ARC_E_ALIGN
    assert call_batch(lib, logits=FAKE + 2, dtype=0) == sampler.ARC_E_ALIGN
    assert call_batch(lib, logits=FAKE + 1, dtype=2) == sampler.ARC_E_ALIGN  # fp16: 2-byte elements
    assert call_batch(lib, params=FAKE + 4) == sampler.ARC_E_ALIGN
    assert call_batch(lib, opts=sampler.Options(0, 129, 0, 0, None)) == sampler.ARC_E_OPTION
    assert call_batch(lib, opts=sampler.Options(0, -1, 0, 0, None)) == sampler.ARC_E_OPTION
    assert call_batch(lib, ws=None) == sampler.ARC_E_WORKSPACE
    assert call_batch(lib, ws=FAKE + 8) == sampler.ARC_E_ALIGN
    assert call_batch(lib, opts=sampler.Options(0x80, 0, 0, 0, None)) == sampler.ARC_E_OPTION
    assert call_batch(lib, opts=sampler.Options(0x4, 0, 0, 0, None)) == sampler.ARC_E_OPTION
    # both defined flags together are a valid option set (checked without CUDA by the plan)
    both = sampler.Options(sampler.ARC_OPT_STEP_AUTOINC | sampler.ARC_OPT_FORCE_BISECTION, 0, 0, 0, None)
    geom = sampler.Geometry()
    assert lib.arc_sample_plan(2, 1000, 1, 0, ctypes.byref(both), ctypes.byref(geom)) == sampler.ARC_OK
    assert lib.arc_sample_workspace_bytes(2, 1000, 1, 0, ctypes.byref(both)) > 0
    assert call_batch(lib, opts=sampler.Options(0, 0, -1, 0, None)) == sampler.ARC_E_OPTION
    # top-n log-probabilities: 1..64 ids, and an output pointer with them
    assert call_batch(lib, opts=sampler.Options(0, 0, 0, 5, None, None)) == sampler.ARC_E_OPTION
    assert call_batch(lib, opts=sampler.Options(0, 0, 0, -1, None, FAKE)) == sampler.ARC_E_OPTION
    assert call_batch(lib, opts=sampler.Options(0, 0, 0, 65, None, FAKE)) == sampler.ARC_E_OPTION
    assert sampler.ARC_MAX_TOP_N == 64 and sampler.TOP_LOGPROB_DTYPE.itemsize == 8
    assert lib.arc_sample_abi_version() == 3
    g = lib.arc_sample_greedy
    assert g(None, 2, 8, 8, 1, FAKE, None, None) == sampler.ARC_E_NULL
    assert g(FAKE, 2, 8, 4, 1, FAKE, None, None) == sampler.ARC_E_SHAPE
    assert g(FAKE, 2, 8, 8, 7, FAKE, None, None) == sampler.ARC_E_DTYPE


def test_plan_geometry(lib):
    # the mixed B=256 bf16 batch: 16 slices per row of 8,080 logits (16,160 B) each
    g = sampler.plan(256, workloads.VOCAB_V4, workloads.DTYPE_BF16)
    assert (g.ctas_per_row, g.slice_elems, g.grid_ctas, g.threads) == (16, 8080, 4096, 256)
    assert g.frac_bits == 62 - 17
    assert g.launches == 2 and g.workspace_bytes == 256 * 16 * 1664
    # a single row: one launch, a cluster of 16 CTAs sharing the row (their
    # summaries combined in distributed shared memory, no workspace)
    g1 = sampler.plan(1, workloads.VOCAB_V4, workloads.DTYPE_BF16)
    assert (g1.launches, g1.ctas_per_row, g1.grid_ctas, g1.workspace_bytes) == (1, 16, 16, 0)
    # up to 8 such rows take the cluster kernel; more take two launches with
    # the fewest slices a row allows (16 for bf16 at V = 129,280)
    assert sampler.plan(8, workloads.VOCAB_V4, workloads.DTYPE_BF16).launches == 1
    g9 = sampler.plan(9, workloads.VOCAB_V4, workloads.DTYPE_BF16)
    assert g9.launches == 2 and g9.ctas_per_row == 16
    g20 = sampler.plan(20, workloads.VOCAB_V4, workloads.DTYPE_BF16)
    assert g20.launches == 2 and g20.ctas_per_row == 16
    # small vocabularies too take the fewest slices (one here)
    assert sampler.plan(64, 20_000, workloads.DTYPE_BF16).ctas_per_row == 3
    # an explicit slice count always takes the two kernels
    assert sampler.plan(1, workloads.VOCAB_V4, workloads.DTYPE_BF16, ctas_per_row=32).launches == 2
    # fp32 rows of 129,280 need 32 slices: more than a cluster holds
    assert sampler.plan(1, workloads.VOCAB_V4, workloads.DTYPE_F32).launches == 2
    # fp16 rows slice like bf16 rows (8 logits per 16-byte vector)
    g16 = sampler.plan(256, workloads.VOCAB_V4, workloads.DTYPE_F16)
    assert (g16.ctas_per_row, g16.slice_elems, g16.grid_ctas) == (16, 8080, 4096)
    # fp32 slices hold half as many logits
    assert sampler.plan(64, workloads.VOCAB_V4, workloads.DTYPE_F32).ctas_per_row == 32
    # finish CTAs per row: one while the batch fills the SMs (two finish CTAs
    # per SM), else a cluster of up to 8 while each keeps >= 2,048 vectors
    assert g.finish_ctas == 1 and g1.finish_ctas == 1
    assert sampler.plan(64, workloads.VOCAB_V4, workloads.DTYPE_F32).finish_ctas == 4
    assert sampler.plan(152, workloads.VOCAB_V4, workloads.DTYPE_F32).finish_ctas == 2
    assert sampler.plan(153, workloads.VOCAB_V4, workloads.DTYPE_F32).finish_ctas == 1
    assert sampler.plan(20, workloads.VOCAB_V4, workloads.DTYPE_BF16).finish_ctas == 4
    assert sampler.plan(1, workloads.VOCAB_V4, workloads.DTYPE_F32).finish_ctas == 8
    assert sampler.plan(2, 5_000, workloads.DTYPE_F32, ctas_per_row=4).finish_ctas == 1
    assert sampler.plan(2, 20_000, workloads.DTYPE_F32, ctas_per_row=8).finish_ctas == 2
    # small vocabularies stay on one CTA (which scans and finishes its row)
    g4 = sampler.plan(4, 1024, workloads.DTYPE_F32)
    assert (g4.ctas_per_row, g4.launches) == (1, 1)
    # a forced geometry too small for the row is refused
    with pytest.raises(sampler.ArcError) as e:
        sampler.plan(1, workloads.VOCAB_V4, workloads.DTYPE_BF16, ctas_per_row=1)
    assert e.value.rc == sampler.ARC_E_UNSUPPORTED
    # history support reserves bitmap + patch space
    g2 = sampler.plan(512, workloads.VOCAB_V4, workloads.DTYPE_BF16, has_history=True, max_hist_len=256)
    assert g2.smem_bytes > g.smem_bytes
    # every slice covers the row with no empty CTA: (s-1)*L < V <= s*L
    for B, V, dt in [(3, 1, 1), (7, 9, 0), (1, 12345, 1), (33, 4097, 0), (2, 200_000, 1), (5, 1_000_000, 1)]:
        gg = sampler.plan(B, V, dt)
        assert (gg.ctas_per_row - 1) * gg.slice_elems < V <= gg.ctas_per_row * gg.slice_elems
        assert gg.slice_elems % (8 if dt == 1 else 4) == 0
        assert gg.slice_elems <= 4 * 256 * (8 if dt == 1 else 4)
    # the workspace covers every automatic geometry
    for B, V, dt in [(256, workloads.VOCAB_V4, 1), (1, workloads.VOCAB_V4, 1), (64, workloads.VOCAB_V4, 0)]:
        ws = sampler.workspace_bytes(B, V, dt)
        assert ws >= sampler.plan(B, V, dt).workspace_bytes and ws > 0
        # and the two-kernel geometry the library falls back to when a device
        # cannot schedule the cluster
        assert ws >= sampler.plan(B, V, dt, ctas_per_row=sampler.plan(B, V, dt).ctas_per_row).workspace_bytes
    assert sampler.workspace_bytes(0, 10, 1) == 0


def test_workload_generators_are_deterministic():
    a = workloads.mixed_batch(B=8, V=1000)
    b = workloads.mixed_batch(B=8, V=1000)
    assert a.logits.tobytes() == b.logits.tobytes()
    assert a.params.tobytes() == b.params.tobytes()
    # bf16 rounding is round-to-nearest-even
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], dtype=np.float32)
    bits = workloads.f32_to_bf16_bits(x)
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F62]
    assert np.array_equal(workloads.bf16_bits_to_f32(bits)[:4], np.array([1.0, 1.0, 1.015625, -2.5], np.float32))
