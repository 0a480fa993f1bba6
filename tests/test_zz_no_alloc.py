"""arc_sample_batch_static, the entry point that allocates nothing: it must give
exactly what arc_sample_batch gives with a caller-owned workspace.

Collected last (file name) so that it runs both alone and after every other
GPU test on the same device context."""
import numpy as np
import pytest

from device_logits_sampling_gb300 import sampler, workloads


def test_static_rejects_bad_arguments_before_cuda():
    lib = sampler.load()
    opts = sampler.make_options()
    # NULL logits / out: refused before any CUDA call (works without a GPU)
    rc = lib.arc_sample_batch_static(None, 4, 1024, 1024, 0, None, None, None, None, None, opts, None)
    assert rc == sampler.ARC_E_NULL
    rc = lib.arc_sample_batch_static(16, 0, 1024, 1024, 0, 16, None, None, 16, None, opts, None)
    assert rc == sampler.ARC_E_SHAPE


def _run(S, w, static, ctas_per_row=0):
    import torch

    logits = S.logits_tensor(w)
    prm = S.params_tensor(w.params)
    offs, ids = S.history_tensors(w)
    out = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dbg = S.debug_tensor(w.B)
    if static:
        S.sample_batch_static(logits, prm, out, hist_offsets=offs, hist_ids=ids, err_word=err, debug=dbg,
                              ctas_per_row=ctas_per_row)
    else:
        S.sample_batch(logits, prm, out, hist_offsets=offs, hist_ids=ids, err_word=err, debug=dbg,
                       ctas_per_row=ctas_per_row)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item()), S.debug_records(dbg)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mixed_batch", "small_fp32", "penalized_batch"])
def test_static_matches_workspace_call_two_calls_in_a_row(cuda_lib, name):
    w = getattr(workloads, name)()
    ref_tok, ref_err, ref_dbg = _run(cuda_lib, w, static=False)
    for _ in range(2):
        tok, err, dbg = _run(cuda_lib, w, static=True)
        assert np.array_equal(tok, ref_tok)
        assert err == ref_err
        assert np.array_equal(dbg, ref_dbg)


def _largest_accepted(S, V, dtype):
    """The largest B whose planned workspace fits the library's static array."""
    lo, hi = 1, 1 << 16
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if S.plan(mid, V, dtype).workspace_bytes <= S.ARC_STATIC_WORKSPACE_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_static_limits_are_the_documented_ones():
    # B x slices-per-row x 1,664 B <= 16 MiB: 16 bf16 slices or 32 fp32 slices
    # per row at V = 129,280 (host-only planning, no GPU)
    S = sampler
    S.load()
    assert _largest_accepted(S, 129_280, workloads.DTYPE_BF16) == 630
    assert _largest_accepted(S, 129_280, workloads.DTYPE_F16) == 630
    assert _largest_accepted(S, 129_280, workloads.DTYPE_F32) == 315


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,B_max", [(workloads.DTYPE_BF16, 630), (workloads.DTYPE_F32, 315)])
def test_static_at_its_limit_and_one_past_it(cuda_lib, dtype, B_max):
    """The largest accepted batch matches arc_sample_batch token for token; one
    more row is refused with nothing enqueued."""
    import torch

    S = cuda_lib
    V = 129_280
    w = workloads.random_case(seed=77 + dtype, B=B_max, V=V, dtype=dtype)
    ref_tok, ref_err, _ = _run(S, w, static=False)
    tok, err, _ = _run(S, w, static=True)
    assert np.array_equal(tok, ref_tok) and err == ref_err
    B = B_max + 1
    tdt = torch.bfloat16 if dtype == workloads.DTYPE_BF16 else torch.float32
    logits = torch.zeros((B, V), dtype=tdt, device="cuda")
    prm = S.params_tensor(workloads.make_params(B))
    out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    rc = S.sample_batch_static(logits, prm, out, check=False)
    assert rc == sampler.ARC_E_WORKSPACE
    torch.cuda.synchronize()
    assert int((out != -7).sum().item()) == 0  # nothing was enqueued


@pytest.mark.gpu
def test_static_after_a_different_shape(cuda_lib):
    """Calls of different shapes share the array: each matches arc_sample_batch."""
    S = cuda_lib
    shapes = [(40, 129_280, workloads.DTYPE_BF16), (6, 20_000, workloads.DTYPE_F32),
              (300, 50_000, workloads.DTYPE_BF16)]
    for i, (B, V, dt) in enumerate(shapes):
        w = workloads.random_case(seed=500 + i, B=B, V=V, dtype=dt)
        ref_tok, ref_err, ref_dbg = _run(S, w, static=False)
        tok, err, dbg = _run(S, w, static=True)
        assert np.array_equal(tok, ref_tok) and err == ref_err
        assert np.array_equal(dbg, ref_dbg)
