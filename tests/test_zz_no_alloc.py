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


@pytest.mark.gpu
def test_static_refuses_a_shape_beyond_its_scratch(cuda_lib):
    import torch

    S = cuda_lib
    B, V = 1024, 129_280  # 1024 rows x 16 slices x 656 B > ARC_STATIC_WORKSPACE_BYTES
    assert S.plan(B, V, workloads.DTYPE_BF16).workspace_bytes > S.ARC_STATIC_WORKSPACE_BYTES
    logits = torch.zeros((B, V), dtype=torch.bfloat16, device="cuda")
    prm = S.params_tensor(workloads.make_params(B))
    out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    rc = S.sample_batch_static(logits, prm, out, check=False)
    assert rc == sampler.ARC_E_WORKSPACE
    torch.cuda.synchronize()
    assert int((out != -7).sum().item()) == 0  # nothing was enqueued
