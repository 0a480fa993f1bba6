"""Python binding of libarcsample.so (include/arc_sample.h): argument marshalling only.

Every step of sampling runs in the library's CUDA kernels.  Tensors are
PyTorch CUDA tensors used purely as device memory; the library never sees a
torch type, only raw pointers, sizes and the current CUDA stream.  There is
no fallback: if the library is not built, `load()` raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .workloads import DTYPE_BF16, DTYPE_F16, DTYPE_F32, ROW_PARAMS_DTYPE

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libarcsample.so")

ARC_OK = 0
ARC_E_NULL = -1
ARC_E_SHAPE = -2
ARC_E_DTYPE = -3
ARC_E_ALIGN = -4
ARC_E_UNSUPPORTED = -5
ARC_E_OPTION = -6
ARC_E_CUDA = -7
ARC_E_WORKSPACE = -8

ARC_ERR_PARAM = 0x1
ARC_ERR_HIST_ID = 0x2
ARC_ERR_NAN = 0x4
ARC_ERR_DEGENERATE = 0x8
ARC_ERR_HIST_CAP = 0x10
ARC_ERR_TIMEOUT = 0x20
ARC_ERR_INTERNAL = 0x40

ARC_OPT_STEP_AUTOINC = 0x1
ARC_OPT_FORCE_BISECTION = 0x2
ARC_STATIC_WORKSPACE_BYTES = 16 << 20  # scratch compiled into the library (arc_sample_batch_static)

# arc_row_debug, 72 bytes
ROW_DEBUG_DTYPE = np.dtype(
    [
        ("mode", "<i4"), ("err", "<u4"), ("token", "<i4"), ("passes", "<i4"),
        ("kappa_k", "<u4"), ("iota_k", "<i4"), ("kappa_r", "<u4"), ("iota_r", "<i4"),
        ("max_z", "<f4"), ("frac_bits", "<i4"),
        ("rbits", "<u8"), ("mass_k", "<u8"), ("mass_r", "<u8"), ("target", "<u8"),
    ],
    align=True,
)
assert ROW_DEBUG_DTYPE.itemsize == 72


class Options(ctypes.Structure):
    _fields_ = [
        ("flags", ctypes.c_uint32),
        ("ctas_per_row", ctypes.c_int32),
        ("max_hist_len", ctypes.c_int32),
        ("top_n", ctypes.c_int32),
        ("debug", ctypes.c_void_p),
        ("top_logprobs", ctypes.c_void_p),
    ]


# arc_top_logprob, 8 bytes
TOP_LOGPROB_DTYPE = np.dtype([("id", "<i4"), ("logprob", "<f4")])
ARC_MAX_TOP_N = 64


class Geometry(ctypes.Structure):
    _fields_ = [
        ("ctas_per_row", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("slice_elems", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("grid_ctas", ctypes.c_int64),
        ("frac_bits", ctypes.c_int32),
        ("launches", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("finish_ctas", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class CommitTarget(ctypes.Structure):
    """arc_commit_target (arc_decode.h), 56 bytes."""
    _fields_ = [
        ("next_ids", ctypes.c_void_p),
        ("positions", ctypes.c_void_p),
        ("owners", ctypes.c_void_p),
        ("ring", ctypes.c_void_p),
        ("head", ctypes.c_void_p),
        ("fault_word", ctypes.c_void_p),
        ("max_position", ctypes.c_int32),
        ("capacity", ctypes.c_uint32),
    ]


_lib = None

# exported symbol -> (restype, argtypes)
SIGNATURES = {
    "arc_sample_batch": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(Options), ctypes.c_void_p]),
    "arc_sample_batch_static": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.POINTER(Options), ctypes.c_void_p]),
    "arc_sample_workspace_bytes": (ctypes.c_size_t, [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(Options)]),
    "arc_sample_greedy": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "arc_sample_plan": (ctypes.c_int, [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.POINTER(Options), ctypes.POINTER(Geometry)]),
    "arc_sample_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "arc_sample_abi_version": (ctypes.c_int, []),
    # arc_decode.h
    "arc_decode_commit": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "arc_sample_batch_commit": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(Options), ctypes.POINTER(CommitTarget),
        ctypes.c_void_p]),
    "arc_ring_drain": (ctypes.c_int64, [
        ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint64]),
    "arc_stream_idle": (ctypes.c_int, [ctypes.c_void_p]),
    "arc_ring_alloc": (ctypes.c_int, [ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p),
                                      ctypes.POINTER(ctypes.c_void_p)]),
    "arc_ring_free": (ctypes.c_int, [ctypes.c_void_p]),
}


def load(path: str | None = None):
    """Load libarcsample.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the sampler has no CPU fallback)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def strerror(rc: int) -> str:
    return load().arc_sample_strerror(rc).decode()


class ArcError(RuntimeError):
    def __init__(self, rc: int):
        super().__init__(f"arc_sample error {rc}: {strerror(rc)}")
        self.rc = rc


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.float16:
        return DTYPE_F16
    raise TypeError(f"logits must be bfloat16, float16 or float32, not {t.dtype}")


def _stream(stream) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def params_tensor(params: np.ndarray, device="cuda"):
    """Device copy of an arc_row_params array (uint8 tensor, 48 bytes per row)."""
    import torch

    arr = np.ascontiguousarray(params, dtype=ROW_PARAMS_DTYPE)
    return torch.from_numpy(arr.view(np.uint8).copy()).to(device)


def debug_tensor(B: int, device="cuda"):
    import torch

    return torch.zeros(B * ROW_DEBUG_DTYPE.itemsize, dtype=torch.uint8, device=device)


def debug_records(t) -> np.ndarray:
    """Host view of a debug tensor as arc_row_debug records."""
    return t.cpu().numpy().view(ROW_DEBUG_DTYPE)


def make_options(ctas_per_row=0, max_hist_len=0, autoinc=False, debug=None, force_bisection=False,
                 top_n=0, top_logprobs=None) -> Options:
    flags = (ARC_OPT_STEP_AUTOINC if autoinc else 0) | (ARC_OPT_FORCE_BISECTION if force_bisection else 0)
    return Options(flags, int(ctas_per_row), int(max_hist_len), int(top_n), _ptr(debug), _ptr(top_logprobs))


def top_logprobs_tensor(B: int, n: int, device="cuda"):
    """Device output for top_n log-probabilities: arc_top_logprob [B][n] as bytes."""
    import torch

    return torch.zeros(B * n * TOP_LOGPROB_DTYPE.itemsize, dtype=torch.uint8, device=device)


def top_logprobs_records(t, n: int) -> np.ndarray:
    """Host view [B, n] of a top-n log-probability tensor (fields id, logprob)."""
    return t.cpu().numpy().view(TOP_LOGPROB_DTYPE).reshape(-1, n)


def workspace_bytes(B: int, V: int, dtype: int, has_history=False, ctas_per_row=0, max_hist_len=0) -> int:
    opts = make_options(ctas_per_row, max_hist_len)
    return int(load().arc_sample_workspace_bytes(int(B), int(V), int(dtype), int(bool(has_history)),
                                                 ctypes.byref(opts)))


def workspace_tensor(B: int, V: int, dtype: int, has_history=False, ctas_per_row=0, max_hist_len=0,
                     device="cuda"):
    """A zero-filled device workspace for arc_sample_batch (uint8 tensor)."""
    import torch

    n = workspace_bytes(B, V, dtype, has_history, ctas_per_row, max_hist_len)
    if n == 0:
        raise ValueError("arc_sample_workspace_bytes rejected the shape or options")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sample_batch(logits, params, out, hist_offsets=None, hist_ids=None, err_word=None, debug=None,
                 workspace=None, ctas_per_row=0, max_hist_len=0, autoinc=False, stream=None,
                 check=True, force_bisection=False, top_n=0, top_logprobs=None) -> int:
    """arc_sample_batch on CUDA tensors: logits [B, V] (row stride >= V), params uint8
    [B*48], out int32 [B], optional CSR history (int32), err_word uint32 [1], debug uint8
    [B*72], workspace uint8 (zero-filled once; allocated here when None)."""
    B, V = int(logits.shape[0]), int(logits.shape[1])
    ld = int(logits.stride(0)) if B > 1 else V
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    if workspace is None:
        workspace = workspace_tensor(B, V, _dtype_code(logits), hist_offsets is not None, ctas_per_row,
                                     max_hist_len, device=logits.device)
    opts = make_options(ctas_per_row, max_hist_len, autoinc, debug, force_bisection, top_n, top_logprobs)
    rc = load().arc_sample_batch(_ptr(logits), B, V, ld, _dtype_code(logits), _ptr(params),
                                 _ptr(hist_offsets), _ptr(hist_ids), _ptr(out), _ptr(err_word),
                                 _ptr(workspace), int(workspace.numel()), ctypes.byref(opts),
                                 _stream(stream))
    if check and rc != ARC_OK:
        raise ArcError(rc)
    return rc


def sample_batch_static(logits, params, out, hist_offsets=None, hist_ids=None, err_word=None, debug=None,
                        ctas_per_row=0, max_hist_len=0, autoinc=False, stream=None, check=True,
                        top_n=0, top_logprobs=None) -> int:
    """arc_sample_batch_static: as sample_batch, with the library's own scratch
    array instead of a workspace (nothing is allocated for the call)."""
    B, V = int(logits.shape[0]), int(logits.shape[1])
    ld = int(logits.stride(0)) if B > 1 else V
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    opts = make_options(ctas_per_row, max_hist_len, autoinc, debug, top_n=top_n, top_logprobs=top_logprobs)
    rc = load().arc_sample_batch_static(_ptr(logits), B, V, ld, _dtype_code(logits), _ptr(params),
                                        _ptr(hist_offsets), _ptr(hist_ids), _ptr(out), _ptr(err_word),
                                        ctypes.byref(opts), _stream(stream))
    if check and rc != ARC_OK:
        raise ArcError(rc)
    return rc


def sample_greedy(logits, out, err_word=None, stream=None, check=True) -> int:
    B, V = int(logits.shape[0]), int(logits.shape[1])
    ld = int(logits.stride(0)) if B > 1 else V
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    rc = load().arc_sample_greedy(_ptr(logits), B, V, ld, _dtype_code(logits), _ptr(out),
                                  _ptr(err_word), _stream(stream))
    if check and rc != ARC_OK:
        raise ArcError(rc)
    return rc


def plan(B: int, V: int, dtype: int, has_history=False, ctas_per_row=0, max_hist_len=0) -> Geometry:
    g = Geometry()
    opts = make_options(ctas_per_row, max_hist_len)
    rc = load().arc_sample_plan(int(B), int(V), int(dtype), int(bool(has_history)), ctypes.byref(opts),
                                ctypes.byref(g))
    if rc != ARC_OK:
        raise ArcError(rc)
    return g


def logits_tensor(wl, device="cuda", ld: int | None = None):
    """Device tensor of a Workload's logits (bf16 from bit patterns), optional padded row stride."""
    import torch

    if wl.dtype == DTYPE_BF16:
        host = torch.from_numpy(np.ascontiguousarray(wl.logits).view(np.int16)).view(torch.bfloat16)
    elif wl.dtype == DTYPE_F16:
        host = torch.from_numpy(np.ascontiguousarray(wl.logits).view(np.int16)).view(torch.float16)
    else:
        host = torch.from_numpy(np.ascontiguousarray(wl.logits, dtype=np.float32))
    if ld is None or ld == wl.V:
        return host.to(device)
    full = torch.zeros((wl.B, ld), dtype=host.dtype)
    full[:, : wl.V] = host
    return full.to(device)[:, : wl.V]


def history_tensors(wl, device="cuda"):
    import torch

    if wl.hist_offsets is None:
        return None, None
    offs = torch.from_numpy(np.ascontiguousarray(wl.hist_offsets, dtype=np.int32)).to(device)
    ids_np = np.ascontiguousarray(wl.hist_ids, dtype=np.int32)
    if ids_np.size == 0:
        ids_np = np.zeros(1, dtype=np.int32)
    ids = torch.from_numpy(ids_np).to(device)
    return offs, ids
