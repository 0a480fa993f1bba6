"""fp64 CPU oracle for on-device logits sampling.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
cpu_baseline / --impl reference legs of bench.py, never by the product path.
"""
from .sampler import (  # noqa: F401
    ERR_DEGENERATE, ERR_HIST_ID, ERR_NAN, ERR_PARAM,
    MODE_FILTERED, MODE_GREEDY, MODE_INERT, MODE_INVALID,
    RowResult, apply_penalties, draw_bits, draw_many, inverse_cdf, params_valid,
    row_mode, sample_batch, sample_row, sample_row_u, splitmix64, top_k_mask,
    top_logprobs, top_p_cutoff, uniform,
)
from . import decode_commit  # noqa: F401,E402
