"""Chunked gated delta rule (GDN) on NVIDIA GB300: a C-ABI CUDA library (libgdn.so,
include/gdn.h) with a thin ctypes binding.

    from chunked_gated_delta_06_gb300 import chunk_fwd, chunk_bwd, decode_step

The library is loaded on first use; it must have been built with
``python -m chunked_gated_delta_06_gb300.build``.
"""
from .binding import (GDN_DTYPE_BF16, GDN_DTYPE_F32, GdnError, GdnProblem,  # noqa: F401
                      chunk_bwd, chunk_bwd_gated, chunk_fwd, chunk_fwd_gated,
                      check_indices, chunk_prefill_paged, decode_step,
                      gdn_check_indices, gdn_chunk_prefill_paged,
                      gdn_chunk_scan_plan,
                      decode_step_gated, gdn_chunk_bwd_gated, gdn_chunk_fwd_gated,
                      gdn_decode_step_gated,
                      gdn_chunk_bwd, gdn_chunk_fwd, gdn_chunk_saved_bytes,
                      gdn_chunk_workspace_bytes, gdn_decode_step, lib, make_problem,
                      status_string)
from .autograd import chunk_gated_delta_rule  # noqa: E402,F401
