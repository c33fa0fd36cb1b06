"""The plan of the forward state scan (gdn_chunk_scan_plan, a pure host function):
split only where a few long sequences would leave the GPU idle, never for the
packed training workloads, and the same plan on every call."""
import numpy as np

import chunked_gated_delta_06_gb300 as gdn
from chunked_gated_delta_06_gb300 import binding, build, workloads as W


def _plan(lengths, H, HV, scan_segment_chunks=0):
    build.build()
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    p, keep = binding.make_problem(cu, H, HV, cu_dev_ptr=0x1000, scan_segment_chunks=scan_segment_chunks)
    st, seg_len, nseg = gdn.gdn_chunk_scan_plan(p)
    assert st == binding.GDN_OK
    return seg_len, nseg, gdn.gdn_chunk_workspace_bytes(p, 0)


def test_packed_training_workloads_are_not_split():
    assert _plan(W.varlen_lengths(0, 32768, 1, 8192), 16, 32)[:2] == (0, 1)
    assert _plan([4096] * 4, 16, 32)[:2] == (0, 1)
    assert _plan([65536], 16, 64)[:2] == (0, 1)  # 128 scan CTAs already: too little gain


def test_a_long_sequence_with_few_heads_is_split():
    seg_len, nseg, _ = _plan([8192], 2, 4)
    assert seg_len > 0 and nseg >= 3
    assert nseg == -(-128 // seg_len)


def test_short_sequences_are_never_split():
    assert _plan([64 * 20], 1, 1)[:2] == (0, 1)
    assert _plan([100] * 50, 1, 2)[:2] == (0, 1)


def test_the_split_adds_exactly_its_segment_buffers_to_the_workspace():
    seg_len, nseg, ws = _plan([8192], 2, 4)
    # the same token count in sequences too short to split: the workspace differs only by
    # the segment buffers (N x (S - 1) x HV x (K x 2K + K x V) fp32), up to 256-byte rounding
    seg_len2, nseg2, ws2 = _plan([64] * 128, 2, 4)
    assert seg_len2 == 0
    table_diff = 3 * 128 * 4 + 128 * 4  # the chunk table and sequence order of 128 sequences
    bufs = 1 * (nseg - 1) * 4 * (128 * 256 + 128 * 128) * 4
    assert abs((ws - ws2) - (bufs - table_diff)) <= 8 * 256


def test_the_plan_is_a_pure_function_of_the_problem():
    assert _plan([3000, 7000, 500], 2, 4) == _plan([3000, 7000, 500], 2, 4)


def test_the_plan_query_rejects_an_invalid_problem():
    cu = np.array([0, 5, 3], dtype=np.int32)
    p, keep = binding.make_problem(cu, 2, 4, cu_dev_ptr=0x1000)
    st, _, _ = gdn.gdn_chunk_scan_plan(p)
    assert st == binding.GDN_ERR_INVALID_ARG


def test_the_problem_field_overrides_the_plan():
    assert _plan([8192], 2, 4, scan_segment_chunks=-1)[:2] == (0, 1)
    assert _plan([8192], 2, 4, scan_segment_chunks=16)[:2] == (16, 8)
    assert _plan(W.varlen_lengths(0, 32768, 1, 8192), 16, 32, scan_segment_chunks=16)[0] == 16
    assert _plan([8192], 2, 4, scan_segment_chunks=64)[:2] == (0, 1)  # two segments: nothing to gain


def test_the_environment_no_longer_changes_the_plan(monkeypatch):
    # the plan (and so the bits) depends on the call's arguments only
    before = _plan([8192], 2, 4)
    monkeypatch.setenv("GDN_SCAN_SEGMENT_CHUNKS", "0")
    assert _plan([8192], 2, 4) == before


def test_an_invalid_scan_field_is_rejected():
    cu = np.array([0, 8192], dtype=np.int32)
    p, keep = binding.make_problem(cu, 2, 4, cu_dev_ptr=0x1000, scan_segment_chunks=-2)
    assert gdn.gdn_chunk_scan_plan(p)[0] == binding.GDN_ERR_INVALID_ARG
    assert gdn.gdn_chunk_workspace_bytes(p, 0) == 0
