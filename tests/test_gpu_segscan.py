"""GPU parity of the segment-parallel state scans (a long sequence cut into
segments: pass 1 scans the first segment -- the last one in the reverse scan --
beside the pre-scans of the transitions of the inner segments, k_seg_stitch forms
the segments' start states, pass 2 re-scans them; "[Cake 1/13] gdn: ...", Review items: pre-scan + stitch; "Qwen3.5-397B RL
trainer on 128 v7x", GDN context-parallel m-scan).  Each case asserts that the
plan really splits, then compares with the fp64 oracle, whose per-token forward
has no segments at all.  Tolerance: |x - ref| <= 1e-2 max|ref| + 1e-2 |ref|.
"""
import numpy as np
import pytest

import chunked_gated_delta_06_gb300 as gdn_pkg
from chunked_gated_delta_06_gb300 import binding
from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import close, compare_units, oracle_chunk, run_chunk, run_chunk_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


def _plan(wl, scan_segment_chunks=0):
    p, keep = binding.make_problem(wl.cu_seqlens, wl.H, wl.HV, cu_dev_ptr=0x1000,
                                   scan_segment_chunks=scan_segment_chunks)
    st, seg_len, nseg = gdn_pkg.gdn_chunk_scan_plan(p)
    assert st == 0
    return seg_len, nseg


def test_split_forward_and_backward_match_the_oracle():
    wl = W.chunk_workload("seg_one_long", [8192], 2, 4, seed=41, h0=True, backward=True, d_ht=True)
    seg_len, nseg = _plan(wl)
    assert seg_len > 0 and nseg >= 3
    compare_units(run_chunk(wl, torch), oracle_chunk(wl), wl)


def test_split_forward_with_unsplit_neighbours_matches_the_oracle():
    # one sequence long enough to split, one that fits one segment, one in between
    wl = W.chunk_workload("seg_mixed", [5000, 100, 2500], 2, 4, seed=42, h0=True, backward=False)
    seg_len, nseg = _plan(wl)
    assert seg_len > 0 and nseg >= 3
    assert 100 <= 64 * seg_len  # the short sequence is a single segment
    compare_units(run_chunk(wl, torch), oracle_chunk(wl), wl)


def test_split_scan_is_bitwise_repeatable_and_recompute_gives_the_same_bits():
    wl = W.chunk_workload("seg_det", [6000, 300], 2, 4, seed=43, h0=True, backward=True, d_ht=True)
    assert _plan(wl)[0] > 0
    a = run_chunk_raw(wl, torch)
    b = run_chunk_raw(wl, torch)
    c = run_chunk_raw(wl, torch, recompute=True)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key
            assert torch.equal(a[key], c[key]), key


def test_split_paged_prefill_matches_the_oracle():
    import oracle
    wl = W.chunk_workload("seg_paged", [7000, 64], 2, 4, seed=44, backward=False)
    assert _plan(wl)[0] > 0
    slots = 4
    pool0 = (0.1 * np.random.default_rng(45).standard_normal((slots, 4, 128, 128))).astype(np.float32)
    idx = np.array([3, 1], dtype=np.int32)
    bf = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    pool = torch.from_numpy(pool0).cuda()
    o = gdn_pkg.chunk_prefill_paged(bf(wl.q_bits), bf(wl.k_bits), bf(wl.v_bits),
                                    torch.from_numpy(wl.g).cuda(), bf(wl.beta_bits), wl.cu_seqlens,
                                    torch.from_numpy(wl.cu_seqlens).cuda(), pool,
                                    torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    o_ref, pool_ref, bad = oracle.prefill_paged(wl.q, wl.k, wl.v, wl.g, wl.beta, wl.cu_seqlens,
                                                pool0, idx)
    close("o", o.float().cpu().numpy(), o_ref)
    close("pool", pool.cpu().numpy()[[1, 3]], pool_ref[[1, 3]])


def test_split_and_plain_scans_agree():
    # the split is driven through the ABI: scan_segment_chunks = -1 never splits
    wl = W.chunk_workload("seg_vs_plain", [8192, 700], 2, 4, seed=46, h0=True, backward=True,
                          d_ht=True)
    assert _plan(wl)[0] > 0
    split = run_chunk(wl, torch)
    assert _plan(wl, scan_segment_chunks=-1) == (0, 1)
    plain = run_chunk(wl, torch, scan_segment_chunks=-1)
    for key in ("o", "ht", "dq", "dk", "dv", "dg", "dbeta", "dh0"):
        close(key, split[key], plain[key])
