"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases run the oracle on everything; they span several chunks with ragged
tails, empty sequences, grouped value heads r = 1, 2, 4 and both gate recipes.
The full-size workloads run on the GPU in the configuration the bench times and
are compared on sampled (sequence, value head) units that the oracle computes
one by one (units are independent), plus bitwise run-to-run determinism.
Tolerance per tensor: |x - ref| <= 1e-2 max|ref| + 1e-2 |ref|.
"""
import numpy as np
import pytest

from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import compare_units, oracle_chunk, run_chunk, run_chunk_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


SMALL = [
    # name, lengths, H, HV, gate, h0, d_ht
    ("ragged_r2_softplus", [1, 63, 64, 65, 130, 200], 2, 4, "softplus", True, True),
    ("ragged_r1_logsigmoid", [129, 7, 64], 2, 2, "logsigmoid", True, False),
    ("ragged_r4_empty_seqs", [0, 100, 0, 191, 0], 1, 4, "softplus", False, True),
    ("single_token_seqs", [1, 1, 1], 1, 2, "logsigmoid", True, True),
]


def test_many_short_sequences_match_oracle():
    # 400 sequences of 1 .. 80 tokens: a chunk table and scan grid far wider than the
    # small cases, with a partial chunk at the end of almost every sequence
    lengths = np.random.default_rng(6).integers(1, 81, size=400).tolist()
    wl = W.chunk_workload("many_short", lengths, 1, 2, seed=7, gate="softplus", h0=True,
                          backward=True, d_ht=True)
    compare_units(run_chunk(wl, torch), oracle_chunk(wl), wl)


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_fwd_bwd_matches_oracle(case):
    name, lengths, H, HV, gate, h0, dht = case
    wl = W.chunk_workload(name, lengths, H, HV, seed=3, gate=gate, h0=h0, backward=True, d_ht=dht)
    gpu = run_chunk(wl, torch)
    ref = oracle_chunk(wl)
    compare_units(gpu, ref, wl)


def test_fwd_t256_matches_oracle():
    wl = W.fwd_t256()
    gpu = run_chunk(wl, torch)
    ref = oracle_chunk(wl)
    compare_units(gpu, ref, wl)


def test_empty_call_passes_the_state_through():
    wl = W.chunk_workload("empty", [0, 0], 1, 2, seed=4, h0=True, backward=True, d_ht=True)
    gpu = run_chunk(wl, torch)
    assert gpu["o"].shape == (0, 2, 128)
    np.testing.assert_array_equal(gpu["ht"], wl.h0)
    np.testing.assert_array_equal(gpu["dh0"], wl.d_ht)


def test_repeated_runs_are_bit_identical():
    wl = W.chunk_workload("det", [300, 77, 64], 2, 4, seed=5, h0=True, backward=True, d_ht=True)
    a = run_chunk_raw(wl, torch)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = run_chunk_raw(wl, torch)
    s.synchronize()
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key


def _sampled(wl, seqs, key_heads=None, value_heads=None, skip=()):
    gpu = run_chunk(wl, torch)
    ref = oracle_chunk(wl, seqs=seqs, key_heads=key_heads, value_heads=value_heads)
    return compare_units(gpu, ref, wl, skip=skip)


def test_fb_4x4096_sampled_units():
    wl = W.fb_4x4096()
    _sampled(wl, seqs=[0, 3], key_heads=[0, 15])


def test_fb_32k_varlen_sampled_units():
    wl = W.fb_32k_varlen()
    lens = np.diff(wl.cu_seqlens)
    seqs = [int(np.argmin(lens)), int(np.argmax(lens))]
    _sampled(wl, seqs=seqs, key_heads=[7])


def test_fb_65536_long_sampled_key_head():
    wl = W.fb_65536_long()
    # all four value heads (36 .. 39) of key head 9 of the single 65536-token sequence:
    # o, final state, dv, dg, dbeta, dh0 per value head, and dq, dk of the key head
    # (its sum over the four value heads) over all 1024 chunks
    _sampled(wl, seqs=[0], key_heads=[9])


def test_fb_32k_varlen_repeats_bit_for_bit():
    wl = W.fb_32k_varlen()
    a = run_chunk_raw(wl, torch)
    b = run_chunk_raw(wl, torch)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key


def test_hundred_repeats_of_the_32k_varlen_step_are_bit_identical():
    """fwd + bwd of the 32K varlen pack 100 times (every tenth on a side stream):
    every output of every run equals the first run's bit for bit."""
    import chunked_gated_delta_06_gb300 as gdn
    from gpu_helpers import to_dev
    wl = W.fb_32k_varlen()
    d = to_dev(wl, torch)
    side = torch.cuda.Stream()

    def step():
        o, ht, ctx = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.cu_seqlens, d["cu_dev"],
                                   initial_state=d["h0"], output_final_state=True, for_backward=True)
        gr = gdn.chunk_bwd(ctx, d["q"], d["k"], d["v"], d["g"], d["beta"], d["d_o"],
                           d_final_state=d["d_ht"], initial_state=d["h0"])
        return dict(o=o, ht=ht, **gr)

    first = step()
    for i in range(1, 100):
        if i % 10 == 0:
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                out = step()
            torch.cuda.current_stream().wait_stream(side)
        else:
            out = step()
        for key, ref in first.items():
            if ref is not None:
                assert torch.equal(out[key], ref), (i, key)
