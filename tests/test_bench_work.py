"""The bench's algorithmic work formulas against the figures they are built from
("[Cake 1/13] gdn", Performance: the chunked form's contractions per token and
value head; the call's own inputs and outputs for the bytes), on CPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


@pytest.mark.parametrize("r, f_fwd", [(1, 182955), (2, 166571), (4, 158379)])
def test_forward_flops_per_token_and_value_head(bench, r, f_fwd):
    # 4CK/r + 2C(K + 2V) + 6KV + 2C^2/3 with C = 64, K = V = 128, rounded to a flop
    f, _ = bench.step_work(T=1, H=1, HV=r, N=1, backward=False, h0=False, final_state=False)
    assert round(f / r) == f_fwd
    fb, _ = bench.step_work(T=1, H=1, HV=r, N=1, backward=True, h0=False, final_state=False)
    assert fb == pytest.approx(3 * f)


def test_headline_totals(bench):
    # 32768 tokens, H = 16, HV = 32: 5.24e11 flops; 24,768 bytes per token forward and
    # 41,344 backward, plus the fp32 states of 11 sequences (h0 read twice, final state, dh0)
    f, b = bench.step_work(32768, 16, 32, 11, True, True, True, False)
    assert f == pytest.approx(5.24e11, rel=1e-3)
    states = 11 * 32 * 128 * 128 * 4
    assert b == 32768 * (24768 + 41344) + 4 * states
    f1, b1 = bench.step_work(256, 2, 2, 1, False, False, True, False)
    assert f1 == pytest.approx(256 * 2 * 182955, rel=1e-5)   # about 9.4e7
    assert b1 == 256 * (2 * 2 * 256 + 2 * 256 + 2 * 6 + 2 * 256) + 2 * 128 * 128 * 4


def test_decode_bytes(bench):
    # 230 active rows of 256, HV = 32: the state read and written once per active (row,
    # value head), 0.965 GB, plus q, k, v, o and g, beta of every row
    state = 230 * 32 * 2 * 128 * 128 * 4
    assert state == pytest.approx(0.965e9, rel=1e-3)
    tokens = 256 * (2 * 16 * 128 * 2 + 32 * 128 * 2 * 2 + 32 * 8)
    assert bench.decode_bytes(230, 256, 16, 32) == state + tokens
