"""GPU checks of the call variants of the chunk path ("[Cake 1/13] gdn: chunked
gated delta rule, det and fast, with KCP and FLA-CP", API and flags and
Performance (3/5)):

* recompute-state mode: gdn_chunk_bwd without a saved buffer rebuilds w, u, h and
  v_new itself and returns the same bits as the backward of a saved forward;
* fp32 beta (GDN_DTYPE_F32): parity with the fp64 oracle on the exact fp32
  values, dbeta returned in fp32, the same bits as the bf16 path when the fp32
  values are bf16 numbers, and different bits when they are not (beta is never
  rounded inside).
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


def _bitwise(a, b, keys=None):
    for key in keys or a:
        if a[key] is not None:
            assert b[key] is not None, key
            assert a[key].dtype == b[key].dtype, key
            assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("lengths, H, HV, h0, dht", [
    ([1, 63, 64, 65, 130, 200], 2, 4, True, True),
    ([0, 100, 0, 191, 0], 1, 4, False, False),
])
def test_recompute_mode_gives_the_saved_mode_bits(lengths, H, HV, h0, dht):
    wl = W.chunk_workload("recompute", lengths, H, HV, seed=11, h0=h0, backward=True, d_ht=dht)
    saved = run_chunk_raw(wl, torch)
    again = run_chunk_raw(wl, torch, recompute=True)
    _bitwise(saved, again)


def test_recompute_mode_at_the_4x4096_workload():
    wl = W.fb_4x4096()
    _bitwise(run_chunk_raw(wl, torch), run_chunk_raw(wl, torch, recompute=True))


@pytest.mark.parametrize("lengths, H, HV, gate", [
    ([1, 63, 64, 65, 130, 200], 2, 4, "softplus"),
    ([129, 7, 64], 2, 2, "logsigmoid"),
    ([0, 100, 191], 1, 4, "softplus"),
])
def test_fp32_beta_matches_the_oracle(lengths, H, HV, gate):
    wl = W.chunk_workload("beta_f32", lengths, H, HV, seed=12, gate=gate, h0=True, backward=True,
                          d_ht=True, beta_dtype="f32")
    raw = run_chunk_raw(wl, torch)
    assert raw["dbeta"].dtype == torch.float32
    gpu = {k_: (None if v_ is None else v_.float().cpu().numpy().astype(np.float64))
           for k_, v_ in raw.items()}
    compare_units(gpu, oracle_chunk(wl), wl)


def test_fp32_beta_holding_bf16_values_gives_the_bf16_bits():
    wl = W.chunk_workload("beta_bf16", [1, 63, 64, 65, 130, 200], 2, 4, seed=13, h0=True,
                          backward=True, d_ht=True)
    ref = run_chunk_raw(wl, torch)
    wl.beta_f32 = W.bf16_value(wl.beta_bits).copy()  # the same numbers, stored as fp32
    got = run_chunk_raw(wl, torch)
    _bitwise(ref, got, keys=("o", "ht", "dq", "dk", "dv", "dg", "dh0"))
    assert got["dbeta"].dtype == torch.float32
    # dbeta itself: the bf16 output is the fp32 output rounded once
    assert torch.equal(got["dbeta"].to(torch.bfloat16), ref["dbeta"])


def test_fp32_beta_is_not_rounded_inside():
    wl = W.chunk_workload("beta_f32", [300, 77], 2, 4, seed=14, h0=True, backward=True,
                          beta_dtype="f32")
    assert not np.array_equal(wl.beta_f32, W.bf16_value(wl.beta_bits))
    full = run_chunk_raw(wl, torch)
    wl.beta_f32 = W.bf16_value(wl.beta_bits).copy()
    rounded = run_chunk_raw(wl, torch)
    assert not torch.equal(full["o"], rounded["o"])
    assert not torch.equal(full["dk"], rounded["dk"])
