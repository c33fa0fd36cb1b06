"""The device status word of the chunk calls (gdn_problem.device_status): the
pages ask for failures to be reported, not silent ("[Cake 1/13] gdn: chunked
gated delta rule, det and fast, with KCP and FLA-CP", API and flags).

- a valid forward + backward leaves the word at 0;
- a device copy of cu_seqlens that disagrees with the host copy sets bit 1, and
  the kernels then see an empty chunk table (no access outside the buffers, the
  context stays usable);
- the bounded wait the tensor-core kernels use gives up and sets bit 2, shown by
  gdn_selftest_bounded_wait on a barrier that nothing arrives on (no GPU fault,
  no hang: the wait has a 2 ms limit).
"""
import numpy as np
import pytest

import chunked_gated_delta_06_gb300 as gdn
from chunked_gated_delta_06_gb300 import binding
from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import compare_units, oracle_chunk, run_chunk, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


def _fwd_bwd(wl, cu_dev, status):
    d = to_dev(wl, torch)
    o, ht, ctx = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.cu_seqlens, cu_dev,
                               initial_state=d["h0"], for_backward=True, device_status=status)
    gdn.chunk_bwd(ctx, d["q"], d["k"], d["v"], d["g"], d["beta"], d["d_o"],
                  d_final_state=d["d_ht"], initial_state=d["h0"])
    torch.cuda.synchronize()


def test_a_valid_call_leaves_the_status_word_at_zero():
    wl = W.chunk_workload("status_ok", [70, 130, 1], 2, 4, seed=21, h0=True, backward=True, d_ht=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _fwd_bwd(wl, torch.from_numpy(wl.cu_seqlens).cuda(), status)
    assert int(status.item()) == 0


@pytest.mark.parametrize("cu_dev", [
    [0, 150, 200],   # same total and chunk count, but one sequence longer than any on the host
    [0, 100, 190],   # a different total
    [0, 120, 100],   # decreasing
], ids=["longer_sequence", "other_total", "decreasing"])
def test_a_device_cu_seqlens_that_disagrees_sets_bit_1(cu_dev):
    # host: two sequences of 100 tokens (two chunks each)
    wl = W.chunk_workload("status_cu", [100, 100], 2, 4, seed=22, h0=True, backward=True, d_ht=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _fwd_bwd(wl, torch.tensor(cu_dev, dtype=torch.int32, device="cuda"), status)
    assert int(status.item()) & binding.GDN_DEVICE_CU_SEQLENS_MISMATCH
    # the context is still usable: a valid call afterwards matches the oracle
    compare_units(run_chunk(wl, torch), oracle_chunk(wl), wl)


def test_the_bounded_wait_gives_up_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = binding.gdn_selftest_bounded_wait(status.data_ptr(), 2_000_000,
                                           torch.cuda.current_stream().cuda_stream)
    assert st == binding.GDN_OK
    torch.cuda.synchronize()
    assert int(status.item()) == binding.GDN_DEVICE_WAIT_TIMEOUT
    # the context is still usable
    wl = W.chunk_workload("after_wait", [64, 3], 1, 2, seed=23, backward=True)
    compare_units(run_chunk(wl, torch), oracle_chunk(wl), wl)


def test_the_selftest_rejects_bad_arguments():
    s = torch.cuda.current_stream().cuda_stream
    assert binding.gdn_selftest_bounded_wait(None, 2_000_000, s) == binding.GDN_ERR_INVALID_ARG
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert binding.gdn_selftest_bounded_wait(status.data_ptr(), 10, s) == binding.GDN_ERR_INVALID_ARG
    assert binding.gdn_selftest_bounded_wait(status.data_ptr(), 10 ** 10, s) == binding.GDN_ERR_INVALID_ARG
    assert binding.gdn_selftest_bounded_wait(status.data_ptr() + 2, 10 ** 6, s) == binding.GDN_ERR_INVALID_ARG
    np.testing.assert_array_equal(status.cpu().numpy(), [0, 0])
