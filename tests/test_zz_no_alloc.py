"""gdn_chunk_fwd_noalloc: the forward for callers that cannot allocate device
memory at call time (a pre-planned memory arena that forbids allocations
after start-up, a host plugin handed only its input and output buffers, a
latency-critical path that must avoid cudaMalloc's implicit synchronisation).

The entry point keeps its scratch in a fixed device array inside libgdn.so.
These checks call it through the C ABI twice in a row (the second call reuses
the array the first one left behind) and compare both results with the
regular gdn_chunk_fwd, which uses a caller workspace.  Both run the same
kernels in the same order on the same inputs, so the results must be the same
bits (the check is torch.equal, stricter than the parity tolerance).  A problem
whose workspace exceeds the array is rejected before any launch.  This file is
collected last on purpose.
"""
import pytest

from chunked_gated_delta_06_gb300 import binding
from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


def _outputs(wl, dev):
    T, N = wl.T, wl.N
    o = torch.empty((T, wl.HV, wl.V), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, wl.HV, wl.K, wl.V), dtype=torch.float32, device=dev)
    return o, ht


def test_no_alloc_forward_matches_the_workspace_forward_twice_in_a_row():
    wl = W.chunk_workload("noalloc", [70, 1, 130, 64], 2, 4, seed=11, gate="softplus", h0=True,
                          backward=False)
    d = to_dev(wl, torch)
    P = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    p, keep = binding.make_problem(wl.cu_seqlens, wl.H, wl.HV, cu_dev_ptr=d["cu_dev"].data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    # reference: the regular entry point with a torch-allocated workspace
    o_ref, ht_ref = _outputs(wl, "cuda")
    ws = torch.empty(binding.gdn_chunk_workspace_bytes(p, 0), dtype=torch.uint8, device="cuda")
    st = binding.gdn_chunk_fwd(p, P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]),
                               P(d["h0"]), P(o_ref), P(ht_ref), None, P(ws), ws.numel(), stream)
    assert st == binding.GDN_OK, binding.status_string(st)
    torch.cuda.synchronize()
    for _ in range(2):
        o, ht = _outputs(wl, "cuda")
        st = binding.gdn_chunk_fwd_noalloc(p, P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]),
                                           P(d["beta"]), P(d["h0"]), P(o), P(ht), stream)
        assert st == binding.GDN_OK, binding.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), "o differs from the workspace forward"
        assert torch.equal(ht, ht_ref), "final state differs from the workspace forward"


def test_no_alloc_forward_rejects_problems_beyond_its_scratch():
    # 4096 tokens x 32 value heads needs far more than the fixed 64 MiB scratch
    p, keep = binding.make_problem([0, 4096], 16, 32, cu_dev_ptr=0x1000)
    assert binding.gdn_chunk_workspace_bytes(p, 0) > (64 << 20)
    fake = 0x10000  # never dereferenced: the size check comes first
    st = binding.gdn_chunk_fwd_noalloc(p, fake, fake, fake, fake, fake, None, fake, None, None)
    assert st == binding.GDN_ERR_WORKSPACE_TOO_SMALL
