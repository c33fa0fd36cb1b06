"""GPU checks of chunk_gated_delta_rule, the differentiable call with the pages' shape
([1, T, H, K] packed inputs, cu_seqlens, initial / final state): its forward and
its autograd gradients are the bits of gdn_chunk_fwd / gdn_chunk_bwd, with and
without the recompute-state option."""
import numpy as np
import pytest

from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import run_chunk_raw

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


@pytest.mark.parametrize("recompute", [False, True])
def test_autograd_gives_the_c_abi_bits(recompute):
    import chunked_gated_delta_06_gb300 as gdn
    wl = W.chunk_workload("autograd", [1, 63, 64, 65, 200], 2, 4, seed=51, h0=True, backward=True,
                          d_ht=True)
    ref = run_chunk_raw(wl, torch)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)

    q, k, v, beta = bf(wl.q_bits), bf(wl.k_bits), bf(wl.v_bits), bf(wl.beta_bits)
    g = torch.from_numpy(wl.g).cuda()
    h0 = torch.from_numpy(wl.h0).cuda()
    for x in (q, k, v, g, beta, h0):
        x.requires_grad_(True)
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    o, ht = gdn.chunk_gated_delta_rule(q[None], k[None], v[None], g[None], beta[None],
                                       initial_state=h0, output_final_state=True, cu_seqlens=cu,
                                       cu_seqlens_cpu=wl.cu_seqlens, recompute_state=recompute)
    assert o.shape == (1, wl.T, wl.HV, 128)
    assert torch.equal(o[0], ref["o"]) and torch.equal(ht, ref["ht"])
    d_o, d_ht = bf(wl.do_bits), torch.from_numpy(wl.d_ht).cuda()
    torch.autograd.backward([o[0], ht], [d_o, d_ht])
    torch.cuda.synchronize()
    for name, t in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta), ("dh0", h0)):
        assert t.grad is not None, name
        assert torch.equal(t.grad, ref[name]), name


def test_autograd_without_states():
    """No initial state, no final state: ht is None, h0 gets no gradient, and the
    other gradients are those of gdn_chunk_bwd with no d_final_state."""
    import chunked_gated_delta_06_gb300 as gdn
    wl = W.chunk_workload("autograd_nostate", [0, 129, 7, 64], 2, 2, seed=52, h0=False,
                          backward=True, d_ht=False)
    ref = run_chunk_raw(wl, torch)

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)

    q, k, v, beta = bf(wl.q_bits), bf(wl.k_bits), bf(wl.v_bits), bf(wl.beta_bits)
    g = torch.from_numpy(wl.g).cuda()
    for x in (q, k, v, g, beta):
        x.requires_grad_(True)
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    o, ht = gdn.chunk_gated_delta_rule(q, k, v, g, beta, cu_seqlens=cu)
    assert ht is None and o.shape == (wl.T, wl.HV, 128)
    assert torch.equal(o, ref["o"])
    o.backward(bf(wl.do_bits))
    torch.cuda.synchronize()
    for name, t in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta)):
        assert torch.equal(t.grad, ref[name]), name
