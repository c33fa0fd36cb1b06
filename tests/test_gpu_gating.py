"""GPU parity of the fused-gating entry points ("C6: GDN decode-step goldens and
recurrent/conv state contract", What and Provider: beta = sigmoid(b) and
g = -exp(A_log) softplus(a + dt_bias) computed in fp32 inside the kernels, softplus
threshold 20) against the fp64 oracle: oracle.gate_fwd, the rule, oracle.gate_bwd.
Tolerance per tensor: |x - ref| <= 1e-2 max|ref| + 1e-2 |ref|.
"""
import numpy as np
import pytest

from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    build.build()


def _bf(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def _run(wl, gi, recompute=False):
    import chunked_gated_delta_06_gb300 as gdn
    q, k, v, d_o = _bf(wl.q_bits), _bf(wl.k_bits), _bf(wl.v_bits), _bf(wl.do_bits)
    a, b = _bf(gi.a_bits), _bf(gi.b_bits)
    A = torch.from_numpy(gi.A_log).cuda()
    dt = torch.from_numpy(gi.dt_bias).cuda()
    h0 = None if wl.h0 is None else torch.from_numpy(wl.h0).cuda()
    dht = None if wl.d_ht is None else torch.from_numpy(wl.d_ht).cuda()
    cu_dev = torch.from_numpy(wl.cu_seqlens).cuda()
    o, ht, ctx = gdn.chunk_fwd_gated(q, k, v, a, b, A, dt, wl.cu_seqlens, cu_dev, initial_state=h0,
                                     for_backward=not recompute)
    out = dict(o=o, ht=ht)
    out.update(gdn.chunk_bwd_gated(ctx, q, k, v, a, b, A, dt, d_o, d_final_state=dht,
                                   initial_state=h0))
    torch.cuda.synchronize()
    return out


def _oracle(wl, gi):
    import oracle
    g, beta = oracle.gate_fwd(gi.a, gi.b, gi.A_log, gi.dt_bias)
    o, ht = oracle.fwd(wl.q, wl.k, wl.v, g, beta, wl.cu_seqlens, h0=wl.h0)
    gr = oracle.bwd(wl.q, wl.k, wl.v, g, beta, wl.cu_seqlens, wl.d_o, d_ht=wl.d_ht, h0=wl.h0)
    ch = oracle.gate_bwd(gi.a, gi.b, gi.A_log, gi.dt_bias, gr["dg"], gr["dbeta"])
    return dict(o=o, ht=ht, dq=gr["dq"], dk=gr["dk"], dv=gr["dv"], dh0=gr["dh0"], **ch)


CASES = [
    # name, lengths, H, HV, h0, d_ht
    ("ragged_r2", [1, 63, 64, 65, 130, 200], 2, 4, True, True),
    ("ragged_r1", [129, 7, 64], 2, 2, False, False),
    ("ragged_r4_empty", [0, 100, 0, 191], 1, 4, True, False),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_gated_fwd_bwd_matches_the_oracle(case):
    name, lengths, H, HV, h0, dht = case
    wl = W.chunk_workload(name, lengths, H, HV, seed=21, h0=h0, backward=True, d_ht=dht)
    gi = W.gate_inputs(wl.T, HV, seed=22)
    got = {k_: v_.float().cpu().numpy().astype(np.float64) for k_, v_ in _run(wl, gi).items()}
    ref = _oracle(wl, gi)
    for key in ("o", "ht", "dq", "dk", "dv", "dh0", "da", "db", "dA_log", "ddt_bias"):
        close(key, got[key], ref[key])


def test_gated_recompute_mode_gives_the_saved_mode_bits():
    wl = W.chunk_workload("gated", [300, 77, 64], 2, 4, seed=23, h0=True, backward=True, d_ht=True)
    gi = W.gate_inputs(wl.T, 4, seed=24)
    a, b = _run(wl, gi), _run(wl, gi, recompute=True)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_gated_backward_without_tokens_returns_zero_parameter_gradients():
    wl = W.chunk_workload("empty", [0, 0], 1, 2, seed=25, h0=True, backward=True, d_ht=True)
    gi = W.gate_inputs(0, 2, seed=26)
    out = _run(wl, gi)
    assert torch.equal(out["dA_log"], torch.zeros(2, device="cuda"))
    assert torch.equal(out["ddt_bias"], torch.zeros(2, device="cuda"))
    np.testing.assert_array_equal(out["dh0"].cpu().numpy(), wl.d_ht)


def test_gated_decode_matches_the_oracle():
    import oracle
    import chunked_gated_delta_06_gb300 as gdn
    dw = W.decode_workload(B=64, H=4, HV=8, num_slots=96, seed=27)
    gi = W.gate_inputs(dw.B, dw.HV, seed=28)
    pool = torch.from_numpy(dw.pool).cuda()
    idx = torch.from_numpy(dw.state_indices).cuda()
    o = gdn.decode_step_gated(_bf(dw.q_bits), _bf(dw.k_bits), _bf(dw.v_bits), _bf(gi.a_bits),
                              _bf(gi.b_bits), torch.from_numpy(gi.A_log).cuda(),
                              torch.from_numpy(gi.dt_bias).cuda(), pool, idx)
    torch.cuda.synchronize()
    g, beta = oracle.gate_fwd(gi.a, gi.b, gi.A_log, gi.dt_bias)
    o_ref, pool_ref, bad = oracle.decode(dw.q, dw.k, dw.v, g, beta, dw.pool, dw.state_indices)
    assert bad == 0
    close("o", o.float().cpu().numpy(), o_ref)
    live = sorted(set(int(s) for s in dw.state_indices if s > 0))
    close("pool", pool.cpu().numpy()[live], pool_ref[live])
