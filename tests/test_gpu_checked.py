"""The bounds-checked build (nvcc -DGDN_CHECKED, libgdn_checked.so), which stands in
for the race / out-of-bounds sanitizers the pages run on their kernels ("cake_gdn:
deterministic chunked GDN training kernels", Validation of the round-13 kernels:
synccheck and racecheck).  In it every direct global access of the chunk and decode
kernels is range-checked against its buffer's extent; an access outside sets bit 4
(GDN_DEVICE_INDEX_OUT_OF_RANGE) of the status word and is skipped, never trapping.

The small ragged cases of the parity tests (empty and one-token sequences, partial
chunks, r = 1, 2, 4, both gate recipes), a split scan, the fused gate, the paged
prefill and a decode batch run through the checked build: the status word must stay
0 and the results must match the fp64 oracle within the usual tolerance.
"""
import numpy as np
import pytest

import chunked_gated_delta_06_gb300 as gdn
from chunked_gated_delta_06_gb300 import binding
from chunked_gated_delta_06_gb300 import workloads as W
from gpu_helpers import close, compare_units, oracle_chunk, run_chunk

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    # name, lengths, H, HV, gate, h0, d_ht, scan_segment_chunks
    ("ragged_r2_softplus", [1, 63, 64, 65, 130, 200], 2, 4, "softplus", True, True, 0),
    ("ragged_r1_logsigmoid", [129, 7, 64], 2, 2, "logsigmoid", True, False, 0),
    ("ragged_r4_empty_seqs", [0, 100, 0, 191, 0], 1, 4, "softplus", False, True, 0),
    ("single_token_seqs", [1, 1, 1], 1, 2, "logsigmoid", True, True, 0),
    ("split_scan", [1500, 70], 1, 2, "softplus", True, True, 4),
]


@pytest.fixture(scope="module")
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_gated_delta_06_gb300 import build
    return build.build(checked=True)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_checked_build_small_cases(checked_lib, case):
    name, lengths, H, HV, gate, h0, dht, seg = case
    wl = W.chunk_workload(name, lengths, H, HV, seed=31, gate=gate, h0=h0, backward=True, d_ht=dht)
    with binding.use_library(checked_lib):
        # run_chunk passes a status word and asserts it stays 0
        gpu = run_chunk(wl, torch, scan_segment_chunks=seg)
        gpu_rc = run_chunk(wl, torch, recompute=True, scan_segment_chunks=seg)
    compare_units(gpu, oracle_chunk(wl), wl)
    for key in gpu:
        if gpu[key] is not None:
            np.testing.assert_array_equal(gpu[key], gpu_rc[key])


def test_checked_build_gated_paged_and_decode(checked_lib):
    import oracle
    wl = W.chunk_workload("checked_gate", [70, 1, 130], 2, 4, seed=32, backward=True, h0=True, d_ht=True)
    gi = W.gate_inputs(wl.T, wl.HV, seed=33)
    bf = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    q, k, v = bf(wl.q_bits), bf(wl.k_bits), bf(wl.v_bits)
    a_, b_ = bf(gi.a_bits), bf(gi.b_bits)
    A_log, dt_bias = torch.from_numpy(gi.A_log).cuda(), torch.from_numpy(gi.dt_bias).cuda()
    h0 = torch.from_numpy(wl.h0).cuda()
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    dstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    with binding.use_library(checked_lib):
        o, ht, ctx = gdn.chunk_fwd_gated(q, k, v, a_, b_, A_log, dt_bias, wl.cu_seqlens, cu,
                                         initial_state=h0, for_backward=True, device_status=status)
        gr = gdn.chunk_bwd_gated(ctx, q, k, v, a_, b_, A_log, dt_bias, bf(wl.do_bits),
                                 d_final_state=torch.from_numpy(wl.d_ht).cuda(), initial_state=h0)
        # paged prefill over a pool (slots 3 and 1 resumed, one null slot)
        slots = 5
        pool0 = (0.1 * np.random.default_rng(34).standard_normal((slots, wl.HV, 128, 128))).astype(np.float32)
        pool = torch.from_numpy(pool0).cuda()
        idx = np.array([3, 0, 1], dtype=np.int32)
        g = torch.from_numpy(wl.g).cuda()
        beta = bf(wl.beta_bits)
        op = gdn.chunk_prefill_paged(q, k, v, g, beta, wl.cu_seqlens, cu, pool, torch.from_numpy(idx).cuda(),
                                     device_status=pstatus, problem_status=status)
        # a decode batch on the pool
        dw = W.decode_workload("checked_decode", B=8, H=2, HV=4, num_slots=12, seed=35)
        dpool = torch.from_numpy(dw.pool).cuda()
        od = gdn.decode_step(bf(dw.q_bits), bf(dw.k_bits), bf(dw.v_bits), torch.from_numpy(dw.g).cuda(),
                             torch.from_numpy(dw.beta).cuda(), dpool, torch.from_numpy(dw.state_indices).cuda(),
                             device_status=dstatus)
        torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(pstatus.item()) == 0 and int(dstatus.item()) == 0
    # the gated call against the oracle's gated form
    g_ref, beta_ref = oracle.gate_fwd(gi.a, gi.b, gi.A_log, gi.dt_bias)
    ro, rht = oracle.fwd(wl.q, wl.k, wl.v, g_ref, beta_ref, wl.cu_seqlens, h0=wl.h0)
    close("o", o.float().cpu().numpy(), ro)
    close("final_state", ht.cpu().numpy(), rht)
    o_ref, pool_ref, _ = oracle.prefill_paged(wl.q, wl.k, wl.v, wl.g, wl.beta, wl.cu_seqlens, pool0, idx)
    close("paged o", op.float().cpu().numpy(), o_ref)
    close("paged pool", pool.cpu().numpy(), pool_ref)
    rod, rpool, _ = oracle.decode(dw.q, dw.k, dw.v, dw.g, dw.beta, dw.pool, dw.state_indices)
    close("decode o", od.float().cpu().numpy(), rod)
    close("decode pool", dpool.cpu().numpy(), rpool)
    assert gr["dq"].shape == q.shape
