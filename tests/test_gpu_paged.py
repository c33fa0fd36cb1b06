"""GPU checks of the paged chunk prefill ("Replace Qwen3.5 FLA paths with Attention
Gym", GDN prefill ablation and Paged-state continuity): gdn_chunk_prefill_paged
reads each sequence's initial state from a slot of the decode pool
[slots, HV, V, K] and writes its final state back in place.

* the bits of gdn_chunk_fwd with the slots gathered (transposed) as initial
  states and the final states scattered back;
* parity with the oracle on a batch that mixes resumed, fresh-with-slot, null
  and out-of-range slots, with continuation lengths 1, 63, 64, 65 and 527;
* a prefill continued through a slot agrees with one call over the whole
  sequence, and a decode step after the prefill reads the state it left.
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
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _dev(wl):
    return dict(q=_bf(wl.q_bits), k=_bf(wl.k_bits), v=_bf(wl.v_bits),
                g=torch.from_numpy(wl.g).cuda(), beta=_bf(wl.beta_bits),
                cu=torch.from_numpy(wl.cu_seqlens).cuda())


def _pool(slots, HV, seed):
    r = np.random.default_rng(seed)
    return (0.1 * r.standard_normal((slots, HV, 128, 128))).astype(np.float32)


LENGTHS = [1, 63, 64, 65, 527, 40]


def test_paged_prefill_gives_the_bits_of_the_gathered_call():
    import chunked_gated_delta_06_gb300 as gdn
    wl = W.chunk_workload("paged", LENGTHS, 2, 4, seed=31, backward=False)
    d = _dev(wl)
    slots = 12
    pool0 = _pool(slots, 4, 32)
    idx = np.array([5, 0, 9, 3, 11, 7], dtype=np.int32)
    resume = np.array([1, 1, 0, 1, 1, 1], dtype=np.int32)
    pool = torch.from_numpy(pool0).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.chunk_prefill_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.cu_seqlens, d["cu"],
                                pool, torch.from_numpy(idx).cuda(), torch.from_numpy(resume).cuda(),
                                device_status=status)
    # the same forward with explicit states
    h0 = np.zeros((wl.N, 4, 128, 128), np.float32)
    for n, (s, rs) in enumerate(zip(idx, resume)):
        if s > 0 and rs:
            h0[n] = pool0[s].transpose(0, 2, 1)
    o2, ht, _ = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.cu_seqlens, d["cu"],
                              initial_state=torch.from_numpy(h0).cuda(), output_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    assert int(status.item()) == 0
    want = pool0.copy()
    htn = ht.cpu().numpy()
    for n, s in enumerate(idx):
        if s > 0:
            want[s] = htn[n].transpose(0, 2, 1)
    np.testing.assert_array_equal(pool.cpu().numpy(), want)


def test_paged_prefill_matches_the_oracle_with_null_and_out_of_range_slots():
    import oracle
    import chunked_gated_delta_06_gb300 as gdn
    wl = W.chunk_workload("paged", LENGTHS, 2, 4, seed=33, backward=False)
    d = _dev(wl)
    slots = 8
    pool0 = _pool(slots, 4, 34)
    idx = np.array([2, -1, 6, 8, 0, 5], dtype=np.int32)   # 8 is out of range
    resume = np.array([1, 1, 0, 1, 1, 1], dtype=np.int32)
    pool = torch.from_numpy(pool0).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = gdn.chunk_prefill_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.cu_seqlens, d["cu"],
                                pool, torch.from_numpy(idx).cuda(), torch.from_numpy(resume).cuda(),
                                device_status=status)
    torch.cuda.synchronize()
    o_ref, pool_ref, bad = oracle.prefill_paged(wl.q, wl.k, wl.v, wl.g, wl.beta, wl.cu_seqlens,
                                                pool0, idx, has_initial_state=resume)
    assert bad == 1 and int(status.item()) == 1
    close("o", o.float().cpu().numpy(), o_ref)
    got = pool.cpu().numpy()
    close("pool", got[[2, 5, 6]], pool_ref[[2, 5, 6]])
    np.testing.assert_array_equal(got[[0, 1, 3, 4, 7]], pool0[[0, 1, 3, 4, 7]])


def test_paged_prefill_continuation_then_decode():
    import oracle
    import chunked_gated_delta_06_gb300 as gdn
    # one 1584-token sequence prefilled in two calls (cut at 1056) through slot 3, then a
    # decode step on the slot; against one oracle call over all 1585 tokens
    full = W.chunk_workload("cont", [1585], 1, 2, seed=35, backward=False)
    slots = 4
    pool = torch.zeros((slots, 2, 128, 128), dtype=torch.float32, device="cuda")
    idx = torch.tensor([3], dtype=torch.int32, device="cuda")
    outs = []
    for i, (a, b) in enumerate([(0, 1056), (1056, 1584)]):
        part = W.ChunkWorkload(name="part", cu_seqlens=np.array([0, b - a], np.int32), H=1, HV=2,
                               K=128, V=128, q_bits=full.q_bits[a:b], k_bits=full.k_bits[a:b],
                               v_bits=full.v_bits[a:b], g=full.g[a:b], beta_bits=full.beta_bits[a:b],
                               h0=None, do_bits=None, d_ht=None, backward=False)
        d = _dev(part)
        resume = torch.tensor([i], dtype=torch.int32, device="cuda")
        outs.append(gdn.chunk_prefill_paged(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                            part.cu_seqlens, d["cu"], pool, idx, resume))
    t = 1584
    od = gdn.decode_step(_bf(full.q_bits[t:t + 1]), _bf(full.k_bits[t:t + 1]),
                         _bf(full.v_bits[t:t + 1]), torch.from_numpy(full.g[t:t + 1]).cuda(),
                         torch.from_numpy(full.beta[t:t + 1]).cuda(), pool, idx)
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle.fwd(full.q, full.k, full.v, full.g, full.beta, full.cu_seqlens)
    got = torch.cat(outs + [od]).float().cpu().numpy()
    close("o", got, o_ref)
    close("state", pool[3].cpu().numpy(), ht_ref[0].transpose(0, 2, 1))
