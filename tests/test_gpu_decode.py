"""GPU parity of the decode step against the fp64 oracle, on the full
256-row / [512, 32, 128, 128] pool workload and on small cases: sampled rows
match the oracle, null rows (index <= 0) are zero and leave every slot
untouched, an out-of-range index is flagged and skipped, and a row's result does
not depend on its batch position (bitwise)."""
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


def _run(wl, pool_dev, idx=None, status=None):
    import chunked_gated_delta_06_gb300 as gdn
    idx = wl.state_indices if idx is None else idx
    o = gdn.decode_step(_bf(wl.q_bits), _bf(wl.k_bits), _bf(wl.v_bits),
                        torch.from_numpy(wl.g).cuda(), torch.from_numpy(wl.beta).cuda(), pool_dev,
                        torch.from_numpy(idx).cuda(), device_status=status)
    torch.cuda.synchronize()
    return o


def _oracle_rows(wl, rows):
    """Oracle decode for the rows (b, hv) listed, on a pool of just their slots."""
    import oracle
    out = {}
    for b, hv in rows:
        slot = int(wl.state_indices[b])
        h = hv // (wl.HV // wl.H)
        sub = np.zeros((2, 1, wl.V, wl.K))
        if slot > 0:
            sub[1, 0] = wl.pool[slot, hv]
        o, newpool, _ = oracle.decode(wl.q[b:b + 1, h:h + 1], wl.k[b:b + 1, h:h + 1],
                                      wl.v[b:b + 1, hv:hv + 1], wl.g[b:b + 1, hv:hv + 1],
                                      wl.beta[b:b + 1, hv:hv + 1], sub,
                                      np.array([1 if slot > 0 else 0], np.int32))
        out[(b, hv)] = (o[0, 0], newpool[1, 0])
    return out


def test_decode_256_sampled_rows_match_oracle():
    wl = W.decode_workload()
    pool = torch.from_numpy(wl.pool).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = _run(wl, pool, status=status).float().cpu().numpy()
    assert int(status.item()) == 0
    r = np.random.default_rng(7)
    active = np.nonzero(wl.state_indices > 0)[0]
    null = np.nonzero(wl.state_indices <= 0)[0]
    rows = [(int(b), int(r.integers(wl.HV))) for b in r.choice(active, 24, replace=False)]
    rows += [(int(b), int(r.integers(wl.HV))) for b in null[:4]]
    ref = _oracle_rows(wl, rows)
    newpool = pool.cpu().numpy()
    for (b, hv), (o_ref, s_ref) in ref.items():
        close("o[%d,%d]" % (b, hv), o[b, hv], o_ref)
        slot = int(wl.state_indices[b])
        if slot > 0:
            close("state[%d,%d]" % (slot, hv), newpool[slot, hv], s_ref)
    # null rows are exact zeros; slots not named by an active row are untouched
    assert np.all(o[null] == 0)
    touched = set(int(s) for s in wl.state_indices if s > 0)
    untouched = np.array([s for s in range(wl.pool.shape[0]) if s not in touched])
    np.testing.assert_array_equal(newpool[untouched], wl.pool[untouched])


def test_decode_flags_out_of_range_indices_and_skips_them():
    wl = W.decode_workload("small", B=6, H=2, HV=4, num_slots=8, null_frac=0.0, seed=3)
    idx = wl.state_indices.copy()
    idx[2] = 8      # == num_slots: out of range
    idx[4] = -3     # null
    pool = torch.from_numpy(wl.pool).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = _run(wl, pool, idx=idx, status=status).float().cpu().numpy()
    assert int(status.item()) == 1
    assert np.all(o[2] == 0) and np.all(o[4] == 0)
    newpool = pool.cpu().numpy()
    live = set(int(s) for i, s in enumerate(idx) if 0 < s < 8)
    for s in range(8):
        if s not in live:
            np.testing.assert_array_equal(newpool[s], wl.pool[s])


def test_decode_row_is_independent_of_batch_position():
    wl = W.decode_workload("inv", B=16, H=2, HV=4, num_slots=40, null_frac=0.0, seed=9)
    pool = torch.from_numpy(wl.pool).cuda()
    o_all = _run(wl, pool).cpu()
    pool_after = pool.clone()
    # row 5 alone, on a fresh copy of the pool
    b = 5
    single = W.DecodeWorkload(name="one", H=wl.H, HV=wl.HV, K=wl.K, V=wl.V,
                              q_bits=wl.q_bits[b:b + 1], k_bits=wl.k_bits[b:b + 1],
                              v_bits=wl.v_bits[b:b + 1], g=wl.g[b:b + 1], beta=wl.beta[b:b + 1],
                              pool=wl.pool, state_indices=wl.state_indices[b:b + 1])
    pool2 = torch.from_numpy(wl.pool).cuda()
    o_one = _run(single, pool2).cpu()
    assert torch.equal(o_all[b], o_one[0])
    s = int(wl.state_indices[b])
    assert torch.equal(pool_after[s], pool2[s])
