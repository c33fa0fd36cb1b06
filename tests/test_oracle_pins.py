"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each check ties the oracle to something the pages or the mathematics fix:
hand-worked examples (tests/golden/), closed forms of the recurrence, finite
differences of the forward for the hand-derived backward, the chunked (WY) form
at several chunk sizes against the per-token form, and invariances (splitting a
sequence across calls, grouped value heads, packing order, decode = one-token
chunk call).  ``test_every_planted_mistake_fails_a_pin`` plants mistakes in the
oracle and requires each to break at least one of these checks.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, lengths, H, HV, K, V, gate="logsigmoid", h0=True, scale_g=1.0):
    r = np.random.default_rng(seed)
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = r.standard_normal((T, H, K))
    k = r.standard_normal((T, H, K))
    v = r.standard_normal((T, HV, V))
    x = r.standard_normal((T, HV))
    if gate == "logsigmoid":
        g = np.minimum(x, 0) - np.log1p(np.exp(-np.abs(x)))
    else:  # strong decays, as the softplus gate of the benchmark workloads
        g = -np.log1p(np.exp(x)) * np.exp(r.uniform(0, 2.7, size=(HV,)))[None]
    g = g * scale_g
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, HV))))
    N = len(lengths)
    hz = 0.3 * r.standard_normal((N, HV, K, V)) if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu=cu, h0=hz)


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / den)


# ----------------------------------------------------------------------------- golden
@pytest.mark.parametrize("fname", ["delta_rule_hand_worked.json", "l2norm_epsilon.json"])
def test_hand_worked_golden(fname):
    check_golden(fname)


def check_golden(fname):
    with open(os.path.join(GOLD, fname)) as f:
        d = json.load(f)
    i = d["inputs"]
    o, ht = oracle.fwd(np.array(i["q"]), np.array(i["k"]), np.array(i["v"]), np.array(i["g"]),
                       np.array(i["beta"]), i["cu_seqlens"], scale=i["scale"],
                       h0=np.array(i["h0"]), use_l2norm=i["use_l2norm"])
    np.testing.assert_allclose(o, np.array(d["expected"]["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht, np.array(d["expected"]["final_state"]), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- closed forms
def check_beta_zero_is_pure_decay():
    """beta = 0: S_L = exp(sum g) S_0 and o_t = exp(sum_{i<=t} g_i) S_0 qhat_t."""
    c = _rand_case(1, [7], 1, 2, 5, 3)
    c["beta"][:] = 0.0
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"], scale=0.7)
    G = np.cumsum(c["g"], axis=0)  # [T, HV]
    assert _rel(ht, np.exp(G[-1])[None, :, None, None] * c["h0"]) < 1e-13
    qn = c["q"] / np.sqrt((c["q"] ** 2).sum(-1, keepdims=True) + 1e-6) * 0.7  # [T,1,K]
    for hv in range(2):
        S0 = c["h0"][0, hv].T  # V x K
        exp_o = np.exp(G[:, hv])[:, None] * (qn[:, 0, :] @ S0.T)
        assert _rel(o[:, hv], exp_o) < 1e-13


def test_beta_zero_is_pure_decay():
    check_beta_zero_is_pure_decay()


def check_unit_key_overwrites_one_column():
    """g = 0, beta = 1, key e_j (norm off): column j of S becomes v, other columns unchanged."""
    K, V = 6, 4
    r = np.random.default_rng(2)
    h0 = r.standard_normal((1, 1, K, V))
    j = 3
    k = np.zeros((1, 1, K)); k[0, 0, j] = 1.0
    q = r.standard_normal((1, 1, K))
    v = r.standard_normal((1, 1, V))
    o, ht = oracle.fwd(q, k, v, np.zeros((1, 1)), np.ones((1, 1)), [0, 1], h0=h0,
                       use_l2norm=False, scale=1.0)
    S0 = h0[0, 0].T
    S1 = ht[0, 0].T
    expect = S0.copy(); expect[:, j] = v[0, 0]
    # exact up to the rounding of S'_j + (v - S'_j)
    np.testing.assert_allclose(S1, expect, rtol=0, atol=1e-14)
    untouched = [c for c in range(K) if c != j]
    np.testing.assert_array_equal(S1[:, untouched], S0[:, untouched])
    np.testing.assert_allclose(o[0, 0], expect @ q[0, 0], rtol=1e-14, atol=1e-14)


def test_unit_key_overwrites_one_column():
    check_unit_key_overwrites_one_column()


def check_orthonormal_keys_are_recalled():
    """g = 0, beta = 1, orthonormal keys written in turn: S k_i = v_i afterwards."""
    K, V, T = 8, 5, 6
    r = np.random.default_rng(3)
    Qm, _ = np.linalg.qr(r.standard_normal((K, K)))
    keys = Qm[:, :T].T  # T orthonormal rows
    v = r.standard_normal((T, 1, V))
    h0 = r.standard_normal((1, 1, K, V))
    q = np.zeros((T, 1, K))
    _, ht = oracle.fwd(q, keys[:, None, :], v, np.zeros((T, 1)), np.ones((T, 1)), [0, T], h0=h0,
                       use_l2norm=False, scale=1.0)
    S = ht[0, 0].T
    for i in range(T):
        np.testing.assert_allclose(S @ keys[i], v[i, 0], rtol=0, atol=1e-12)


def test_orthonormal_keys_are_recalled():
    check_orthonormal_keys_are_recalled()


def check_keys_are_not_scaled():
    """scale multiplies q only: S1 = v khat^T with khat = k / sqrt(|k|^2 + 1e-6)."""
    K, V = 4, 3
    k = np.zeros((1, 1, K)); k[0, 0, 1] = 2.0
    q = np.zeros((1, 1, K)); q[0, 0, 1] = 1.0
    v = np.arange(1.0, V + 1).reshape(1, 1, V)
    s = 0.25
    o, ht = oracle.fwd(q, k, v, np.zeros((1, 1)), np.ones((1, 1)), [0, 1], scale=s)
    kh = 2.0 / np.sqrt(4.0 + 1e-6)
    qh = s / np.sqrt(1.0 + 1e-6)
    np.testing.assert_allclose(ht[0, 0, 1], v[0, 0] * kh, rtol=1e-15)
    np.testing.assert_allclose(o[0, 0], v[0, 0] * kh * qh, rtol=1e-15)


def test_keys_are_not_scaled():
    check_keys_are_not_scaled()


# ----------------------------------------------------------------------------- chunked form
CHUNK_LENGTHS = [1, 63, 64, 65, 130]


def check_chunked_form_equals_per_token(C, gate="softplus", K=8, V=8, lengths=CHUNK_LENGTHS,
                                        H=2, HV=4, tol=1e-11):
    c = _rand_case(4 + C, lengths, H, HV, K, V, gate=gate)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"])
    ch = oracle.fwd_chunked(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], C, h0=c["h0"])
    assert _rel(ch["o"], o) < tol, _rel(ch["o"], o)
    assert _rel(ch["ht"], ht) < tol, _rel(ch["ht"], ht)


@pytest.mark.parametrize("C", [1, 2, 3, 16, 64])
@pytest.mark.parametrize("gate", ["softplus", "logsigmoid"])
def test_chunked_form_equals_per_token(C, gate):
    check_chunked_form_equals_per_token(C, gate)


def test_chunked_form_equals_per_token_at_head_dim_128():
    check_chunked_form_equals_per_token(64, "softplus", K=128, V=128, lengths=[70, 64], H=1, HV=2)


def test_chunked_intermediates_reproduce_the_state_passing():
    """h_chunks[c] is the state after the previous chunk; v_new is the WY delta."""
    c = _rand_case(11, [130, 5], 1, 2, 8, 8)
    ch = oracle.fwd_chunked(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], 64, h0=c["h0"],
                            want_chunks=True)
    # chunk 1 of sequence 0 starts after 64 tokens: compare with a per-token call on them
    _, ht64 = oracle.fwd(c["q"][:64], c["k"][:64], c["v"][:64], c["g"][:64], c["beta"][:64],
                         [0, 64], h0=c["h0"][:1])
    assert _rel(ch["h_chunks"][1], ht64[0]) < 1e-12
    np.testing.assert_array_equal(ch["h_chunks"][0], c["h0"][0])
    np.testing.assert_array_equal(ch["h_chunks"][3], c["h0"][1])


# ----------------------------------------------------------------------------- backward
def _loss_and_grads(c, Wo, Wht, use_l2norm, scale):
    def loss(**over):
        a = dict(c); a.update(over)
        o, ht = oracle.fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["cu"], h0=a["h0"],
                           use_l2norm=use_l2norm, scale=scale, threads=1)
        return float((o * Wo).sum() + (ht * Wht).sum())
    gr = oracle.bwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], Wo, d_ht=Wht, h0=c["h0"],
                    use_l2norm=use_l2norm, scale=scale, threads=1)
    return loss, gr


def check_backward_matches_finite_differences(use_l2norm=True, seed=5, K=4, V=4, lengths=(4, 5),
                                              H=1, HV=2, sample=None, eps=1e-5, tol=1e-6):
    c = _rand_case(seed, list(lengths), H, HV, K, V)
    r = np.random.default_rng(seed + 100)
    T = c["q"].shape[0]
    N = len(lengths)
    Wo = r.standard_normal((T, HV, V))
    Wht = r.standard_normal((N, HV, K, V))
    scale = 0.8
    loss, gr = _loss_and_grads(c, Wo, Wht, use_l2norm, scale)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    for name, gname in names.items():
        x = c[name]
        flat = np.arange(x.size)
        if sample is not None and x.size > sample:
            flat = r.choice(x.size, size=sample, replace=False)
        an = gr[gname].reshape(-1)[flat]
        fd = np.empty(len(flat))
        for n_, i in enumerate(flat):
            xp = x.copy().reshape(-1); xp[i] += eps
            xm = x.copy().reshape(-1); xm[i] -= eps
            fd[n_] = (loss(**{name: xp.reshape(x.shape)}) - loss(**{name: xm.reshape(x.shape)})) / (2 * eps)
        err = np.linalg.norm(fd - an) / max(np.linalg.norm(fd), 1e-30)
        assert err < tol, (name, err)


@pytest.mark.parametrize("use_l2norm", [True, False])
def test_backward_matches_finite_differences(use_l2norm):
    check_backward_matches_finite_differences(use_l2norm)


def test_backward_matches_finite_differences_grouped_heads():
    check_backward_matches_finite_differences(True, seed=9, K=3, V=5, lengths=(3, 1, 4), H=2, HV=4)


def test_backward_matches_finite_differences_at_head_dim_128():
    check_backward_matches_finite_differences(True, seed=7, K=128, V=128, lengths=(3,), H=1, HV=1,
                                              sample=12)


def test_backward_crosses_the_checkpoint_segments():
    """Sequences longer than the oracle's 64-token recompute segments."""
    check_backward_matches_finite_differences(True, seed=13, K=2, V=3, lengths=(70,), H=1, HV=1,
                                              sample=25)


# ----------------------------------------------------------------------------- invariances
def check_split_call_equals_one_call():
    c = _rand_case(21, [50], 1, 2, 6, 5)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"])
    s = 23
    o1, h1 = oracle.fwd(c["q"][:s], c["k"][:s], c["v"][:s], c["g"][:s], c["beta"][:s], [0, s],
                        h0=c["h0"])
    o2, h2 = oracle.fwd(c["q"][s:], c["k"][s:], c["v"][s:], c["g"][s:], c["beta"][s:], [0, 50 - s],
                        h0=h1)
    assert _rel(np.concatenate([o1, o2]), o) < 1e-13
    assert _rel(h2, ht) < 1e-13
    # backward: gradient of the first half's final state = dh0 of the second half
    r = np.random.default_rng(22)
    do = r.standard_normal(o.shape)
    full = oracle.bwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], do, h0=c["h0"])
    b2 = oracle.bwd(c["q"][s:], c["k"][s:], c["v"][s:], c["g"][s:], c["beta"][s:], [0, 50 - s],
                    do[s:], h0=h1)
    b1 = oracle.bwd(c["q"][:s], c["k"][:s], c["v"][:s], c["g"][:s], c["beta"][:s], [0, s], do[:s],
                    d_ht=b2["dh0"], h0=c["h0"])
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert _rel(np.concatenate([b1[key], b2[key]]), full[key]) < 1e-12, key
    assert _rel(b1["dh0"], full["dh0"]) < 1e-12


def test_split_call_equals_one_call():
    check_split_call_equals_one_call()


def check_grouped_heads_equal_repeated_keys():
    """HV = r H reads key head hv // r: same as H' = HV with q, k repeated r times."""
    H, r_, K, V = 2, 3, 4, 5
    c = _rand_case(31, [9, 4], H, H * r_, K, V)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"])
    qr = np.repeat(c["q"], r_, axis=1)
    kr = np.repeat(c["k"], r_, axis=1)
    o2, ht2 = oracle.fwd(qr, kr, c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"])
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ht, ht2, rtol=1e-13, atol=1e-13)
    do = np.random.default_rng(32).standard_normal(o.shape)
    g1 = oracle.bwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], do, h0=c["h0"])
    g2 = oracle.bwd(qr, kr, c["v"], c["g"], c["beta"], c["cu"], do, h0=c["h0"])
    T = c["q"].shape[0]
    np.testing.assert_allclose(g1["dq"], g2["dq"].reshape(T, H, r_, K).sum(2), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g1["dk"], g2["dk"].reshape(T, H, r_, K).sum(2), rtol=1e-12, atol=1e-12)


def test_grouped_heads_equal_repeated_keys():
    check_grouped_heads_equal_repeated_keys()


def test_packing_order_is_irrelevant():
    c = _rand_case(41, [5, 9, 3], 1, 1, 4, 4)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"])
    perm = [2, 0, 1]
    segs = [np.arange(c["cu"][i], c["cu"][i + 1]) for i in range(3)]
    idx = np.concatenate([segs[p] for p in perm])
    lens = [len(segs[p]) for p in perm]
    cu2 = np.concatenate([[0], np.cumsum(lens)])
    o2, ht2 = oracle.fwd(c["q"][idx], c["k"][idx], c["v"][idx], c["g"][idx], c["beta"][idx], cu2,
                         h0=c["h0"][perm])
    np.testing.assert_allclose(o2, o[idx], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(ht2, ht[perm], rtol=1e-14, atol=1e-14)


def test_empty_call_passes_the_state_through():
    c = _rand_case(42, [0, 0], 1, 2, 4, 4)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], h0=c["h0"])
    assert o.shape == (0, 2, 4)
    np.testing.assert_array_equal(ht, c["h0"])


# ----------------------------------------------------------------------------- decode
def check_decode_equals_one_token_chunk_call():
    """Decode on a V-major pool = a one-token chunk call per row with h0 = pool[slot]^T."""
    B, H, HV, K, V, slots = 5, 2, 4, 6, 3, 9
    r = np.random.default_rng(51)
    q = r.standard_normal((B, H, K)); k = r.standard_normal((B, H, K))
    v = r.standard_normal((B, HV, V))
    g = -np.abs(r.standard_normal((B, HV))); beta = r.uniform(0, 1, (B, HV))
    pool = r.standard_normal((slots, HV, V, K))
    idx = np.array([3, 0, 7, -2, 1], dtype=np.int32)
    o, newpool, bad = oracle.decode(q, k, v, g, beta, pool, idx, scale=0.6)
    assert bad == 0
    for b in range(B):
        if idx[b] <= 0:
            assert np.all(o[b] == 0)
            continue
        h0 = np.transpose(pool[idx[b]], (0, 2, 1))[None]  # [1, HV, K, V]
        o1, ht = oracle.fwd(q[b:b + 1], k[b:b + 1], v[b:b + 1], g[b:b + 1], beta[b:b + 1], [0, 1],
                            h0=h0, scale=0.6)
        np.testing.assert_allclose(o[b], o1[0], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(newpool[idx[b]], np.transpose(ht[0], (0, 2, 1)), rtol=1e-13,
                                   atol=1e-13)
    untouched = [s for s in range(slots) if s not in set(idx[idx > 0].tolist())]
    np.testing.assert_array_equal(newpool[untouched], pool[untouched])


def test_decode_equals_one_token_chunk_call():
    check_decode_equals_one_token_chunk_call()


def test_decode_counts_out_of_range_slots_and_skips_them():
    B, H, HV, K, V, slots = 3, 1, 2, 4, 4, 4
    r = np.random.default_rng(52)
    pool = r.standard_normal((slots, HV, V, K))
    idx = np.array([1, 4, 9], dtype=np.int32)
    o, newpool, bad = oracle.decode(r.standard_normal((B, H, K)), r.standard_normal((B, H, K)),
                                    r.standard_normal((B, HV, V)), np.zeros((B, HV)),
                                    np.ones((B, HV)), pool, idx)
    assert bad == 2
    assert np.all(o[1:] == 0)
    np.testing.assert_array_equal(newpool[2:], pool[2:])


# ----------------------------------------------------------------------------- fused gating
def check_gate_closed_forms():
    # softplus(0) = ln 2; above the threshold 20 softplus is the identity; far below it
    # softplus(x) = e^x to within e^{2x}; sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4,
    # sigmoid(x) + sigmoid(-x) = 1
    A = np.array([0.0, 0.7, -1.3, 2.0])
    dt = np.array([0.0, 0.5, 0.25, -1.0])
    a = np.array([[0.0 - 0.0, 30.0 - 0.5, -40.0 - 0.25, 20.5 + 1.0]])
    b = np.array([[0.0, np.log(3.0), 2.5, -2.5]])
    g, beta = oracle.gate_fwd(a, b, A, dt)
    assert g[0, 0] == pytest.approx(-np.log(2.0), rel=1e-15)
    assert g[0, 1] == -np.exp(0.7) * 30.0
    assert g[0, 2] == pytest.approx(-np.exp(-1.3) * np.exp(-40.0), rel=1e-12)
    assert g[0, 3] == -np.exp(2.0) * 20.5
    assert beta[0, 0] == 0.5
    assert beta[0, 1] == pytest.approx(0.75, rel=1e-15)
    assert beta[0, 2] + beta[0, 3] == pytest.approx(1.0, rel=1e-15)


def check_gate_backward_matches_finite_differences():
    r = np.random.default_rng(61)
    n, HV = 5, 3
    A = r.uniform(-1, 1.5, size=HV)
    dt = r.uniform(-1, 1, size=HV)
    a = r.uniform(-6, 6, size=(n, HV))
    a[2, 1] = 26.0 - dt[1]  # above the softplus threshold: derivative exactly 1
    b = r.uniform(-4, 4, size=(n, HV))
    wg, wb = r.standard_normal((n, HV)), r.standard_normal((n, HV))

    def loss(a_, b_, A_, dt_):
        g, beta = oracle.gate_fwd(a_, b_, A_, dt_)
        return float((wg * g).sum() + (wb * beta).sum())

    gr = oracle.gate_bwd(a, b, A, dt, wg, wb)
    eps = 1e-6
    for name, x, ref in (("a", a, gr["da"]), ("b", b, gr["db"]), ("A_log", A, gr["dA_log"]),
                         ("dt_bias", dt, gr["ddt_bias"])):
        fd = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += eps
            xm[i] -= eps
            args_p = dict(a_=a, b_=b, A_=A, dt_=dt)
            args_m = dict(args_p)
            key = {"a": "a_", "b": "b_", "A_log": "A_", "dt_bias": "dt_"}[name]
            args_p[key], args_m[key] = xp, xm
            fd[i] = (loss(**args_p) - loss(**args_m)) / (2 * eps)
        np.testing.assert_allclose(ref, fd, rtol=1e-6, atol=1e-8, err_msg=name)


def check_gated_rule_gradients_through_the_gate():
    # the composition the gated entry points compute: g, beta from a, b, then the rule;
    # d loss / d (a, b, A_log, dt_bias) by the chain rule against central differences
    r = np.random.default_rng(62)
    lengths, H, HV, K, V = [5, 4], 1, 2, 4, 4
    c = _rand_case(63, lengths, H, HV, K, V, h0=True)
    T = sum(lengths)
    A = r.uniform(-0.5, 1.0, size=HV)
    dt = r.uniform(-0.5, 0.5, size=HV)
    a = r.standard_normal((T, HV))
    b = r.standard_normal((T, HV))
    dO = r.standard_normal((T, HV, V))

    def loss(a_, b_, A_, dt_):
        g, beta = oracle.gate_fwd(a_, b_, A_, dt_)
        o, _ = oracle.fwd(c["q"], c["k"], c["v"], g, beta, c["cu"], h0=c["h0"], threads=1)
        return float((dO * o).sum())

    g, beta = oracle.gate_fwd(a, b, A, dt)
    gr = oracle.bwd(c["q"], c["k"], c["v"], g, beta, c["cu"], dO, h0=c["h0"], threads=1)
    ch = oracle.gate_bwd(a, b, A, dt, gr["dg"], gr["dbeta"])
    eps = 1e-6
    for (t, h) in [(0, 0), (3, 1), (5, 0), (8, 1)]:
        for name, x in (("a", a), ("b", b)):
            xp, xm = x.copy(), x.copy()
            xp[t, h] += eps
            xm[t, h] -= eps
            if name == "a":
                fd = (loss(xp, b, A, dt) - loss(xm, b, A, dt)) / (2 * eps)
            else:
                fd = (loss(a, xp, A, dt) - loss(a, xm, A, dt)) / (2 * eps)
            assert ch["d" + name][t, h] == pytest.approx(fd, rel=1e-5, abs=1e-8), (name, t, h)
    for h in range(HV):
        Ap, Am = A.copy(), A.copy()
        Ap[h] += eps
        Am[h] -= eps
        fd = (loss(a, b, Ap, dt) - loss(a, b, Am, dt)) / (2 * eps)
        assert ch["dA_log"][h] == pytest.approx(fd, rel=1e-5, abs=1e-8)
        dp, dm = dt.copy(), dt.copy()
        dp[h] += eps
        dm[h] -= eps
        fd = (loss(a, b, A, dp) - loss(a, b, A, dm)) / (2 * eps)
        assert ch["ddt_bias"][h] == pytest.approx(fd, rel=1e-5, abs=1e-8)


def test_gate_closed_forms():
    check_gate_closed_forms()


def test_gate_backward_matches_finite_differences():
    check_gate_backward_matches_finite_differences()


def test_gated_rule_gradients_through_the_gate():
    check_gated_rule_gradients_through_the_gate()


# ----------------------------------------------------------------------------- paged prefill
def check_paged_prefill_one_token_equals_decode():
    # a one-token prefill that resumes a slot is the decode step on that slot: the two
    # read the pool through different code (transpose + chunk call vs the decode rule)
    r = np.random.default_rng(71)
    B, H, HV, K, V, slots = 3, 1, 2, 4, 4, 6
    pool = 0.5 * r.standard_normal((slots, HV, V, K))
    q, k = r.standard_normal((B, H, K)), r.standard_normal((B, H, K))
    v = r.standard_normal((B, HV, V))
    g = -np.abs(r.standard_normal((B, HV)))
    beta = 1 / (1 + np.exp(-r.standard_normal((B, HV))))
    idx = np.array([4, 1, 5], dtype=np.int32)
    cu = np.arange(B + 1, dtype=np.int32)
    o, newpool, bad = oracle.prefill_paged(q, k, v, g, beta, cu, pool, idx, scale=0.7)
    od, pool_d, bad_d = oracle.decode(q, k, v, g, beta, pool, idx, scale=0.7)
    assert bad == bad_d == 0
    np.testing.assert_allclose(o, od, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(newpool, pool_d, rtol=1e-12, atol=1e-12)


def check_paged_prefill_continues_a_sequence():
    # "Paged-state continuity": a sequence prefilled in two calls through its slot
    # gives the outputs and final state of one call over the whole sequence
    c = _rand_case(72, [23], 1, 2, 4, 4, h0=False)
    slots = 3
    pool = np.zeros((slots, 2, 4, 4))
    idx = np.array([2], dtype=np.int32)
    o_all, ht_all = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"])
    for cut in (1, 9, 22):
        parts = [(0, cut), (cut, 23)]
        p = pool.copy()
        outs = []
        for i, (a, b) in enumerate(parts):
            sl = slice(a, b)
            o, p, _ = oracle.prefill_paged(c["q"][sl], c["k"][sl], c["v"][sl], c["g"][sl],
                                           c["beta"][sl], np.array([0, b - a], dtype=np.int32), p,
                                           idx, has_initial_state=np.array([i > 0]))
            outs.append(o)
        np.testing.assert_allclose(np.concatenate(outs), o_all, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(p[2], ht_all[0].transpose(0, 2, 1), rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(p[[0, 1]], pool[[0, 1]])


def check_paged_prefill_fresh_and_null_slots():
    c = _rand_case(73, [5, 4, 6], 1, 2, 4, 4, h0=False)
    r = np.random.default_rng(74)
    slots = 5
    pool = r.standard_normal((slots, 2, 4, 4))
    idx = np.array([3, 0, 7], dtype=np.int32)        # fresh with a slot, none, out of range
    o, newpool, bad = oracle.prefill_paged(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"], pool,
                                           idx, has_initial_state=np.array([0, 1, 1]))
    o0, ht0 = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu"])  # all from zeros
    assert bad == 1
    np.testing.assert_allclose(o, o0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(newpool[3], ht0[0].transpose(0, 2, 1), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(newpool[[0, 1, 2, 4]], pool[[0, 1, 2, 4]])


def test_paged_prefill_one_token_equals_decode():
    check_paged_prefill_one_token_equals_decode()


def test_paged_prefill_continues_a_sequence():
    check_paged_prefill_continues_a_sequence()


def test_paged_prefill_fresh_and_null_slots():
    check_paged_prefill_fresh_and_null_slots()


# ----------------------------------------------------------------------------- discrimination
PINS = [
    lambda: check_golden("delta_rule_hand_worked.json"),
    lambda: check_golden("l2norm_epsilon.json"),
    check_beta_zero_is_pure_decay,
    check_unit_key_overwrites_one_column,
    check_orthonormal_keys_are_recalled,
    check_keys_are_not_scaled,
    lambda: check_chunked_form_equals_per_token(16),
    lambda: check_backward_matches_finite_differences(True),
    check_split_call_equals_one_call,
    check_grouped_heads_equal_repeated_keys,
    check_decode_equals_one_token_chunk_call,
    check_gate_closed_forms,
    check_gate_backward_matches_finite_differences,
    check_paged_prefill_one_token_equals_decode,
    check_paged_prefill_continues_a_sequence,
]

# 1 decay after the write, 2 prediction from the undecayed state, 3 output before the write,
# 4 scale on k too, 5 epsilon outside the sqrt, 6 sign of dp flipped (backward), 7 key head hv % H,
# 8 dbeta -> db through beta instead of beta (1 - beta), 9 da through softplus instead of its slope,
# 10 paged prefill reads and writes the slots without transposing, 11 chunked form: the
# decay in A as e^{G_j - G_i}, 12 chunked form: the state update's decay factor e^{G_j - G_L},
# 13 decode step without the decay
MUTATIONS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13]


@pytest.mark.parametrize("m", MUTATIONS)
def test_every_planted_mistake_fails_a_pin(m):
    oracle.set_mutation(m)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    oracle.set_mutation(0)
    assert failed >= 1, "planted mistake %d passed every pin" % m
