"""Shared helpers of the GPU parity tests: upload a seeded workload, run the
CUDA path through the C ABI, slice units for the oracle, compare within the
per-tensor tolerance |x - ref| <= 1e-2 max|ref| + 1e-2 |ref|."""
from __future__ import annotations

import numpy as np

ATOL_REL = 1e-2  # times max|ref| of the tensor
RTOL = 1e-2


def close(name, got, ref, atol_rel=ATOL_REL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    assert np.all(np.isfinite(got)), "%s: non-finite values" % name
    m = np.abs(ref).max()
    err = np.abs(got - ref)
    bound = atol_rel * m + rtol * np.abs(ref)
    worst = float((err / np.maximum(bound, 1e-300)).max())
    assert worst <= 1.0, "%s: error %.3g of its bound (max|err| %.3g, max|ref| %.3g)" % (
        name, worst, err.max(), m)
    return worst


def to_dev(wl, torch):
    """Upload a ChunkWorkload; returns a dict of device tensors."""
    dev = "cuda"

    def bf(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    beta = bf(wl.beta_bits) if wl.beta_f32 is None else torch.from_numpy(wl.beta_f32).to(dev)
    d = dict(q=bf(wl.q_bits), k=bf(wl.k_bits), v=bf(wl.v_bits),
             g=torch.from_numpy(wl.g).to(dev), beta=beta,
             h0=None if wl.h0 is None else torch.from_numpy(wl.h0).to(dev),
             cu_dev=torch.from_numpy(wl.cu_seqlens).to(dev))
    d["d_o"] = None if wl.do_bits is None else bf(wl.do_bits)
    d["d_ht"] = None if wl.d_ht is None else torch.from_numpy(wl.d_ht).to(dev)
    return d


def run_chunk(wl, torch, backward=None, recompute=False, scan_segment_chunks=0):
    """Run gdn_chunk_fwd (+ gdn_chunk_bwd) on a workload; returns numpy float64 results."""
    out = run_chunk_raw(wl, torch, backward=backward, recompute=recompute,
                        scan_segment_chunks=scan_segment_chunks)
    return {k_: (None if v_ is None else v_.float().cpu().numpy().astype(np.float64))
            for k_, v_ in out.items()}


def run_chunk_raw(wl, torch, backward=None, recompute=False, scan_segment_chunks=0):
    """Like run_chunk but returns the device tensors (for bitwise comparisons).
    recompute: the forward keeps no saved buffer and the backward rebuilds it.
    Every call passes a device status word and asserts that the kernels left it 0."""
    import chunked_gated_delta_06_gb300 as gdn
    backward = wl.backward if backward is None else backward
    d = to_dev(wl, torch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, ht, ctx = gdn.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], wl.cu_seqlens, d["cu_dev"],
                               initial_state=d["h0"], output_final_state=True,
                               for_backward=backward and not recompute, device_status=status,
                               scan_segment_chunks=scan_segment_chunks)
    out = dict(o=o, ht=ht)
    if backward:
        out.update(gdn.chunk_bwd(ctx, d["q"], d["k"], d["v"], d["g"], d["beta"], d["d_o"],
                                 d_final_state=d["d_ht"], initial_state=d["h0"]))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %d after a valid call" % int(status.item())
    return out


def oracle_chunk(wl, backward=None, seqs=None, key_heads=None, value_heads=None, threads=None):
    """Oracle on the (sequence, value head) units selected.

    seqs: sequence indices (default all); key_heads: the key heads whose value
    heads are all taken (dq/dk are complete for them); value_heads: explicit value
    heads (default: all of key_heads, or every head).  Returns results indexed
    like the full problem restricted to the selection, plus the selection itself."""
    import oracle
    backward = wl.backward if backward is None else backward
    N = wl.N
    seqs = list(range(N)) if seqs is None else list(seqs)
    r = wl.HV // wl.H
    if value_heads is None:
        if key_heads is None:
            key_heads = list(range(wl.H))
        value_heads = [h * r + j for h in key_heads for j in range(r)]
    kh = sorted({hv // r for hv in value_heads})
    # slice tokens of the chosen sequences, in order
    cu = wl.cu_seqlens
    tok = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs]) if seqs else np.zeros(0, int)
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    cu2 = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    # the oracle needs HV' = r' H' with head map hv // r'; use one key head per value head
    q = wl.q[tok][:, [hv // r for hv in value_heads]]
    k = wl.k[tok][:, [hv // r for hv in value_heads]]
    v = wl.v[tok][:, value_heads]
    g = wl.g[tok][:, value_heads]
    beta = wl.beta[tok][:, value_heads]
    h0 = None if wl.h0 is None else wl.h0[seqs][:, value_heads]
    o, ht = oracle.fwd(q, k, v, g, beta, cu2, h0=h0, threads=threads)
    res = dict(o=o, ht=ht, tok=tok, seqs=seqs, value_heads=value_heads, key_heads=kh)
    if backward:
        d_o = wl.d_o[tok][:, value_heads]
        d_ht = None if wl.d_ht is None else wl.d_ht[seqs][:, value_heads]
        gr = oracle.bwd(q, k, v, g, beta, cu2, d_o, d_ht=d_ht, h0=h0, threads=threads)
        # gr["dq"] is per value head here (H' = HV'); sum per key head in value-head order
        dq = np.zeros((len(tok), len(kh), wl.K))
        dk = np.zeros((len(tok), len(kh), wl.K))
        for i, hv in enumerate(value_heads):
            dq[:, kh.index(hv // r)] += gr["dq"][:, i]
            dk[:, kh.index(hv // r)] += gr["dk"][:, i]
        res.update(dq=dq, dk=dk, dv=gr["dv"], dg=gr["dg"], dbeta=gr["dbeta"], dh0=gr["dh0"])
    return res


def compare_units(gpu, ref, wl, skip=()):
    """Compare the GPU results restricted to the oracle's selection."""
    tok, seqs, vh, kh = ref["tok"], ref["seqs"], ref["value_heads"], ref["key_heads"]
    worst = {}
    worst["o"] = close("o", gpu["o"][tok][:, vh], ref["o"])
    if gpu.get("ht") is not None:
        worst["ht"] = close("final_state", gpu["ht"][seqs][:, vh], ref["ht"])
    if "dv" in ref and gpu.get("dv") is not None:
        for name in ("dv", "dg", "dbeta"):
            if name not in skip:
                worst[name] = close(name, gpu[name][tok][:, vh], ref[name])
        if "dh0" not in skip and gpu.get("dh0") is not None:
            worst["dh0"] = close("dh0", gpu["dh0"][seqs][:, vh], ref["dh0"])
        if "dqdk" not in skip:
            worst["dq"] = close("dq", gpu["dq"][tok][:, kh], ref["dq"])
            worst["dk"] = close("dk", gpu["dk"][tok][:, kh], ref["dk"])
    return worst
