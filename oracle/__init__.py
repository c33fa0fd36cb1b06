"""fp64 CPU oracle of the gated delta rule (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
oracle imports nothing from the product package.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, no code shared with
the CUDA library); this module compiles it with gcc, converts numpy arrays to
contiguous float64 and splits the independent (sequence, value head) work units
over host threads.  See the header of ``gdn_oracle.c`` for the pages each step
follows.

Every input is given as it is stored on the device (bf16 values widened to
float64 exactly), so the oracle sees the same numbers as the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_gdn_oracle.so (gcc, -O2, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.gdn_oracle_set_mutation.argtypes = [ctypes.c_int]
            lib.gdn_oracle_get_mutation.restype = ctypes.c_int
            common = [ctypes.c_int, _I, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_double, ctypes.c_int]
            lib.gdn_oracle_fwd.argtypes = common + [_D] * 7 + [_D, ctypes.c_int, ctypes.c_int]
            lib.gdn_oracle_bwd.argtypes = common + [_D] * 6 + [_D] * 2 + [_D] * 6 + [ctypes.c_int] * 2
            lib.gdn_oracle_fwd_chunked.argtypes = (common + [ctypes.c_int] + [_D] * 6 + [_D] * 4
                                                   + [ctypes.c_int] * 2)
            lib.gdn_oracle_decode.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_int]
                                              + [_D] * 6 + [ctypes.c_int, _I, _D]
                                              + [ctypes.c_int] * 2)
            lib.gdn_oracle_decode.restype = ctypes.c_int
            lib.gdn_oracle_gate_fwd.argtypes = [ctypes.c_int] * 2 + [_D] * 6
            lib.gdn_oracle_gate_bwd.argtypes = [ctypes.c_int] * 2 + [_D] * 10
            _lib = lib
    return _lib


def set_mutation(m: int) -> None:
    """Plant mistake number ``m`` in the oracle (0 = none).  Tests only."""
    _load().gdn_oracle_set_mutation(int(m))


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(_D)


def _parallel(n_units: int, fn, threads: int | None):
    threads = threads or os.cpu_count() or 1
    threads = max(1, min(threads, n_units))
    if threads == 1:
        fn(0, n_units)
        return
    bounds = np.linspace(0, n_units, threads + 1).astype(int)
    with ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(fn, int(b), int(e)) for b, e in zip(bounds[:-1], bounds[1:]) if e > b]
        for f in futs:
            f.result()


def _shapes(q, v, cu):
    T, H, K = q.shape
    _, HV, V = v.shape
    assert HV % H == 0, "HV must be a multiple of H"
    N = len(cu) - 1
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    return T, H, HV, K, V, N


def _scale(scale, K):
    return float(scale) if scale is not None and scale > 0 else 1.0 / np.sqrt(K)


def fwd(q, k, v, g, beta, cu_seqlens, scale=None, h0=None, use_l2norm=True, threads=None):
    """Per-token forward.  Returns (o [T,HV,V], final_state [N,HV,K,V])."""
    lib = _load()
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, H, HV, K, V, N = _shapes(q, v, cu)
    o = np.zeros((T, HV, V))
    ht = np.zeros((N, HV, K, V))
    s = _scale(scale, K)
    cup = cu.ctypes.data_as(_I)

    def run(b, e):
        lib.gdn_oracle_fwd(N, cup, H, HV, K, V, s, int(use_l2norm), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht), b, e)

    _parallel(N * HV, run, threads)
    return o, ht


def bwd(q, k, v, g, beta, cu_seqlens, d_o, d_ht=None, scale=None, h0=None, use_l2norm=True,
        threads=None):
    """Per-token backward.  Returns dict dq, dk [T,H,K], dv [T,HV,V], dg, dbeta [T,HV], dh0."""
    lib = _load()
    q, k, v, g, beta, h0, d_o, d_ht = map(_f64, (q, k, v, g, beta, h0, d_o, d_ht))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, H, HV, K, V, N = _shapes(q, v, cu)
    s = _scale(scale, K)
    dq_part = np.zeros((T, HV, K))
    dk_part = np.zeros((T, HV, K))
    dv = np.zeros((T, HV, V))
    dg = np.zeros((T, HV))
    dbeta = np.zeros((T, HV))
    dh0 = np.zeros((N, HV, K, V))
    cup = cu.ctypes.data_as(_I)

    def run(b, e):
        lib.gdn_oracle_bwd(N, cup, H, HV, K, V, s, int(use_l2norm), _ptr(q), _ptr(k), _ptr(v),
                           _ptr(g), _ptr(beta), _ptr(h0), _ptr(d_o), _ptr(d_ht), _ptr(dq_part),
                           _ptr(dk_part), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), b, e)

    _parallel(N * HV, run, threads)
    r = HV // H
    # gradients of q and k: fixed-order sum over the r value heads of each key head
    dq = dq_part.reshape(T, H, r, K).sum(axis=2)
    dk = dk_part.reshape(T, H, r, K).sum(axis=2)
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)


def fwd_chunked(q, k, v, g, beta, cu_seqlens, chunk, scale=None, h0=None, use_l2norm=True,
                want_chunks=False, threads=None):
    """Chunked WY forward at any chunk size.  Returns dict o, ht (and h_chunks, v_new)."""
    lib = _load()
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, H, HV, K, V, N = _shapes(q, v, cu)
    s = _scale(scale, K)
    o = np.zeros((T, HV, V))
    ht = np.zeros((N, HV, K, V))
    nchunks = int(sum((int(cu[i + 1] - cu[i]) + chunk - 1) // chunk for i in range(N)))
    hc = np.zeros((nchunks, HV, K, V)) if want_chunks else None
    vn = np.zeros((T, HV, V)) if want_chunks else None
    cup = cu.ctypes.data_as(_I)

    def run(b, e):
        lib.gdn_oracle_fwd_chunked(N, cup, H, HV, K, V, s, int(use_l2norm), int(chunk), _ptr(q),
                                   _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                                   _ptr(ht), _ptr(hc), _ptr(vn), b, e)

    _parallel(N * HV, run, threads)
    out = dict(o=o, ht=ht)
    if want_chunks:
        out.update(h_chunks=hc, v_new=vn)
    return out


def decode(q, k, v, g, beta, pool, state_indices, scale=None, use_l2norm=True, threads=None):
    """Decode step.  pool [num_slots,HV,V,K] is copied, updated and returned with o.

    Returns (o [B,HV,V], new_pool, n_out_of_range)."""
    lib = _load()
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    pool = np.array(pool, dtype=np.float64, copy=True, order="C")
    idx = np.ascontiguousarray(np.asarray(state_indices, dtype=np.int32))
    B, H, K = q.shape
    _, HV, V = v.shape
    s = _scale(scale, K)
    o = np.zeros((B, HV, V))
    bad = [0]
    lock = threading.Lock()

    def run(b, e):
        n = lib.gdn_oracle_decode(B, H, HV, K, V, s, int(use_l2norm), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(g), _ptr(beta), _ptr(pool), pool.shape[0],
                                  idx.ctypes.data_as(_I), _ptr(o), b, e)
        with lock:
            bad[0] += n

    # rows of one slot must not run on two threads; repeated indices are a caller error
    _parallel(B * HV, run, threads)
    return o, pool, bad[0] // max(HV, 1)


def gate_fwd(a, b, A_log, dt_bias):
    """Fused gating: g = -exp(A_log) softplus(a + dt_bias) (threshold 20), beta = sigmoid(b).
    a, b [..., HV]; A_log, dt_bias [HV].  Returns (g, beta) shaped like a."""
    lib = _load()
    a, b, A_log, dt_bias = map(_f64, (a, b, A_log, dt_bias))
    HV = a.shape[-1]
    n = a.size // HV if HV else 0
    g = np.zeros(a.shape)
    beta = np.zeros(a.shape)
    lib.gdn_oracle_gate_fwd(n, HV, _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g), _ptr(beta))
    return g, beta


def gate_bwd(a, b, A_log, dt_bias, dg, dbeta):
    """Backward of gate_fwd.  Returns dict da, db (shaped like a), dA_log, ddt_bias [HV]
    (sums over every row in row order)."""
    lib = _load()
    a, b, A_log, dt_bias, dg, dbeta = map(_f64, (a, b, A_log, dt_bias, dg, dbeta))
    HV = a.shape[-1]
    n = a.size // HV if HV else 0
    da, db = np.zeros(a.shape), np.zeros(a.shape)
    dA, ddt = np.zeros(HV), np.zeros(HV)
    lib.gdn_oracle_gate_bwd(n, HV, _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(dg), _ptr(dbeta),
                            _ptr(da), _ptr(db), _ptr(dA), _ptr(ddt))
    return dict(da=da, db=db, dA_log=dA, ddt_bias=ddt)


def prefill_paged(q, k, v, g, beta, cu_seqlens, pool, state_indices, has_initial_state=None,
                  scale=None, use_l2norm=True, threads=None):
    """Paged chunk prefill ("Replace Qwen3.5 FLA paths with Attention Gym", GDN prefill
    ablation and Paged-state continuity): the forward whose states live in a decode
    pool [num_slots, HV, V, K] (S itself; the chunk call's state is its transpose).
    Sequence n starts from the transpose of pool[idx[n]] when 0 < idx[n] < num_slots and
    has_initial_state[n] is nonzero (or not given), else from zeros; its final state is
    written back, transposed, to every slot 0 < idx[n] < num_slots.

    Returns (o [T,HV,V], new_pool, number of indices >= num_slots)."""
    pool = np.array(pool, dtype=np.float64, copy=True, order="C")
    idx = np.asarray(state_indices, dtype=np.int64)
    cu = np.asarray(cu_seqlens)
    N = len(cu) - 1
    slots, HV, V, K = pool.shape
    transpose = _load().gdn_oracle_get_mutation() != 10
    h0 = np.zeros((N, HV, K, V))
    for n in range(N):
        s = int(idx[n])
        if 0 < s < slots and (has_initial_state is None or has_initial_state[n]):
            h0[n] = pool[s].transpose(0, 2, 1) if transpose else pool[s]
    o, ht = fwd(q, k, v, g, beta, cu, scale=scale, h0=h0, use_l2norm=use_l2norm, threads=threads)
    for n in range(N):
        s = int(idx[n])
        if 0 < s < slots:
            pool[s] = ht[n].transpose(0, 2, 1) if transpose else ht[n]
    return o, pool, int((idx >= slots).sum())
