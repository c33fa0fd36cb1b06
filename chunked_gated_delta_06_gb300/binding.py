"""ctypes binding of libgdn (include/gdn.h): argument marshalling only.

The functions named like the C entry points (``gdn_chunk_fwd`` ...) forward raw
pointers and sizes.  ``chunk_fwd`` / ``chunk_bwd`` / ``decode_step`` take torch
CUDA tensors, allocate outputs and scratch with torch (plumbing) and call the
C entry points on the current torch stream.  Every step of the computation runs
in libgdn's CUDA kernels; there is no other path.  If libgdn.so is missing the
first call raises, telling the user to build it.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "gdn.h")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE_TOO_SMALL, GDN_ERR_CUDA = range(5)
GDN_DTYPE_BF16, GDN_DTYPE_F32 = 0, 1
GDN_DEVICE_CU_SEQLENS_MISMATCH, GDN_DEVICE_WAIT_TIMEOUT, GDN_DEVICE_INDEX_OUT_OF_RANGE = 1, 2, 4


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


class GdnKernelTimer(ctypes.Structure):
    _fields_ = [
        ("capacity", ctypes.c_int32),
        ("count", ctypes.c_int32),
        ("start_events", ctypes.POINTER(ctypes.c_void_p)),
        ("stop_events", ctypes.POINTER(ctypes.c_void_p)),
        ("kernel_ids", ctypes.POINTER(ctypes.c_int32)),
    ]


class GdnProblem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("num_k_heads", ctypes.c_int32),
        ("num_v_heads", ctypes.c_int32),
        ("head_dim_k", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("beta_dtype", ctypes.c_int32),
        ("cu_seqlens_host", ctypes.POINTER(ctypes.c_int32)),
        ("cu_seqlens_dev", ctypes.c_void_p),
        ("device_status", ctypes.c_void_p),
        ("scan_segment_chunks", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t


def lib():
    """Load libgdn.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libgdn.so not found at %s: build it with "
                                   "`python -m chunked_gated_delta_06_gb300.build`" % LIB_PATH)
            _lib = load_library(LIB_PATH)
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Route every call of this module through another build of the library (the
    bounds-checked libgdn_checked.so, say) inside the `with` block."""
    global _lib
    other = load_library(path)
    with _lock:
        saved, _lib = _lib, other
    try:
        yield other
    finally:
        with _lock:
            _lib = saved


def load_library(path):
    """ctypes handle of a build of libgdn with every entry point's signature set."""
    L = ctypes.CDLL(path)
    P = ctypes.POINTER(GdnProblem)
    L.gdn_status_string.argtypes = [ctypes.c_int]
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_chunk_saved_bytes.argtypes = [P]
    L.gdn_chunk_saved_bytes.restype = _sz
    L.gdn_chunk_scan_plan.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.gdn_chunk_scan_plan.restype = ctypes.c_int
    L.gdn_chunk_workspace_bytes.argtypes = [P, ctypes.c_int]
    L.gdn_chunk_workspace_bytes.restype = _sz
    L.gdn_chunk_fwd.argtypes = [P] + [_vp] * 10 + [_sz, _vp]
    L.gdn_chunk_fwd.restype = ctypes.c_int
    L.gdn_chunk_bwd.argtypes = [P] + [_vp] * 16 + [_sz, _vp]
    L.gdn_chunk_bwd.restype = ctypes.c_int
    L.gdn_decode_step.argtypes = ([ctypes.c_int32] * 5 + [ctypes.c_float] + [_vp] * 6
                                  + [ctypes.c_int32] + [_vp] * 3 + [_vp])
    L.gdn_decode_step.restype = ctypes.c_int
    T = ctypes.POINTER(GdnKernelTimer)
    L.gdn_chunk_fwd_timed.argtypes = [P] + [_vp] * 10 + [_sz, _vp, T]
    L.gdn_chunk_fwd_timed.restype = ctypes.c_int
    L.gdn_chunk_bwd_timed.argtypes = [P] + [_vp] * 16 + [_sz, _vp, T]
    L.gdn_chunk_bwd_timed.restype = ctypes.c_int
    L.gdn_decode_step_timed.argtypes = L.gdn_decode_step.argtypes + [T]
    L.gdn_decode_step_timed.restype = ctypes.c_int
    L.gdn_chunk_fwd_gated.argtypes = [P] + [_vp] * 12 + [_sz, _vp]
    L.gdn_chunk_fwd_gated.restype = ctypes.c_int
    L.gdn_chunk_bwd_gated.argtypes = [P] + [_vp] * 20 + [_sz, _vp]
    L.gdn_chunk_bwd_gated.restype = ctypes.c_int
    L.gdn_decode_step_gated.argtypes = ([ctypes.c_int32] * 5 + [ctypes.c_float] + [_vp] * 8
                                        + [ctypes.c_int32] + [_vp] * 3 + [_vp])
    L.gdn_decode_step_gated.restype = ctypes.c_int
    L.gdn_chunk_prefill_paged.argtypes = [P] + [_vp] * 6 + [ctypes.c_int32] + [_vp] * 5 + [_sz, _vp]
    L.gdn_chunk_prefill_paged.restype = ctypes.c_int
    L.gdn_chunk_fwd_noalloc.argtypes = [P] + [_vp] * 8 + [_vp]
    L.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
    L.gdn_check_indices.argtypes = [_vp, ctypes.c_int32, ctypes.c_int32, _vp]
    L.gdn_check_indices.restype = ctypes.c_int
    L.gdn_selftest_bounded_wait.argtypes = [_vp, ctypes.c_uint64, _vp]
    L.gdn_selftest_bounded_wait.restype = ctypes.c_int
    L.gdn_kernel_name.argtypes = [ctypes.c_int32]
    L.gdn_kernel_name.restype = ctypes.c_char_p
    return L


def header_functions() -> list[str]:
    """Names of the functions include/gdn.h declares."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(gdn_\w+)\s*\(", txt, re.M)))


def status_string(s: int) -> str:
    return lib().gdn_status_string(int(s)).decode()


def kernel_name(i: int) -> str:
    return lib().gdn_kernel_name(int(i)).decode()


class KernelTimer:
    """Event pairs the *_timed entry points record around each kernel launch."""

    def __init__(self, capacity: int = 64):
        import torch
        self.capacity = capacity
        self.starts = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        self.stops = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.starts + self.stops:
            e.record()  # materialise the CUDA events
        torch.cuda.synchronize()
        self._sa = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.starts])
        self._so = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.stops])
        self._ids = (ctypes.c_int32 * capacity)()
        self.struct = GdnKernelTimer(capacity, 0, self._sa, self._so, self._ids)

    def reset(self):
        self.struct.count = 0

    def records(self):
        """[(kernel name, milliseconds)] of the launches recorded since reset (synchronises)."""
        import torch
        torch.cuda.synchronize()
        return [(kernel_name(self._ids[i]), self.starts[i].elapsed_time(self.stops[i]))
                for i in range(self.struct.count)]


# ----------------------------------------------------------------------------- raw entry points
def make_problem(cu_host, H, HV, K=128, V=128, scale=0.0, cu_dev_ptr=0, beta_dtype=GDN_DTYPE_BF16,
                 device_status_ptr=0, scan_segment_chunks=0):
    """Build a GdnProblem; returns (problem, keepalive) -- keep both alive during the call.
    device_status_ptr: a device int32 the kernels OR GDN_DEVICE_* bits into (0: none);
    scan_segment_chunks: 0 = the library's scan plan, -1 = never split, L > 0 = force L."""
    cu = np.ascontiguousarray(np.asarray(cu_host, dtype=np.int32))
    p = GdnProblem()
    p.num_seqs = len(cu) - 1
    p.total_tokens = int(cu[-1]) if len(cu) else 0
    p.num_k_heads, p.num_v_heads, p.head_dim_k, p.head_dim_v = H, HV, K, V
    p.scale = float(scale)
    p.beta_dtype = int(beta_dtype)
    p.cu_seqlens_host = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if len(cu) else None
    p.cu_seqlens_dev = cu_dev_ptr or None
    p.device_status = device_status_ptr or None
    p.scan_segment_chunks = int(scan_segment_chunks)
    return p, cu


def gdn_chunk_saved_bytes(p: GdnProblem) -> int:
    return int(lib().gdn_chunk_saved_bytes(ctypes.byref(p)))


def gdn_chunk_scan_plan(p: GdnProblem):
    """(status, seg_len, num_segments) of the forward state scan of a problem."""
    sl, ns = ctypes.c_int32(), ctypes.c_int32()
    st = int(lib().gdn_chunk_scan_plan(ctypes.byref(p), ctypes.byref(sl), ctypes.byref(ns)))
    return st, int(sl.value), int(ns.value)


def gdn_chunk_workspace_bytes(p: GdnProblem, for_backward: int) -> int:
    return int(lib().gdn_chunk_workspace_bytes(ctypes.byref(p), int(for_backward)))


def gdn_chunk_fwd(p, q, k, v, g, beta, initial_state, o, final_state, saved, workspace, ws_bytes,
                  stream, timer=None) -> int:
    if timer is not None:
        return int(lib().gdn_chunk_fwd_timed(ctypes.byref(p), q, k, v, g, beta, initial_state, o,
                                             final_state, saved, workspace, ws_bytes, stream,
                                             ctypes.byref(timer.struct)))
    return int(lib().gdn_chunk_fwd(ctypes.byref(p), q, k, v, g, beta, initial_state, o,
                                   final_state, saved, workspace, ws_bytes, stream))


def gdn_chunk_fwd_noalloc(p, q, k, v, g, beta, initial_state, o, final_state, stream) -> int:
    return int(lib().gdn_chunk_fwd_noalloc(ctypes.byref(p), q, k, v, g, beta, initial_state, o,
                                           final_state, stream))


def gdn_chunk_bwd(p, q, k, v, g, beta, initial_state, saved, d_o, d_final_state, dq, dk, dv, dg,
                  dbeta, dh0, workspace, ws_bytes, stream, timer=None) -> int:
    if timer is not None:
        return int(lib().gdn_chunk_bwd_timed(ctypes.byref(p), q, k, v, g, beta, initial_state,
                                             saved, d_o, d_final_state, dq, dk, dv, dg, dbeta,
                                             dh0, workspace, ws_bytes, stream,
                                             ctypes.byref(timer.struct)))
    return int(lib().gdn_chunk_bwd(ctypes.byref(p), q, k, v, g, beta, initial_state, saved, d_o,
                                   d_final_state, dq, dk, dv, dg, dbeta, dh0, workspace, ws_bytes,
                                   stream))


def gdn_chunk_prefill_paged(p, q, k, v, g, beta, state_pool, num_slots, state_indices,
                            has_initial_state, o, device_status, workspace, ws_bytes, stream) -> int:
    return int(lib().gdn_chunk_prefill_paged(ctypes.byref(p), q, k, v, g, beta, state_pool,
                                             num_slots, state_indices, has_initial_state, o,
                                             device_status, workspace, ws_bytes, stream))


def gdn_chunk_fwd_gated(p, q, k, v, a, b, A_log, dt_bias, initial_state, o, final_state, saved,
                        workspace, ws_bytes, stream) -> int:
    return int(lib().gdn_chunk_fwd_gated(ctypes.byref(p), q, k, v, a, b, A_log, dt_bias,
                                         initial_state, o, final_state, saved, workspace, ws_bytes,
                                         stream))


def gdn_chunk_bwd_gated(p, q, k, v, a, b, A_log, dt_bias, initial_state, saved, d_o, d_final_state,
                        dq, dk, dv, da, db, dA_log, ddt_bias, dh0, workspace, ws_bytes,
                        stream) -> int:
    return int(lib().gdn_chunk_bwd_gated(ctypes.byref(p), q, k, v, a, b, A_log, dt_bias,
                                         initial_state, saved, d_o, d_final_state, dq, dk, dv, da,
                                         db, dA_log, ddt_bias, dh0, workspace, ws_bytes, stream))


def gdn_decode_step_gated(batch, H, HV, K, V, scale, q, k, v, a, b, A_log, dt_bias, state_pool,
                          num_slots, state_indices, o, device_status, stream) -> int:
    return int(lib().gdn_decode_step_gated(batch, H, HV, K, V, scale, q, k, v, a, b, A_log,
                                           dt_bias, state_pool, num_slots, state_indices, o,
                                           device_status, stream))


def gdn_decode_step(batch, H, HV, K, V, scale, q, k, v, g, beta, state_pool, num_slots,
                    state_indices, o, device_status, stream, timer=None) -> int:
    if timer is not None:
        return int(lib().gdn_decode_step_timed(batch, H, HV, K, V, scale, q, k, v, g, beta,
                                               state_pool, num_slots, state_indices, o,
                                               device_status, stream, ctypes.byref(timer.struct)))
    return int(lib().gdn_decode_step(batch, H, HV, K, V, scale, q, k, v, g, beta, state_pool,
                                     num_slots, state_indices, o, device_status, stream))


def gdn_selftest_bounded_wait(device_status, limit_ns, stream) -> int:
    return int(lib().gdn_selftest_bounded_wait(device_status, int(limit_ns), stream))


def gdn_check_indices(state_indices, batch, num_slots, bad_row) -> int:
    return int(lib().gdn_check_indices(state_indices, batch, num_slots, bad_row))


def check_indices(state_indices, num_slots):
    """gdn_check_indices on a host array (numpy, list or CPU tensor) of decode slot
    indices.  Returns -1 when every active (> 0) index is < num_slots and unique,
    else the first offending row."""
    idx = np.ascontiguousarray(
        state_indices.numpy() if hasattr(state_indices, "numpy") else state_indices, dtype=np.int32)
    bad = ctypes.c_int32(-1)
    st = gdn_check_indices(idx.ctypes.data if idx.size else None, idx.size, int(num_slots),
                           ctypes.byref(bad))
    if st != GDN_OK and bad.value < 0:
        raise GdnError(st, "gdn_check_indices")
    return bad.value


# ----------------------------------------------------------------------------- torch helpers
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(st, where):
    if st != GDN_OK:
        raise GdnError(st, where)


def beta_dtype_of(beta):
    """GDN_DTYPE_* of a torch beta tensor (bf16 or fp32)."""
    import torch
    if beta.dtype == torch.bfloat16:
        return GDN_DTYPE_BF16
    if beta.dtype == torch.float32:
        return GDN_DTYPE_F32
    raise TypeError("beta must be bfloat16 or float32, not %s" % beta.dtype)


class ChunkContext:
    """Problem description plus the saved buffer of one forward (for the backward);
    saved stays None after a forward without for_backward, and the backward then
    runs in recompute-state mode."""

    def __init__(self, cu_host, cu_dev, H, HV, scale, beta_dtype=GDN_DTYPE_BF16, device_status=None,
                 scan_segment_chunks=0):
        self.cu_host = np.ascontiguousarray(np.asarray(cu_host, dtype=np.int32))
        self.cu_dev = cu_dev
        self.H, self.HV, self.scale = H, HV, scale
        self.device_status = device_status
        self.problem, self._keep = make_problem(self.cu_host, H, HV, scale=scale or 0.0,
                                                cu_dev_ptr=cu_dev.data_ptr(), beta_dtype=beta_dtype,
                                                device_status_ptr=_ptr(device_status) or 0,
                                                scan_segment_chunks=scan_segment_chunks)
        self.saved = None


def chunk_fwd(q, k, v, g, beta, cu_host, cu_dev, scale=None, initial_state=None,
              output_final_state=True, for_backward=False, workspace=None, device_status=None,
              scan_segment_chunks=0):
    """gdn_chunk_fwd on torch tensors.  Returns (o, final_state or None, ctx).
    device_status: an int32 device tensor the kernels OR GDN_DEVICE_* bits into (the
    backward of ctx uses it too); scan_segment_chunks: the problem field of that name."""
    import torch
    T, H, K = q.shape
    HV = v.shape[1]
    ctx = ChunkContext(cu_host, cu_dev, H, HV, scale, beta_dtype_of(beta), device_status,
                       scan_segment_chunks)
    p = ctx.problem
    N = p.num_seqs
    dev = q.device
    o = torch.empty((T, HV, v.shape[2]), dtype=torch.bfloat16, device=dev)
    ht = torch.empty((N, HV, K, v.shape[2]), dtype=torch.float32, device=dev) if output_final_state else None
    nws = gdn_chunk_workspace_bytes(p, 0)
    if nws == 0:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_chunk_workspace_bytes")
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    saved = None
    if for_backward:
        saved = torch.empty(gdn_chunk_saved_bytes(p), dtype=torch.uint8, device=dev)
    st = gdn_chunk_fwd(p, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                       _ptr(o), _ptr(ht), _ptr(saved), _ptr(workspace), workspace.numel(),
                       _stream())
    _check(st, "gdn_chunk_fwd")
    ctx.saved = saved
    ctx.workspace = workspace
    return o, ht, ctx


def chunk_bwd(ctx, q, k, v, g, beta, d_o, d_final_state=None, initial_state=None,
              want_dh0=True, workspace=None):
    """gdn_chunk_bwd on torch tensors.  Returns dict dq, dk, dv, dg, dbeta, dh0.
    Without a saved buffer in ctx (forward run without for_backward) this is the
    recompute-state mode: the call rebuilds the forward's tensors itself."""
    import torch
    T, H, K = q.shape
    HV = v.shape[1]
    p = ctx.problem
    dev = q.device
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty((T, HV), dtype=torch.float32, device=dev)
    dbeta = torch.empty((T, HV), dtype=beta.dtype, device=dev)
    dh0 = torch.empty((p.num_seqs, HV, K, v.shape[2]), dtype=torch.float32, device=dev) if want_dh0 else None
    nws = gdn_chunk_workspace_bytes(p, 1 if ctx.saved is not None else 2)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    st = gdn_chunk_bwd(p, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                       _ptr(ctx.saved), _ptr(d_o), _ptr(d_final_state), _ptr(dq), _ptr(dk),
                       _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(workspace),
                       workspace.numel(), _stream())
    _check(st, "gdn_chunk_bwd")
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)


def decode_step(q, k, v, g, beta, state_pool, state_indices, scale=None, device_status=None):
    """gdn_decode_step on torch tensors (state_pool updated in place).  Returns o."""
    import torch
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    o = torch.empty((B, HV, V), dtype=torch.bfloat16, device=q.device)
    st = gdn_decode_step(B, H, HV, K, V, float(scale or 0.0), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                         _ptr(beta), _ptr(state_pool), state_pool.shape[0], _ptr(state_indices),
                         _ptr(o), _ptr(device_status), _stream())
    _check(st, "gdn_decode_step")
    return o


def chunk_fwd_gated(q, k, v, a, b, A_log, dt_bias, cu_host, cu_dev, scale=None, initial_state=None,
                    output_final_state=True, for_backward=False, workspace=None, device_status=None):
    """gdn_chunk_fwd_gated on torch tensors (g and beta from the fused gate).
    Returns (o, final_state or None, ctx); ctx feeds chunk_bwd_gated."""
    import torch
    T, H, K = q.shape
    HV = v.shape[1]
    ctx = ChunkContext(cu_host, cu_dev, H, HV, scale, device_status=device_status)
    p = ctx.problem
    dev = q.device
    o = torch.empty((T, HV, v.shape[2]), dtype=torch.bfloat16, device=dev)
    ht = (torch.empty((p.num_seqs, HV, K, v.shape[2]), dtype=torch.float32, device=dev)
          if output_final_state else None)
    nws = gdn_chunk_workspace_bytes(p, 0)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    saved = torch.empty(gdn_chunk_saved_bytes(p), dtype=torch.uint8, device=dev) if for_backward else None
    st = gdn_chunk_fwd_gated(p, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                             _ptr(dt_bias), _ptr(initial_state), _ptr(o), _ptr(ht), _ptr(saved),
                             _ptr(workspace), workspace.numel(), _stream())
    _check(st, "gdn_chunk_fwd_gated")
    ctx.saved = saved
    ctx.workspace = workspace
    return o, ht, ctx


def chunk_bwd_gated(ctx, q, k, v, a, b, A_log, dt_bias, d_o, d_final_state=None,
                    initial_state=None, want_dh0=True, workspace=None):
    """gdn_chunk_bwd_gated on torch tensors.  Returns dict dq, dk, dv, da, db, dA_log,
    ddt_bias, dh0 (recompute-state mode when ctx holds no saved buffer)."""
    import torch
    T, H, K = q.shape
    HV = v.shape[1]
    p = ctx.problem
    dev = q.device
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    da = torch.empty((T, HV), dtype=torch.bfloat16, device=dev)
    db = torch.empty((T, HV), dtype=torch.bfloat16, device=dev)
    dA_log = torch.empty((HV,), dtype=torch.float32, device=dev)
    ddt_bias = torch.empty((HV,), dtype=torch.float32, device=dev)
    dh0 = (torch.empty((p.num_seqs, HV, K, v.shape[2]), dtype=torch.float32, device=dev)
           if want_dh0 else None)
    nws = gdn_chunk_workspace_bytes(p, 1 if ctx.saved is not None else 2)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
    st = gdn_chunk_bwd_gated(p, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(A_log),
                             _ptr(dt_bias), _ptr(initial_state), _ptr(ctx.saved), _ptr(d_o),
                             _ptr(d_final_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da), _ptr(db),
                             _ptr(dA_log), _ptr(ddt_bias), _ptr(dh0), _ptr(workspace),
                             workspace.numel(), _stream())
    _check(st, "gdn_chunk_bwd_gated")
    return dict(dq=dq, dk=dk, dv=dv, da=da, db=db, dA_log=dA_log, ddt_bias=ddt_bias, dh0=dh0)


def decode_step_gated(q, k, v, a, b, A_log, dt_bias, state_pool, state_indices, scale=None,
                      device_status=None):
    """gdn_decode_step_gated on torch tensors (state_pool updated in place).  Returns o."""
    import torch
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    o = torch.empty((B, HV, V), dtype=torch.bfloat16, device=q.device)
    st = gdn_decode_step_gated(B, H, HV, K, V, float(scale or 0.0), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(state_pool),
                               state_pool.shape[0], _ptr(state_indices), _ptr(o),
                               _ptr(device_status), _stream())
    _check(st, "gdn_decode_step_gated")
    return o


def chunk_prefill_paged(q, k, v, g, beta, cu_host, cu_dev, state_pool, state_indices,
                        has_initial_state=None, scale=None, device_status=None, workspace=None,
                        problem_status=None):
    """gdn_chunk_prefill_paged on torch tensors: sequence n starts from pool slot
    state_indices[n] (zeros when the slot is <= 0 or has_initial_state[n] == 0) and its
    final state is written back to that slot in place.  Returns o.  device_status is the
    call's slot-status word; problem_status the kernels' status word of gdn_problem."""
    import torch
    T, H, K = q.shape
    HV = v.shape[1]
    ctx = ChunkContext(cu_host, cu_dev, H, HV, scale, beta_dtype_of(beta), device_status=problem_status)
    p = ctx.problem
    o = torch.empty((T, HV, v.shape[2]), dtype=torch.bfloat16, device=q.device)
    nws = gdn_chunk_workspace_bytes(p, 0)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=q.device)
    st = gdn_chunk_prefill_paged(p, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool),
                                 state_pool.shape[0], _ptr(state_indices), _ptr(has_initial_state),
                                 _ptr(o), _ptr(device_status), _ptr(workspace), workspace.numel(),
                                 _stream())
    _check(st, "gdn_chunk_prefill_paged")
    return o
