"""Host-only checks of the C ABI: the library loads, exports every function
include/gdn.h declares, sizes its buffers as documented and rejects invalid
arguments before any CUDA call (no GPU needed: no call here reaches a launch)."""
import ctypes

import numpy as np
import pytest

import chunked_gated_delta_06_gb300 as gdn
from chunked_gated_delta_06_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_library_exports_every_declared_function(lib):
    names = binding.header_functions()
    assert {"gdn_chunk_fwd", "gdn_chunk_bwd", "gdn_decode_step", "gdn_chunk_saved_bytes",
            "gdn_chunk_workspace_bytes", "gdn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_bounds_checked_build_exports_the_same_functions():
    # nvcc -DGDN_CHECKED: the same entry points; its kernels only add range checks
    path = build.build(checked=True)
    checked = binding.load_library(path)
    for n in binding.header_functions():
        assert hasattr(checked, n), n
    p, keep = _problem([0, 5])
    assert checked.gdn_chunk_workspace_bytes(ctypes.byref(p), 1) == binding.lib().gdn_chunk_workspace_bytes(
        ctypes.byref(p), 1)


def test_status_strings(lib):
    for s in range(5):
        assert gdn.status_string(s).startswith("GDN_")
    assert "unknown" in gdn.status_string(99)


def _problem(cu, H=2, HV=4, K=128, V=128, scale=0.0, dev=0x1000, beta_dtype=0):
    return binding.make_problem(cu, H, HV, K, V, scale, cu_dev_ptr=dev, beta_dtype=beta_dtype)


def test_saved_and_workspace_sizes(lib):
    cu = [0, 1, 64, 200]  # chunks: 1 + 1 + 3 = 5
    p, keep = _problem(cu)
    T, H, HV, C = 200, 2, 4, 5
    D = 128

    def al(x):
        return (x + 255) // 256 * 256
    # per-chunk h (bf16), v_new (bf16 per token), w^T per chunk (bf16 [C, HV, 128, 64]),
    # the WY inverses (bf16 [C, HV, 64, 64]), r_q, r_k (per key head), G (per value head),
    # the scans' scalar records (fp32 [C, HV, 132]: 64 + 64 per-token scalars, e^{G_L}, pad)
    saved = (al(C * HV * D * D * 2) + al(T * HV * D * 2) + al(C * HV * D * 64 * 2)
             + al(C * HV * 64 * 64 * 2) + al(T * H * 4) + al(T * H * 4) + al(T * HV * 4)
             + al(C * HV * 132 * 4))
    assert gdn.gdn_chunk_saved_bytes(p) == saved
    fwd_ws = gdn.gdn_chunk_workspace_bytes(p, 0)
    assert fwd_ws >= saved + C * HV * D * 64 * 2  # and u^T per chunk
    bwd_ws = gdn.gdn_chunk_workspace_bytes(p, 1)
    # dv_loc, dv_new, dW (bf16 per value head); the key heads' summed dkhat terms (bf16);
    # per-chunk dh (bf16)
    assert bwd_ws >= 3 * T * HV * D * 2 + T * H * D * 2 + C * HV * D * D * 2
    # recompute-state mode: the backward scratch followed by the saved tensors
    assert gdn.gdn_chunk_workspace_bytes(p, 2) == bwd_ws + saved
    assert gdn.gdn_chunk_workspace_bytes(p, 3) == 0
    assert gdn.gdn_chunk_workspace_bytes(p, -1) == 0
    # the beta dtype changes no buffer size (beta and dbeta are the caller's)
    p32, keep32 = _problem(cu, beta_dtype=binding.GDN_DTYPE_F32)
    assert gdn.gdn_chunk_saved_bytes(p32) == saved
    assert gdn.gdn_chunk_workspace_bytes(p32, 2) == bwd_ws + saved


@pytest.mark.parametrize("mut, status", [
    (dict(K=64), binding.GDN_ERR_UNSUPPORTED),
    (dict(V=256), binding.GDN_ERR_UNSUPPORTED),
    (dict(H=3, HV=4), binding.GDN_ERR_UNSUPPORTED),
    (dict(cu=[0, 5, 3]), binding.GDN_ERR_INVALID_ARG),
    (dict(cu=[1, 5]), binding.GDN_ERR_INVALID_ARG),
    (dict(dev=0), binding.GDN_ERR_INVALID_ARG),
    (dict(beta_dtype=2), binding.GDN_ERR_INVALID_ARG),
    (dict(beta_dtype=-1), binding.GDN_ERR_INVALID_ARG),
])
def test_invalid_problems_are_rejected_before_any_launch(lib, mut, status):
    kw = dict(cu=[0, 5, 9], H=2, HV=4, K=128, V=128, dev=0x1000)
    kw.update(mut)
    p, keep = _problem(kw.pop("cu"), **kw)
    assert gdn.gdn_chunk_saved_bytes(p) == 0
    assert gdn.gdn_chunk_workspace_bytes(p, 0) == 0
    fake = 0x10000  # never dereferenced: validation fails first
    st = gdn.gdn_chunk_fwd(p, fake, fake, fake, fake, fake, None, fake, None, None, fake, 1 << 40, None)
    assert st == status
    st = gdn.gdn_chunk_bwd(p, fake, fake, fake, fake, fake, None, fake, fake, None, fake, fake, fake,
                           fake, fake, None, fake, 1 << 40, None)
    assert st == status


def test_missing_buffers_are_rejected(lib):
    p, keep = _problem([0, 5])
    fake = 0x10000
    # null q
    assert gdn.gdn_chunk_fwd(p, None, fake, fake, fake, fake, None, fake, None, None, fake, 1 << 40,
                             None) == binding.GDN_ERR_INVALID_ARG
    # misaligned workspace
    assert gdn.gdn_chunk_fwd(p, fake, fake, fake, fake, fake, None, fake, None, None, fake + 16,
                             1 << 40, None) == binding.GDN_ERR_INVALID_ARG
    # workspace too small
    assert gdn.gdn_chunk_fwd(p, fake, fake, fake, fake, fake, None, fake, None, None, fake, 1024,
                             None) == binding.GDN_ERR_WORKSPACE_TOO_SMALL
    # backward without the saved buffer is recompute-state mode: its workspace must also
    # hold the forward's tensors (checked before any launch)
    ws1 = gdn.gdn_chunk_workspace_bytes(p, 1)
    assert gdn.gdn_chunk_bwd(p, fake, fake, fake, fake, fake, None, None, fake, None, fake, fake,
                             fake, fake, fake, None, fake, ws1, None) == binding.GDN_ERR_WORKSPACE_TOO_SMALL
    # fp32 beta must be 4-byte aligned, bf16 beta 2-byte aligned
    p32, keep32 = _problem([0, 5], beta_dtype=binding.GDN_DTYPE_F32)
    assert gdn.gdn_chunk_fwd(p32, fake, fake, fake, fake, fake + 2, None, fake, None, None, fake,
                             1 << 40, None) == binding.GDN_ERR_INVALID_ARG
    assert gdn.gdn_chunk_fwd(p, fake, fake, fake, fake, fake + 1, None, fake, None, None, fake,
                             1 << 40, None) == binding.GDN_ERR_INVALID_ARG
    # null problem
    assert lib.gdn_chunk_saved_bytes(None) == 0


def test_decode_argument_checks(lib):
    fake = 0x10000
    args = dict(batch=4, H=2, HV=4, K=128, V=128, scale=0.0)

    def call(**over):
        a = dict(args); a.update(over)
        return gdn.gdn_decode_step(a["batch"], a["H"], a["HV"], a["K"], a["V"], a["scale"], fake, fake,
                                   fake, fake, fake, a.get("pool", fake), a.get("slots", 8),
                                   a.get("idx", fake), fake, None, None)
    assert call(K=64) == binding.GDN_ERR_UNSUPPORTED
    assert call(H=3) == binding.GDN_ERR_UNSUPPORTED
    assert call(batch=-1) == binding.GDN_ERR_INVALID_ARG
    assert call(slots=0) == binding.GDN_ERR_INVALID_ARG
    assert call(idx=None) == binding.GDN_ERR_INVALID_ARG
    assert call(pool=fake + 4) == binding.GDN_ERR_INVALID_ARG
    assert call(batch=0) == binding.GDN_OK  # nothing to do, nothing launched


def test_problem_struct_layout_matches_the_header(lib):
    # int32, int64, 4 x int32, float, int32, 2 pointers: offsets as a C compiler lays them
    # out (beta_dtype fills what was the padding before the pointers)
    P = binding.GdnProblem
    assert P.total_tokens.offset == 8
    assert P.scale.offset == 32
    assert P.beta_dtype.offset == 36
    assert P.cu_seqlens_host.offset == 40
    assert P.cu_seqlens_dev.offset == 48
    assert P.device_status.offset == 56
    assert P.scan_segment_chunks.offset == 64
    assert ctypes.sizeof(P) == 72


def test_gated_calls_check_their_arguments_before_any_launch(lib):
    fake = 0x10000
    p, keep = _problem([0, 5])
    big = 1 << 40

    def fwd(pp=p, a=fake, b=fake, A=fake, dt=fake):
        return gdn.gdn_chunk_fwd_gated(pp, fake, fake, fake, a, b, A, dt, None, fake, None, None,
                                       fake, big, None)

    def bwd(pp=p, a=fake, b=fake, A=fake, dt=fake, da=fake, db=fake, dA=fake, ddt=fake):
        return gdn.gdn_chunk_bwd_gated(pp, fake, fake, fake, a, b, A, dt, None, fake, fake, None,
                                       fake, fake, fake, da, db, dA, ddt, None, fake, big, None)

    assert fwd(A=None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(a=None) == binding.GDN_ERR_INVALID_ARG
    assert fwd(b=fake + 1) == binding.GDN_ERR_INVALID_ARG      # bf16 must be 2-byte aligned
    assert fwd(dt=fake + 2) == binding.GDN_ERR_INVALID_ARG     # fp32 must be 4-byte aligned
    p32, keep32 = _problem([0, 5], beta_dtype=binding.GDN_DTYPE_F32)
    assert fwd(pp=p32) == binding.GDN_ERR_INVALID_ARG          # a and b are bf16
    assert bwd(dA=None) == binding.GDN_ERR_INVALID_ARG
    assert bwd(ddt=None) == binding.GDN_ERR_INVALID_ARG
    assert bwd(da=None) == binding.GDN_ERR_INVALID_ARG
    assert bwd(db=fake + 1) == binding.GDN_ERR_INVALID_ARG
    # the workspace check still comes before any launch
    assert gdn.gdn_chunk_bwd_gated(p, fake, fake, fake, fake, fake, fake, fake, None, fake, fake,
                                   None, fake, fake, fake, fake, fake, fake, fake, None, fake, 1024,
                                   None) == binding.GDN_ERR_WORKSPACE_TOO_SMALL

    def dec(**over):
        a = dict(batch=4, a=fake, b=fake, A=fake, dt=fake)
        a.update(over)
        return gdn.gdn_decode_step_gated(a["batch"], 2, 4, 128, 128, 0.0, fake, fake, fake, a["a"],
                                         a["b"], a["A"], a["dt"], fake, 8, fake, fake, None, None)
    assert dec(a=None) == binding.GDN_ERR_INVALID_ARG
    assert dec(A=None) == binding.GDN_ERR_INVALID_ARG
    assert dec(b=fake + 1) == binding.GDN_ERR_INVALID_ARG
    assert dec(batch=0) == binding.GDN_OK


def test_paged_prefill_checks_its_arguments_before_any_launch(lib):
    fake = 0x10000
    p, keep = _problem([0, 5, 9])

    def call(pool=fake, slots=8, idx=fake, resume=None, status=None, ws=1 << 40):
        return gdn.gdn_chunk_prefill_paged(p, fake, fake, fake, fake, fake, pool, slots, idx, resume,
                                           fake, status, fake, ws, None)
    assert call(pool=None) == binding.GDN_ERR_INVALID_ARG
    assert call(pool=fake + 4) == binding.GDN_ERR_INVALID_ARG
    assert call(slots=0) == binding.GDN_ERR_INVALID_ARG
    assert call(idx=None) == binding.GDN_ERR_INVALID_ARG
    assert call(idx=fake + 2) == binding.GDN_ERR_INVALID_ARG
    assert call(resume=fake + 1) == binding.GDN_ERR_INVALID_ARG
    assert call(ws=1024) == binding.GDN_ERR_WORKSPACE_TOO_SMALL


def test_differentiable_call_takes_packed_batches_only():
    torch = pytest.importorskip("torch")
    assert callable(gdn.chunk_gated_delta_rule)
    x = torch.zeros((2, 4, 1, 128), dtype=torch.bfloat16)
    gb = torch.zeros((2, 4, 1))
    with pytest.raises(ValueError, match="B must be 1"):
        gdn.chunk_gated_delta_rule(x, x, x, gb, gb)


def test_index_check_finds_repeats_and_out_of_range_slots(lib):
    assert gdn.check_indices(np.array([3, 0, -1, 0, 5, 1], np.int32), 6) == -1
    assert gdn.check_indices([], 1) == -1
    assert gdn.check_indices([0, 0, -7], 1) == -1          # null rows may repeat
    assert gdn.check_indices([4, 2, 9, 2, 2], 10) == 3     # later row of the first repeat
    assert gdn.check_indices([4, 2, 10, 2], 10) == 2       # index == num_slots
    assert gdn.check_indices(np.array([63, 64, 127, 128, 64]), 200) == 4  # across bit words
    # the bench's decode batch: 256 draws without repeat from 1..511, some set to 0
    from chunked_gated_delta_06_gb300 import workloads as W
    dw = W.decode_workload(B=256, H=1, HV=1, num_slots=512, seed=3)
    assert gdn.check_indices(dw.state_indices, 512) == -1
    bad = ctypes.c_int32(7)
    assert binding.gdn_check_indices(None, 3, 8, ctypes.byref(bad)) == binding.GDN_ERR_INVALID_ARG
    assert binding.gdn_check_indices(None, 0, 0, None) == binding.GDN_ERR_INVALID_ARG
    assert binding.gdn_check_indices(None, 0, 8, ctypes.byref(bad)) == binding.GDN_OK
    assert bad.value == -1


def test_sizes_at_the_largest_token_count(lib):
    """T = 2^31 - 1 in one sequence: the chunk count and every size are computed
    without overflow (no launch: size queries and the scan plan only)."""
    T = 2**31 - 1
    p, keep = _problem([0, T], H=1, HV=1)
    C = (T + 63) // 64
    saved = gdn.gdn_chunk_saved_bytes(p)
    # h_c (bf16 per chunk), v_new rows (bf16), w^T per chunk (bf16), T per chunk (bf16),
    # r_q, r_k, G (fp32), the scans' scalar records (fp32, 132 per chunk), each rounded up
    # to 256 bytes
    need = (C * 128 * 128 * 2 + T * 128 * 2 + C * 128 * 64 * 2 + C * 64 * 64 * 2 + 3 * T * 4
            + C * 132 * 4)
    assert need <= saved <= need + 8 * 256
    for mode in (0, 1, 2):
        assert gdn.gdn_chunk_workspace_bytes(p, mode) > 0
    st, seg_len, nseg = gdn.gdn_chunk_scan_plan(p)
    assert st == binding.GDN_OK and nseg >= 1
