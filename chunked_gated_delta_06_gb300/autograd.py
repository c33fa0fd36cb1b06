"""The chunk path as a differentiable PyTorch function, with the call shape of the
pages' op ("[Cake 1/13] gdn: chunked gated delta rule, det and fast, with KCP and
FLA-CP", API and flags: chunk_gated_delta_rule(q, k, v, g, beta, scale,
initial_state, output_final_state, cu_seqlens, cu_seqlens_cpu, ...), packed B = 1,
in-kernel q/k L2 norm, the recompute-state option).

Argument marshalling only: the forward calls gdn_chunk_fwd and the backward
gdn_chunk_bwd through the C ABI (binding.chunk_fwd / chunk_bwd).
"""
from __future__ import annotations

import numpy as np

from . import binding


def _function():
    import torch

    class ChunkGatedDeltaRule(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, g, beta, initial_state, cu_host, cu_dev, scale, output_final_state,
                    recompute_state):
            ctx.set_materialize_grads(False)
            o, ht, c = binding.chunk_fwd(q, k, v, g, beta, cu_host, cu_dev, scale=scale,
                                         initial_state=initial_state,
                                         output_final_state=output_final_state,
                                         for_backward=not recompute_state)
            ctx.gdn = c
            ctx.has_h0 = initial_state is not None
            ctx.save_for_backward(q, k, v, g, beta, initial_state)
            return o, ht

        @staticmethod
        def backward(ctx, d_o, d_ht):
            q, k, v, g, beta, h0 = ctx.saved_tensors
            if d_o is None:
                d_o = torch.zeros((q.shape[0], v.shape[1], v.shape[2]), dtype=torch.bfloat16,
                                  device=q.device)
            gr = binding.chunk_bwd(ctx.gdn, q, k, v, g, beta, d_o.to(torch.bfloat16).contiguous(),
                                   d_final_state=None if d_ht is None else d_ht.float().contiguous(),
                                   initial_state=h0, want_dh0=ctx.has_h0)
            return (gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], gr["dh0"], None, None, None,
                    None, None)

    return ChunkGatedDeltaRule


_FN = None


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                           cu_seqlens=None, cu_seqlens_cpu=None, recompute_state=False):
    """o [B=1, T, HV, V] (and the final state [N, HV, K, V] when output_final_state).

    q, k: bf16 [1, T, H, 128] or [T, H, 128]; v: bf16 [.., T, HV, 128]; g: fp32 [.., T, HV];
    beta: bf16 or fp32 [.., T, HV]; initial_state: fp32 [N, HV, 128, 128] or None;
    cu_seqlens: int32 device [N + 1] (default: one sequence), cu_seqlens_cpu: the same
    boundaries on the host (read from cu_seqlens when not given: one device-to-host copy).
    recompute_state: the backward rebuilds w, u, h and v_new instead of keeping them."""
    import torch
    global _FN
    if _FN is None:
        _FN = _function()
    batched = q.dim() == 4
    if batched:
        if q.shape[0] != 1:
            raise ValueError("packed sequences only: B must be 1 (use cu_seqlens)")
        q, k, v, g, beta = q[0], k[0], v[0], g[0], beta[0]
    T = q.shape[0]
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    if cu_seqlens_cpu is None:
        cu_seqlens_cpu = cu_seqlens.cpu()
    cu_host = np.asarray(cu_seqlens_cpu.cpu() if hasattr(cu_seqlens_cpu, "cpu") else cu_seqlens_cpu,
                         dtype=np.int32)
    o, ht = _FN.apply(q.contiguous(), k.contiguous(), v.contiguous(), g.contiguous(), beta.contiguous(),
                      initial_state, cu_host, cu_seqlens.to(torch.int32).contiguous(), scale,
                      output_final_state, recompute_state)
    if batched:
        o = o.unsqueeze(0)
    return o, ht
