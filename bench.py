#!/usr/bin/env python
"""Benchmark of the chunked gated delta rule on GB300.

One step = gdn_chunk_fwd (keeping the saved tensors) + gdn_chunk_bwd on the
packed varlen workload (32768 tokens, lengths ~U[1,8192], H=16, HV=32,
K=V=128, fp32 initial state, dh0 out), inputs resident in HBM.  The same JSON
line carries the decode-step bandwidth on the 256-row / [512,32,128,128]
pool workload, the per-kernel roofline of the dominant kernel, an end-to-end
number through host buffers, and the fp64 CPU oracle as a baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica of the workload (no data-path
collective: the (sequence, head) units are independent); the time is the max
over ranks and `value` counts every rank's tokens.
"""
from __future__ import annotations

import argparse
import csv
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

from collections import defaultdict

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd tokens/s (T=32K packed, H=16, HV=32, K=V=128); decode state GB/s"
C, D = 64, 128


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p["bf16_tflops_sustained"]), source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------- algorithmic work
def kernel_work(name, T, H, HV, N, C_total):
    """Algorithmic (flops, bytes) of one launch of a kernel on a problem.

    Flops count the contractions of the chunked form per (token, value head)
    with chunk C = 64, K = V = 128, r = HV / H (masking and padding excluded);
    bytes count the tensors the kernel must read or write once."""
    r = HV // H
    TV = T * HV
    f = dict(
        intra=(2 * C * D / r + 2 * C * D + 2 * C * D + 2 * C * C / 3) * TV,
        state=4 * D * D * TV,
        out=(2 * C * D / r + 2 * C * D + 2 * D * D) * TV,
        dvloc=(2 * C * D / r + 2 * C * D) * TV,
        bstate=6 * D * D * TV,
        bintra_a=(6 * D * D + 8 * C * D) * TV,
        bintra_b=(14 * C * D + 4 * C * C) * TV,
    ).get(name, 0.0)
    bf = 2
    b = dict(
        plan=4 * (N + 1 + 3 * C_total),
        prep=T * H * D * bf * 2 + TV * 4 * 2 + T * H * 8,
        # k, v, G, beta, r_k, r_q in; w^T, u^T, T and the scans' scalar records out
        intra=T * H * D * bf + TV * D * bf + TV * 6 + T * H * 8 + TV * D * bf * 2 + C_total * HV * C * C * 2
        + C_total * HV * 132 * 4,
        state=TV * D * bf * 3 + T * H * D * bf + C_total * HV * D * D * bf + N * HV * D * D * 8
        + C_total * HV * 132 * 4,
        out=T * H * D * bf * 2 + TV * D * bf * 2 + C_total * HV * D * D * bf,
        dvloc=T * H * D * bf * 2 + TV * D * bf * 2,
        bstate=T * H * D * bf * 2 + TV * D * bf * 4 + C_total * HV * D * D * bf + C_total * HV * 132 * 4,
        # q, k; dO, dv_new, v_new in and dW out; dG; h_c, dh_c; dq and the summed dkhat out
        bintra_a=T * H * D * bf * 4 + TV * D * bf * 4 + TV * 4 + C_total * HV * D * D * bf * 2,
        # k and the h / dh' dkhat terms in, dk out; v, dW, dv_new in and dv out; beta, G, dG,
        # dg / dbeta; r_k; T
        bintra_b=T * H * D * bf * 3 + TV * D * bf * 4 + TV * 12 + T * H * 4 + C_total * HV * C * C * 2,
    ).get(name, 0.0)
    return f, b


def step_work(T, H, HV, N, backward=True, h0=True, final_state=True, d_final_state=False):
    """Algorithmic (flops, minimum bytes) of a whole call on a problem.

    Flops: per (token, value head) the forward's contractions of the chunked form,
    4CK/r (K K^T and Q K^T once per key head) + 2C(K + 2V) (w, u, the intra part of o)
    + 6KV (v_new, the state update, the inter part of o) + 2C^2/3 (the triangular
    inverse); the backward counts twice the forward.  Bytes: the call's own inputs
    and outputs, each moved once (q, k, v, g, beta, o; then dO, dq, dk, dv, dg,
    dbeta; the fp32 states), none of the per-chunk intermediates."""
    r = HV // H
    f_fwd = (4 * C * D / r + 2 * C * (D + 2 * D) + 6 * D * D + 2 * C * C / 3) * T * HV
    st = N * HV * D * D * 4
    io = 2 * T * H * D * 2 + T * HV * D * 2 + T * HV * 6          # q, k, v, g, beta
    fwd_b = io + T * HV * D * 2 + st * (h0 + final_state)          # + o, h0, final state
    if not backward:
        return f_fwd, fwd_b
    bwd_b = (io + T * HV * D * 2 + 2 * T * H * D * 2 + T * HV * D * 2 + T * HV * 6
             + st * (h0 + h0 + d_final_state))                      # dO; dq, dk, dv, dg, dbeta; h0, dh0, dht
    return 3 * f_fwd, fwd_b + bwd_b


def step_fractions(flops, nbytes, seconds, peaks):
    """A call against both measured peaks: tensor (sustained bf16) and HBM (copy)."""
    return {"tflops": flops / seconds / 1e12, "gbs": nbytes / seconds / 1e9,
            "tensor_frac": flops / seconds / 1e12 / peaks["bf16_sustained"],
            "hbm_frac": nbytes / seconds / 1e9 / peaks["hbm"],
            "algorithmic_flops": flops, "min_bytes": nbytes}


# kernel name -> source file (the DRAM-traffic record is valid only for the source it was taken on)
KERNEL_SOURCE = {
    "intra": "gdn_intra_tc.cu", "state": "gdn_state_tc.cu", "out": "gdn_out_tc.cu",
    "dvloc": "gdn_out_tc.cu", "bstate": "gdn_bstate_tc.cu", "bintra_a": "gdn_bintra_tc.cu",
    "bintra_b": "gdn_bintra_b_tc.cu", "decode": "gdn_decode.cu", "prep": "gdn_chunk.cu",
    "plan": "gdn_chunk.cu",
}


def _source_hash(kernel):
    import hashlib
    f = KERNEL_SOURCE.get(kernel)
    if not f:
        return None
    path = os.path.join(ROOT, "chunked_gated_delta_06_gb300", "csrc", f)
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def measured_traffic(kernel, units):
    """DRAM bytes per launch from the committed ncu record (profiles/kernel_traffic.json),
    scaled by the work units of this launch; None when the kernel source changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "kernel_traffic.json")) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_sha256_16") != _source_hash(kernel):
        return None
    return rec["bytes_per_unit"] * units


def roofline(kernel, flops, nbytes, seconds, peaks, units):
    """Roofline of one kernel: bound = the resource its algorithmic work needs the
    longest on (tensor at the sustained bf16 peak, HBM at the copy peak)."""
    t_tc = flops / (peaks["bf16_sustained"] * 1e12) if flops else 0.0
    t_hbm = nbytes / (peaks["hbm"] * 1e9) if nbytes else 0.0
    if t_tc >= t_hbm and flops:
        r = {"kernel": kernel, "bound": "tensor", "achieved": flops / seconds / 1e12,
             "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
             "peak_source": "bf16_tflops_sustained (%s)" % peaks["source"],
             "algorithmic_flops": flops}
    else:
        r = {"kernel": kernel, "bound": "hbm", "achieved": nbytes / seconds / 1e9,
             "peak": peaks["hbm"], "unit": "GB/s", "peak_source": "hbm_gbs (%s)" % peaks["source"]}
    r["algorithmic_bytes"] = nbytes
    r["frac"] = r["achieved"] / r["peak"]
    r["traffic"] = measured_traffic(kernel, units)
    return r


def decode_bytes(n_active, B, H, HV):
    return n_active * HV * 2 * D * D * 4 + B * (2 * H * D * 2 + HV * D * 2 * 2 + HV * 8)


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------- helpers
def _bf(torch, bits, dev):
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)


# training-step variants ("[Cake 1/13] gdn: chunked gated delta rule, det and fast, with
# KCP and FLA-CP", Performance (3/5): fwd+bwd = one training step; ckpt = forward,
# recomputed forward and backward of a checkpointed step; the recompute-state option
# of API and flags rebuilds w, u, h and v_new inside the backward)
STEP_MODES = {
    "saved": "gdn_chunk_fwd (saving for backward) + gdn_chunk_bwd",
    "recompute": "gdn_chunk_fwd (no saved buffer) + gdn_chunk_bwd in recompute-state mode",
    "ckpt": "gdn_chunk_fwd (no saved buffer) + gdn_chunk_fwd (saving) + gdn_chunk_bwd",
    "gated": "gdn_chunk_fwd_gated (saving) + gdn_chunk_bwd_gated: g, beta from the fused gate",
    "fwd": "gdn_chunk_fwd (o and the final state; no backward follows)",
}


class ChunkRunner:
    """Device buffers of one chunk workload and one training step through the C ABI
    (mode: a key of STEP_MODES; beta in fp32 when the workload carries fp32 beta)."""

    def __init__(self, torch, wl, dev, mode="saved", scan_segment_chunks=0):
        import chunked_gated_delta_06_gb300 as gdn
        self.torch, self.gdn, self.wl, self.dev, self.mode = torch, gdn, wl, dev, mode
        T, H, HV, N = wl.T, wl.H, wl.HV, wl.N
        self.q, self.k, self.v = _bf(torch, wl.q_bits, dev), _bf(torch, wl.k_bits, dev), _bf(torch, wl.v_bits, dev)
        self.g = torch.from_numpy(wl.g).to(dev)
        f32 = wl.beta_f32 is not None
        self.beta = torch.from_numpy(wl.beta_f32).to(dev) if f32 else _bf(torch, wl.beta_bits, dev)
        self.h0 = None if wl.h0 is None else torch.from_numpy(wl.h0).to(dev)
        self.d_o = None if mode == "fwd" else _bf(torch, wl.do_bits, dev)
        self.d_ht = None if wl.d_ht is None else torch.from_numpy(wl.d_ht).to(dev)
        self.cu_dev = torch.from_numpy(wl.cu_seqlens).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.p, self._keep = gdn.make_problem(wl.cu_seqlens, H, HV, cu_dev_ptr=self.cu_dev.data_ptr(),
                                              beta_dtype=gdn.GDN_DTYPE_F32 if f32 else gdn.GDN_DTYPE_BF16,
                                              device_status_ptr=self.status.data_ptr(),
                                              scan_segment_chunks=scan_segment_chunks)
        e = lambda *s, dt=torch.float32: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        self.o = e(T, HV, D, dt=torch.bfloat16)
        self.ht = e(N, HV, D, D)
        self.saved = (None if mode in ("recompute", "fwd") else
                      e(gdn.gdn_chunk_saved_bytes(self.p), dt=torch.uint8))
        self.ws_f = e(gdn.gdn_chunk_workspace_bytes(self.p, 0), dt=torch.uint8)
        if mode == "fwd":
            return
        self.ws_b = e(gdn.gdn_chunk_workspace_bytes(self.p, 2 if mode == "recompute" else 1), dt=torch.uint8)
        self.dq, self.dk = torch.empty_like(self.q), torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.dg = e(T, HV)
        self.dbeta = e(T, HV, dt=torch.float32 if f32 else torch.bfloat16)
        self.dh0 = e(N, HV, D, D)
        if mode == "gated":  # pre-activations and parameters of the fused gate
            from chunked_gated_delta_06_gb300 import workloads as W
            gi = W.gate_inputs(T, HV, seed=wl.notes.get("seed", 0))
            self.ga, self.gb = _bf(torch, gi.a_bits, dev), _bf(torch, gi.b_bits, dev)
            self.A_log = torch.from_numpy(gi.A_log).to(dev)
            self.dt_bias = torch.from_numpy(gi.dt_bias).to(dev)
            self.da, self.db = e(T, HV, dt=torch.bfloat16), e(T, HV, dt=torch.bfloat16)
            self.dA_log, self.ddt_bias = e(HV), e(HV)

    def _fwd(self, saved, s, timer):
        gdn, P = self.gdn, lambda t: None if t is None else t.data_ptr()  # noqa: E731
        st = gdn.gdn_chunk_fwd(self.p, P(self.q), P(self.k), P(self.v), P(self.g), P(self.beta),
                               P(self.h0), P(self.o), P(self.ht), P(saved), P(self.ws_f),
                               self.ws_f.numel(), s, timer)
        if st:
            raise gdn.GdnError(st, "gdn_chunk_fwd")

    def _gated_step(self, s):
        gdn, P = self.gdn, lambda t: None if t is None else t.data_ptr()  # noqa: E731
        gate = (P(self.ga), P(self.gb), P(self.A_log), P(self.dt_bias))
        st = gdn.gdn_chunk_fwd_gated(self.p, P(self.q), P(self.k), P(self.v), *gate, P(self.h0),
                                     P(self.o), P(self.ht), P(self.saved), P(self.ws_f),
                                     self.ws_f.numel(), s)
        if st:
            raise gdn.GdnError(st, "gdn_chunk_fwd_gated")
        st = gdn.gdn_chunk_bwd_gated(self.p, P(self.q), P(self.k), P(self.v), *gate, P(self.h0),
                                     P(self.saved), P(self.d_o), P(self.d_ht), P(self.dq), P(self.dk),
                                     P(self.dv), P(self.da), P(self.db), P(self.dA_log),
                                     P(self.ddt_bias), P(self.dh0), P(self.ws_b), self.ws_b.numel(), s)
        if st:
            raise gdn.GdnError(st, "gdn_chunk_bwd_gated")

    def step(self, timer=None, stream=None):
        gdn, P = self.gdn, lambda t: None if t is None else t.data_ptr()  # noqa: E731
        s = (stream or self.torch.cuda.current_stream()).cuda_stream
        if self.mode == "gated":
            return self._gated_step(s)
        if self.mode == "fwd":
            return self._fwd(None, s, timer)
        if self.mode == "ckpt":
            self._fwd(None, s, timer)  # the forward of the checkpointed step keeps nothing
        self._fwd(self.saved, s, timer)
        st = gdn.gdn_chunk_bwd(self.p, P(self.q), P(self.k), P(self.v), P(self.g), P(self.beta),
                               P(self.h0), P(self.saved), P(self.d_o), P(self.d_ht), P(self.dq),
                               P(self.dk), P(self.dv), P(self.dg), P(self.dbeta), P(self.dh0),
                               P(self.ws_b), self.ws_b.numel(), s, timer)
        if st:
            raise gdn.GdnError(st, "gdn_chunk_bwd")

    def check_status(self):
        """The kernels' status word after the steps so far (must stay 0)."""
        st = int(self.status.item())
        if st:
            raise RuntimeError("device status %d after the timed steps" % st)

    def inputs(self):
        return [x for x in (self.q, self.k, self.v, self.g, self.beta, self.h0, self.d_o, self.d_ht)
                if x is not None]

    def outputs(self):
        if self.mode == "fwd":
            return [self.o, self.ht]
        return [self.o, self.ht, self.dq, self.dk, self.dv, self.dg, self.dbeta, self.dh0]


L2_FLUSH_BYTES = 512 << 20


def _time_steps(torch, fn, steps, flush=True):
    """Per-step device times in ms ("cake_gdn: deterministic chunked GDN training
    kernels", section 2, Operator level, Method): before every step a 512 MiB memset
    evicts L2 (outside the timed region), then CUDA events on the launching stream
    bracket the step alone.  Returns the list of per-step times."""
    buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda") if flush else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        if buf is not None:
            buf.zero_()
        starts[i].record()
        fn()
        stops[i].record()
    torch.cuda.synchronize()
    del buf
    return [a.elapsed_time(b) for a, b in zip(starts, stops)]


def _time_loop(torch, fn, steps, flush=True):
    """Median per-step time (ms) under the protocol of _time_steps."""
    return statistics.median(_time_steps(torch, fn, steps, flush))


def _kernel_table(torch, runner_step, steps, capacity, flush=True):
    """Per-kernel device times (ms) of `steps` steps, each after an L2 flush:
    {kernel name: [duration of each launch]}."""
    from chunked_gated_delta_06_gb300.binding import KernelTimer
    timer = KernelTimer(capacity)
    buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda") if flush else None
    per = {}
    for _ in range(steps):
        if buf is not None:
            buf.zero_()
        timer.reset()
        runner_step(timer)
        for name, ms in timer.records():
            per.setdefault(name, []).append(ms)
    del buf
    return per


def _cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


# ---------------------------------------------------------------------------- CPU oracle
def oracle_sample(wl, target_tokens):
    """A bounded sample of a chunk workload: whole sequences in packing order until
    target_tokens (the last one cut), every value head."""
    from chunked_gated_delta_06_gb300 import workloads as W
    cu = wl.cu_seqlens
    lens, tot = [], 0
    for n in range(wl.N):
        L = int(cu[n + 1] - cu[n])
        take = min(L, target_tokens - tot)
        if take <= 0:
            break
        lens.append(take)
        tot += take
    idx = np.concatenate([np.arange(cu[n], cu[n] + lens[n]) for n in range(len(lens))])
    return idx, lens


def run_oracle_sample(wl, target_tokens, threads=None):
    import oracle
    idx, lens = oracle_sample(wl, target_tokens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = len(lens)
    h0 = None if wl.h0 is None else wl.h0[:n]
    d_ht = None if wl.d_ht is None else wl.d_ht[:n]
    q, k, v, g, beta, d_o = wl.q[idx], wl.k[idx], wl.v[idx], wl.g[idx], wl.beta[idx], wl.d_o[idx]
    threads = threads or os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, g, beta, cu, h0=h0, threads=threads)
    oracle.bwd(q, k, v, g, beta, cu, d_o, d_ht=d_ht, h0=h0, threads=threads)
    dt = time.perf_counter() - t0
    return int(cu[-1]), dt, threads, min(threads, n * wl.HV)


def aggregate_over_ranks(ms_per_step, tokens_per_rank):
    """Whole-job timing of replicas: the step time is the max over ranks (the job
    finishes with its slowest rank) and the token count is the sum over ranks.
    Uses the default torch.distributed group when one is initialised (NCCL on
    GPUs, gloo on CPU); a single process returns its own numbers."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms_per_step, tokens_per_rank
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_per_step], dtype=torch.float64, device=dev)
    n = torch.tensor([tokens_per_rank], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def bench_reference(args):
    """The oracle (fp64 CPU) on the same workload, metric and unit: every step runs
    fwd+bwd on a bounded sample of the workload (its first --ref-tokens tokens, whole
    sequences in packing order, every value head); value and ms_per_step are those of
    the sample actually run."""
    rank, world, _ = _dist()
    if rank != 0:
        return
    from chunked_gated_delta_06_gb300 import workloads as W
    import oracle
    oracle.build()
    wl = W.CHUNK_CONFIGS[args.workload](seed=0)
    vals, secs = [], []
    tok = used = 0
    for i in range(args.warmup + args.steps):
        tok, dt, thr, used = run_oracle_sample(wl, args.ref_tokens)
        if i >= args.warmup:
            vals.append(tok / dt)
            secs.append(dt)
    v = statistics.median(vals)
    sample = ("first %d tokens of the packed %s workload (whole sequences in packing "
              "order, last cut), all %d value heads, fwd+bwd per step" % (tok, args.workload, wl.HV))
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "T": wl.T, "num_seqs": wl.N, "H": wl.H, "HV": wl.HV,
                       "K": wl.K, "V": wl.V, "chunk": C,
                       "sample_tokens_per_step": tok,
                       "parallelism": "single" if world == 1 else "rank 0 alone (host cores)"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "cpu_model": _cpu_model(), "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- ncu summaries
# (profiles/ holds what these print for the committed captures)
def ncu_launches(path, skip_first=0):
    """Per kernel of an ncu launch list (--metrics gpu__time_duration.sum --csv): launches,
    total and mean device time, share of the total."""
    rows = []
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        rows.append(r)
    rows = rows[skip_first:]
    agg = defaultdict(lambda: [0, 0.0])
    for r in rows:
        name = r["Kernel Name"].replace("(anonymous namespace)", "anon")
        if "FillFunctor" in name:  # torch's memset: the L2 flush between timed steps
            name = "torch fill (L2 flush)"
        else:
            name = re.sub(r"\(.*", "", name).split("::")[-1].strip()
        scale = {"ns": 1e-6, "us": 1e-3, "usecond": 1e-3, "nsecond": 1e-6, "ms": 1.0,
                 "msecond": 1.0}.get(r["Metric Unit"], 1e-6)
        agg[name][0] += 1
        agg[name][1] += float(r["Metric Value"].replace(",", "")) * scale
    total = sum(v[1] for v in agg.values())
    out = ["%-28s %8s %12s %10s %7s" % ("kernel", "launches", "total ms", "mean ms", "share")]
    for name, (n, ms) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        out.append("%-28s %8d %12.3f %10.4f %6.1f%%" % (name, n, ms, ms / n, 100 * ms / total))
    out.append("%-28s %8d %12.3f" % ("total", sum(v[0] for v in agg.values()), total))
    return "\n".join(out)


def ncu_report(path):
    """Per captured launch of a --set full report: duration, DRAM bytes, DRAM throughput,
    tensor-pipe activity, warps active, registers, grid and the largest warp stalls."""
    out = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(out.splitlines()))
    hdr, units, data = rows[0], rows[1], rows[2:]

    def get(r, m):
        return r[hdr.index(m)] if m in hdr else ""

    def unit(r, m):
        return units[hdr.index(m)] if m in hdr else ""

    stall = [c for c in hdr if c.startswith("smsp__average_warps_issue_stalled_")
             and c.endswith("_per_issue_active.ratio")]
    lines = []
    for r in data:
        name = re.sub(r"\(.*", "", r[hdr.index("Kernel Name")].replace("(anonymous namespace)", "anon"))
        name = name.split("::")[-1].strip()
        tops = sorted(((float(get(r, c) or 0), c[len("smsp__average_warps_issue_stalled_"):-len(
            "_per_issue_active.ratio")]) for c in stall), reverse=True)[:4]
        lines.append(
            "%s: %s %s; DRAM read %s %s, write %s %s (%s %% of peak); tensor pipe %s %% of active; "
            "warps active %s %%; %s regs/thread; grid %s block %s; stalls (cycles/issue): %s" % (
                name, get(r, "gpu__time_duration.sum"), unit(r, "gpu__time_duration.sum"),
                get(r, "dram__bytes_read.sum"), unit(r, "dram__bytes_read.sum"),
                get(r, "dram__bytes_write.sum"), unit(r, "dram__bytes_write.sum"),
                get(r, "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed"),
                get(r, "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"),
                get(r, "sm__warps_active.avg.pct_of_peak_sustained_active"),
                get(r, "launch__registers_per_thread"), get(r, "launch__grid_size"),
                get(r, "launch__block_size"),
                ", ".join("%s %.2f" % (n, v) for v, n in tops)))
    return "\n".join(lines)


NCU_KERNELS = {  # ncu kernel name -> bench kernel name (its source: KERNEL_SOURCE)
    "k_intra_tc": "intra", "k_state_tc": "state", "k_state_tc<0>": "state",
    "k_out_tc<1>": "out", "k_out_tc<true>": "out", "k_out_tc<0>": "dvloc", "k_out_tc<false>": "dvloc",
    "k_bstate_tc": "bstate", "k_bstate_tc<0>": "bstate", "k_bintra_a_tc": "bintra_a",
    "k_bintra_b_tc": "bintra_b", "k_decode": "decode", "k_prep": "prep",
    "k_plan": "plan",
}


def ncu_traffic(path, units):
    """JSON record of DRAM bytes (read + write) per work unit of every known kernel in a
    --set full (or dram-metric) report, with the hash of its source at capture time."""
    out = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(out.splitlines()))
    hdr, data = rows[0], rows[2:]
    units_row = rows[1]
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    rec = {}
    for r in data:
        name = re.sub(r"\(.*", "", r[hdr.index("Kernel Name")].replace("(anonymous namespace)", "anon"))
        name = name.split("::")[-1].strip()
        if name not in NCU_KERNELS:
            continue
        kname = NCU_KERNELS[name]
        rd = float(r[hdr.index("dram__bytes_read.sum")]) * scale[units_row[hdr.index("dram__bytes_read.sum")]]
        wr = float(r[hdr.index("dram__bytes_write.sum")]) * scale[units_row[hdr.index("dram__bytes_write.sum")]]
        sha = _source_hash(kname)
        rec[kname] = {"bytes_per_unit": (rd + wr) / units, "captured_units": units,
                      "capture": os.path.basename(path), "source_sha256_16": sha}
    return json.dumps(rec, indent=1, sort_keys=True)



# ---------------------------------------------------------------------------- main bench
def bench_ours(args):
    import torch
    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = "cuda:%d" % local
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))
    from chunked_gated_delta_06_gb300 import build as B
    B.build()
    from chunked_gated_delta_06_gb300 import workloads as W
    peaks = _peaks()

    wl = W.CHUNK_CONFIGS[args.workload](seed=rank)
    T, H, HV, N = wl.T, wl.H, wl.HV, wl.N
    C_total = int(sum((int(wl.cu_seqlens[i + 1] - wl.cu_seqlens[i]) + C - 1) // C for i in range(N)))
    run = ChunkRunner(torch, wl, dev, scan_segment_chunks=args.scan_segment_chunks)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    step_ms = _time_steps(torch, run.step, args.steps)
    clk = clocks.stop()
    barrier()
    run.check_status()
    ms, total_tokens = aggregate_over_ranks(statistics.median(step_ms), T)
    value = total_tokens / (ms / 1e3)

    # per-kernel durations (the same steps with the kernel timer, each after an L2
    # flush; median per kernel), launches per step
    ksteps = max(3, min(args.steps, 10))
    per = _kernel_table(torch, run.step, ksteps, 64)
    launches_per_step = sum(len(v) for v in per.values()) // ksteps
    ktab = {k: {"ms": statistics.median(v), "launches_per_step": len(v) // ksteps}
            for k, v in per.items()}
    dom = max(ktab, key=lambda k: ktab[k]["ms"] * ktab[k]["launches_per_step"])
    fl, by = kernel_work(dom, T, H, HV, N, C_total)
    dom_roof = roofline(dom, fl, by, ktab[dom]["ms"] / 1e3, peaks, C_total * HV)
    step_bytes = 0
    for k in ktab:
        f_, b_ = kernel_work(k, T, H, HV, N, C_total)
        step_bytes += b_ * ktab[k]["launches_per_step"]
        ktab[k]["tflops"] = f_ / (ktab[k]["ms"] / 1e3) / 1e12 if f_ else None
        ktab[k]["gbs"] = b_ / (ktab[k]["ms"] / 1e3) / 1e9 if b_ else None
        ktab[k]["tensor_frac"] = (ktab[k]["tflops"] / peaks["bf16_sustained"]) if f_ else None
        ktab[k]["hbm_frac"] = (ktab[k]["gbs"] / peaks["hbm"]) if b_ else None
        ktab[k]["algorithmic_bytes"] = b_

    sf, sb = step_work(T, H, HV, N, True, wl.h0 is not None, True, wl.d_ht is not None)
    srf = step_fractions(sf, sb, ms / 1e3, peaks)
    # the headline roofline is the whole step on the tensor cores (the target is half of
    # the sustained bf16 peak); the kernel with the largest share of the step follows
    # with its own bound and its ncu DRAM traffic
    traffic = [measured_traffic(k, C_total * HV) for k in ktab if k not in ("plan",)]
    roof = {"scope": "whole fwd+bwd step (every kernel of gdn_chunk_fwd + gdn_chunk_bwd)",
            "bound": "tensor", "achieved": srf["tflops"], "peak": peaks["bf16_sustained"],
            "unit": "TFLOP/s", "frac": srf["tensor_frac"], "target_frac": 0.5,
            "peak_source": "bf16_tflops_sustained (%s)" % peaks["source"],
            "algorithmic_flops": sf,
            "traffic": (sum(traffic) if traffic and all(t is not None for t in traffic) else None),
            "kernel_bytes_per_step": step_bytes,
            "dominant_kernel": dom_roof}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_mean": statistics.mean(step_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": args.workload, "T": T, "num_seqs": N, "H": H, "HV": HV,
                       "K": D, "V": D, "chunk": C, "chunks": C_total,
                       "step": "gdn_chunk_fwd (saving for backward) + gdn_chunk_bwd",
                       "l2": "512 MiB memset before every timed step (outside the timed region); "
                             "the median of the per-step CUDA-event times",
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": roof, "kernels": ktab, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk}
    line["step_roofline"] = srf

    # the other chunk workloads of the method's configurations, each timed the same
    # way (per-step CUDA events after an L2 flush, the median), with the whole call
    # against both peaks
    if not args.no_workloads:
        others = {}
        for name in ("fwd_t256", "fb_4x4096", "fb_65536_long"):
            if name == args.workload:
                continue
            owl = W.CHUNK_CONFIGS[name](seed=rank)
            mode = "saved" if owl.backward else "fwd"
            orun = ChunkRunner(torch, owl, dev, mode=mode)
            for _ in range(max(3, args.warmup)):
                orun.step()
            barrier()
            osteps = max(3, min(args.steps, 10))
            oms, otok = aggregate_over_ranks(_time_loop(torch, orun.step, osteps), owl.T)
            barrier()
            of, ob = step_work(owl.T, owl.H, owl.HV, owl.N, owl.backward, owl.h0 is not None, True,
                               owl.d_ht is not None)
            others[name] = {"value": otok / (oms / 1e3), "unit": "tokens/s", "ms_per_step": oms,
                            "steps": osteps, "step": STEP_MODES[mode],
                            "config": {"T": owl.T, "num_seqs": owl.N, "H": owl.H, "HV": owl.HV,
                                       "initial_state": owl.h0 is not None,
                                       "d_final_state": owl.d_ht is not None},
                            **step_fractions(of, ob, oms / 1e3, peaks)}
            del orun, owl
        line["workloads"] = others

    # the other training-step forms on the same workload: recompute-state mode,
    # the checkpointed step, and fp32 beta (same kernels; device-timed like value)
    if not args.no_variants:
        vsteps = max(3, min(args.steps, 10))
        variants = {}
        for name, vwl, mode in (("recompute", wl, "recompute"), ("ckpt", wl, "ckpt"),
                                ("beta_f32", W.with_fp32_beta(wl), "saved"),
                                ("gated", wl, "gated")):
            vr = ChunkRunner(torch, vwl, dev, mode=mode)
            for _ in range(max(2, min(args.warmup, 3))):
                vr.step()
            barrier()
            vms, _ = aggregate_over_ranks(_time_loop(torch, vr.step, vsteps), T)
            barrier()
            variants[name] = {"value": total_tokens / (vms / 1e3), "unit": "tokens/s",
                              "ms_per_step": vms, "steps": vsteps, "step": STEP_MODES[mode],
                              "beta": ("sigmoid(b), b bf16" if mode == "gated" else
                                       "fp32" if vwl.beta_f32 is not None else "bf16")}
            del vr
        line["variants"] = variants

    # paged chunk prefill at the largest case of the pages' GDN prefill ablation
    # ("Replace Qwen3.5 FLA paths with Attention Gym": N = 64 sequences, T = 8192 packed
    # tokens, 8 key / 16 value heads, states resumed from and written back to pool
    # slots in place; warm cache, repeated calls on fixed pointers, as there)
    if not args.no_prefill:
        import chunked_gated_delta_06_gb300 as gdn
        pw = W.chunk_workload("prefill_64x128", [128] * 64, 8, 16, seed=rank, backward=False)
        pr = np.random.default_rng([rank, 99])
        slots = 2 * pw.N + 1
        ppool = torch.from_numpy((0.1 * pr.standard_normal((slots, pw.HV, D, D))).astype(np.float32)).to(dev)
        pidx = torch.from_numpy(pr.choice(np.arange(1, slots), size=pw.N, replace=False).astype(np.int32)).to(dev)
        pq, pk, pv = _bf(torch, pw.q_bits, dev), _bf(torch, pw.k_bits, dev), _bf(torch, pw.v_bits, dev)
        pg_, pb = torch.from_numpy(pw.g).to(dev), _bf(torch, pw.beta_bits, dev)
        pcu = torch.from_numpy(pw.cu_seqlens).to(dev)
        pp, pkeep = gdn.make_problem(pw.cu_seqlens, pw.H, pw.HV, cu_dev_ptr=pcu.data_ptr())
        po = torch.empty((pw.T, pw.HV, D), dtype=torch.bfloat16, device=dev)
        pws = torch.empty(gdn.gdn_chunk_workspace_bytes(pp, 0), dtype=torch.uint8, device=dev)

        def pstep():
            st = gdn.gdn_chunk_prefill_paged(pp, pq.data_ptr(), pk.data_ptr(), pv.data_ptr(),
                                             pg_.data_ptr(), pb.data_ptr(), ppool.data_ptr(), slots,
                                             pidx.data_ptr(), None, po.data_ptr(), None,
                                             pws.data_ptr(), pws.numel(),
                                             torch.cuda.current_stream().cuda_stream)
            if st:
                raise gdn.GdnError(st, "gdn_chunk_prefill_paged")

        for _ in range(max(3, args.warmup)):
            pstep()
        psteps = max(args.steps, 20)
        pms = _time_loop(torch, pstep, psteps, flush=False)  # warm, as the pages' ablation
        line["prefill_paged"] = {
            "metric": "paged chunk prefill us per call", "value": pms * 1e3, "unit": "us",
            "higher_is_better": False, "tokens_per_s": pw.T / (pms / 1e3), "steps": psteps,
            "config": {"workload": "prefill_64x128", "N": pw.N, "T": pw.T, "H": pw.H, "HV": pw.HV,
                       "slots": slots, "cache": "warm (repeated calls on fixed pointers)",
                       "step": "gdn_chunk_prefill_paged, every sequence resumed from its slot"}}
        del ppool, pws

    # segment-parallel state scans: one long sequence with few value heads (the case
    # the plain scans leave the GPU idle in), fwd+bwd with the planned split and with
    # the split turned off (scan_segment_chunks = -1), device-timed
    if not args.no_segscan:
        import chunked_gated_delta_06_gb300 as gdn
        sw = W.chunk_workload("fb_1x65536_hv16", [65536], 8, 16, seed=rank, h0=True, backward=True,
                              d_ht=True)
        seg = {}
        for label, field in (("split", 0), ("plain", -1)):
            sr = ChunkRunner(torch, sw, dev, scan_segment_chunks=field)
            _, seg_len, nseg = gdn.gdn_chunk_scan_plan(sr.p)
            for _ in range(3):
                sr.step()
            sms = _time_loop(torch, sr.step, 5)
            sper = _kernel_table(torch, sr.step, 3, 32)
            scan = {k_: statistics.median(v) * (len(v) // 3) for k_, v in sper.items()
                    if k_ in ("state", "bstate", "seg_stitch")}
            sr.check_status()
            seg[label] = {"ms_per_step": sms, "tokens_per_s": sw.T / (sms / 1e3), "seg_len": seg_len,
                          "segments": nseg, "scan_ms": scan}
            del sr
        line["segscan"] = {"config": {"workload": "fb_1x65536_hv16", "T": sw.T, "N": 1, "H": sw.H,
                                      "HV": sw.HV, "step": STEP_MODES["saved"]}, **seg}

    # decode state bandwidth
    if not args.no_decode:
        dw = W.decode_workload(seed=rank)
        pool = torch.from_numpy(dw.pool).to(dev)
        qd, kd, vd = _bf(torch, dw.q_bits, dev), _bf(torch, dw.k_bits, dev), _bf(torch, dw.v_bits, dev)
        gd, bd = torch.from_numpy(dw.g).to(dev), torch.from_numpy(dw.beta).to(dev)
        idx = torch.from_numpy(dw.state_indices).to(dev)
        od = torch.empty((dw.B, dw.HV, D), dtype=torch.bfloat16, device=dev)
        import chunked_gated_delta_06_gb300 as gdn

        def dstep(timer=None):
            st = gdn.gdn_decode_step(dw.B, dw.H, dw.HV, D, D, 0.0, qd.data_ptr(), kd.data_ptr(),
                                     vd.data_ptr(), gd.data_ptr(), bd.data_ptr(), pool.data_ptr(),
                                     pool.shape[0], idx.data_ptr(), od.data_ptr(), None,
                                     torch.cuda.current_stream().cuda_stream, timer)
            if st:
                raise gdn.GdnError(st, "gdn_decode_step")

        for _ in range(max(3, args.warmup)):
            dstep()
        dsteps = max(args.steps, 20)
        dms = _time_loop(torch, dstep, dsteps)
        n_active = int((dw.state_indices > 0).sum())
        nb = decode_bytes(n_active, dw.B, dw.H, dw.HV)
        dper = _kernel_table(torch, dstep, 10, 4)
        kms = statistics.median(dper["decode"])
        line["decode"] = {
            "metric": "decode state GB/s", "value": nb / (dms / 1e3) / 1e9, "unit": "GB/s",
            "ms_per_step": dms, "steps": dsteps,
            "config": {"workload": "decode_256", "B": dw.B, "active": n_active, "H": dw.H,
                       "HV": dw.HV, "pool": list(dw.pool.shape), "bytes_per_step": nb,
                       "l2": "state pool (1.07 GB) larger than L2"},
            "roofline": {"kernel": "decode", "bound": "hbm", "achieved": nb / (kms / 1e3) / 1e9,
                         "peak": peaks["hbm"], "unit": "GB/s", "frac": nb / (kms / 1e3) / 1e9 / peaks["hbm"],
                         "traffic": measured_traffic("decode", n_active * dw.HV),
                         "peak_source": "hbm_gbs (%s)" % peaks["source"]}}
        del pool

    # end to end through host buffers: every step uploads its inputs from pinned host
    # memory, runs fwd+bwd through the C ABI and reads every result back.  As in a
    # training input pipeline the uploads, the compute and the read-backs run on three
    # streams over two device buffer sets, so step n+1's upload and step n-1's
    # read-back overlap step n's compute; all of them lie inside the timed region.
    if not args.no_e2e:
        runs = [run, ChunkRunner(torch, wl, dev)]
        h_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x.cpu()) for x in run.inputs()]
        h_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in run.outputs()]
        s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ran = [ev(), ev()]     # buffer set b: compute done (its inputs may be overwritten)
        down = [ev(), ev()]    # buffer set b: results read back (its outputs may be overwritten)
        for b in range(2):
            ran[b].record(s_run)
            down[b].record(s_down)

        def e2e_steps(n):
            for i in range(n):
                b = i & 1
                r = runs[b]
                up = ev()
                s_up.wait_event(ran[b])
                with torch.cuda.stream(s_up):
                    for d_, h_ in zip(r.inputs(), h_in):
                        d_.copy_(h_, non_blocking=True)
                up.record(s_up)
                s_run.wait_event(up)
                s_run.wait_event(down[b])
                r.step(stream=s_run)
                ran[b].record(s_run)
                s_down.wait_event(ran[b])
                with torch.cuda.stream(s_down):
                    for h_, d_ in zip(h_out, r.outputs()):
                        h_.copy_(d_, non_blocking=True)
                down[b].record(s_down)

        e2e_steps(2)
        nsteps = max(3, args.steps)
        t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0e.record(s_up)
        s_run.wait_event(t0e)
        s_down.wait_event(t0e)
        e2e_steps(nsteps)
        s_down.wait_event(ran[0])
        s_down.wait_event(ran[1])
        t1e.record(s_down)
        torch.cuda.synchronize()
        ems = t0e.elapsed_time(t1e) / nsteps
        # the same copies with no compute: one step's uploads and read-backs at once
        # (the floor the copy engines set for the pipelined step)
        def copies_only():
            with torch.cuda.stream(s_up):
                for d_, h_ in zip(run.inputs(), h_in):
                    d_.copy_(h_, non_blocking=True)
            with torch.cuda.stream(s_down):
                for h_, d_ in zip(h_out, run.outputs()):
                    h_.copy_(d_, non_blocking=True)
        copies_only()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(s_up)
        s_down.wait_event(c0)
        for _ in range(3):
            copies_only()
        s_up.synchronize()
        c1.record(s_down)
        s_up.wait_event(c1)
        torch.cuda.synchronize()
        copy_ms = c0.elapsed_time(c1) / 3
        line["e2e"] = {"value": T * world / (ems / 1e3), "unit": "tokens/s",
                       "ms_per_step": ems,
                       "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in run.inputs())),
                       "d2h_bytes_per_step": int(sum(x.numel() * x.element_size() for x in run.outputs())),
                       "copies_alone_ms_per_step": copy_ms,
                       "pipeline": "uploads, compute and read-backs on three streams over two buffer sets"}
        del runs

    # the oracle on the host cores (rank 0, single GPU only)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, dt, thr, used = run_oracle_sample(wl, args.ref_tokens)
        line["cpu_baseline"] = {
            "value": tok / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "cpu_model": _cpu_model(),
            "sample": "first %d tokens of the workload (whole sequences in packing order), all "
                      "32 value heads, fwd+bwd, %.1f s on %d threads" % (tok, dt, used)}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="fb_32k_varlen",
                    choices=["fb_32k_varlen", "fb_4x4096", "fb_65536_long", "fb_8192"],
                    help="chunk workload of the fwd+bwd step (the headline is fb_32k_varlen)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the paged-prefill timing")
    ap.add_argument("--no-segscan", action="store_true", help="skip the segment-parallel scan timing")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the recompute-state, checkpointed-step and fp32-beta timings")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the timings of the other chunk workloads (256-token forward, "
                         "4x4096, 1x65536 with 64 value heads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scan-segment-chunks", type=int, default=0,
                    help="gdn_problem.scan_segment_chunks of the timed workload: 0 = the library's "
                         "plan, -1 = never split, L > 0 = segments of L chunks")
    ap.add_argument("--ref-tokens", type=int, default=2048,
                    help="tokens of the workload the oracle runs per baseline sample")
    ap.add_argument("--ncu-launches", metavar="CSV", help="print the per-kernel summary of an ncu launch "
                    "list (--metrics gpu__time_duration.sum --csv) and exit")
    ap.add_argument("--ncu-report", metavar="REP", help="print a per-launch summary of an ncu report and exit")
    ap.add_argument("--ncu-traffic", nargs="+", metavar="REP UNITS",
                    help="print the DRAM-bytes-per-unit record of ncu reports (pairs of report and the "
                         "work units of its captured launches) and exit")
    ap.add_argument("--skip-first", type=int, default=0, help="launches to skip in --ncu-launches")
    args = ap.parse_args()
    if args.ncu_launches:
        print(ncu_launches(args.ncu_launches, args.skip_first))
        return
    if args.ncu_report:
        print(ncu_report(args.ncu_report))
        return
    if args.ncu_traffic:
        rec = {}
        for r, u in zip(args.ncu_traffic[0::2], args.ncu_traffic[1::2]):
            rec.update(json.loads(ncu_traffic(r, float(u))))
        print(json.dumps(rec, indent=1, sort_keys=True))
        return
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
