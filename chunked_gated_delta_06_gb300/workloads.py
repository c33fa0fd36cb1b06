"""Seeded synthetic workloads for the chunked gated delta rule.

This module only draws inputs: it holds none of the method's arithmetic, and it
is the one piece shared by the CUDA path's tests / bench and the fp64 oracle.
Every array comes from its own counter-based numpy stream
``default_rng([seed, stream])``, so a workload is the same bytes on any host
(x86 or Arm) and an array's values do not depend on which other arrays were drawn.

The recipes follow the five workloads the library is measured on (the shapes and
value distributions of the operator benchmarks in "cake_gdn: deterministic
chunked GDN training kernels", section 2, and the decode state contract of "C6:
GDN decode-step goldens ..."):

* ``fwd_t256``            1 sequence, T=256, H=HV=2, forward only, zero state.
* ``fb_4x4096``           4 x 4096 tokens packed, H=16, HV=32, forward+backward.
* ``fb_32k_varlen``       32768 packed tokens, lengths ~U[1,8192], H=16, HV=32,
                          fp32 initial state, final state and dh0 returned.
* ``fb_65536_long``       1 x 65536 tokens, H=16, HV=64, initial state, dO and
                          d(final state).
* ``decode_256``          256 rows, H=16, HV=32, fp32 pool [512,32,128,128].

bf16 values are produced by round-to-nearest-even of float32 draws; arrays are
kept both as their bf16 bit patterns (uint16, for upload) and as the float32
values those bits denote (for the oracle).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# stream numbers of default_rng([seed, stream])
S_LEN, S_Q, S_K, S_V, S_G, S_BETA, S_ALOG, S_H0, S_DO, S_DHT, S_POOL, S_IDX, S_GATE = range(13)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even; NaN kept quiet."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values they denote (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _normal(seed, stream, shape, scale=1.0):
    a = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _logsigmoid(x):
    x = x.astype(np.float64)
    return (np.minimum(x, 0.0) - np.log1p(np.exp(-np.abs(x)))).astype(np.float32)


def _softplus(x):
    x = x.astype(np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


@dataclass
class ChunkWorkload:
    """Inputs of one chunk_gated_delta_rule call (packed, B = 1)."""
    name: str
    cu_seqlens: np.ndarray           # int32 [N+1]
    H: int
    HV: int
    K: int
    V: int
    q_bits: np.ndarray               # uint16 [T,H,K]
    k_bits: np.ndarray               # uint16 [T,H,K]
    v_bits: np.ndarray               # uint16 [T,HV,V]
    g: np.ndarray                    # float32 [T,HV]
    beta_bits: np.ndarray            # uint16 [T,HV] (bf16 beta)
    h0: np.ndarray | None            # float32 [N,HV,K,V] or None
    do_bits: np.ndarray | None       # uint16 [T,HV,V] or None (forward only)
    d_ht: np.ndarray | None          # float32 [N,HV,K,V] or None
    backward: bool = True
    want_final: bool = True
    notes: dict = field(default_factory=dict)
    beta_f32: np.ndarray | None = None  # float32 [T,HV]: fp32 beta (then beta_bits is unused)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return len(self.cu_seqlens) - 1

    # float32 views of the bf16 inputs (exact values the device sees)
    @property
    def q(self):
        return bf16_value(self.q_bits)

    @property
    def k(self):
        return bf16_value(self.k_bits)

    @property
    def v(self):
        return bf16_value(self.v_bits)

    @property
    def beta(self):
        return self.beta_f32 if self.beta_f32 is not None else bf16_value(self.beta_bits)

    @property
    def d_o(self):
        return None if self.do_bits is None else bf16_value(self.do_bits)


@dataclass
class DecodeWorkload:
    """Inputs of one decode step over a slot-indexed fp32 state pool."""
    name: str
    H: int
    HV: int
    K: int
    V: int
    q_bits: np.ndarray               # uint16 [B,H,K]
    k_bits: np.ndarray               # uint16 [B,H,K]
    v_bits: np.ndarray               # uint16 [B,HV,V]
    g: np.ndarray                    # float32 [B,HV]
    beta: np.ndarray                 # float32 [B,HV]
    pool: np.ndarray                 # float32 [num_slots,HV,V,K]
    state_indices: np.ndarray        # int32 [B]

    @property
    def B(self) -> int:
        return int(self.state_indices.shape[0])

    @property
    def q(self):
        return bf16_value(self.q_bits)

    @property
    def k(self):
        return bf16_value(self.k_bits)

    @property
    def v(self):
        return bf16_value(self.v_bits)


def varlen_lengths(seed: int, total: int, lo: int, hi: int) -> list[int]:
    """Lengths ~U[lo, hi] (integers) drawn until their sum reaches total; last clipped."""
    r = _rng(seed, S_LEN)
    out, s = [], 0
    while s < total:
        L = int(r.integers(lo, hi + 1))
        L = min(L, total - s)
        out.append(L)
        s += L
    return out


def chunk_workload(name: str, lengths, H: int, HV: int, *, seed: int = 0, K: int = 128,
                   V: int = 128, gate: str = "softplus", h0: bool = False, backward: bool = True,
                   d_ht: bool = False, h0_std: float = 0.1, beta_dtype: str = "bf16") -> ChunkWorkload:
    """General recipe.

    gate = "logsigmoid":  g = logsigmoid(N(0,1))                      (per token, head)
    gate = "softplus":    g = -softplus(N(0,1) + dt_bias) * exp(A_log),
                          A_log ~ U(0, 2.7) per value head, dt_bias = 0
    beta = sigmoid(N(0,1)) rounded to bf16 (beta_dtype "bf16") or kept in fp32
    (beta_dtype "f32"); q, k, v, dO ~ N(0,1) rounded to bf16;
    h0 ~ h0_std * N(0,1) fp32 per sequence; d(final state) ~ N(0,1) fp32.
    """
    lengths = [int(x) for x in lengths]
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    N = len(lengths)
    q = bf16_bits(_normal(seed, S_Q, (T, H, K)))
    k = bf16_bits(_normal(seed, S_K, (T, H, K)))
    v = bf16_bits(_normal(seed, S_V, (T, HV, V)))
    gn = _normal(seed, S_G, (T, HV))
    if gate == "logsigmoid":
        g = _logsigmoid(gn)
    elif gate == "softplus":
        a_log = _rng(seed, S_ALOG).uniform(0.0, 2.7, size=(HV,))
        dt_bias = np.zeros((HV,))
        g = (-_softplus(gn.astype(np.float64) + dt_bias[None, :]) * np.exp(a_log)[None, :]).astype(
            np.float32)
    else:
        raise ValueError(gate)
    beta32 = _sigmoid(_normal(seed, S_BETA, (T, HV)))
    beta = bf16_bits(beta32)
    if beta_dtype not in ("bf16", "f32"):
        raise ValueError(beta_dtype)
    h0a = _normal(seed, S_H0, (N, HV, K, V), h0_std) if h0 else None
    do = bf16_bits(_normal(seed, S_DO, (T, HV, V))) if backward else None
    dht = _normal(seed, S_DHT, (N, HV, K, V)) if (backward and d_ht) else None
    return ChunkWorkload(name=name, cu_seqlens=cu, H=H, HV=HV, K=K, V=V, q_bits=q, k_bits=k,
                         v_bits=v, g=g, beta_bits=beta, h0=h0a, do_bits=do, d_ht=dht,
                         backward=backward, notes=dict(gate=gate, seed=seed, beta_dtype=beta_dtype),
                         beta_f32=beta32 if beta_dtype == "f32" else None)


def with_fp32_beta(wl: ChunkWorkload) -> ChunkWorkload:
    """The same workload with beta kept in fp32: the draw that the bf16 beta is the
    rounding of (same seed and stream)."""
    import dataclasses
    T, HV = wl.T, wl.HV
    beta32 = _sigmoid(_normal(wl.notes.get("seed", 0), S_BETA, (T, HV)))
    notes = dict(wl.notes, beta_dtype="f32")
    return dataclasses.replace(wl, beta_f32=beta32, notes=notes)


@dataclass
class GateInputs:
    """Pre-activations and parameters of the fused gate for n rows of HV heads."""
    a_bits: np.ndarray               # uint16 [n,HV] bf16 gate pre-activation
    b_bits: np.ndarray               # uint16 [n,HV] bf16 beta pre-activation
    A_log: np.ndarray                # float32 [HV]
    dt_bias: np.ndarray              # float32 [HV]

    @property
    def a(self):
        return bf16_value(self.a_bits)

    @property
    def b(self):
        return bf16_value(self.b_bits)


def gate_inputs(n: int, HV: int, seed: int = 0, over_threshold: int = 3) -> GateInputs:
    """a, b ~ N(0,1) rounded to bf16 with ``over_threshold`` entries of a set to 24 (past
    the softplus threshold of 20 even after dt_bias), A_log ~ U(0, 2.7) and
    dt_bias ~ U(-1, 1) per value head, fp32 (the gate recipe of the chunk workloads,
    with the gate computed by the kernels)."""
    r = _rng(seed, S_GATE)
    a = r.standard_normal(size=(n, HV), dtype=np.float32)
    b = r.standard_normal(size=(n, HV), dtype=np.float32)
    if n * HV and over_threshold:
        flat = r.choice(n * HV, size=min(over_threshold, n * HV), replace=False)
        a.reshape(-1)[flat] = 24.0
    A_log = r.uniform(0.0, 2.7, size=HV).astype(np.float32)
    dt_bias = r.uniform(-1.0, 1.0, size=HV).astype(np.float32)
    return GateInputs(a_bits=bf16_bits(a), b_bits=bf16_bits(b), A_log=A_log, dt_bias=dt_bias)


def fwd_t256(seed: int = 0) -> ChunkWorkload:
    """Forward only, 1 sequence, T=256, H=HV=2, logsigmoid gate, zero initial state."""
    return chunk_workload("fwd_t256", [256], 2, 2, seed=seed, gate="logsigmoid", h0=False,
                          backward=False)


def fb_4x4096(seed: int = 0) -> ChunkWorkload:
    """4 equal sequences of 4096 packed (T=16384), H=16, HV=32, zero initial state."""
    return chunk_workload("fb_4x4096", [4096] * 4, 16, 32, seed=seed, gate="softplus", h0=False,
                          backward=True)


def fb_32k_varlen(seed: int = 0) -> ChunkWorkload:
    """32768 packed tokens, lengths ~U[1,8192], H=16, HV=32, initial state, dh0 out."""
    lengths = varlen_lengths(seed, 32768, 1, 8192)
    return chunk_workload("fb_32k_varlen", lengths, 16, 32, seed=seed, gate="softplus", h0=True,
                          backward=True, d_ht=False)


def fb_65536_long(seed: int = 0) -> ChunkWorkload:
    """1 x 65536 tokens, H=16, HV=64, initial state, dO and d(final state)."""
    return chunk_workload("fb_65536_long", [65536], 16, 64, seed=seed, gate="softplus", h0=True,
                          backward=True, d_ht=True)


def decode_workload(name: str = "decode_256", B: int = 256, H: int = 16, HV: int = 32,
                    num_slots: int = 512, null_frac: float = 0.1, seed: int = 0, K: int = 128,
                    V: int = 128, pool_std: float = 0.1) -> DecodeWorkload:
    """Decode recipe: indices drawn without repeat from 1..num_slots-1, round(null_frac*B)
    of them set to 0 (null); q,k,v ~ N(0,1) bf16; g = logsigmoid(N(0,1)) fp32;
    beta = sigmoid(N(0,1)) fp32; pool ~ pool_std * N(0,1) fp32 [num_slots,HV,V,K]."""
    r = _rng(seed, S_IDX)
    idx = r.choice(np.arange(1, num_slots, dtype=np.int32), size=B, replace=False).astype(np.int32)
    n_null = int(round(null_frac * B))
    if n_null:
        idx[r.choice(B, size=n_null, replace=False)] = 0
    q = bf16_bits(_normal(seed, S_Q, (B, H, K)))
    k = bf16_bits(_normal(seed, S_K, (B, H, K)))
    v = bf16_bits(_normal(seed, S_V, (B, HV, V)))
    g = _logsigmoid(_normal(seed, S_G, (B, HV)))
    beta = _sigmoid(_normal(seed, S_BETA, (B, HV)))
    pool = _normal(seed, S_POOL, (num_slots, HV, V, K), pool_std)
    return DecodeWorkload(name=name, H=H, HV=HV, K=K, V=V, q_bits=q, k_bits=k, v_bits=v, g=g,
                          beta=beta, pool=pool, state_indices=idx)


def fb_8192(seed: int = 0) -> ChunkWorkload:
    """1 x 8192 tokens, H=16, HV=32, initial state: a profiling-size case of the same
    value recipe (inputs about 200 MB, above the 129 MB L2)."""
    return chunk_workload("fb_8192", [8192], 16, 32, seed=seed, gate="softplus", h0=True,
                          backward=True, d_ht=False)


CHUNK_CONFIGS = {
    "fwd_t256": fwd_t256,
    "fb_4x4096": fb_4x4096,
    "fb_32k_varlen": fb_32k_varlen,
    "fb_65536_long": fb_65536_long,
    "fb_8192": fb_8192,
}
