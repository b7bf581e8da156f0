"""Seeded synthetic inputs for the KDA / Gated DeltaNet step.

This module is shared by the tests, the benchmark and the oracle harness.  It
holds none of the method's arithmetic: it only draws numbers and rounds them
to the storage types the step reads (fp32, bf16).

Generator.  One counter-based stream per tensor: the i-th 64-bit word of a
stream is splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; Vigna's public-domain splitmix64) of
``key + (i + 1) * 0x9E3779B97F4A7C15``, where ``key`` mixes the seed with a
stable name of the tensor.  Uniforms take the top 53 bits; normals use the
cosine branch of Box-Muller on two consecutive uniforms.  Values are drawn in
fp64, rounded to fp32, and, for bf16 tensors, rounded again to bf16 with
round-to-nearest-even; every consumer sees the rounded value.

Distributions (the KDA / GDN workloads): q/k/v/f/beta/z ~ N(0, 1);
conv weights ~ N(0, 0.25); A_log ~ U(0, ln 16); dt_bias ~ N(0, 0.5);
norm weight = 1 + N(0, 0.1); initial state ~ N(0, 0.02); conv state ~ N(0, 1).
The second parameter of N is the standard deviation.
"""

from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22  # elements drawn per numpy pass, bounds temporary memory


def _mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, *names) -> np.uint64:
    """Stable 64-bit key for (seed, tensor name, indices...)."""
    h = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    for n in names:
        tag = zlib.crc32(str(n).encode()) & 0xFFFFFFFF
        h = _mix64(h ^ np.uint64(tag) + _GOLDEN)
    return np.uint64(h[0])


def _words(key: np.uint64, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GOLDEN)


def _uniform01(key: np.uint64, start: int, n: int) -> np.ndarray:
    """Uniforms in (0, 1]: top 53 bits, plus one ulp so log() is finite."""
    w = _words(key, start, n)
    return ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(key: np.uint64, n: int) -> np.ndarray:
    """n standard normals (fp64), Box-Muller cosine branch."""
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _BLOCK):
        m = min(_BLOCK, n - s)
        u = _uniform01(key, 2 * s, 2 * m)
        out[s:s + m] = np.sqrt(-2.0 * np.log(u[0::2])) * np.cos(2.0 * np.pi * u[1::2])
    return out


def uniform(key: np.uint64, n: int, lo: float, hi: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _BLOCK):
        m = min(_BLOCK, n - s)
        out[s:s + m] = lo + (hi - lo) * _uniform01(key, s, m)
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 values exactly representable in bf16 (the value a bf16 load sees)."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Shape:
    """Sizes of one call of the step.

    B sequences, T tokens per call, H_qk query/key heads, H_v value heads,
    d_k / d_v head widths, K conv taps.  ``kda`` selects the per-key-channel
    decay (Kimi Delta Attention); otherwise the decay is one scalar per head
    (Gated DeltaNet).  ``lb_gate`` (with ``kda``) selects the lower-bound form
    of the per-channel decay, ``sigmoid_out`` the sigmoid output gate.
    ``bf16_in`` stores q/k/v/f/beta/z as bf16.
    """
    B: int
    T: int
    H_qk: int
    H_v: int
    d_k: int
    d_v: int
    K: int = 4
    kda: bool = True
    bf16_in: bool = True
    chunk: int = 64
    eps_l2: float = 1e-6
    eps_norm: float = 1e-6
    lb_gate: bool = False
    sigmoid_out: bool = False

    @property
    def C(self) -> int:
        """conv channels: q and k of every qk head, then v of every value head."""
        return 2 * self.H_qk * self.d_k + self.H_v * self.d_v

    @property
    def f_width(self) -> int:
        """gate logits per (token, value head): d_k for KDA, 1 for GDN."""
        return self.d_k if self.kda else 1

    @property
    def q_scale(self) -> float:
        """d_k^-1/2 rounded once to fp32; both sides use this exact value."""
        return float(np.float32(1.0 / math.sqrt(self.d_k)))


# The five workloads.  Names describe what they are.
WORKLOADS: Dict[str, dict] = {
    # Tiny GDN decode: 8 sequential single-token steps, fp32 everywhere.
    "tiny_gdn_decode": dict(shape=Shape(B=1, T=1, H_qk=2, H_v=2, d_k=16, d_v=16,
                                        kda=False, bf16_in=False), steps=8, layers=1),
    # KDA single-sequence decode: 34 independent layers x 256 tokens.
    "kda_decode_b1_34layers": dict(shape=Shape(B=1, T=1, H_qk=32, H_v=32, d_k=128, d_v=128),
                                   steps=256, layers=34),
    # KDA batched decode: 64 sequences, one step per launch, 100 steps.
    "kda_decode_b64": dict(shape=Shape(B=64, T=1, H_qk=32, H_v=32, d_k=128, d_v=128),
                           steps=100, layers=1),
    # KDA verify: 32 sequences x 4 tokens, per-token states for rollback.
    "kda_verify_b32_t4": dict(shape=Shape(B=32, T=4, H_qk=32, H_v=32, d_k=128, d_v=128),
                              steps=1, layers=1),
    # GDN chunked prefill: 4 sequences x 4096 tokens, 16 qk heads shared by 32 value heads.
    "gdn_prefill_b4_t4096": dict(shape=Shape(B=4, T=4096, H_qk=16, H_v=32, d_k=128, d_v=128,
                                             kda=False, chunk=64), steps=1, layers=1),
}


@dataclasses.dataclass
class Params:
    """Per-layer parameters (fp32)."""
    conv_w: np.ndarray   # [C, K]
    A_log: np.ndarray    # [H_v]
    dt_bias: np.ndarray  # [H_v, d_k] (KDA) or [H_v] (GDN)
    norm_w: np.ndarray   # [d_v]


@dataclasses.dataclass
class Inputs:
    """Pre-projected rows for one call (values as fp32; exact bf16 values when bf16_in)."""
    qkv: np.ndarray   # [B, T, C]
    f: np.ndarray     # [B, T, H_v, f_width]
    beta: np.ndarray  # [B, T, H_v]   (logits)
    z: np.ndarray     # [B, T, H_v, d_v]


@dataclasses.dataclass
class State:
    conv: np.ndarray   # [B, K-1, C] fp32, oldest row first
    S: np.ndarray      # [B, H_v, d_k, d_v] fp32


def _f32(x: np.ndarray, shape) -> np.ndarray:
    return x.astype(np.float32).reshape(shape)


def make_params(shape: Shape, seed: int = 0, layer: int = 0, slow_decay: bool = False) -> Params:
    s = shape
    conv_w = _f32(0.25 * normal(stream_key(seed, "conv_w", layer), s.C * s.K), (s.C, s.K))
    if s.lb_gate:
        # lower-bound gate g = lb * sigmoid(-a f): the per-head scale a in A_log's place,
        # the bound lb <= 0 in dt_bias's (slow decay: a small bound)
        A_log = _f32(uniform(stream_key(seed, "lb_a", layer), s.H_v, 0.5, 2.0), (s.H_v,))
        lo, hi = (-0.2, -0.02) if slow_decay else (-4.0, -0.5)
        dt_bias = _f32(uniform(stream_key(seed, "lb_bound", layer), s.H_v, lo, hi), (s.H_v,))
    else:
        if slow_decay:
            # exp(A_log) in [0.02, 0.1]: with softplus of O(1) the log-decay is |g| <~ 0.1.
            A_log = _f32(uniform(stream_key(seed, "A_log_slow", layer), s.H_v,
                                 math.log(0.02), math.log(0.1)), (s.H_v,))
        else:
            A_log = _f32(uniform(stream_key(seed, "A_log", layer), s.H_v, 0.0, math.log(16.0)),
                         (s.H_v,))
        dt_shape = (s.H_v, s.d_k) if s.kda else (s.H_v,)
        dt_bias = _f32(0.5 * normal(stream_key(seed, "dt_bias", layer), int(np.prod(dt_shape))),
                       dt_shape)
    norm_w = _f32(1.0 + 0.1 * normal(stream_key(seed, "norm_w", layer), s.d_v), (s.d_v,))
    return Params(conv_w, A_log, dt_bias, norm_w)


def make_inputs(shape: Shape, seed: int = 0, layer: int = 0, step: int = 0,
                slow_decay: bool = False) -> Inputs:
    """Inputs of call ``step`` of layer ``layer``.

    With ``slow_decay`` the gate logits are a per-(head, channel) rate plus a
    small per-token jitter (rate ~ N(-1, 0.5), jitter ~ N(0, 0.1)), so a slow
    channel stays slow across tokens and state carries over chunk boundaries.
    """
    s = shape
    rnd = round_bf16 if s.bf16_in else (lambda a: a)
    qkv = rnd(_f32(normal(stream_key(seed, "qkv", layer, step), s.B * s.T * s.C),
                   (s.B, s.T, s.C)))
    fshape = (s.B, s.T, s.H_v, s.f_width)
    if slow_decay:
        rate = normal(stream_key(seed, "f_rate", layer), s.H_v * s.f_width)
        rate = (-1.0 + 0.5 * rate).reshape(1, 1, s.H_v, s.f_width)
        jit = 0.1 * normal(stream_key(seed, "f_jitter", layer, step), int(np.prod(fshape)))
        f = rnd(_f32(rate + jit.reshape(fshape), fshape))
    else:
        f = rnd(_f32(normal(stream_key(seed, "f", layer, step), int(np.prod(fshape))), fshape))
    beta = rnd(_f32(normal(stream_key(seed, "beta", layer, step), s.B * s.T * s.H_v),
                    (s.B, s.T, s.H_v)))
    z = rnd(_f32(normal(stream_key(seed, "z", layer, step), s.B * s.T * s.H_v * s.d_v),
                 (s.B, s.T, s.H_v, s.d_v)))
    return Inputs(qkv, f, beta, z)


def make_state(shape: Shape, seed: int = 0, layer: int = 0) -> State:
    s = shape
    conv = _f32(normal(stream_key(seed, "conv_state", layer), s.B * (s.K - 1) * s.C),
                (s.B, s.K - 1, s.C))
    S = _f32(0.02 * normal(stream_key(seed, "state", layer), s.B * s.H_v * s.d_k * s.d_v),
             (s.B, s.H_v, s.d_k, s.d_v))
    return State(conv, S)


@dataclasses.dataclass
class LayerWeights:
    """Projection weights of one KDA layer, bf16 values held in fp32 arrays."""
    d_model: int
    rank: int
    w_qkv: np.ndarray   # [C, d_model]
    w_fa: np.ndarray    # [rank, d_model]
    w_fb: np.ndarray    # [H_v * d_k, rank]
    w_ga: np.ndarray    # [rank, d_model]
    w_gb: np.ndarray    # [H_v * d_v, rank]
    w_beta: np.ndarray  # [H_v, d_model]
    w_o: np.ndarray     # [d_model, H_v * d_v]

    FIELDS = ("w_qkv", "w_fa", "w_fb", "w_ga", "w_gb", "w_beta", "w_o")


def make_layer_weights(shape: Shape, d_model: int, rank: int, seed: int = 0,
                       layer: int = 0) -> LayerWeights:
    """Each weight ~ N(0, 1/fan_in), rounded to bf16, so unit-variance inputs give
    unit-variance rows: the step sees q/k/v/f/beta/z of the distributions above."""
    s = shape

    def w(name, rows, cols):
        x = normal(stream_key(seed, "proj", name, layer), rows * cols) / math.sqrt(cols)
        return round_bf16(_f32(x, (rows, cols)))

    return LayerWeights(d_model, rank,
                        w("qkv", s.C, d_model), w("fa", rank, d_model),
                        w("fb", s.H_v * s.d_k, rank), w("ga", rank, d_model),
                        w("gb", s.H_v * s.d_v, rank), w("beta", s.H_v, d_model),
                        w("o", d_model, s.H_v * s.d_v))


def make_layer_input(shape: Shape, d_model: int, seed: int = 0, layer: int = 0,
                     step: int = 0) -> np.ndarray:
    """Layer input rows [B, d_model] ~ N(0, 1), rounded to bf16."""
    return round_bf16(_f32(normal(stream_key(seed, "layer_x", layer, step), shape.B * d_model),
                           (shape.B, d_model)))


def with_tokens(shape: Shape, T: int, B: Optional[int] = None) -> Shape:
    return dataclasses.replace(shape, T=T, B=shape.B if B is None else B)
