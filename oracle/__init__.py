"""fp64 CPU oracle of the KDA / Gated DeltaNet step (ctypes loader).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke check
and by the benchmark's CPU-baseline leg.  The product path never imports it.
The C source (``gdn_oracle.c``) shares no code with the CUDA path.

``build()`` compiles the C source with gcc into ``oracle/_build``; ``load()``
returns the ctypes library; ``run()`` / ``run_chunked()`` are numpy wrappers.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_OUT = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT, "libgdn_oracle.so")

# -ffp-contract=off: no fused multiply-add, so x86 and Arm builds round alike.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
          "-fno-fast-math"]


def build(src: str = _SRC, out: str = _LIB, extra=()) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, *extra, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H_qk", ctypes.c_int),
                ("H_v", ctypes.c_int), ("d_k", ctypes.c_int), ("d_v", ctypes.c_int),
                ("K", ctypes.c_int), ("gate", ctypes.c_int), ("out_gate", ctypes.c_int),
                ("q_scale", ctypes.c_double),
                ("eps_l2", ctypes.c_double), ("eps_norm", ctypes.c_double)]


_P = ctypes.c_void_p
_cache = {}


def load(path: Optional[str] = None):
    path = path or _LIB
    if path in _cache:
        return _cache[path]
    if path == _LIB and (not os.path.exists(_LIB) or
                         os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        build()
    lib = ctypes.CDLL(path)
    for name in ("gdn_oracle_silu", "gdn_oracle_sigmoid", "gdn_oracle_softplus"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_double
        fn.argtypes = [ctypes.c_double]
    lib.gdn_oracle_l2norm.argtypes = [ctypes.c_int, _P, ctypes.c_double, ctypes.c_double, _P]
    lib.gdn_oracle_log_decay.argtypes = [ctypes.c_int, _P, _P, ctypes.c_double, _P]
    lib.gdn_oracle_delta_step.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_double,
                                          _P, _P, _P, _P]
    lib.gdn_oracle_log_decay_lb.argtypes = [ctypes.c_int, _P, ctypes.c_double, ctypes.c_double, _P]
    lib.gdn_oracle_gated_rmsnorm.argtypes = [ctypes.c_int, _P, _P, _P, ctypes.c_double, ctypes.c_int,
                                             _P]
    lib.gdn_oracle_conv.argtypes = [ctypes.POINTER(Shape), _P, _P, _P, _P]
    lib.gdn_oracle_run.restype = ctypes.c_int
    lib.gdn_oracle_run.argtypes = [ctypes.POINTER(Shape)] + [_P] * 13 + [ctypes.c_int]
    lib.gdn_oracle_run_chunked.restype = ctypes.c_int
    lib.gdn_oracle_run_chunked.argtypes = ([ctypes.POINTER(Shape), ctypes.c_int] + [_P] * 12 +
                                           [ctypes.c_int])
    _cache[path] = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def make_shape(shape) -> Shape:
    """ctypes shape from any object with the synth.Shape fields."""
    lb = getattr(shape, "lb_gate", False)
    gate = 2 if lb else (1 if shape.kda else 0)
    out_gate = 1 if getattr(shape, "sigmoid_out", False) else 0
    return Shape(shape.B, shape.T, shape.H_qk, shape.H_v, shape.d_k, shape.d_v, shape.K,
                 gate, out_gate, shape.q_scale, shape.eps_l2, shape.eps_norm)


def run(shape, params, inputs, conv_state, state, *, hist: bool = False, o_raw: bool = False,
        nthreads: Optional[int] = None, lib=None):
    """T sequential steps.  Returns dict(y, conv_state, state[, state_hist][, o_raw]).

    ``conv_state`` / ``state`` are copied (fp64) and the advanced copies returned.
    """
    lib = lib or load()
    s = shape
    cs = _f64(conv_state).copy()
    S = _f64(state).copy()
    y = np.empty((s.B, s.T, s.H_v, s.d_v), dtype=np.float64)
    o = np.empty_like(y) if o_raw else None
    H = np.empty((s.T, s.B, s.H_v, s.d_k, s.d_v), dtype=np.float64) if hist else None
    keep = [_f32(inputs.qkv), _f32(inputs.f), _f32(inputs.beta), _f32(inputs.z),
            _f32(params.conv_w), _f32(params.A_log), _f32(params.dt_bias), _f32(params.norm_w)]
    sh = make_shape(s)
    rc = lib.gdn_oracle_run(ctypes.byref(sh), *[_ptr(a) for a in keep], _ptr(cs), _ptr(S),
                            _ptr(y), _ptr(o), _ptr(H), nthreads or os.cpu_count() or 1)
    if rc != 0:
        raise ValueError(f"oracle rejected the shape (rc={rc})")
    out = dict(y=y, conv_state=cs, state=S)
    if hist:
        out["state_hist"] = H
    if o_raw:
        out["o_raw"] = o
    return out


def run_chunked(shape, params, inputs, conv_state, state, chunk: int, *, o_raw: bool = False,
                nthreads: Optional[int] = None, lib=None):
    lib = lib or load()
    s = shape
    cs = _f64(conv_state).copy()
    S = _f64(state).copy()
    y = np.empty((s.B, s.T, s.H_v, s.d_v), dtype=np.float64)
    o = np.empty_like(y) if o_raw else None
    keep = [_f32(inputs.qkv), _f32(inputs.f), _f32(inputs.beta), _f32(inputs.z),
            _f32(params.conv_w), _f32(params.A_log), _f32(params.dt_bias), _f32(params.norm_w)]
    sh = make_shape(s)
    rc = lib.gdn_oracle_run_chunked(ctypes.byref(sh), chunk, *[_ptr(a) for a in keep], _ptr(cs),
                                    _ptr(S), _ptr(y), _ptr(o), nthreads or os.cpu_count() or 1)
    if rc != 0:
        raise ValueError(f"oracle rejected the shape (rc={rc})")
    out = dict(y=y, conv_state=cs, state=S)
    if o_raw:
        out["o_raw"] = o
    return out


def project(x, w):
    """A linear projection, y[b][n] = sum_k x[b][k] w[n][k], in fp64 (the layer's
    q/k/v, gate, beta and output projections around the step, "Thirty tiny
    kernels per layer", the KDA decode budget)."""
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64).T


def layer_decode(shape, params, weights, x, conv_state, state, nthreads: Optional[int] = None,
                 lib=None):
    """One decode token of a whole KDA layer: the projections (fp64), the step on
    the projected rows, the output projection.  f = f_b(f_a(x)), z = g_b(g_a(x))
    (the low-rank gate chains), qkv and beta straight from x.  The rows enter the
    step as fp32, the width the step's C interface takes.  Returns dict(rows=...,
    y, x_out, conv_state, state)."""
    s = shape
    assert s.T == 1 and s.kda
    W = weights
    qkv = project(x, W.w_qkv)
    f = project(project(x, W.w_fa), W.w_fb)
    z = project(project(x, W.w_ga), W.w_gb)
    beta = project(x, W.w_beta)

    class _Rows:
        pass

    rows = _Rows()
    rows.qkv = qkv.reshape(s.B, 1, s.C)
    rows.f = f.reshape(s.B, 1, s.H_v, s.d_k)
    rows.beta = beta.reshape(s.B, 1, s.H_v)
    rows.z = z.reshape(s.B, 1, s.H_v, s.d_v)
    out = run(s, params, rows, conv_state, state, nthreads=nthreads, lib=lib)
    out["x_out"] = project(out["y"].reshape(s.B, s.H_v * s.d_v), W.w_o)
    out["rows"] = dict(qkv=qkv, f=f, beta=beta, z=z)
    return out


def conv(shape, qkv, conv_w, conv_state, lib=None):
    """a1 alone: returns (xhat [B,T,C], advanced conv_state)."""
    lib = lib or load()
    s = shape
    cs = _f64(conv_state).copy()
    xh = np.empty((s.B, s.T, s.C), dtype=np.float64)
    q = _f32(qkv)
    w = _f32(conv_w)
    sh = make_shape(s)
    lib.gdn_oracle_conv(ctypes.byref(sh), _ptr(q), _ptr(w), _ptr(cs), _ptr(xh))
    return xh, cs


def delta_step(S, alpha, beta, k, v, q, lib=None):
    """a5 + a6 on one [d_k, d_v] state; returns (S_new, o)."""
    lib = lib or load()
    S = _f64(S).copy()
    d_k, d_v = S.shape
    o = np.empty(d_v, dtype=np.float64)
    a, kk, vv, qq = _f64(alpha), _f64(k), _f64(v), _f64(q)
    lib.gdn_oracle_delta_step(d_k, d_v, _ptr(S), _ptr(a), float(beta), _ptr(kk), _ptr(vv),
                              _ptr(qq), _ptr(o))
    return S, o


def l2norm(x, scale, eps, lib=None):
    lib = lib or load()
    x = _f64(x)
    out = np.empty_like(x)
    lib.gdn_oracle_l2norm(x.size, _ptr(x), float(scale), float(eps), _ptr(out))
    return out


def log_decay(f, dt_bias, A_log, lib=None):
    lib = lib or load()
    f = _f64(f)
    d = _f64(dt_bias)
    g = np.empty_like(f)
    lib.gdn_oracle_log_decay(f.size, _ptr(f), _ptr(d), float(A_log), _ptr(g))
    return g


def log_decay_lb(f, a, lb, lib=None):
    lib = lib or load()
    f = _f64(f)
    g = np.empty_like(f)
    lib.gdn_oracle_log_decay_lb(f.size, _ptr(f), float(a), float(lb), _ptr(g))
    return g


def gated_rmsnorm(o, z, w, eps, sigmoid_gate: bool = False, lib=None):
    lib = lib or load()
    o, z, w = _f64(o), _f64(z), _f64(w)
    y = np.empty_like(o)
    lib.gdn_oracle_gated_rmsnorm(o.size, _ptr(o), _ptr(z), _ptr(w), float(eps),
                                 1 if sigmoid_gate else 0, _ptr(y))
    return y
