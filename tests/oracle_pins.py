"""Pins of the fp64 oracle to facts the definition fixes independently of it.

Each ``pin_*(lib)`` raises AssertionError when the oracle library ``lib``
disagrees with a closed form, a special case, a brute-force matrix product
on a tiny size, or an invariant.  The same functions run against planted
mutants of the oracle (tests/test_oracle_mutants.py): every mutant must fail
at least one pin.

Sources of the facts (the pages' definitions):
  * "Thirty tiny kernels per layer": the decode-step op list and the pure
    step function (conv window of the last K-1 rows + current row, SiLU,
    L2 norm of q with the head_dim^-1/2 scale and of k, safe gate, sigmoid
    beta, delta-rule update, gated RMS norm).
  * The delta-rule update S <- (I - beta k k^T) Diag(exp g) S + beta k v^T and
    readout o = S^T q, and g = -exp(A_log) softplus(f + dt_bias).
  * "llama.cpp PR #84", chunked KDA prefill: the chunked form must equal the
    recurrent one.
"""

from __future__ import annotations

import math
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synth  # noqa: E402


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        raise AssertionError(f"{what}: shape {a.shape} != {b.shape}")
    err = np.max(np.abs(a - b)) if a.size else 0.0
    tol = atol + rtol * (np.max(np.abs(b)) if b.size else 0.0)
    if not err <= tol:
        raise AssertionError(f"{what}: max|err| {err:.3e} > {tol:.3e}")


def _silu(x):
    return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------- scalar maps

def pin_scalars(lib):
    ln3 = math.log(3.0)
    _close(lib.gdn_oracle_sigmoid(0.0), 0.5, what="sigmoid(0)")
    _close(lib.gdn_oracle_sigmoid(ln3), 0.75, what="sigmoid(ln 3) = 3/4")
    _close(lib.gdn_oracle_sigmoid(-ln3), 0.25, what="sigmoid(-ln 3) = 1/4")
    _close(lib.gdn_oracle_silu(0.0), 0.0, what="silu(0)")
    _close(lib.gdn_oracle_silu(ln3), 0.75 * ln3, what="silu(ln 3)")
    _close(lib.gdn_oracle_silu(-ln3), -0.25 * ln3, what="silu(-ln 3)")
    _close(lib.gdn_oracle_softplus(0.0), math.log(2.0), what="softplus(0) = ln 2")
    _close(lib.gdn_oracle_softplus(math.log(math.e - 1.0)), 1.0, what="softplus(ln(e-1)) = 1")
    for x in (0.3, 2.0, 7.5, 31.0):
        # softplus(x) - softplus(-x) = x
        _close(lib.gdn_oracle_softplus(x) - lib.gdn_oracle_softplus(-x), x,
               what=f"softplus odd part at {x}")
    _close(lib.gdn_oracle_softplus(-50.0), math.exp(-50.0), rtol=1e-12, atol=0.0,
           what="softplus(-50) = e^-50 (no cut-off)")


# ---------------------------------------------------------------- a2

def pin_l2norm(lib):
    _close(oracle.l2norm([3.0, 4.0], 1.0, 0.0, lib=lib), [0.6, 0.8], what="l2norm 3-4-5")
    _close(oracle.l2norm([3.0, 4.0], 0.25, 0.0, lib=lib), [0.15, 0.2], what="l2norm scaled")
    rng = np.random.default_rng(1)
    x = rng.normal(size=37)
    out = oracle.l2norm(x, 0.125, 0.0, lib=lib)
    _close(np.linalg.norm(out), 0.125, what="|l2norm(x)| = scale")
    _close(out / np.linalg.norm(out), x / np.linalg.norm(x), what="l2norm keeps direction")
    # eps enters under the root: |x|^2 = 25, eps = 11 -> 1/6
    _close(oracle.l2norm([3.0, 4.0], 1.0, 11.0, lib=lib), [0.5, 4.0 / 6.0], what="l2norm eps")


# ---------------------------------------------------------------- a3

def pin_log_decay(lib):
    g = oracle.log_decay([0.0, 1.0, math.log(math.e - 1.0)], [0.0, -1.0, 0.0], 0.0, lib=lib)
    _close(g, [-math.log(2.0), -math.log(2.0), -1.0], what="g = -softplus(f + dt_bias) at A_log 0")
    g = oracle.log_decay([math.log(math.e - 1.0)], [0.0], math.log(2.0), lib=lib)
    _close(g, [-2.0], what="g = -exp(A_log) at softplus 1")
    g = oracle.log_decay([0.5, -3.0], [0.25, 1.0], -800.0, lib=lib)
    _close(np.exp(g), [1.0, 1.0], atol=0.0, rtol=0.0, what="exp(A_log) -> 0 gives alpha = 1")
    g = oracle.log_decay([40.0], [0.0], math.log(3.0), lib=lib)
    _close(g, [-120.0], rtol=1e-15, what="softplus(x) ~ x for large x")


def pin_log_decay_lb(lib):
    """Lower-bound gate g = lb sigmoid(-a f): closed forms and limits."""
    g = oracle.log_decay_lb([0.0, 0.0], 1.7, -3.0, lib=lib)
    _close(g, [-1.5, -1.5], what="f = 0 gives lb / 2")
    g = oracle.log_decay_lb([math.log(3.0)], 1.0, -2.0, lib=lib)
    _close(g, [-0.5], what="sigmoid(-ln 3) = 1/4")
    f = np.array([0.3, -1.2, 2.5])
    _close(oracle.log_decay_lb(f, 0.8, -1.6, lib=lib) + oracle.log_decay_lb(-f, 0.8, -1.6, lib=lib),
           np.full(3, -1.6), what="g(f) + g(-f) = lb")
    _close(oracle.log_decay_lb(f, 2.0, -1.6, lib=lib), oracle.log_decay_lb(2.0 * f, 1.0, -1.6, lib=lib),
           what="a scales f")
    g = oracle.log_decay_lb([800.0, -800.0], 1.0, -2.5, lib=lib)
    _close(np.exp(g), [1.0, math.exp(-2.5)], atol=0.0, rtol=1e-15,
           what="alpha -> 1 for large a f, exp(lb) for large -a f")


# ---------------------------------------------------------------- a5 + a6

def pin_delta_identity(lib):
    rng = np.random.default_rng(2)
    S = rng.normal(size=(3, 5))
    for i in range(3):
        q = np.zeros(3)
        q[i] = 1.0
        S2, o = oracle.delta_step(S, np.ones(3), 0.0, rng.normal(size=3), rng.normal(size=5), q,
                                  lib=lib)
        _close(S2, S, rtol=0, atol=0, what="beta 0, alpha 1: state unchanged")
        _close(o, S[i, :], what="o = S^T e_i is row i of S (row = key channel)")


def pin_delta_unit_key(lib):
    rng = np.random.default_rng(3)
    for trial in range(5):
        S = rng.normal(size=(4, 6))
        k = rng.normal(size=4)
        k /= np.linalg.norm(k)
        v = rng.normal(size=6)
        S2, _ = oracle.delta_step(S, np.ones(4), 1.0, k, v, rng.normal(size=4), lib=lib)
        _close(S2.T @ k, v, what="beta 1, |k| = 1, alpha 1: S^T k = v")


def pin_delta_full_decay(lib):
    rng = np.random.default_rng(4)
    S = rng.normal(size=(3, 4))
    k, v, q = rng.normal(size=3), rng.normal(size=4), rng.normal(size=3)
    S2, o = oracle.delta_step(S, np.zeros(3), 0.7, k, v, q, lib=lib)
    _close(S2, 0.7 * np.outer(k, v), what="alpha 0: S = beta k v^T")
    _close(o, 0.7 * v * float(k @ q), what="alpha 0: o = beta (k.q) v")


def pin_delta_bruteforce(lib):
    """Six steps against the matrix form (I - b k k^T) Diag(a) S + b k v^T, o = S^T q."""
    rng = np.random.default_rng(5)
    for d_k, d_v in ((2, 3), (3, 2), (4, 4)):
        S = rng.normal(size=(d_k, d_v))
        Sb = S.copy()
        for t in range(6):
            a = rng.uniform(0.05, 1.0, size=d_k)
            b = rng.uniform(0.0, 1.0)
            k, v, q = rng.normal(size=d_k), rng.normal(size=d_v), rng.normal(size=d_k)
            Sb = (np.eye(d_k) - b * np.outer(k, k)) @ np.diag(a) @ Sb + b * np.outer(k, v)
            S, o = oracle.delta_step(S, a, b, k, v, q, lib=lib)
            _close(S, Sb, rtol=1e-12, atol=1e-12, what=f"matrix form step {t} ({d_k}x{d_v})")
            _close(o, Sb.T @ q, what=f"readout step {t}")


# ---------------------------------------------------------------- a7

def pin_gated_rmsnorm(lib):
    rng = np.random.default_rng(6)
    o = rng.normal(size=16)
    z = np.full(16, 0.8)
    w = np.full(16, 1.3)
    y = oracle.gated_rmsnorm(o, z, w, 0.0, lib=lib)
    _close(np.mean(y ** 2), (1.3 * _silu(0.8)) ** 2, what="mean(y^2) = (w silu z)^2")
    zz, ww = rng.normal(size=16), rng.normal(size=16)
    _close(oracle.gated_rmsnorm(3.0 * o, zz, ww, 0.0, lib=lib),
           oracle.gated_rmsnorm(o, zz, ww, 0.0, lib=lib), what="scale invariance")
    e = np.zeros(16)
    e[5] = -2.0
    y = oracle.gated_rmsnorm(e, zz, ww, 0.0, lib=lib)
    want = np.zeros(16)
    want[5] = -4.0 * ww[5] * _silu(zz[5])  # rms = 2 / sqrt(16) = 1/2
    _close(y, want, what="one-hot o")
    # eps under the root: mean(o^2) = 4/16, eps = 3/4 -> rms 1
    y = oracle.gated_rmsnorm(e, np.full(16, 50.0), np.ones(16), 0.75, lib=lib)
    _close(y[5], -2.0 * _silu(50.0), what="rmsnorm eps")


def pin_gated_rmsnorm_sigmoid(lib):
    """Sigmoid output gate: z = 0 halves, and y(z) / y(-z) = e^z."""
    rng = np.random.default_rng(16)
    o, w = rng.normal(size=8), rng.normal(size=8)
    half = oracle.gated_rmsnorm(o, np.zeros(8), w, 0.0, sigmoid_gate=True, lib=lib)
    r = 1.0 / np.sqrt(np.mean(o ** 2))
    _close(half, 0.5 * o * r * w, what="sigmoid(0) = 1/2")
    z = rng.normal(size=8)
    yp = oracle.gated_rmsnorm(o, z, w, 0.0, sigmoid_gate=True, lib=lib)
    ym = oracle.gated_rmsnorm(o, -z, w, 0.0, sigmoid_gate=True, lib=lib)
    _close(yp / ym, np.exp(z), what="sigmoid(z) / sigmoid(-z) = e^z")
    y3 = oracle.gated_rmsnorm(o, np.full(8, math.log(3.0)), w, 0.0, sigmoid_gate=True, lib=lib)
    _close(y3, 0.75 * o * r * w, what="sigmoid(ln 3) = 3/4")


# ---------------------------------------------------------------- a1

def pin_conv(lib):
    shape = synth.Shape(B=2, T=6, H_qk=1, H_v=1, d_k=2, d_v=2, K=4, kda=False, bf16_in=False)
    rng = np.random.default_rng(7)
    C = shape.C
    qkv = rng.normal(size=(2, 6, C)).astype(np.float32)
    cs = rng.normal(size=(2, 3, C)).astype(np.float32)
    X = np.concatenate([cs, qkv], axis=1).astype(np.float64)   # [B, 9, C]
    for tap, scale in ((3, 1.0), (0, 1.0), (1, 2.0)):
        w = np.zeros((C, 4), dtype=np.float32)
        w[:, tap] = scale
        xh, cs2 = oracle.conv(shape, qkv, w, cs, lib=lib)
        _close(xh, _silu(scale * X[:, tap:tap + 6, :]), what=f"one-hot tap {tap}")
        _close(cs2, X[:, 6:9, :], rtol=0, atol=0, what="conv state = last K-1 rows")
    # taps add: w = [1, 0, 0, 1] -> silu(X[t] + X[t+3])
    w = np.zeros((C, 4), dtype=np.float32)
    w[:, 0] = 1.0
    w[:, 3] = 1.0
    xh, _ = oracle.conv(shape, qkv, w, cs, lib=lib)
    _close(xh, _silu(X[:, 0:6, :] + X[:, 3:9, :]), what="two taps")


# ---------------------------------------------------------------- whole-step wiring

def _identity_conv_params(shape, A_log, dt_bias):
    w = np.zeros((shape.C, shape.K), dtype=np.float32)
    w[:, shape.K - 1] = 1.0
    return synth.Params(conv_w=w, A_log=np.asarray(A_log, np.float32),
                        dt_bias=np.asarray(dt_bias, np.float32),
                        norm_w=np.linspace(0.5, 1.5, shape.d_v).astype(np.float32))


def _channels(shape, h):
    hq = h // (shape.H_v // shape.H_qk)
    q = slice(hq * shape.d_k, (hq + 1) * shape.d_k)
    k0 = shape.H_qk * shape.d_k
    k = slice(k0 + hq * shape.d_k, k0 + (hq + 1) * shape.d_k)
    v0 = 2 * shape.H_qk * shape.d_k
    v = slice(v0 + h * shape.d_v, v0 + (h + 1) * shape.d_v)
    return q, k, v


def pin_run_write_then_read(lib):
    """beta = 1 then beta = 0 with no decay and S0 = 0 (GVA: 2 value heads per qk head).

    Token 0 writes S = k0 v0^T, so o0 = (k0.q0) v0; token 1 leaves S and reads
    o1 = (k0.q1) v0.  q, k, v are the L2-normalised SiLU of the raw rows
    (identity conv), so both outputs and the final state are closed forms.
    """
    for kda in (True, False):
        sh = synth.Shape(B=2, T=2, H_qk=2, H_v=4, d_k=3, d_v=5, K=4, kda=kda, bf16_in=False,
                         eps_l2=0.0, eps_norm=0.0)
        rng = np.random.default_rng(8)
        qkv = rng.normal(size=(sh.B, sh.T, sh.C)).astype(np.float32)
        inp = synth.Inputs(qkv=qkv,
                           f=rng.normal(size=(sh.B, sh.T, sh.H_v, sh.f_width)).astype(np.float32),
                           beta=np.stack([np.full((sh.B, sh.H_v), 800.0),
                                          np.full((sh.B, sh.H_v), -800.0)], 1).astype(np.float32),
                           z=rng.normal(size=(sh.B, sh.T, sh.H_v, sh.d_v)).astype(np.float32))
        dt = np.zeros((sh.H_v, sh.d_k) if kda else (sh.H_v,), np.float32)
        prm = _identity_conv_params(sh, np.full(sh.H_v, -800.0), dt)
        cs0 = np.zeros((sh.B, sh.K - 1, sh.C), np.float32)
        S0 = np.zeros((sh.B, sh.H_v, sh.d_k, sh.d_v), np.float32)
        out = oracle.run(sh, prm, inp, cs0, S0, o_raw=True, nthreads=3, lib=lib)
        x = _silu(qkv.astype(np.float64))
        for b in range(sh.B):
            for h in range(sh.H_v):
                cq, ck, cv = _channels(sh, h)
                q = [x[b, t, cq] * sh.q_scale / np.linalg.norm(x[b, t, cq]) for t in range(2)]
                k0 = x[b, 0, ck] / np.linalg.norm(x[b, 0, ck])
                v0 = x[b, 0, cv]
                _close(out["state"][b, h], np.outer(k0, v0), what=f"S = k0 v0^T b{b} h{h}")
                for t in range(2):
                    o = float(k0 @ q[t]) * v0
                    _close(out["o_raw"][b, t, h], o, what=f"o{t} b{b} h{h}")
                    rms = np.sqrt(np.mean(o ** 2))
                    y = o / rms * prm.norm_w * _silu(inp.z[b, t, h].astype(np.float64))
                    _close(out["y"][b, t, h], y, what=f"y{t} b{b} h{h}")


def pin_run_decay_only(lib):
    """beta = 0: S_t = Diag(prod alpha) S0 with alpha = exp(-exp(A_log) softplus(f + dt_bias)),
    or alpha = exp(lb sigmoid(-a f)) for the lower-bound gate (a in A_log, lb in dt_bias)."""
    for kda, lb in ((True, False), (False, False), (True, True)):
        sh = synth.Shape(B=2, T=3, H_qk=1, H_v=2, d_k=4, d_v=3, K=4, kda=kda, bf16_in=False,
                         eps_l2=0.0, eps_norm=1e-6, lb_gate=lb)
        rng = np.random.default_rng(9)
        qkv = rng.normal(size=(sh.B, sh.T, sh.C)).astype(np.float32)
        f = rng.normal(size=(sh.B, sh.T, sh.H_v, sh.f_width)).astype(np.float32)
        inp = synth.Inputs(qkv=qkv, f=f,
                           beta=np.full((sh.B, sh.T, sh.H_v), -800.0, np.float32),
                           z=rng.normal(size=(sh.B, sh.T, sh.H_v, sh.d_v)).astype(np.float32))
        A_log = np.array([0.3, -0.4], np.float32) if not lb else np.array([1.5, 0.7], np.float32)
        dt = (rng.normal(size=(sh.H_v, sh.d_k) if kda else (sh.H_v,)).astype(np.float32)
              if not lb else np.array([-2.0, -0.6], np.float32))
        prm = _identity_conv_params(sh, A_log, dt)
        cs0 = np.zeros((sh.B, sh.K - 1, sh.C), np.float32)
        S0 = rng.normal(size=(sh.B, sh.H_v, sh.d_k, sh.d_v)).astype(np.float32)
        out = oracle.run(sh, prm, inp, cs0, S0, o_raw=True, hist=True, lib=lib)
        x = _silu(qkv.astype(np.float64))
        for b in range(sh.B):
            for h in range(sh.H_v):
                cq, _, _ = _channels(sh, h)
                S = S0[b, h].astype(np.float64)
                for t in range(sh.T):
                    fb = f[b, t, h].astype(np.float64)
                    dth = dt[h].astype(np.float64)
                    if lb:
                        a = np.exp(dth * (1.0 / (1.0 + np.exp(float(A_log[h]) * fb))))
                    else:
                        sp = np.logaddexp(0.0, fb + dth)            # softplus, library form
                        a = np.exp(-math.exp(float(A_log[h])) * sp)
                    a = np.broadcast_to(a, (sh.d_k,))
                    S = a[:, None] * S
                    q = x[b, t, cq] * sh.q_scale / np.linalg.norm(x[b, t, cq])
                    _close(out["state_hist"][t, b, h], S, what=f"decayed S t{t} b{b} h{h}")
                    _close(out["o_raw"][b, t, h], S.T @ q, what=f"o t{t} b{b} h{h}")


# ---------------------------------------------------------------- composition invariants

def _case(sh, seed, slow=False):
    prm = synth.make_params(sh, seed=seed, slow_decay=slow)
    inp = synth.make_inputs(sh, seed=seed, slow_decay=slow)
    st = synth.make_state(sh, seed=seed)
    return prm, inp, st


def pin_verify_equals_steps(lib):
    """One T-token call with per-token states == T single-token calls chained."""
    for kda in (True, False):
        sh = synth.Shape(B=2, T=5, H_qk=2, H_v=4, d_k=4, d_v=6, kda=kda, bf16_in=False)
        prm, inp, st = _case(sh, 11)
        full = oracle.run(sh, prm, inp, st.conv, st.S, hist=True, lib=lib)
        one = dataclass_replace_T(sh, 1)
        cs, S = st.conv.astype(np.float64), st.S.astype(np.float64)
        for t in range(sh.T):
            sl = synth.Inputs(qkv=inp.qkv[:, t:t + 1], f=inp.f[:, t:t + 1],
                              beta=inp.beta[:, t:t + 1], z=inp.z[:, t:t + 1])
            r = _run64(one, prm, sl, cs, S, lib)
            cs, S = r["conv_state"], r["state"]
            _close(r["y"][:, 0], full["y"][:, t], rtol=0, atol=0, what=f"y token {t}")
            _close(S, full["state_hist"][t], rtol=0, atol=0, what=f"state after token {t}")
        _close(cs, full["conv_state"], rtol=0, atol=0, what="conv state after T")
        _close(S, full["state"], rtol=0, atol=0, what="state after T")


def dataclass_replace_T(sh, T):
    import dataclasses
    return dataclasses.replace(sh, T=T)


def _run64(sh, prm, inp, cs, S, lib):
    """oracle.run taking fp64 states (keeps full precision when chaining calls)."""
    import ctypes
    cs = np.ascontiguousarray(cs, np.float64).copy()
    S = np.ascontiguousarray(S, np.float64).copy()
    y = np.empty((sh.B, sh.T, sh.H_v, sh.d_v))
    keep = [np.ascontiguousarray(a, np.float32) for a in
            (inp.qkv, inp.f, inp.beta, inp.z, prm.conv_w, prm.A_log, prm.dt_bias, prm.norm_w)]
    shp = oracle.make_shape(sh)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    rc = lib.gdn_oracle_run(ctypes.byref(shp), *[p(a) for a in keep], p(cs), p(S), p(y),
                            None, None, 2)
    assert rc == 0
    return dict(y=y, conv_state=cs, state=S)


def pin_chunked_equals_sequential(lib):
    """The chunked WY/UT form equals T sequential steps (fp64), with a partial last chunk."""
    cases = [(True, 8, 1), (True, 8, 7), (True, 8, 8), (True, 8, 9), (True, 8, 21),
             (False, 8, 21), (True, 64, 65), (False, 64, 130)]
    for kda, chunk, T in cases:
        sh = synth.Shape(B=2, T=T, H_qk=1, H_v=2, d_k=8, d_v=6, kda=kda, bf16_in=False)
        prm, inp, st = _case(sh, 12, slow=True)
        seq = oracle.run(sh, prm, inp, st.conv, st.S, lib=lib)
        chk = oracle.run_chunked(sh, prm, inp, st.conv, st.S, chunk, lib=lib)
        tag = f"kda={kda} chunk={chunk} T={T}"
        _close(chk["y"], seq["y"], rtol=1e-10, atol=1e-12, what="y " + tag)
        _close(chk["state"], seq["state"], rtol=1e-10, atol=1e-12, what="state " + tag)
        _close(chk["conv_state"], seq["conv_state"], rtol=0, atol=0, what="conv " + tag)


def pin_head_permutation(lib):
    """Swapping two value heads of one qk group (with their params) swaps their outputs."""
    sh = synth.Shape(B=1, T=3, H_qk=1, H_v=2, d_k=4, d_v=4, kda=True, bf16_in=False)
    prm, inp, st = _case(sh, 13)
    base = oracle.run(sh, prm, inp, st.conv, st.S, lib=lib)
    p = [1, 0]
    C = sh.C
    v0 = 2 * sh.H_qk * sh.d_k
    perm_ch = np.arange(C)
    perm_ch[v0:] = (v0 + np.arange(sh.H_v * sh.d_v).reshape(sh.H_v, sh.d_v)[p]).ravel()
    inp2 = synth.Inputs(qkv=inp.qkv[:, :, perm_ch], f=inp.f[:, :, p], beta=inp.beta[:, :, p],
                        z=inp.z[:, :, p])
    prm2 = synth.Params(conv_w=prm.conv_w[perm_ch], A_log=prm.A_log[p], dt_bias=prm.dt_bias[p],
                        norm_w=prm.norm_w)
    out = oracle.run(sh, prm2, inp2, st.conv[:, :, perm_ch], st.S[:, p], lib=lib)
    _close(out["y"], base["y"][:, :, p], rtol=0, atol=0, what="permuted y")
    _close(out["state"], base["state"][:, p], rtol=0, atol=0, what="permuted state")


ALL_PINS = [pin_scalars, pin_l2norm, pin_log_decay, pin_log_decay_lb, pin_delta_identity,
            pin_delta_unit_key, pin_delta_full_decay, pin_delta_bruteforce, pin_gated_rmsnorm,
            pin_gated_rmsnorm_sigmoid, pin_conv,
            pin_run_write_then_read, pin_run_decay_only, pin_verify_equals_steps,
            pin_chunked_equals_sequential, pin_head_permutation]
