"""Runs the CUDA path through the C ABI and the oracle on the same seeded inputs."""

from __future__ import annotations

import dataclasses
import os

import numpy as np
import torch

import linear_attention_decode_kda_gb300 as gdn
import oracle
import synth
from synth import device as dev

DECODE_TOL = 1e-3    # max|err| / RMS(ref), fp32 state, decode and verify
PREFILL_TOL = 1e-2   # bf16 tensor-core prefill


def stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def steps_major(a: np.ndarray) -> np.ndarray:
    """[B, T, ...] -> contiguous [T, B, ...] so every step's slice is contiguous."""
    return np.ascontiguousarray(np.swapaxes(a, 0, 1))


def gpu_decode_run(shape1, params, inp, state, *, pdl=False, bf16_out=False, device="cuda"):
    """len(T) decode calls (shape1.T == 1) over inp ([B, T, ...]); returns y, state, conv."""
    steps = inp.qkv.shape[1]
    bf = shape1.bf16_in
    qkv = dev.to_torch(steps_major(inp.qkv), bf, device)
    f = dev.to_torch(steps_major(inp.f if shape1.kda else inp.f[..., 0]), bf, device)
    beta = dev.to_torch(steps_major(inp.beta), bf, device)
    z = dev.to_torch(steps_major(inp.z), bf, device)
    first = synth.Inputs(inp.qkv[:, :1], inp.f[:, :1], inp.beta[:, :1], inp.z[:, :1])
    case = dev.upload(shape1, params, first, state, device=device)
    out = torch.empty((steps, shape1.B, shape1.H_v * shape1.d_v),
                      dtype=torch.bfloat16 if bf16_out else torch.float32, device=device)
    sh = case.abi_shape(bf16_out=bf16_out, pdl=pdl)
    for t in range(steps):
        tens = gdn.tensors_from_torch(qkv=qkv[t], f=f[t], beta=beta[t], z=z[t],
                                      conv_w=case.conv_w, A_log=case.A_log, dt_bias=case.dt_bias,
                                      norm_w=case.norm_w, conv_state=case.conv_state,
                                      state=case.state, out=out[t])
        gdn.gdn_decode_step(sh, tens, stream())
    torch.cuda.synchronize()
    y = out.float().permute(1, 0, 2).reshape(shape1.B, steps, shape1.H_v, shape1.d_v)
    return y, case.state, case.conv_state


def oracle_run(shape1, params, inp, state, **kw):
    T = inp.qkv.shape[1]
    return oracle.run(dataclasses.replace(shape1, T=T), params, inp, state.conv, state.S,
                      nthreads=os.cpu_count(), **kw)


def assert_close(got, ref, tol, what):
    e = dev.rel_err(got, ref)
    assert e <= tol, f"{what}: max|err|/RMS(ref) = {e:.3e} > {tol:.0e}"
    return e


def assert_close_bf16_out(got, ref, what):
    """bf16 outputs: |got - ref| <= 2^-8 |ref| + 1e-3 RMS(ref) elementwise
    (round-to-nearest bf16 is within 2^-9 of the value, plus the fp32 path's error)."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    r = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(r ** 2)))
    bound = 2.0 ** -8 * np.abs(r) + DECODE_TOL * rms
    worst = float(np.max(np.abs(g - r) - bound))
    assert worst <= 0.0, f"{what}: bf16 output off by {worst:.3e} beyond its rounding bound"
