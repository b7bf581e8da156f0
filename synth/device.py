"""Copies a synthetic case to the GPU as torch tensors in the ABI's layouts.

Harness code shared by the GPU tests and the benchmark: it holds none of the
method's arithmetic (only dtype conversion and buffer allocation).
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import Inputs, Params, Shape, State, f32_to_bf16_bits


def to_torch(a: np.ndarray, bf16: bool, device) -> torch.Tensor:
    """fp32 numpy array -> torch tensor (bf16 from the exact bf16 bits, or fp32)."""
    if bf16:
        bits = f32_to_bf16_bits(np.ascontiguousarray(a, np.float32))
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(device) if device is not None else t


@dataclasses.dataclass
class DeviceCase:
    shape: Shape
    qkv: torch.Tensor
    f: torch.Tensor
    beta: torch.Tensor
    z: torch.Tensor
    conv_w: torch.Tensor
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    norm_w: torch.Tensor
    conv_state: torch.Tensor
    state: torch.Tensor
    out: torch.Tensor
    state_hist: Optional[torch.Tensor] = None
    conv_hist: Optional[torch.Tensor] = None

    def abi_tensors(self):
        import linear_attention_decode_kda_gb300 as gdn
        return gdn.tensors_from_torch(qkv=self.qkv, f=self.f, beta=self.beta, z=self.z,
                                      conv_w=self.conv_w, A_log=self.A_log,
                                      dt_bias=self.dt_bias, norm_w=self.norm_w,
                                      conv_state=self.conv_state, state=self.state, out=self.out,
                                      state_hist=self.state_hist, conv_hist=self.conv_hist)

    def abi_shape(self, bf16_out: bool = False, pdl: bool = False):
        import linear_attention_decode_kda_gb300 as gdn
        s = self.shape
        return gdn.make_shape(s.B, s.T, s.H_qk, s.H_v, s.d_k, s.d_v, kda=s.kda,
                              bf16_in=s.bf16_in, bf16_out=bf16_out, conv_K=s.K, chunk=s.chunk,
                              q_scale=s.q_scale, eps_l2=s.eps_l2, eps_norm=s.eps_norm, pdl=pdl,
                              lb_gate=s.lb_gate, sigmoid_gate=s.sigmoid_out)


def upload(shape: Shape, params: Params, inputs: Inputs, state: State, device="cuda",
           bf16_out: bool = False, hist: bool = False, conv_hist: bool = False) -> DeviceCase:
    s = shape
    bf = s.bf16_in
    out = torch.empty((s.B, s.T, s.H_v * s.d_v),
                      dtype=torch.bfloat16 if bf16_out else torch.float32, device=device)
    f = inputs.f if s.kda else inputs.f.reshape(s.B, s.T, s.H_v)
    dc = DeviceCase(
        shape=s,
        qkv=to_torch(inputs.qkv, bf, device), f=to_torch(f, bf, device),
        beta=to_torch(inputs.beta, bf, device), z=to_torch(inputs.z, bf, device),
        conv_w=to_torch(params.conv_w, False, device), A_log=to_torch(params.A_log, False, device),
        dt_bias=to_torch(params.dt_bias, False, device),
        norm_w=to_torch(params.norm_w, False, device),
        conv_state=to_torch(state.conv, False, device), state=to_torch(state.S, False, device),
        out=out)
    if hist:
        dc.state_hist = torch.empty((s.T, s.B, s.H_v, s.d_k, s.d_v), dtype=torch.float32,
                                    device=device)
    if conv_hist:
        dc.conv_hist = torch.empty((s.T, s.B, s.K - 1, s.C), dtype=torch.float32, device=device)
    return dc


def rel_err(got, ref) -> float:
    """max |got - ref| / RMS(ref), both taken to fp64 on the host."""
    if isinstance(got, torch.Tensor):
        got = got.detach().float().cpu().numpy()
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-30)
