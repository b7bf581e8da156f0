"""A whole KDA layer's decode step (gdn_layer_decode: the projections around the
step in four launches) against the oracle's projections and step."""

import dataclasses

import numpy as np
import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import DECODE_TOL, assert_close, stream

import oracle

pytestmark = pytest.mark.gpu

# fp32 projections against fp64, relative to the rows' RMS: a sum of K <= 4096 fp32
# products, in the tensor core's order from 16 batch rows (its partial sums are
# not each rounded to fp32), stays well inside 1e-4
ROW_TOL = 1e-4


def _run(shape, d_model, rank, seed):
    s = dataclasses.replace(shape, bf16_in=False)
    params = synth.make_params(s, seed=seed)
    state = synth.make_state(s, seed=seed)
    W = synth.make_layer_weights(s, d_model, rank, seed=seed)
    x = synth.make_layer_input(s, d_model, seed=seed)
    zero = synth.Inputs(np.zeros((s.B, 1, s.C), np.float32),
                        np.zeros((s.B, 1, s.H_v, s.d_k), np.float32),
                        np.zeros((s.B, 1, s.H_v), np.float32),
                        np.zeros((s.B, 1, s.H_v, s.d_v), np.float32))
    case = dev.upload(s, params, zero, state)
    sh = case.abi_shape()
    wd = {k: dev.to_torch(getattr(W, k), True, "cuda") for k in W.FIELDS}
    wts = gdn.layer_weights_from_torch(d_model, rank, **wd)
    xs = dev.to_torch(x, True, "cuda")
    x_out = torch.empty((s.B, d_model), dtype=torch.float32, device="cuda")
    n = gdn.gdn_layer_workspace_bytes(sh, wts)
    assert n == s.B * 2 * rank * 4
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    gdn.gdn_layer_decode(sh, wts, xs, x_out, case.abi_tensors(), ws.data_ptr(), n, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    ref = oracle.layer_decode(s, params, W, x, state.conv, state.S)
    r = ref["rows"]
    assert_close(case.qkv.reshape(s.B, -1), r["qkv"], ROW_TOL, "qkv rows")
    assert_close(case.f.reshape(s.B, -1), r["f"], ROW_TOL, "f rows")
    assert_close(case.beta.reshape(s.B, -1), r["beta"], ROW_TOL, "beta rows")
    assert_close(case.z.reshape(s.B, -1), r["z"], ROW_TOL, "z rows")
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], DECODE_TOL, "y")
    assert_close(x_out, ref["x_out"], DECODE_TOL, "x_out")
    assert_close(case.state, ref["state"], DECODE_TOL, "state")
    assert_close(case.conv_state, ref["conv_state"], ROW_TOL, "conv_state")
    return x_out, case.out, case.state, case.qkv


@pytest.mark.parametrize("B", [1, 3, 9])
def test_layer_decode_small(B):
    """B = 9 takes two passes over each weight row (8 batch rows a pass)."""
    shape = synth.Shape(B=B, T=1, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True)
    _run(shape, 512, 32, seed=60 + B)


@pytest.mark.parametrize("B,rank", [(16, 64), (70, 64), (17, 32)])
def test_layer_decode_tensor_core_projections(B, rank):
    """From 16 batch rows the projections run on tcgen05 (K a multiple of 64);
    B = 70 takes two column tiles of 64; rank 32 keeps the gate pair on the
    CUDA cores."""
    shape = synth.Shape(B=B, T=1, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True)
    _run(shape, 512, rank, seed=80 + B)


def test_layer_decode_grouped_heads_bounded_gate():
    shape = synth.Shape(B=2, T=1, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, lb_gate=True,
                        sigmoid_out=True)
    _run(shape, 256, 16, seed=70)


def test_layer_decode_b64_h32_d4096():
    """The bench's batched layer: 64 sequences, 32 heads, d_model 4096, rank 128."""
    shape = synth.Shape(B=64, T=1, H_qk=32, H_v=32, d_k=128, d_v=128, kda=True)
    _run(shape, 4096, 128, seed=71)


@pytest.mark.parametrize("B,d_model,H", [(1, 4096, 32), (2, 1024, 8), (3, 1536, 12),
                                          (8, 2048, 8), (4, 2304, 8)])
def test_layer_decode_warp_mma(B, d_model, H):
    """K a multiple of 32 up to 4096 with up to 8 bf16 activation rows (the
    in-projection) or 4 fp32 rows (the output projection, each split into a bf16 value
    and a bf16 remainder): warp-level MMA.  B = 8 keeps the output projection on the
    CUDA-core ring."""
    shape = synth.Shape(B=B, T=1, H_qk=H, H_v=H, d_k=128, d_v=128, kda=True)
    _run(shape, d_model, 64, seed=90 + B)


@pytest.mark.parametrize("B,d_model,H", [(5, 3072, 8), (15, 2048, 16), (12, 1024, 8)])
def test_layer_decode_bulk_copy_ring(B, d_model, H):
    """Rows of 1024 to 4096 past the warp-MMA's batch (fp32 activations from 5 rows,
    bf16 from 9) stream through per-warp rings of bulk copies into CUDA-core FMAs."""
    shape = synth.Shape(B=B, T=1, H_qk=H, H_v=H, d_k=128, d_v=128, kda=True)
    _run(shape, d_model, 64, seed=100 + B)


def test_layer_decode_repeat_is_bitwise():
    """Fixed reduction orders: the same inputs give the same bits."""
    shape = synth.Shape(B=2, T=1, H_qk=8, H_v=8, d_k=128, d_v=128, kda=True)
    a = _run(shape, 1024, 64, seed=110)
    b = _run(shape, 1024, 64, seed=110)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_layer_decode_in_step_gates_past_48kb():
    """Eight value heads on one qk head: a whole head a CTA (step<128,128>), whose gate
    rows at rank 128 take 70 KB of shared memory, past the default 48 KB."""
    shape = synth.Shape(B=2, T=1, H_qk=1, H_v=8, d_k=128, d_v=128, kda=True)
    s = dataclasses.replace(shape, bf16_in=False)
    sh = gdn.make_shape(s.B, s.T, s.H_qk, s.H_v, s.d_k, s.d_v, kda=True, bf16_in=False,
                        q_scale=s.q_scale)
    assert gdn.gdn_kernel_variant(sh, gdn.OP_DECODE) == "step<128,128>"
    _run(shape, 1024, 128, seed=120)
