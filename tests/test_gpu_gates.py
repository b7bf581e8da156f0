"""Gate variants of the GLM KDA ("llama.cpp PR #84"): the lower-bound decay
g = lb sigmoid(-a f) per key channel and the sigmoid output gate, through every
kernel, against the oracle."""

import dataclasses

import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import (DECODE_TOL, PREFILL_TOL, assert_close, gpu_decode_run, oracle_run,
                         stream)

pytestmark = pytest.mark.gpu


def _case(shape, steps, seed=0, slow=False):
    sT = dataclasses.replace(shape, T=steps)
    return (synth.make_params(shape, seed=seed, slow_decay=slow),
            synth.make_inputs(sT, seed=seed, slow_decay=slow),
            synth.make_state(shape, seed=seed))


@pytest.mark.parametrize("B,lb,sig,slow", [
    (64, True, False, False),    # streaming kernel, bounded decay
    (64, False, True, False),    # streaming kernel, sigmoid output gate
    (64, True, True, True),      # both, slow decay (state carried)
    (1, True, True, False),      # column slabs
    (2, True, False, True),
])
def test_decode_gate_variants_match_the_oracle(B, lb, sig, slow):
    shape = synth.Shape(B=B, T=1, H_qk=32, H_v=32, d_k=128, d_v=128, kda=True, lb_gate=lb,
                        sigmoid_out=sig)
    params, inp, state = _case(shape, 12, seed=21, slow=slow)
    y, S, cs = gpu_decode_run(shape, params, inp, state)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")
    assert_close(cs, ref["conv_state"], 0.0, "conv_state")


def test_gdn_sigmoid_gate_grouped_heads():
    shape = synth.Shape(B=4, T=1, H_qk=4, H_v=8, d_k=64, d_v=64, kda=False, sigmoid_out=True)
    params, inp, state = _case(shape, 8, seed=22)
    y, S, _ = gpu_decode_run(shape, params, inp, state)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")


@pytest.mark.parametrize("B", [32, 1])
def test_verify_gate_variants_bitwise_equal_decode(B):
    shape = synth.Shape(B=B, T=4, H_qk=32, H_v=32, d_k=128, d_v=128, kda=True, lb_gate=True,
                        sigmoid_out=True)
    params, inp, state = _case(shape, 4, seed=23)
    case = dev.upload(shape, params, inp, state, hist=True)
    gdn.gdn_verify_T(case.abi_shape(), case.abi_tensors(), stream())
    torch.cuda.synchronize()
    y, S, _ = gpu_decode_run(dataclasses.replace(shape, T=1), params, inp, state)
    assert torch.equal(y.reshape(case.out.shape), case.out)
    assert torch.equal(S, case.state_hist[-1])
    ref = oracle_run(dataclasses.replace(shape, T=1), params, inp, state, hist=True)
    assert_close(case.state_hist, ref["state_hist"], DECODE_TOL, "state_hist")


@pytest.mark.parametrize("shape,tol,variant", [
    # chunked tensor-core prefill with the sigmoid output gate (GDN gate)
    (synth.Shape(B=2, T=200, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, sigmoid_out=True,
                 chunk=32), PREFILL_TOL, "chunked<128,32>"),
    # the 64-token tensor-core kernel
    (synth.Shape(B=2, T=200, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, sigmoid_out=True),
     PREFILL_TOL, "chunked<128,64>"),
    # and the two-kernel form
    (synth.Shape(B=2, T=200, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, sigmoid_out=True,
                 chunk=16), DECODE_TOL, "kda_chunked<16>"),
    # the bounded per-channel gate on the two-kernel chunked form
    (synth.Shape(B=2, T=70, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, lb_gate=True,
                 sigmoid_out=True), DECODE_TOL, "kda_chunked<16>"),
    # and on the recurrent kernel (d = 64 has no chunked form)
    (synth.Shape(B=2, T=40, H_qk=2, H_v=4, d_k=64, d_v=64, kda=True, lb_gate=True,
                 sigmoid_out=True), DECODE_TOL, None),
])
def test_prefill_gate_variants(shape, tol, variant):
    params, inp, state = _case(shape, shape.T, seed=24, slow=True)
    case = dev.upload(shape, params, inp, state)
    sh = case.abi_shape()
    if variant is not None:
        assert gdn.gdn_kernel_variant(sh, gdn.OP_PREFILL) == variant
    n = gdn.gdn_prefill_workspace_bytes(sh)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    gdn.gdn_prefill_chunked(sh, case.abi_tensors(), ws.data_ptr(), n, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    ref = oracle_run(dataclasses.replace(shape, T=1), params, inp, state)
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], tol, "y")
    assert_close(case.state, ref["state"], tol, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")
