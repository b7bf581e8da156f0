"""Verify without per-token states and the in-place commit of accepted tokens
("opus_gdn_qsa" audit, the gdn_step commit / verify modes) against verify with
history (bit for bit: the same per-token arithmetic) and against the oracle."""

import dataclasses

import numpy as np
import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import DECODE_TOL, assert_close, oracle_run, stream

pytestmark = pytest.mark.gpu


def _case(shape, seed=0):
    return (synth.make_params(shape, seed=seed), synth.make_inputs(shape, seed=seed),
            synth.make_state(shape, seed=seed))


def _verify_with_history(shape, params, inp, state):
    case = dev.upload(shape, params, inp, state, hist=True, conv_hist=True)
    gdn.gdn_verify_T(case.abi_shape(), case.abi_tensors(), stream())
    torch.cuda.synchronize()
    return case


# (B, H_qk, H_v): streaming kernel (1024 heads), column slabs (one sequence),
# grouped heads on clustered slabs
SHAPES = [(32, 32, 32), (1, 32, 32), (4, 4, 8)]


@pytest.mark.parametrize("B,H_qk,H_v", SHAPES)
def test_verify_without_history_writes_outputs_only(B, H_qk, H_v):
    shape = synth.Shape(B=B, T=4, H_qk=H_qk, H_v=H_v, d_k=128, d_v=128, kda=True)
    params, inp, state = _case(shape, seed=11)
    ref = _verify_with_history(shape, params, inp, state)
    case = dev.upload(shape, params, inp, state)  # no state_hist, no conv_hist
    S0, cs0 = case.state.clone(), case.conv_state.clone()
    gdn.gdn_verify_T(case.abi_shape(), case.abi_tensors(), stream())
    torch.cuda.synchronize()
    assert torch.equal(case.out, ref.out)
    assert torch.equal(case.state, S0) and torch.equal(case.conv_state, cs0)


@pytest.mark.parametrize("B,H_qk,H_v", SHAPES)
def test_commit_accepted_equals_verify_history(B, H_qk, H_v):
    T = 4
    shape = synth.Shape(B=B, T=T, H_qk=H_qk, H_v=H_v, d_k=128, d_v=128, kda=True)
    params, inp, state = _case(shape, seed=12)
    ref = _verify_with_history(shape, params, inp, state)
    acc = np.arange(B, dtype=np.int32) % (T + 1)          # 0, 1, ..., T, 0, ...
    if B == 1:
        acc[:] = 3
    case = dev.upload(shape, params, inp, state)
    case.out.fill_(float("nan"))
    S0, cs0 = case.state.clone(), case.conv_state.clone()
    accepted = torch.from_numpy(acc).cuda()
    gdn.gdn_commit_accepted(case.abi_shape(), case.abi_tensors(), accepted, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    out = case.out.reshape(B, T, -1)
    ref_out = ref.out.reshape(B, T, -1)
    for b in range(B):
        k = int(acc[b])
        if k == 0:
            assert torch.equal(case.state[b], S0[b]) and torch.equal(case.conv_state[b], cs0[b])
        else:
            assert torch.equal(case.state[b], ref.state_hist[k - 1, b]), f"state b={b} k={k}"
            assert torch.equal(case.conv_state[b], ref.conv_hist[k - 1, b]), f"conv b={b} k={k}"
        assert torch.equal(out[b, :k], ref_out[b, :k])
        assert torch.isnan(out[b, k:]).all(), "rows past the accepted tokens were written"


def test_commit_all_matches_the_oracle_and_leaves_out_alone_when_null():
    shape = synth.Shape(B=32, T=3, H_qk=32, H_v=32, d_k=128, d_v=128, kda=True)
    params, inp, state = _case(shape, seed=13)
    case = dev.upload(shape, params, inp, state)
    t = case.abi_tensors()
    t.out = None
    gdn.gdn_commit_accepted(case.abi_shape(), t, None, stream())
    torch.cuda.synchronize()
    ref = oracle_run(dataclasses.replace(shape, T=1), params, inp, state)
    assert_close(case.state, ref["state"], DECODE_TOL, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")


def test_commit_k_matches_the_oracle_for_k_tokens():
    """Sequences accept 2 of 4 tokens: the state is the oracle's after 2 steps."""
    shape = synth.Shape(B=2, T=4, H_qk=2, H_v=4, d_k=64, d_v=64, kda=False, bf16_in=False)
    params, inp, state = _case(shape, seed=14)
    case = dev.upload(shape, params, inp, state)
    accepted = torch.full((shape.B,), 2, dtype=torch.int32, device="cuda")
    gdn.gdn_commit_accepted(case.abi_shape(), case.abi_tensors(), accepted, stream())
    torch.cuda.synchronize()
    two = synth.Inputs(inp.qkv[:, :2], inp.f[:, :2], inp.beta[:, :2], inp.z[:, :2])
    ref = oracle_run(dataclasses.replace(shape, T=1), params, two, state)
    assert_close(case.state, ref["state"], DECODE_TOL, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")
    assert_close(case.out.reshape(shape.B, 4, shape.H_v, shape.d_v)[:, :2], ref["y"], DECODE_TOL, "y")
