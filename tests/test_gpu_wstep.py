"""The warp-column step kernel (d = 128, from 128 (sequence, head) units): decode
against the oracle for every gate form, grouped heads, input and output types;
verify equal to T decode calls bit for bit; commit of accepted tokens equal to
verify's history.  The recurrence is the one of "Thirty tiny kernels per layer"
(KDA decode) and "llama.cpp PR #84" (gated delta rule with a state column per warp).
"""

import dataclasses

import numpy as np
import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import (DECODE_TOL, assert_close, assert_close_bf16_out, gpu_decode_run,
                         oracle_run, stream)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(shape, steps, seed=0, slow=False):
    sT = dataclasses.replace(shape, T=steps)
    return (synth.make_params(shape, seed=seed, slow_decay=slow),
            synth.make_inputs(sT, seed=seed, slow_decay=slow),
            synth.make_state(shape, seed=seed))


def _shape(B, H_qk, H_v, T=1, **kw):
    return synth.Shape(B=B, T=T, H_qk=H_qk, H_v=H_v, d_k=128, d_v=128, **kw)


def _abi(s):
    return gdn.make_shape(s.B, s.T, s.H_qk, s.H_v, s.d_k, s.d_v, kda=s.kda, bf16_in=s.bf16_in,
                          q_scale=s.q_scale, lb_gate=s.lb_gate, sigmoid_gate=s.sigmoid_out)


# (B, H_qk, H_v, variant): two 64-column slabs a head (clusters of 2 x group), and
# whole heads when a group of 8 value heads shares one qk head
ROUTES = [(4, 16, 32, "wstep<128,64>"), (8, 8, 16, "wstep<128,64>"),
          (4, 8, 32, "wstep<128,64>"), (2, 8, 64, "wstep<128,128>")]


@pytest.mark.parametrize("B,H_qk,H_v,variant", ROUTES)
@pytest.mark.parametrize("kda", [True, False])
def test_decode_matches_the_oracle(B, H_qk, H_v, variant, kda):
    shape = _shape(B, H_qk, H_v, kda=kda)
    assert gdn.gdn_kernel_variant(_abi(shape), gdn.OP_DECODE) == variant
    params, inp, state = _case(shape, 6, seed=31)
    y, S, cs = gpu_decode_run(shape, params, inp, state)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")
    assert_close(cs, ref["conv_state"], 0.0, "conv_state")


@pytest.mark.parametrize("lb,sig", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("H_qk", [32, 16])
def test_gate_variants(lb, sig, H_qk):
    """32 ungrouped heads at B4 stream; pairs of value heads take the warp-column kernel."""
    shape = _shape(4, H_qk, 32, kda=True, lb_gate=lb, sigmoid_out=sig)
    params, inp, state = _case(shape, 8, seed=32, slow=True)
    y, S, cs = gpu_decode_run(shape, params, inp, state)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")
    assert_close(cs, ref["conv_state"], 0.0, "conv_state")


def test_fp32_inputs_and_bf16_out():
    shape = _shape(4, 32, 32, kda=True, bf16_in=False)
    params, inp, state = _case(shape, 3, seed=33)
    y, S, _ = gpu_decode_run(shape, params, inp, state)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")
    shape = _shape(8, 8, 16, kda=True)
    params, inp, state = _case(shape, 3, seed=34)
    y, S, _ = gpu_decode_run(shape, params, inp, state, bf16_out=True)
    ref = oracle_run(shape, params, inp, state)
    assert_close_bf16_out(y, ref["y"], "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")


def test_slow_decay_long_run():
    """Slow per-channel decay (the state survives many tokens), 48 steps."""
    shape = _shape(4, 32, 32, kda=True)
    params, inp, state = _case(shape, 48, seed=35, slow=True)
    y, S, _ = gpu_decode_run(shape, params, inp, state, pdl=True)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("B,H_qk,H_v", [(4, 32, 32), (2, 8, 64)])
def test_verify_equals_decode_bitwise(T, B, H_qk, H_v):
    shape = _shape(B, H_qk, H_v, T=T, kda=True)
    params, inp, state = _case(shape, T, seed=36)
    case = dev.upload(shape, params, inp, state, hist=True, conv_hist=True)
    S0, cs0 = case.state.clone(), case.conv_state.clone()
    gdn.gdn_verify_T(case.abi_shape(), case.abi_tensors(), stream())
    torch.cuda.synchronize()
    assert torch.equal(case.state, S0) and torch.equal(case.conv_state, cs0), "verify wrote state"
    y, S, cs = gpu_decode_run(dataclasses.replace(shape, T=1), params, inp, state)
    assert torch.equal(y.reshape(case.out.shape), case.out)
    assert torch.equal(S, case.state_hist[-1])
    assert torch.equal(cs, case.conv_hist[-1])
    ref = oracle_run(dataclasses.replace(shape, T=1), params, inp, state, hist=True)
    assert_close(case.state_hist, ref["state_hist"], DECODE_TOL, "state_hist")


def test_commit_accepted_equals_verify_history():
    T, B = 4, 8
    shape = _shape(B, 8, 16, T=T, kda=True)
    params, inp, state = _case(shape, T, seed=37)
    ref = dev.upload(shape, params, inp, state, hist=True, conv_hist=True)
    gdn.gdn_verify_T(ref.abi_shape(), ref.abi_tensors(), stream())
    acc = np.arange(B, dtype=np.int32) % (T + 1)
    case = dev.upload(shape, params, inp, state)
    case.out.fill_(float("nan"))
    S0, cs0 = case.state.clone(), case.conv_state.clone()
    gdn.gdn_commit_accepted(case.abi_shape(), case.abi_tensors(), torch.from_numpy(acc).cuda(),
                            stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    out, ref_out = case.out.reshape(B, T, -1), ref.out.reshape(B, T, -1)
    for b in range(B):
        k = int(acc[b])
        if k == 0:
            assert torch.equal(case.state[b], S0[b]) and torch.equal(case.conv_state[b], cs0[b])
        else:
            assert torch.equal(case.state[b], ref.state_hist[k - 1, b]), f"state b={b} k={k}"
            assert torch.equal(case.conv_state[b], ref.conv_hist[k - 1, b]), f"conv b={b} k={k}"
        assert torch.equal(out[b, :k], ref_out[b, :k])
        assert torch.isnan(out[b, k:]).all(), "rows past the accepted tokens were written"
