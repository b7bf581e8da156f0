"""The state and the conv window are the checkpoint: calls resume where the last
one stopped (prefill -> prefill, prefill -> decode), and replaying steps from a
restored state gives the same bits."""

import dataclasses

import numpy as np
import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import DECODE_TOL, PREFILL_TOL, assert_close, gpu_decode_run, oracle_run, stream

pytestmark = pytest.mark.gpu


def _case(shape, steps, seed, slow=True):
    sT = dataclasses.replace(shape, T=steps)
    return (synth.make_params(shape, seed=seed, slow_decay=slow),
            synth.make_inputs(sT, seed=seed, slow_decay=slow),
            synth.make_state(shape, seed=seed))


def _slice(inp, t0, t1):
    return synth.Inputs(inp.qkv[:, t0:t1], inp.f[:, t0:t1], inp.beta[:, t0:t1], inp.z[:, t0:t1])


@pytest.mark.parametrize("B", [64, 1])
def test_replay_from_a_restored_state_is_bitwise_identical(B):
    shape = synth.Shape(B=B, T=1, H_qk=32, H_v=32, d_k=128, d_v=128)
    params, inp, state = _case(shape, 6, seed=31, slow=False)
    y1, S1, c1 = gpu_decode_run(shape, params, inp, state)
    y2, S2, c2 = gpu_decode_run(shape, params, inp, state)
    assert torch.equal(y1, y2) and torch.equal(S1, S2) and torch.equal(c1, c2)


def _prefill(shape, params, inp, S, conv):
    """Prefill of inp's tokens from (S, conv); returns y, state, conv window (device)."""
    T = inp.qkv.shape[1]
    sh = dataclasses.replace(shape, T=T)
    st = synth.State(conv=conv, S=S)
    case = dev.upload(sh, params, inp, st)
    abi = case.abi_shape()
    n = gdn.gdn_prefill_workspace_bytes(abi)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    gdn.gdn_prefill_chunked(abi, case.abi_tensors(), ws.data_ptr(), n, stream())
    torch.cuda.synchronize()
    return case.out.reshape(shape.B, T, shape.H_v, shape.d_v), case.state, case.conv_state


GDN = synth.Shape(B=2, T=1, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False)


def test_prefill_resumes_across_calls():
    params, inp, state = _case(GDN, 130, seed=32)
    y1, S1, c1 = _prefill(GDN, params, _slice(inp, 0, 60), state.S, state.conv)
    y2, S2, c2 = _prefill(GDN, params, _slice(inp, 60, 130), S1.cpu().numpy(), c1.cpu().numpy())
    ref = oracle_run(GDN, params, inp, state)
    assert_close(torch.cat([y1, y2], 1), ref["y"], PREFILL_TOL, "y")
    assert_close(S2, ref["state"], PREFILL_TOL, "state")
    assert_close(c2, ref["conv_state"], 0.0, "conv_state")


def test_decode_resumes_after_prefill():
    params, inp, state = _case(GDN, 108, seed=33)
    y1, S1, c1 = _prefill(GDN, params, _slice(inp, 0, 100), state.S, state.conv)
    st = synth.State(conv=c1.cpu().numpy(), S=S1.cpu().numpy())
    y2, S2, c2 = gpu_decode_run(GDN, params, _slice(inp, 100, 108), st)
    ref = oracle_run(GDN, params, inp, state)
    assert_close(torch.cat([y1, y2], 1), ref["y"], PREFILL_TOL, "y")
    assert_close(S2, ref["state"], PREFILL_TOL, "state")
    assert_close(c2, ref["conv_state"], 0.0, "conv_state")
    # the decode steps themselves, against the oracle from the prefill's state
    ref_tail = oracle_run(GDN, params, _slice(inp, 100, 108), st)
    assert_close(y2, ref_tail["y"], DECODE_TOL, "y after prefill")
    assert np.isfinite(S2.cpu().numpy()).all()
