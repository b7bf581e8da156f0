"""Snapshot tails of the chunked prefill ("llama.cpp PR #84", the chunked
prefill's snapshot slots): with state_hist / conv_hist set, gdn_prefill_chunked
also returns the state and the conv window after each of the last n = min(T, 4)
tokens, so a caller can roll back to any of them.

Each snapshot is compared with the oracle's state after that token (its
sequential run with per-token states) at the decode bar, 1e-3 (the 32-token
kernel's head at its own 1e-2 bar), and each window
bit for bit with the oracle's window after a run of that many tokens; outputs,
final state and final window are checked as for the plain prefill."""

import dataclasses

import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import DECODE_TOL, PREFILL_TOL, assert_close, oracle_run, stream

pytestmark = pytest.mark.gpu


def _inputs_upto(inp, k):
    return synth.Inputs(inp.qkv[:, :k], inp.f[:, :k], inp.beta[:, :k], inp.z[:, :k])


def _run(shape, seed, *, with_state=True, with_conv=True, static=False, variant=None,
         y_tol=DECODE_TOL, s_tol=DECODE_TOL):
    params = synth.make_params(shape, seed=seed, slow_decay=True)
    inp = synth.make_inputs(shape, seed=seed, slow_decay=True)
    state = synth.make_state(shape, seed=seed)
    case = dev.upload(shape, params, inp, state)
    n = min(shape.T, 4)
    C = shape.C
    sh_t = torch.full((n, shape.B, shape.H_v, shape.d_k, shape.d_v), float("nan"), device="cuda")
    ch_t = torch.full((n, shape.B, 3, C), float("nan"), device="cuda")
    tens = case.abi_tensors()
    tens.state_hist = sh_t.data_ptr() if with_state else None
    tens.conv_hist = ch_t.data_ptr() if with_conv else None
    sh = case.abi_shape()
    if variant is not None:
        assert gdn.gdn_kernel_variant(sh, gdn.OP_PREFILL) == variant
    if static:
        gdn.gdn_prefill_chunked_static(sh, tens, stream())
    else:
        nb = gdn.gdn_prefill_workspace_bytes(sh)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
        gdn.gdn_prefill_chunked(sh, tens, ws.data_ptr(), nb, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()

    ref = oracle_run(shape, params, inp, state, hist=True)
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], y_tol, "y")
    assert_close(case.state, ref["state"], s_tol, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")
    T = shape.T
    for k in range(n):
        tok = T - n + k  # the snapshot after this token
        if with_state:
            assert_close(sh_t[k], ref["state_hist"][tok], s_tol, f"state_hist[{k}]")
        if with_conv:
            part = oracle_run(dataclasses.replace(shape, T=tok + 1), params, _inputs_upto(inp, tok + 1),
                              state)
            assert_close(ch_t[k], part["conv_state"], 0.0, f"conv_hist[{k}]")
    if with_state:
        assert torch.equal(sh_t[n - 1], case.state), "the last snapshot is the final state"
    if with_conv:
        assert torch.equal(ch_t[n - 1], case.conv_state), "the last window is the final window"


def test_gdn_chunk64_head_and_recurrent_tail():
    shape = synth.Shape(B=2, T=200, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=64)
    _run(shape, 70, variant="chunked<128,64>", y_tol=PREFILL_TOL)


def test_kda_two_kernel_head_and_recurrent_tail():
    shape = synth.Shape(B=2, T=100, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    _run(shape, 71, variant="kda_chunked<16>")


def test_gdn_chunk32_head():
    """The 32-token kernel's states carry its tensor-core prefill error (the 1e-2
    bar); the tail adds the recurrent kernel's."""
    shape = synth.Shape(B=3, T=77, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=32)
    _run(shape, 72, variant="chunked<128,32>", y_tol=PREFILL_TOL, s_tol=PREFILL_TOL)


@pytest.mark.parametrize("T", [1, 3, 4, 5, 6])
def test_short_runs(T):
    """T <= 4: every token is a snapshot (no head); T = 5, 6: a head of one or two
    tokens, on the 64-token kernel (GDN) and on the recurrent kernel (KDA)."""
    _run(synth.Shape(B=2, T=T, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=64), 73 + T,
         y_tol=PREFILL_TOL)
    _run(synth.Shape(B=2, T=T, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, chunk=64), 80 + T)


def test_recurrent_head_at_d64():
    """d = 64 has no chunked form: head and tail both on the recurrent kernel."""
    shape = synth.Shape(B=2, T=40, H_qk=2, H_v=4, d_k=64, d_v=64, kda=True, chunk=64)
    _run(shape, 90)


def test_state_only_and_window_only():
    shape = synth.Shape(B=2, T=70, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    _run(shape, 91, with_conv=False)
    _run(shape, 92, with_state=False)


def test_static_scratch_entry_point_takes_snapshots_too():
    shape = synth.Shape(B=1, T=90, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    _run(shape, 93, static=True)
