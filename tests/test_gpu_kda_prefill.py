"""Chunked prefill with the per-channel decay (KDA) on the two-kernel form
("llama.cpp PR #84", chunked KDA prefill: an intra-chunk stage over all chunks,
then a state stage over the chunks), against T sequential oracle steps.

The intra-chunk kernel computes in fp32 and the state kernel's tcgen05 products
take split-fp16 operands (hi + lo, about 22 significant bits), so the path is held
to the decode bar (1e-3), tighter than the tensor-core prefill's 1e-2."""

import dataclasses

import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import DECODE_TOL, assert_close, assert_close_bf16_out, oracle_run, stream

pytestmark = pytest.mark.gpu

VARIANT = "kda_chunked<16>"


def _case(shape, seed, slow):
    return (synth.make_params(shape, seed=seed, slow_decay=slow),
            synth.make_inputs(shape, seed=seed, slow_decay=slow),
            synth.make_state(shape, seed=seed))


def _run(shape, params, inp, state, bf16_out=False):
    case = dev.upload(shape, params, inp, state, bf16_out=bf16_out)
    sh = case.abi_shape(bf16_out=bf16_out)
    assert gdn.gdn_kernel_variant(sh, gdn.OP_PREFILL) == VARIANT
    n = gdn.gdn_prefill_workspace_bytes(sh)
    nchunk = -(-shape.T // 16)
    assert n >= shape.B * shape.H_v * nchunk * 16 * 128 * 4 * 4
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    gdn.gdn_prefill_chunked(sh, case.abi_tensors(), ws.data_ptr(), n, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    return case


def _check(shape, seed=0, slow=False, bf16_out=False, tol=DECODE_TOL):
    params, inp, state = _case(shape, seed, slow)
    case = _run(shape, params, inp, state, bf16_out)
    ref = oracle_run(shape, params, inp, state)
    y = case.out.reshape(ref["y"].shape)
    if bf16_out:
        assert_close_bf16_out(y, ref["y"], "y")
    else:
        assert_close(y, ref["y"], tol, "y")
    assert_close(case.state, ref["state"], tol, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")


# lengths: one partial chunk, exact chunks, a token past a chunk, several chunks
# with a ragged tail
@pytest.mark.parametrize("T", [5, 16, 17, 33, 100, 130])
@pytest.mark.parametrize("slow", [False, True])
def test_kda_prefill_ragged_lengths(T, slow):
    shape = synth.Shape(B=2, T=T, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    _check(shape, seed=40 + T, slow=slow)


@pytest.mark.parametrize("H_qk,H_v", [(2, 8), (1, 4)])
def test_kda_prefill_grouped_heads(H_qk, H_v):
    """Value heads sharing q/k heads; the group's first head writes the q/k window."""
    shape = synth.Shape(B=3, T=70, H_qk=H_qk, H_v=H_v, d_k=128, d_v=128, kda=True, chunk=64)
    _check(shape, seed=41, slow=True)


def test_kda_prefill_bounded_gate_and_sigmoid_output():
    shape = synth.Shape(B=2, T=90, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, lb_gate=True,
                        sigmoid_out=True, chunk=64)
    _check(shape, seed=42, slow=True)


def test_kda_prefill_bf16_out():
    shape = synth.Shape(B=2, T=50, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    _check(shape, seed=43, slow=True, bf16_out=True)


def test_kda_prefill_f32_inputs():
    shape = synth.Shape(B=2, T=45, H_qk=2, H_v=2, d_k=128, d_v=128, kda=True, bf16_in=False,
                        chunk=64)
    _check(shape, seed=44, slow=True)


@pytest.mark.parametrize("bf16_in,chunk", [(False, 64), (True, 16)])
def test_per_head_gate_on_the_two_kernel_form(bf16_in, chunk):
    """Per-head decay shapes the tensor-core kernel does not take (fp32 rows, or a
    chunk length it does not run) take the same two kernels."""
    shape = synth.Shape(B=2, T=77, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False,
                        bf16_in=bf16_in, chunk=chunk)
    _check(shape, seed=45, slow=True)


def test_misaligned_output_gate_rows_take_the_recurrent_kernel():
    """The state kernel brings z in by TMA (16-byte aligned base); a z that is only
    element-aligned runs on the recurrent kernel instead, with the same results."""
    shape = synth.Shape(B=2, T=40, H_qk=2, H_v=2, d_k=128, d_v=128, kda=True, chunk=64)
    params, inp, state = _case(shape, 47, True)
    case = dev.upload(shape, params, inp, state)
    buf = torch.empty(case.z.numel() + 8, dtype=case.z.dtype, device="cuda")
    zv = buf[1:1 + case.z.numel()].view(case.z.shape)
    zv.copy_(case.z)
    case.z = zv
    assert zv.data_ptr() % 16 != 0
    sh = case.abi_shape()
    n = gdn.gdn_prefill_workspace_bytes(sh)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    gdn.gdn_prefill_chunked(sh, case.abi_tensors(), ws.data_ptr(), n, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    ref = oracle_run(shape, params, inp, state)
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], DECODE_TOL, "y")
    assert_close(case.state, ref["state"], DECODE_TOL, "state")


def test_kda_prefill_resumes_across_calls_and_matches_one_call():
    """Two calls (60 + 70 tokens, so the second starts mid-chunk in sequence
    terms) from the first call's state and window agree with one 130-token call."""
    shape = synth.Shape(B=2, T=130, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    params, inp, state = _case(shape, 46, True)
    one = _run(shape, params, inp, state)

    def part(a, b):
        return synth.Inputs(inp.qkv[:, a:b], inp.f[:, a:b], inp.beta[:, a:b], inp.z[:, a:b])

    s1 = dataclasses.replace(shape, T=60)
    c1 = _run(s1, params, part(0, 60), state)
    st = synth.State(conv=c1.conv_state.cpu().numpy(), S=c1.state.cpu().numpy())
    c2 = _run(dataclasses.replace(shape, T=70), params, part(60, 130), st)
    y = torch.cat([c1.out.reshape(2, 60, -1), c2.out.reshape(2, 70, -1)], 1)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y.reshape(ref["y"].shape), ref["y"], DECODE_TOL, "y (two calls)")
    assert_close(c2.state, ref["state"], DECODE_TOL, "state (two calls)")
    assert torch.equal(c2.conv_state, one.conv_state)
    assert_close(one.state, ref["state"], DECODE_TOL, "state (one call)")


def test_kda_prefill_b4_t4096_every_head():
    """The full-size KDA prefill (4 sequences x 4096 tokens x 32 heads) in the launch
    the bench times, against the oracle's 4096 sequential steps on every (sequence,
    head) unit: all outputs and all final states."""
    shape = synth.Shape(B=4, T=4096, H_qk=32, H_v=32, d_k=128, d_v=128, kda=True, chunk=64)
    params, inp, state = _case(shape, 0, False)
    case = _run(shape, params, inp, state)
    ref = oracle_run(shape, params, inp, state)
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], DECODE_TOL, "y")
    assert_close(case.state, ref["state"], DECODE_TOL, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")
