"""The 64-token chunked prefill on tcgen05 ("chunked<128,64>": per-head decay,
d = 128, bf16 rows), against T sequential oracle steps ("llama.cpp PR #84", the
chunked prefill; the per-token step of "Thirty tiny kernels per layer").

Every product takes split-fp16 operands (about 22 significant bits) with fp32
accumulation; the bar is the bf16 tensor-core prefill's, max|err| / RMS(ref) <=
1e-2, on outputs and final states, and the conv window is exact."""

import dataclasses

import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev

from gpu_harness import PREFILL_TOL, assert_close, assert_close_bf16_out, oracle_run, stream

pytestmark = pytest.mark.gpu

VARIANT = "chunked<128,64>"


def _case(shape, seed, slow):
    return (synth.make_params(shape, seed=seed, slow_decay=slow),
            synth.make_inputs(shape, seed=seed, slow_decay=slow),
            synth.make_state(shape, seed=seed))


def _run(shape, params, inp, state, bf16_out=False, variant=VARIANT):
    case = dev.upload(shape, params, inp, state, bf16_out=bf16_out)
    sh = case.abi_shape(bf16_out=bf16_out)
    assert gdn.gdn_kernel_variant(sh, gdn.OP_PREFILL) == variant
    assert gdn.gdn_prefill_workspace_bytes(sh) == 0
    gdn.gdn_prefill_chunked(sh, case.abi_tensors(), 0, 0, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    return case


def _check(shape, seed=0, slow=False, bf16_out=False):
    params, inp, state = _case(shape, seed, slow)
    case = _run(shape, params, inp, state, bf16_out)
    ref = oracle_run(shape, params, inp, state)
    y = case.out.reshape(ref["y"].shape)
    if bf16_out:
        assert_close_bf16_out(y, ref["y"], "y")
    else:
        assert_close(y, ref["y"], PREFILL_TOL, "y")
    assert_close(case.state, ref["state"], PREFILL_TOL, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")


# shorter than the conv window, one partial chunk, exact chunks, one past a
# chunk, several chunks with a ragged tail
@pytest.mark.parametrize("T", [1, 2, 3, 17, 64, 128, 129, 250])
@pytest.mark.parametrize("slow", [False, True])
def test_ragged_lengths(T, slow):
    shape = synth.Shape(B=2, T=T, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=64)
    _check(shape, seed=60 + T, slow=slow)


@pytest.mark.parametrize("H_qk,H_v", [(4, 4), (1, 2), (2, 8), (1, 8)])
def test_head_groups(H_qk, H_v):
    """Value heads sharing a qk head run as a thread-block cluster (up to 8 CTAs);
    the group's first head writes the shared q/k conv window."""
    shape = synth.Shape(B=3, T=100, H_qk=H_qk, H_v=H_v, d_k=128, d_v=128, kda=False, chunk=64)
    _check(shape, seed=61, slow=True)


def test_bf16_out():
    shape = synth.Shape(B=2, T=150, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=64)
    _check(shape, seed=62, slow=True, bf16_out=True)


def test_resumes_across_calls():
    """Two calls (90 + 110 tokens, the second starting mid-chunk in sequence terms)
    from the first call's state and window match the oracle over all 200 tokens."""
    shape = synth.Shape(B=2, T=200, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=64)
    params, inp, state = _case(shape, 63, True)

    def part(a, b):
        return synth.Inputs(inp.qkv[:, a:b], inp.f[:, a:b], inp.beta[:, a:b], inp.z[:, a:b])

    c1 = _run(dataclasses.replace(shape, T=90), params, part(0, 90), state)
    st = synth.State(conv=c1.conv_state.cpu().numpy(), S=c1.state.cpu().numpy())
    c2 = _run(dataclasses.replace(shape, T=110), params, part(90, 200), st)
    y = torch.cat([c1.out.reshape(2, 90, -1), c2.out.reshape(2, 110, -1)], 1)
    ref = oracle_run(shape, params, inp, state)
    assert_close(y.reshape(ref["y"].shape), ref["y"], PREFILL_TOL, "y (two calls)")
    assert_close(c2.state, ref["state"], PREFILL_TOL, "state (two calls)")
    assert_close(c2.conv_state, ref["conv_state"], 0.0, "conv_state (two calls)")


def test_repeat_calls_are_bitwise_identical():
    """The same inputs give the same bits on a second call (no order-dependent
    reduction, no stale shared memory)."""
    shape = synth.Shape(B=4, T=300, H_qk=4, H_v=8, d_k=128, d_v=128, kda=False, chunk=64)
    params, inp, state = _case(shape, 64, False)
    a = _run(shape, params, inp, state)
    b = _run(shape, params, inp, state)
    assert torch.equal(a.out, b.out)
    assert torch.equal(a.state, b.state)
    assert torch.equal(a.conv_state, b.conv_state)


def test_unaligned_rows_take_the_recurrent_kernel():
    """q/k/v rows arrive by TMA (16-byte aligned base); rows that are only
    element-aligned run on the recurrent kernel, with the same results."""
    shape = synth.Shape(B=2, T=80, H_qk=2, H_v=2, d_k=128, d_v=128, kda=False, chunk=64)
    params, inp, state = _case(shape, 65, True)
    case = dev.upload(shape, params, inp, state)
    buf = torch.empty(case.qkv.numel() + 8, dtype=case.qkv.dtype, device="cuda")
    qv = buf[1:1 + case.qkv.numel()].view(case.qkv.shape)
    qv.copy_(case.qkv)
    case.qkv = qv
    assert qv.data_ptr() % 16 != 0
    sh = case.abi_shape()
    assert gdn.gdn_prefill_workspace_bytes(sh) == 0
    gdn.gdn_prefill_chunked(sh, case.abi_tensors(), 0, 0, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    ref = oracle_run(shape, params, inp, state)
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], PREFILL_TOL, "y")
    assert_close(case.state, ref["state"], PREFILL_TOL, "state")
