"""gdn_prefill_chunked_static: the prefill on the library's static scratch,
for callers that cannot allocate device memory around the call.

Two calls in a row on the static scratch (the second reuses what the first
left there) must match gdn_prefill_chunked with a caller workspace bit for
bit: the same kernels run on the same inputs.  The file sorts last so the
GPU test also runs after every other test has used the device."""

import ctypes

import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from synth import device as dev


def _shape(**kw):
    base = dict(B=2, T=100, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, bf16_in=True,
                q_scale=0.08838835)
    base.update(kw)
    return gdn.make_shape(**base)


def _fake_tensors():
    names = [n for n, _ in gdn.GdnTensors._fields_]
    return gdn.GdnTensors(**{n: 0x10000 + 0x1000 * i for i, n in enumerate(names)})


def test_scratch_limit_is_checked_before_anything_is_queued():
    """A shape whose workspace exceeds the scratch is refused on the host."""
    lib = gdn.load()
    s = _shape(B=1, T=1024, H_qk=32, H_v=32)
    assert gdn.gdn_prefill_workspace_bytes(s) > gdn.PREFILL_STATIC_SCRATCH_BYTES
    rc = lib.gdn_prefill_chunked_static(ctypes.byref(s), ctypes.byref(_fake_tensors()), None)
    assert rc == gdn.GDN_ERR_WORKSPACE
    # 480 tokens of one 32-head sequence (30 chunks of 16) are the most that fit
    s = _shape(B=1, T=480, H_qk=32, H_v=32)
    assert gdn.gdn_prefill_workspace_bytes(s) <= gdn.PREFILL_STATIC_SCRATCH_BYTES
    s.T = 481
    assert gdn.gdn_prefill_workspace_bytes(s) > gdn.PREFILL_STATIC_SCRATCH_BYTES
    # the ordinary argument checks come first, as in gdn_prefill_chunked
    assert lib.gdn_prefill_chunked_static(None, ctypes.byref(_fake_tensors()), None) == \
        gdn.GDN_ERR_NULL
    s = _shape(T=0)
    assert lib.gdn_prefill_chunked_static(ctypes.byref(s), ctypes.byref(_fake_tensors()),
                                          None) == gdn.GDN_ERR_SHAPE


def _upload(shape, seed):
    params = synth.make_params(shape, seed=seed, slow_decay=True)
    inp = synth.make_inputs(shape, seed=seed, slow_decay=True)
    state = synth.make_state(shape, seed=seed)
    return dev.upload(shape, params, inp, state)


def _call(case, static):
    sh = case.abi_shape()
    st = torch.cuda.current_stream().cuda_stream
    if static:
        gdn.gdn_prefill_chunked_static(sh, case.abi_tensors(), st)
    else:
        n = gdn.gdn_prefill_workspace_bytes(sh)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
        gdn.gdn_prefill_chunked(sh, case.abi_tensors(), ws.data_ptr(), n, st)
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    return case


@pytest.mark.gpu
def test_two_static_calls_in_a_row_match_the_workspace_entry_point():
    first = synth.Shape(B=2, T=100, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True)
    second = synth.Shape(B=3, T=61, H_qk=2, H_v=4, d_k=128, d_v=128, kda=True, lb_gate=True)
    assert gdn.gdn_kernel_variant(_abi(first), gdn.OP_PREFILL) == "kda_chunked<16>"
    runs = [(first, 50), (second, 51)]
    cases = [_upload(s, seed) for s, seed in runs]
    torch.cuda.synchronize()
    _call(cases[0], True)                  # the first call may load the module
    free_before = torch.cuda.mem_get_info()[0]
    _call(cases[1], True)                  # the second call in a row
    assert torch.cuda.mem_get_info()[0] == free_before, "the static call allocated device memory"
    for (s, seed), a in zip(runs, cases):
        b = _call(_upload(s, seed), False)
        assert torch.equal(a.out, b.out), f"out differs for {s}"
        assert torch.equal(a.state, b.state), f"state differs for {s}"
        assert torch.equal(a.conv_state, b.conv_state), f"conv_state differs for {s}"


def _abi(shape):
    return gdn.make_shape(B=shape.B, T=shape.T, H_qk=shape.H_qk, H_v=shape.H_v, d_k=shape.d_k,
                          d_v=shape.d_v, kda=shape.kda, bf16_in=shape.bf16_in,
                          q_scale=shape.q_scale)
