"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Bar: max|err| / RMS(ref) <= 1e-3 for every output and final state of the
fp32-state decode and verify paths; verify equals T decode calls bit for bit.
"""

import dataclasses

import numpy as np
import pytest
import torch

import linear_attention_decode_kda_gb300 as gdn
import synth
from gpu_harness import (DECODE_TOL, PREFILL_TOL, assert_close, assert_close_bf16_out,
                         gpu_decode_run, oracle_run, stream)
from synth import device as dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(shape, steps, seed=0, layer=0, slow=False):
    """Params, state and `steps` tokens ([B, steps, ...]) of one layer."""
    sT = dataclasses.replace(shape, T=steps)
    return (synth.make_params(shape, seed=seed, layer=layer, slow_decay=slow),
            synth.make_inputs(sT, seed=seed, layer=layer, slow_decay=slow),
            synth.make_state(shape, seed=seed, layer=layer))


def _check_decode(shape, steps, tol=DECODE_TOL, **kw):
    params, inp, state = _case(shape, steps, slow=kw.pop("slow", False))
    y, S, cs = gpu_decode_run(shape, params, inp, state, **kw)
    ref = oracle_run(shape, params, inp, state)
    return (assert_close(y, ref["y"], tol, "y"), assert_close(S, ref["state"], tol, "state"),
            assert_close(cs, ref["conv_state"], 0.0, "conv_state"))


# ---------------------------------------------------------------- workloads at full size

def test_tiny_gdn_decode_8_steps():
    spec = synth.WORKLOADS["tiny_gdn_decode"]
    _check_decode(spec["shape"], spec["steps"])


def test_kda_batched_decode_b64_100_steps():
    spec = synth.WORKLOADS["kda_decode_b64"]
    _check_decode(spec["shape"], spec["steps"])


@pytest.mark.parametrize("pdl", [False, True])
def test_kda_decode_b1_34_layers(pdl):
    """34 independent layers stepped token-major for 256 tokens (PDL as the benchmark runs it)."""
    spec = synth.WORKLOADS["kda_decode_b1_34layers"]
    shape, layers, steps = spec["shape"], spec["layers"], spec["steps"]
    if not pdl:
        layers, steps = 3, 24
    cases = [_case(shape, steps, layer=l) for l in range(layers)]
    bf = shape.bf16_in
    from gpu_harness import steps_major
    dev_in, dev_st = [], []
    for params, inp, state in cases:
        first = synth.Inputs(inp.qkv[:, :1], inp.f[:, :1], inp.beta[:, :1], inp.z[:, :1])
        c = dev.upload(shape, params, first, state)
        dev_st.append(c)
        dev_in.append([dev.to_torch(steps_major(x), bf, "cuda") for x in
                       (inp.qkv, inp.f, inp.beta, inp.z)])
    outs = [torch.empty((steps, 1, shape.H_v * shape.d_v), device="cuda") for _ in cases]
    sh = dev_st[0].abi_shape(pdl=pdl)
    for t in range(steps):
        for l in range(layers):
            c, (q, f, b, z) = dev_st[l], dev_in[l]
            tens = gdn.tensors_from_torch(qkv=q[t], f=f[t], beta=b[t], z=z[t], conv_w=c.conv_w,
                                          A_log=c.A_log, dt_bias=c.dt_bias, norm_w=c.norm_w,
                                          conv_state=c.conv_state, state=c.state, out=outs[l][t])
            gdn.gdn_decode_step(sh, tens, stream())
    torch.cuda.synchronize()
    for l, (params, inp, state) in enumerate(cases):
        ref = oracle_run(shape, params, inp, state)
        y = outs[l].permute(1, 0, 2).reshape(ref["y"].shape)
        assert_close(y, ref["y"], DECODE_TOL, f"y layer {l}")
        assert_close(dev_st[l].state, ref["state"], DECODE_TOL, f"state layer {l}")
        assert_close(dev_st[l].conv_state, ref["conv_state"], 0.0, f"conv layer {l}")


def _verify(shape, seed=0, conv_hist=True, bf16_out=False, slow=False):
    params, inp, state = _case(shape, shape.T, seed=seed, slow=slow)
    case = dev.upload(shape, params, inp, state, hist=True, conv_hist=conv_hist,
                      bf16_out=bf16_out)
    S0 = case.state.clone()
    cs0 = case.conv_state.clone()
    gdn.gdn_verify_T(case.abi_shape(bf16_out=bf16_out), case.abi_tensors(), stream())
    torch.cuda.synchronize()
    assert torch.equal(case.state, S0) and torch.equal(case.conv_state, cs0), "verify wrote state"
    return params, inp, state, case


def test_kda_verify_b32_t4_matches_oracle_and_decode_bitwise():
    shape = synth.WORKLOADS["kda_verify_b32_t4"]["shape"]
    params, inp, state, case = _verify(shape)
    ref = oracle_run(shape, params, inp, state, hist=True)
    assert_close(case.out.reshape(ref["y"].shape), ref["y"], DECODE_TOL, "y")
    assert_close(case.state_hist, ref["state_hist"], DECODE_TOL, "state_hist")
    # conv window after each token: rows t+1..t+3 of [conv_state; qkv]
    X = np.concatenate([state.conv, inp.qkv], axis=1)
    for t in range(shape.T):
        np.testing.assert_array_equal(case.conv_hist[t].cpu().numpy(), X[:, t + 1:t + 4])
    # the same tokens as four decode calls: bit for bit
    one = dataclasses.replace(shape, T=1)
    y, S, cs = gpu_decode_run(one, params, inp, state)
    assert torch.equal(y.reshape(case.out.shape), case.out), "verify y != 4 decode steps"
    assert torch.equal(S, case.state_hist[-1]), "verify state != 4 decode steps"
    assert torch.equal(cs, case.conv_hist[-1])


# ---------------------------------------------------------------- tiling variants and edges

@pytest.mark.parametrize("B,D,kda", [(10, 128, True), (5, 128, True), (3, 128, False),
                                     (1, 128, True), (2, 64, True), (1, 64, False),
                                     (3, 32, True), (1, 16, True)])
def test_decode_each_slab_variant(B, D, kda):
    shape = synth.Shape(B=B, T=1, H_qk=32 if D == 128 else 8, H_v=32 if D == 128 else 8,
                        d_k=D, d_v=D, kda=kda)
    _check_decode(shape, 5)


@pytest.mark.parametrize("group", [2, 4])
def test_decode_gva(group):
    shape = synth.Shape(B=3, T=1, H_qk=16 // group, H_v=16, d_k=128, d_v=128, kda=False)
    _check_decode(shape, 4)


def test_decode_fp32_inputs_and_bf16_out():
    shape = synth.Shape(B=4, T=1, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, bf16_in=False)
    _check_decode(shape, 3)
    # bf16 output: each y is rounded once to bf16
    shape = synth.Shape(B=4, T=1, H_qk=4, H_v=4, d_k=128, d_v=128)
    params, inp, state = _case(shape, 3)
    y, S, _ = gpu_decode_run(shape, params, inp, state, bf16_out=True)
    ref = oracle_run(shape, params, inp, state)
    assert_close_bf16_out(y, ref["y"], "y")
    assert_close(S, ref["state"], DECODE_TOL, "state")


def test_decode_slow_decay_long_run():
    """Slow per-channel decay (state survives many tokens), 64 steps."""
    shape = synth.Shape(B=2, T=1, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True)
    _check_decode(shape, 64, slow=True)


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_verify_each_T_bitwise(T):
    shape = synth.Shape(B=3, T=T, H_qk=4, H_v=8, d_k=128, d_v=128, kda=True)
    params, inp, state, case = _verify(shape, seed=3)
    y, S, _ = gpu_decode_run(dataclasses.replace(shape, T=1), params, inp, state)
    assert torch.equal(y.reshape(case.out.shape), case.out)
    assert torch.equal(S, case.state_hist[-1])
    ref = oracle_run(shape, params, inp, state, hist=True)
    assert_close(case.state_hist, ref["state_hist"], DECODE_TOL, "state_hist")


def test_empty_batch_is_a_no_op():
    shape = synth.Shape(B=1, T=1, H_qk=2, H_v=2, d_k=16, d_v=16, kda=False, bf16_in=False)
    params, inp, state = _case(shape, 1)
    case = dev.upload(shape, params, inp, state)
    sh = case.abi_shape()
    sh.B = 0
    gdn.gdn_decode_step(sh, case.abi_tensors(), stream())
    torch.cuda.synchronize()
    assert torch.equal(case.state.cpu(), torch.from_numpy(state.S))


# ---------------------------------------------------------------- prefill

def _prefill(shape, seed=0, slow=False, tol=PREFILL_TOL, bf16_out=False, variant=None):
    params, inp, state = _case(shape, shape.T, seed=seed, slow=slow)
    case = dev.upload(shape, params, inp, state, bf16_out=bf16_out)
    sh = case.abi_shape(bf16_out=bf16_out)
    if variant is not None:
        assert gdn.gdn_kernel_variant(sh, gdn.OP_PREFILL) == variant
    nbytes = gdn.gdn_prefill_workspace_bytes(sh)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    gdn.gdn_prefill_chunked(sh, case.abi_tensors(), ws.data_ptr(), nbytes, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    ref = oracle_run(shape, params, inp, state)
    if bf16_out:
        assert_close_bf16_out(case.out.reshape(ref["y"].shape), ref["y"], "y")
    else:
        assert_close(case.out.reshape(ref["y"].shape), ref["y"], tol, "y")
    assert_close(case.state, ref["state"], tol, "state")
    assert_close(case.conv_state, ref["conv_state"], 0.0, "conv_state")


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 200])
def test_prefill_ragged_lengths(T):
    """The 32-token and the 64-token tensor-core kernels (chunk 32, 64), and the
    two-kernel form (chunk 16)."""
    shape = synth.Shape(B=2, T=T, H_qk=4, H_v=8, d_k=128, d_v=128, kda=False, chunk=32)
    _prefill(shape, slow=True, variant="chunked<128,32>")
    _prefill(dataclasses.replace(shape, chunk=64), slow=True, variant="chunked<128,64>")
    _prefill(dataclasses.replace(shape, chunk=16), slow=True,
             variant="kda_chunked<16>" if T > 4 else None)


@pytest.mark.parametrize("H_qk,H_v", [(4, 4), (2, 8)])
def test_prefill_chunked_head_groups(H_qk, H_v):
    """Ungrouped heads and four value heads per qk head (thread-block cluster of 4)."""
    shape = synth.Shape(B=3, T=130, H_qk=H_qk, H_v=H_v, d_k=128, d_v=128, kda=False, chunk=32)
    _prefill(shape, seed=5, variant="chunked<128,32>")
    _prefill(shape, seed=6, slow=True)
    _prefill(dataclasses.replace(shape, chunk=64), seed=6, slow=True, variant="chunked<128,64>")
    _prefill(dataclasses.replace(shape, chunk=16), seed=6, slow=True, variant="kda_chunked<16>")


def test_prefill_chunked_bf16_out():
    shape = synth.Shape(B=2, T=96, H_qk=2, H_v=4, d_k=128, d_v=128, kda=False, chunk=64)
    _prefill(shape, seed=7, bf16_out=True)


def test_prefill_kda_slow_decay():
    shape = synth.Shape(B=2, T=130, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, chunk=64)
    _prefill(shape, slow=True)


def test_prefill_gdn_b4_t4096():
    """The full-size GDN prefill in the launch the bench times, every output and final
    state against the oracle's 4096 sequential steps."""
    _prefill(synth.WORKLOADS["gdn_prefill_b4_t4096"]["shape"], variant="chunked<128,64>")


def test_stream_shape_with_unaligned_scalars_falls_back_and_matches():
    """A many-head decode whose beta rows are not 16-byte aligned runs on the
    column-slab kernel (the streaming kernel needs aligned chunks); same result."""
    shape = synth.Shape(B=16, T=1, H_qk=32, H_v=32, d_k=128, d_v=128, kda=True)
    params, inp, state = _case(shape, 2)
    from gpu_harness import steps_major
    case = dev.upload(shape, params, synth.Inputs(inp.qkv[:, :1], inp.f[:, :1], inp.beta[:, :1],
                                                  inp.z[:, :1]), state)
    beta_all = dev.to_torch(steps_major(inp.beta), True, "cuda")      # [2, B, 1, H]
    pad = torch.empty(beta_all.numel() + 8, dtype=torch.bfloat16, device="cuda")
    shifted = pad[1:1 + beta_all.numel()].view(beta_all.shape)       # 2-byte offset
    shifted.copy_(beta_all)
    qkv = dev.to_torch(steps_major(inp.qkv), True, "cuda")
    f = dev.to_torch(steps_major(inp.f), True, "cuda")
    z = dev.to_torch(steps_major(inp.z), True, "cuda")
    out = torch.empty((2, shape.B, shape.H_v * shape.d_v), device="cuda")
    sh = case.abi_shape()
    for t in range(2):
        tens = gdn.tensors_from_torch(qkv=qkv[t], f=f[t], beta=shifted[t], z=z[t],
                                      conv_w=case.conv_w, A_log=case.A_log, dt_bias=case.dt_bias,
                                      norm_w=case.norm_w, conv_state=case.conv_state,
                                      state=case.state, out=out[t])
        gdn.gdn_decode_step(sh, tens, stream())
    torch.cuda.synchronize()
    gdn.gdn_device_status()
    ref = oracle_run(shape, params, inp, state)
    y = out.permute(1, 0, 2).reshape(ref["y"].shape)
    assert_close(y, ref["y"], DECODE_TOL, "y")
    assert_close(case.state, ref["state"], DECODE_TOL, "state")


def test_device_status_clean_after_streaming_runs():
    shape = synth.WORKLOADS["kda_decode_b64"]["shape"]
    _check_decode(shape, 2)
    gdn.gdn_device_status()
