"""The C ABI on the host: library loads, exports what include/gdn.h declares,
and rejects bad arguments before launching anything (no GPU needed: every
call here fails validation, so no kernel is queued)."""

import ctypes
import os
import re

import pytest

import linear_attention_decode_kda_gb300 as gdn

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    from linear_attention_decode_kda_gb300 import build
    build.build()
    return gdn.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(gdn.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _shape(**kw):
    base = dict(B=2, T=1, H_qk=4, H_v=4, d_k=128, d_v=128, kda=True, bf16_in=True,
                q_scale=0.08838835)
    base.update(kw)
    return gdn.make_shape(**base)


def _tensors(addr=0x10000):
    names = [n for n, _ in gdn.GdnTensors._fields_]
    return gdn.GdnTensors(**{n: addr + 0x1000 * i for i, n in enumerate(names)})


def _call(lib, op, shape, tensors, ws=None, ws_bytes=0):
    s = ctypes.byref(shape) if shape is not None else None
    t = ctypes.byref(tensors) if tensors is not None else None
    if op == "decode":
        return lib.gdn_decode_step(s, t, None)
    if op == "verify":
        return lib.gdn_verify_T(s, t, None)
    return lib.gdn_prefill_chunked(s, t, ws, ws_bytes, None)


@pytest.mark.parametrize("op", ["decode", "verify", "prefill"])
def test_null_arguments(lib, op):
    assert _call(lib, op, None, _tensors()) == gdn.GDN_ERR_NULL
    assert _call(lib, op, _shape(), None) == gdn.GDN_ERR_NULL
    t = _tensors()
    t.qkv = None
    assert _call(lib, op, _shape(), t) == gdn.GDN_ERR_NULL


@pytest.mark.parametrize("op", ["decode", "verify", "prefill"])
def test_misaligned_pointer(lib, op):
    t = _tensors()
    t.state = t.state + 4
    assert _call(lib, op, _shape(), t) == gdn.GDN_ERR_ALIGN


@pytest.mark.parametrize("kw,want", [
    (dict(B=-1), gdn.GDN_ERR_SHAPE), (dict(H_qk=3, H_v=4), gdn.GDN_ERR_SHAPE),
    (dict(H_qk=0), gdn.GDN_ERR_SHAPE), (dict(d_k=128, d_v=64), gdn.GDN_ERR_UNSUPPORTED),
    (dict(d_k=48, d_v=48), gdn.GDN_ERR_UNSUPPORTED), (dict(conv_K=3), gdn.GDN_ERR_UNSUPPORTED),
    (dict(q_scale=0.0), gdn.GDN_ERR_SHAPE), (dict(B=70000), gdn.GDN_ERR_SHAPE),
])
def test_bad_shapes(lib, kw, want):
    assert _call(lib, "decode", _shape(**kw), _tensors()) == want


def test_bad_enums_and_flags(lib):
    for field, val in (("gate_mode", 7), ("in_dtype", 3), ("out_dtype", -1), ("flags", 8)):
        s = _shape()
        setattr(s, field, val)
        assert _call(lib, "decode", s, _tensors()) == gdn.GDN_ERR_SHAPE, field


def test_token_counts(lib):
    assert _call(lib, "decode", _shape(T=2), _tensors()) == gdn.GDN_ERR_SHAPE
    assert _call(lib, "verify", _shape(T=5), _tensors()) == gdn.GDN_ERR_SHAPE
    assert _call(lib, "verify", _shape(T=0), _tensors()) == gdn.GDN_ERR_SHAPE
    assert _call(lib, "prefill", _shape(T=0), _tensors()) == gdn.GDN_ERR_SHAPE
    t = _tensors()
    t.state_hist = t.state_hist + 4
    assert _call(lib, "verify", _shape(T=2), t) == gdn.GDN_ERR_ALIGN


def test_commit_accepted_checks(lib):
    def commit(shape, tensors, accepted=None):
        return lib.gdn_commit_accepted(ctypes.byref(shape), ctypes.byref(tensors), accepted, None)
    assert commit(_shape(T=0), _tensors()) == gdn.GDN_ERR_SHAPE
    assert commit(_shape(T=5), _tensors()) == gdn.GDN_ERR_SHAPE
    t = _tensors()
    t.qkv = None
    assert commit(_shape(T=2), t) == gdn.GDN_ERR_NULL
    assert commit(_shape(T=2), _tensors(), 0x20002) == gdn.GDN_ERR_ALIGN
    t = _tensors()
    t.out = t.out + 8
    assert commit(_shape(T=2), t) == gdn.GDN_ERR_ALIGN
    assert lib.gdn_commit_accepted(None, ctypes.byref(_tensors()), None, None) == gdn.GDN_ERR_NULL


def test_prefill_workspace_checks(lib):
    s = _shape(T=256, kda=False)
    need = gdn.gdn_prefill_workspace_bytes(s)
    assert need >= 0
    if need > 0:
        assert _call(lib, "prefill", s, _tensors(), None, need) == gdn.GDN_ERR_WORKSPACE
        assert _call(lib, "prefill", s, _tensors(), 0x100000, need - 1) == gdn.GDN_ERR_WORKSPACE
    s.chunk = 0
    assert _call(lib, "prefill", s, _tensors(), 0x100000, need) == gdn.GDN_ERR_SHAPE
    bad = _shape(T=0)
    assert gdn.gdn_prefill_workspace_bytes(bad) == 0


def test_prefill_snapshot_buffers_are_checked(lib):
    """Snapshot tails: state_hist must be 16-byte aligned and conv_hist 4-byte
    aligned, in gdn_prefill_chunked and gdn_prefill_chunked_static alike, before
    anything is queued."""
    s = _shape(T=100, kda=True)
    need = gdn.gdn_prefill_workspace_bytes(s)
    for field, off in (("state_hist", 4), ("conv_hist", 2)):
        t = _tensors()
        setattr(t, field, getattr(t, field) + off)
        assert _call(lib, "prefill", s, t, 0x100000, need) == gdn.GDN_ERR_ALIGN
        s1 = _shape(T=30, kda=True)
        assert lib.gdn_prefill_chunked_static(ctypes.byref(s1), ctypes.byref(t), None) == gdn.GDN_ERR_ALIGN


def test_status_strings(lib):
    for code in range(-7, 1):
        assert gdn.status_string(code).startswith("GDN_")
    assert "unknown" in gdn.status_string(-99)


def test_gate_variants_are_accepted(lib):
    s = _shape(B=64, H_qk=32, H_v=32)
    s.gate_mode = gdn.GDN_GATE_LOWER_BOUND
    s.flags = gdn.GDN_FLAG_SIGMOID_GATE | gdn.GDN_FLAG_PDL
    assert gdn.gdn_kernel_variant(s, gdn.OP_DECODE) == "stream<128>"
    s.T = 64  # the bounded per-channel gate takes the two-kernel chunked form
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "kda_chunked<16>"


def test_prefill_routing_and_workspace(lib):
    """Per-head decay, bf16 rows, d = 128: chunk 64 runs the 64-token tensor-core
    kernel and chunk 32 the 32-token one, neither with a workspace (at any T).
    Other chunks, per-channel decay or fp32 rows at d = 128 and T > 4: the
    two-kernel form, one 34,304-byte block per (sequence, head, 16-token chunk).
    Otherwise the recurrent kernel, no workspace."""
    s = _shape(T=100, kda=False)
    s.chunk = 32
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "chunked<128,32>"
    assert gdn.gdn_prefill_workspace_bytes(s) == 0
    s.chunk = 64
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "chunked<128,64>"
    assert gdn.gdn_prefill_workspace_bytes(s) == 0
    s.T = 3
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "chunked<128,64>"
    s.T = 100
    s.chunk = 16
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "kda_chunked<16>"
    assert gdn.gdn_prefill_workspace_bytes(s) == 2 * 4 * 7 * 34304
    s = _shape(T=100)
    s.chunk = 64
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "kda_chunked<16>"
    assert gdn.gdn_prefill_workspace_bytes(s) == 2 * 4 * 7 * 34304
    s.in_dtype = gdn.GDN_F32
    s.gate_mode = gdn.GDN_GATE_PER_HEAD
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL) == "kda_chunked<16>"
    s = _shape(T=4)
    s.chunk = 64
    assert gdn.gdn_prefill_workspace_bytes(s) == 0
    assert not gdn.gdn_kernel_variant(s, gdn.OP_PREFILL).startswith(("chunked", "kda_chunked"))
    s = _shape(T=100, d_k=64, d_v=64)
    s.chunk = 64
    assert gdn.gdn_prefill_workspace_bytes(s) == 0
    assert gdn.gdn_kernel_variant(s, gdn.OP_PREFILL).startswith("step<64")


def test_variant_choice(lib):
    # B*H_v head units: enough for two CTAs per SM -> streaming CTAs; B=1 -> 16-column slabs
    assert gdn.gdn_kernel_variant(_shape(B=64, H_qk=32, H_v=32), gdn.OP_DECODE) == "stream<128>"
    assert gdn.gdn_kernel_variant(_shape(B=32, H_qk=32, H_v=32), gdn.OP_VERIFY) == "stream<128>"
    assert gdn.gdn_kernel_variant(_shape(B=64, H_qk=16, H_v=32), gdn.OP_DECODE) == "wstep<128,64>"
    assert gdn.gdn_kernel_variant(_shape(B=1, H_qk=32, H_v=32), gdn.OP_DECODE) == "step<128,16>"
    assert gdn.gdn_kernel_variant(_shape(d_k=16, d_v=16), gdn.OP_DECODE) == "step<16,16>"
    assert gdn.gdn_kernel_variant(_shape(d_k=48, d_v=48), gdn.OP_DECODE) is None


@pytest.mark.parametrize("B,H_qk,H_v,want", [
    (1, 32, 32, "step<128,16>"),     # below 64 units: the 8-slab plan
    (2, 32, 32, "step<128,64>"),     # 64 to 127 units: two slabs a head
    (3, 32, 32, "stream<128>"),
    (3, 8, 16, "step<128,32>"),      # 48 grouped units: slabs x group within a cluster of 8
    (4, 32, 32, "stream<128>"),      # more than 64 ungrouped units: the streaming kernel
    (9, 32, 32, "stream<128>"),
    (10, 32, 32, "stream<128>"),
    (4, 8, 32, "wstep<128,64>"),     # grouped heads never stream: from 128 units the
    (8, 8, 16, "wstep<128,64>"),     # warp-column kernel, two slabs
    (2, 8, 64, "wstep<128,128>"),    # a group of 8 value heads: whole heads a CTA
])
def test_decode_routing_by_unit_count(lib, B, H_qk, H_v, want):
    """The d = 128 decode plan by (sequence, head) units (148 SMs when no GPU is present,
    152 on a GB300: the thresholds below sit away from both)."""
    for op in (gdn.OP_DECODE, gdn.OP_VERIFY):
        assert gdn.gdn_kernel_variant(_shape(B=B, H_qk=H_qk, H_v=H_v), op) == want


def test_dependents_start_only_after_the_dependency_wait():
    """Every kernel that takes part in programmatic dependent launch lets its dependents
    start only after its own dependency wait: in each kernel body the trigger follows the
    wait.  A trigger before the wait would let a dependent's pre-wait reads run beside a
    kernel earlier than its immediate predecessor."""
    csrc = os.path.join(ROOT, "linear_attention_decode_kda_gb300", "csrc")
    seen = 0
    for fn in sorted(os.listdir(csrc)):
        if not fn.endswith(".cu"):
            continue
        text = open(os.path.join(csrc, fn)).read()
        for body in re.split(r"__global__", text)[1:]:
            trig = [m.start() for m in re.finditer(r"pdl_launch_dependents\(\)", body)]
            wait = [m.start() for m in re.finditer(r"pdl_wait\(\)", body)]
            if not trig:
                continue
            seen += 1
            assert wait, f"{fn}: a kernel triggers dependents without a dependency wait"
            # only the first kernel body after each __global__ up to the next one is scanned
            assert min(trig) > min(wait), f"{fn}: dependents triggered before the wait"
    assert seen >= 6, seen


def test_product_path_never_touches_the_oracle():
    """The package and its CUDA sources import / include nothing from oracle/."""
    pkg = os.path.join(ROOT, "linear_attention_decode_kda_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".h", ".cuh")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), fn
                assert "gdn_oracle" not in text, fn
    src = open(os.path.join(ROOT, "oracle", "gdn_oracle.c")).read()
    assert not re.search(r'#include\s+"', src), "oracle includes a local header"


def test_layer_decode_argument_checks(lib):
    """gdn_layer_decode refuses, before any launch: the per-head gate, bf16 rows,
    T != 1, missing weights, a short workspace and misaligned rows."""
    def weights(**kw):
        base = dict(d_model=512, rank=32, w_qkv=0x100000, w_fa=0x110000, w_fb=0x120000,
                    w_ga=0x130000, w_gb=0x140000, w_beta=0x150000, w_o=0x160000)
        base.update(kw)
        return gdn.GdnLayerWeights(**base)

    def call(s, w, x=0x170000, x_out=0x180000, t=None, ws=0x190000, ws_bytes=1 << 20):
        t = t or _tensors()
        return lib.gdn_layer_decode(ctypes.byref(s), ctypes.byref(w), x, x_out, ctypes.byref(t),
                                    ws, ws_bytes, None)

    f32 = dict(bf16_in=False)
    s = _shape(**f32)
    assert gdn.gdn_layer_workspace_bytes(s, weights()) == 2 * 2 * 32 * 4
    assert call(_shape(kda=False, **f32), weights()) == gdn.GDN_ERR_SHAPE
    assert call(_shape(), weights()) == gdn.GDN_ERR_SHAPE          # bf16 rows
    assert call(_shape(T=2, **f32), weights()) == gdn.GDN_ERR_SHAPE
    assert call(s, weights(w_fb=0)) == gdn.GDN_ERR_NULL
    assert call(s, weights(rank=12)) == gdn.GDN_ERR_SHAPE
    assert call(s, weights(), ws_bytes=100) == gdn.GDN_ERR_WORKSPACE
    assert call(s, weights(), x=0x170008) == gdn.GDN_ERR_ALIGN
    assert call(s, weights(w_o=0x160004)) == gdn.GDN_ERR_ALIGN


def test_abi_structs_keep_their_tensors_alive():
    """The ABI structs hold raw addresses; the structs built from tensors keep those
    tensors referenced, so a temporary passed in is not freed under a queued kernel."""
    import gc
    import weakref

    import torch

    w = {k: torch.zeros(64, dtype=torch.bfloat16) for k in
         ("w_qkv", "w_fa", "w_fb", "w_ga", "w_gb", "w_beta", "w_o")}
    refs = [weakref.ref(v) for v in w.values()]
    lw = gdn.layer_weights_from_torch(8, 8, **w)
    del w
    gc.collect()
    assert all(r() is not None for r in refs)
    assert lw.w_o == refs[-1]().data_ptr()

    names = ("qkv", "f", "beta", "z", "conv_w", "A_log", "dt_bias", "norm_w", "conv_state",
             "state", "out")
    ts = {n: torch.zeros(16) for n in names}
    trefs = [weakref.ref(v) for v in ts.values()]
    tt = gdn.tensors_from_torch(**ts)
    del ts
    gc.collect()
    assert all(r() is not None for r in trefs)
    assert tt.state == trefs[names.index("state")]().data_ptr()
    del lw, tt
    gc.collect()
    assert all(r() is None for r in refs + trefs)
