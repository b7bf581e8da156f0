"""Python binding of libgdn.so, the KDA / Gated DeltaNet step for GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/gdn.h``.  PyTorch (optional
here) only provides device memory and streams; ``tensors_from_torch`` turns
tensors into the ABI's plain pointers.  If the library is not built this
module raises on first use -- there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

GDN_OK = 0
GDN_ERR_NULL = -1
GDN_ERR_ALIGN = -2
GDN_ERR_SHAPE = -3
GDN_ERR_UNSUPPORTED = -4
GDN_ERR_WORKSPACE = -5
GDN_ERR_CUDA = -6
GDN_ERR_TIMEOUT = -7

GDN_GATE_PER_HEAD = 0
GDN_GATE_PER_CHANNEL = 1
GDN_GATE_LOWER_BOUND = 2
GDN_F32 = 0
GDN_BF16 = 1
GDN_FLAG_PDL = 1
GDN_FLAG_SIGMOID_GATE = 2

OP_DECODE, OP_VERIFY, OP_PREFILL = 0, 1, 2


class GdnShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "T", "H_qk", "H_v", "d_k", "d_v", "conv_K", "chunk", "gate_mode",
                 "in_dtype", "out_dtype", "flags")] + \
               [(n, ctypes.c_float) for n in ("q_scale", "eps_l2", "eps_norm")]


class GdnTensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("qkv", "f", "beta", "z", "conv_w", "A_log", "dt_bias", "norm_w",
                 "conv_state", "state", "out", "state_hist", "conv_hist")]


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


EXPORTS = ("gdn_decode_step", "gdn_verify_T", "gdn_commit_accepted", "gdn_prefill_chunked",
           "gdn_prefill_workspace_bytes", "gdn_prefill_chunked_static", "gdn_layer_decode",
           "gdn_layer_workspace_bytes", "gdn_device_status", "gdn_status_string",
           "gdn_kernel_variant")

# bytes of the library's own scratch behind gdn_prefill_chunked_static
PREFILL_STATIC_SCRATCH_BYTES = 32 << 20

class GdnLayerWeights(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("rank", ctypes.c_int32)] + \
               [(n, ctypes.c_void_p) for n in
                ("w_qkv", "w_fa", "w_fb", "w_ga", "w_gb", "w_beta", "w_o")]


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Loads libgdn.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, S, Tn = ctypes.c_void_p, ctypes.POINTER(GdnShape), ctypes.POINTER(GdnTensors)
    for name in ("gdn_decode_step", "gdn_verify_T"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [S, Tn, P]
    lib.gdn_commit_accepted.restype = ctypes.c_int
    lib.gdn_commit_accepted.argtypes = [S, Tn, P, P]
    lib.gdn_prefill_chunked.restype = ctypes.c_int
    lib.gdn_prefill_chunked.argtypes = [S, Tn, P, ctypes.c_size_t, P]
    lib.gdn_prefill_chunked_static.restype = ctypes.c_int
    lib.gdn_prefill_chunked_static.argtypes = [S, Tn, P]
    W = ctypes.POINTER(GdnLayerWeights)
    lib.gdn_layer_decode.restype = ctypes.c_int
    lib.gdn_layer_decode.argtypes = [S, W, P, P, Tn, P, ctypes.c_size_t, P]
    lib.gdn_layer_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_layer_workspace_bytes.argtypes = [S, W]
    lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_prefill_workspace_bytes.argtypes = [S]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_device_status.restype = ctypes.c_int
    lib.gdn_device_status.argtypes = []
    lib.gdn_kernel_variant.restype = ctypes.c_char_p
    lib.gdn_kernel_variant.argtypes = [S, ctypes.c_int]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != GDN_OK:
        raise GdnError(rc, where)


def gdn_decode_step(shape: GdnShape, tensors: GdnTensors, stream: int = 0) -> None:
    _check(load().gdn_decode_step(ctypes.byref(shape), ctypes.byref(tensors),
                                  ctypes.c_void_p(stream)), "gdn_decode_step")


def gdn_verify_T(shape: GdnShape, tensors: GdnTensors, stream: int = 0) -> None:
    _check(load().gdn_verify_T(ctypes.byref(shape), ctypes.byref(tensors),
                               ctypes.c_void_p(stream)), "gdn_verify_T")


def gdn_commit_accepted(shape: GdnShape, tensors: GdnTensors, accepted=None,
                        stream: int = 0) -> None:
    """accepted: device int32 [B] (a tensor or an address), or None for all T tokens."""
    _check(load().gdn_commit_accepted(ctypes.byref(shape), ctypes.byref(tensors),
                                      ctypes.c_void_p(_ptr(accepted)), ctypes.c_void_p(stream)),
           "gdn_commit_accepted")


def gdn_prefill_chunked(shape: GdnShape, tensors: GdnTensors, workspace: int = 0,
                        workspace_bytes: int = 0, stream: int = 0) -> None:
    _check(load().gdn_prefill_chunked(ctypes.byref(shape), ctypes.byref(tensors),
                                      ctypes.c_void_p(workspace), workspace_bytes,
                                      ctypes.c_void_p(stream)), "gdn_prefill_chunked")


def gdn_prefill_chunked_static(shape: GdnShape, tensors: GdnTensors, stream: int = 0) -> None:
    """gdn_prefill_chunked on the library's static scratch: allocates nothing; calls
    whose work overlaps in time race on the one scratch."""
    _check(load().gdn_prefill_chunked_static(ctypes.byref(shape), ctypes.byref(tensors),
                                             ctypes.c_void_p(stream)), "gdn_prefill_chunked_static")


def gdn_layer_decode(shape: GdnShape, weights: GdnLayerWeights, x, x_out, tensors: GdnTensors,
                     workspace: int = 0, workspace_bytes: int = 0, stream: int = 0) -> None:
    """x: [B, d_model] bf16, x_out: [B, d_model] fp32 (tensors or addresses)."""
    _check(load().gdn_layer_decode(ctypes.byref(shape), ctypes.byref(weights),
                                   ctypes.c_void_p(_ptr(x)), ctypes.c_void_p(_ptr(x_out)),
                                   ctypes.byref(tensors), ctypes.c_void_p(workspace),
                                   workspace_bytes, ctypes.c_void_p(stream)), "gdn_layer_decode")


def gdn_layer_workspace_bytes(shape: GdnShape, weights: GdnLayerWeights) -> int:
    return int(load().gdn_layer_workspace_bytes(ctypes.byref(shape), ctypes.byref(weights)))


def layer_weights_from_torch(d_model: int, rank: int, **w) -> GdnLayerWeights:
    """Weights as bf16 device tensors (keyword per field of GdnLayerWeights).  The
    returned struct holds references to the tensors, so their memory outlives it."""
    lw = GdnLayerWeights(d_model=d_model, rank=rank,
                         **{k: _ptr(w[k]) for k in ("w_qkv", "w_fa", "w_fb", "w_ga", "w_gb",
                                                    "w_beta", "w_o")})
    lw._keep = dict(w)
    return lw


def gdn_prefill_workspace_bytes(shape: GdnShape) -> int:
    return int(load().gdn_prefill_workspace_bytes(ctypes.byref(shape)))


def gdn_device_status() -> None:
    """Raises GdnError if a kernel recorded a bounded-wait time-out (synchronises)."""
    _check(load().gdn_device_status(), "gdn_device_status")


def gdn_kernel_variant(shape: GdnShape, op: int) -> Optional[str]:
    r = load().gdn_kernel_variant(ctypes.byref(shape), op)
    return None if r is None else r.decode()


def make_shape(B: int, T: int, H_qk: int, H_v: int, d_k: int, d_v: int, *, kda: bool,
               bf16_in: bool, bf16_out: bool = False, conv_K: int = 4, chunk: int = 64,
               q_scale: float, eps_l2: float = 1e-6, eps_norm: float = 1e-6,
               pdl: bool = False, lb_gate: bool = False, sigmoid_gate: bool = False) -> GdnShape:
    """lb_gate (with kda): the lower-bound per-channel gate; sigmoid_gate: sigmoid output gate."""
    gate = GDN_GATE_LOWER_BOUND if lb_gate else (GDN_GATE_PER_CHANNEL if kda else GDN_GATE_PER_HEAD)
    flags = (GDN_FLAG_PDL if pdl else 0) | (GDN_FLAG_SIGMOID_GATE if sigmoid_gate else 0)
    return GdnShape(B=B, T=T, H_qk=H_qk, H_v=H_v, d_k=d_k, d_v=d_v, conv_K=conv_K, chunk=chunk,
                    gate_mode=gate, in_dtype=GDN_BF16 if bf16_in else GDN_F32,
                    out_dtype=GDN_BF16 if bf16_out else GDN_F32, flags=flags,
                    q_scale=q_scale, eps_l2=eps_l2, eps_norm=eps_norm)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr()) if hasattr(t, "data_ptr") else int(t)


def tensors_from_torch(*, qkv, f, beta, z, conv_w, A_log, dt_bias, norm_w, conv_state, state,
                       out, state_hist=None, conv_hist=None) -> GdnTensors:
    """Plain device pointers of contiguous tensors (or integer addresses)."""
    for name, t in (("qkv", qkv), ("f", f), ("beta", beta), ("z", z), ("conv_w", conv_w),
                    ("A_log", A_log), ("dt_bias", dt_bias), ("norm_w", norm_w),
                    ("conv_state", conv_state), ("state", state), ("out", out),
                    ("state_hist", state_hist), ("conv_hist", conv_hist)):
        if t is not None and hasattr(t, "is_contiguous") and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    t = GdnTensors(qkv=_ptr(qkv), f=_ptr(f), beta=_ptr(beta), z=_ptr(z), conv_w=_ptr(conv_w),
                   A_log=_ptr(A_log), dt_bias=_ptr(dt_bias), norm_w=_ptr(norm_w),
                   conv_state=_ptr(conv_state), state=_ptr(state), out=_ptr(out),
                   state_hist=_ptr(state_hist), conv_hist=_ptr(conv_hist))
    # the struct keeps its tensors alive (it holds only their addresses)
    t._keep = (qkv, f, beta, z, conv_w, A_log, dt_bias, norm_w, conv_state, state, out,
               state_hist, conv_hist)
    return t
