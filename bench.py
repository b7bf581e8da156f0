#!/usr/bin/env python3
"""Throughput of the KDA / Gated DeltaNet step on GB300 (one JSON line).

Metric: delta-rule decode layer-steps/s (one layer-step = one sequence
advanced one token through one layer) and the achieved HBM GB/s of the step
kernel as a fraction of the measured copy bandwidth.

Default workload: KDA single-sequence decode, B=1, H=32, d_k=d_v=128, 34
independent layers stepped token-major (one bench step = one token through
all 34 layers = 34 gdn_decode_step launches, replayed from a CUDA graph with
programmatic dependent launch).  The batched-decode, verify and prefill
workloads are measured in the same run and reported under "workloads".

Timing: W untimed steps, then K steps, each bracketed by CUDA events on the
launching stream with an L2 flush (a 512 MiB memset) before it; the reported
time is the sum of the K step times.  `e2e` repeats the steps through the same
C ABI with the step's inputs copied from pinned host memory and its outputs
copied back inside the timed region.

`--impl reference` times the fp64 CPU oracle (the slow reference arm: there is no
installable implementation of the method to compare against) on the host cores
for the same workload and metric.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "delta-rule decode layer-steps/s and achieved HBM GB/s (fraction of GB300 peak)"
UNIT = "layer-steps/s"
DEFAULT_WORKLOAD = "kda_decode_b1_34layers"
FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- bytes and peaks

def algorithmic_bytes(s: synth.Shape, mode: str = "decode") -> int:
    """Bytes one call must move at minimum in this ABI's layouts.

    decode / prefill: state read + write, conv window read + write (K-1 rows
    each, shifted layout); verify: state read once, T per-token states
    written, window read; verify_outputs: state and window read only; commit
    (out not written): state and window read + write.  Plus conv weights, the
    inputs, the parameters and the fp32 output where it is written.
    """
    ib = 2 if s.bf16_in else 4
    state = s.B * s.H_v * s.d_k * s.d_v * 4
    conv = s.B * (s.K - 1) * s.C * 4
    st_bytes = {"decode": 2 * state, "prefill": 2 * state, "verify": state * (1 + s.T),
                "verify_outputs": state, "commit": 2 * state}[mode]
    conv_bytes = conv if mode in ("verify", "verify_outputs") else 2 * conv
    inputs = s.B * s.T * (s.C + s.H_v * s.f_width + s.H_v + s.H_v * s.d_v) * ib
    params = s.C * s.K * 4 + s.H_v * 4 + s.H_v * (s.d_k if s.kda else 1) * 4 + s.d_v * 4
    out = 0 if mode == "commit" else s.B * s.T * s.H_v * s.d_v * 4
    return st_bytes + conv_bytes + inputs + params + out


def prefill_flops(s: synth.Shape) -> float:
    """Dense-product FLOPs of the chunked form (per value head and chunk: W, U,
    W S, Q S, A V_new, the state update; per qk head and chunk: K K^T and Q K^T)."""
    C, d = s.chunk, s.d_k
    nch = -(-s.T // C)
    per_v = 2 * C * C * d * 2 + 2 * C * d * d * 3 + 2 * C * C * d
    per_qk = 2 * C * C * d * 2
    return float(s.B * nch * (s.H_v * per_v + s.H_qk * per_qk))


def two_kernel_flops(s: synth.Shape, C: int = 16) -> float:
    """Tensor-core FLOPs of the two-kernel chunked form at chunk C, per (sequence,
    value head, chunk): the state kernel's tcgen05 products W S, e^G Q S and the state
    update (2 C d^2 each) and A V_new (2 C^2 d)."""
    d = s.d_k
    units = s.B * s.H_v * -(-s.T // C)
    return float(units * (3 * 2 * C * d * d + 2 * C * C * d))


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "src": "fallback"}


# The sources each workload's kernels are built from: a traffic figure stays valid
# while these files are unchanged.
_COMMON_SOURCES = ("gdn_internal.h", "gdn_device.cuh")
_STREAM_SOURCES = _COMMON_SOURCES + ("gdn_stream.cu", "gdn_tmap.cu", "gdn_tmap.h")
_STEP_SOURCES = _COMMON_SOURCES + ("gdn_step.cu",)
_PREFILL_SOURCES = _COMMON_SOURCES + ("gdn_kda_prefill.cu", "gdn_prefill.cu", "gdn_prefill.h",
                                      "gdn_tc.cuh", "gdn_tmap.cu", "gdn_tmap.h")
_LAYER_SOURCES = tuple(sorted(set(_STREAM_SOURCES + _STEP_SOURCES + ("gdn_proj.cu", "gdn_tc.cuh"))))


def workload_sources(workload: str):
    if workload in PREFILL_WORKLOADS:
        return _PREFILL_SOURCES
    if workload in LAYER_WORKLOADS:
        return _LAYER_SOURCES
    if workload == "kda_decode_b1_34layers":
        return _STEP_SOURCES
    return _STREAM_SOURCES


def kernel_source_hash(files=None) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_decode_kda_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(csrc)):
        if fn.endswith((".cu", ".h", ".cuh")):
            h.update(fn.encode())
            h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, path: str = None):
    """DRAM bytes per launch from the committed ncu summary, if the kernels are unchanged."""
    p = path or os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("source_sha256_16") != kernel_source_hash(workload_sources(workload)):
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def __enter__(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads (GPU)

class Workload:
    name: str
    shape: synth.Shape
    launches_per_step: int
    units_per_step: int          # layer-steps per bench step
    bytes_per_launch: int
    kernel: str

    def step(self, i):            # queue one step on the current stream
        raise NotImplementedError

    def e2e_step(self, i):
        raise NotImplementedError

    def capture(self, tokens):    # build whatever the timed steps replay (default: nothing)
        pass

    h2d_bytes = 0
    d2h_bytes = 0


def _dev_inputs(shape, layers, tokens, seed=0, slow=False):
    """Per-layer params/states and [tokens, layers, B, ...] input arrays (host)."""
    import torch  # noqa: F401
    params, states, ins = [], [], []
    sT = dataclasses.replace(shape, T=tokens)
    for l in range(layers):
        params.append(synth.make_params(shape, seed=seed, layer=l, slow_decay=slow))
        states.append(synth.make_state(shape, seed=seed, layer=l))
        ins.append(synth.make_inputs(sT, seed=seed, layer=l, slow_decay=slow))
    return params, states, ins


def pack_token_inputs(shape, ins, tokens):
    """Per-layer input arrays -> one packed row per token: [tokens, layers, row] fp32, the
    row holding qkv, f, beta and z of one layer ([B, width] each, token t), every segment
    padded to 16 bytes of the input dtype.  Returns (packed, {name: (offset, width)})."""
    s = shape
    fw = s.f_width if s.kda else 1
    widths = {"qkv": s.C, "f": s.H_v * fw, "beta": s.H_v, "z": s.H_v * s.d_v}
    pad = 8 if s.bf16_in else 4
    seg, off = {}, 0
    for k, w in widths.items():
        seg[k] = (off, w)
        off += -(-(s.B * w) // pad) * pad
    packed = np.zeros((tokens, len(ins), off), np.float32)
    for k, (o, w) in seg.items():
        for l, x in enumerate(ins):
            a = getattr(x, k).reshape(s.B, tokens, w).swapaxes(0, 1)  # [tokens, B, w]
            packed[:, l, o:o + s.B * w] = a.reshape(tokens, s.B * w)
    return packed, seg


class DecodeLayers(Workload):
    """B sequences x `layers` independent layers, one token per step (graphs per token)."""

    def __init__(self, name, spec, device, pdl=True, tokens=None):
        import torch

        import linear_attention_decode_kda_gb300 as gdn
        from synth import device as dev
        self.name = name
        s = spec["shape"]
        self.shape = s
        L = spec["layers"]
        self.tokens = tokens or spec["steps"]
        self.launches_per_step = L
        self.units_per_step = L * s.B
        self.bytes_per_launch = algorithmic_bytes(s)
        params, states, ins = _dev_inputs(s, L, self.tokens)
        bf = s.bf16_in
        # One packed row per token (all layers' qkv, f, beta and z), so a token's inputs
        # are one host-to-device copy.
        packed, self.seg = pack_token_inputs(s, ins, self.tokens)
        self.dev_packed = dev.to_torch(packed, bf, device)
        self.host_packed = dev.to_torch(packed, bf, None).pin_memory()
        del packed
        self.cases = [dev.upload(s, params[l], synth.Inputs(ins[l].qkv[:, :1], ins[l].f[:, :1],
                                                              ins[l].beta[:, :1], ins[l].z[:, :1]),
                                 states[l], device=device) for l in range(L)]
        self.out = torch.empty((self.tokens, L, s.B, s.H_v * s.d_v), device=device)
        self.host_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        self.abi_shape = self.cases[0].abi_shape(pdl=pdl)
        self.kernel = gdn.gdn_kernel_variant(self.abi_shape, gdn.OP_DECODE)
        self.h2d_bytes = self.dev_packed[0].numel() * self.dev_packed.element_size()
        self.d2h_bytes = self.out[0].numel() * 4
        self.graphs, self.e2e_graphs, self.eager_tensors = {}, {}, {}
        self.gdn = gdn

    def _row(self, k, t, l):
        o, w = self.seg[k]
        return self.dev_packed[t, l, o:o + self.shape.B * w]

    def _launch_token(self, t):
        import torch
        st = torch.cuda.current_stream().cuda_stream
        for l in range(len(self.cases)):
            self.gdn.gdn_decode_step(self.abi_shape, self._tensors(t, l), st)

    def _tensors(self, t, l):
        c = self.cases[l]
        return self.gdn.tensors_from_torch(
            qkv=self._row("qkv", t, l), f=self._row("f", t, l), beta=self._row("beta", t, l),
            z=self._row("z", t, l), conv_w=c.conv_w, A_log=c.A_log, dt_bias=c.dt_bias,
            norm_w=c.norm_w, conv_state=c.conv_state, state=c.state, out=self.out[t, l])

    def capture(self, tokens):
        import torch
        for t in tokens:
            if t in self.graphs:
                continue
            self.eager_tensors[t] = [self._tensors(t, l) for l in range(len(self.cases))]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._launch_token(t)
            self.graphs[t] = g
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge):
                self.dev_packed[t].copy_(self.host_packed[t], non_blocking=True)
                self._launch_token(t)
                self.host_out[t].copy_(self.out[t], non_blocking=True)
            self.e2e_graphs[t] = ge

    def step(self, i):
        self.graphs[i % self.tokens].replay()

    def e2e_graph_step(self, i):
        self.e2e_graphs[i % self.tokens].replay()

    def e2e_step(self, i):
        """The token's inputs copied in, one gdn_decode_step call per layer through the
        C ABI (host checks and launch included), the outputs copied back."""
        import torch
        t = i % self.tokens
        st = torch.cuda.current_stream().cuda_stream
        self.dev_packed[t].copy_(self.host_packed[t], non_blocking=True)
        for tens in self.eager_tensors[t]:
            self.gdn.gdn_decode_step(self.abi_shape, tens, st)
        self.host_out[t].copy_(self.out[t], non_blocking=True)


class SingleLaunch(Workload):
    """Batched decode, verify or prefill: one ABI call per step."""

    def __init__(self, name, spec, device, mode, n_inputs=8):
        import torch

        import linear_attention_decode_kda_gb300 as gdn
        from synth import device as dev
        s = spec["shape"]
        op = {"decode": gdn.OP_DECODE, "verify": gdn.OP_VERIFY, "verify_outputs": gdn.OP_VERIFY,
              "commit": gdn.OP_VERIFY, "prefill": gdn.OP_PREFILL}[mode]
        self.name, self.shape, self.op, self.mode, self.gdn = name, s, op, mode, gdn
        self.launches_per_step = 1
        self.units_per_step = s.B * s.T
        self.bytes_per_launch = algorithmic_bytes(s, mode)
        params = synth.make_params(s)
        state = synth.make_state(s)
        n = n_inputs if op == gdn.OP_DECODE else 1
        self.n = n
        inp = synth.make_inputs(dataclasses.replace(s, T=s.T * n))
        bf = s.bf16_in
        fw = s.f_width if s.kda else 1

        def split(a, width):
            # [B, n*T, width] -> [n, B, T, width]
            return np.ascontiguousarray(a.reshape(s.B, n, s.T, width).swapaxes(0, 1))
        host = {"qkv": split(inp.qkv, s.C), "f": split(inp.f, s.H_v * fw),
                "beta": split(inp.beta, s.H_v), "z": split(inp.z, s.H_v * s.d_v)}
        self.dev_in = {k: dev.to_torch(v, bf, device) for k, v in host.items()}
        self.host_in = {k: dev.to_torch(v, bf, None).pin_memory() for k, v in host.items()}
        first = synth.Inputs(inp.qkv[:, :s.T], inp.f[:, :s.T], inp.beta[:, :s.T], inp.z[:, :s.T])
        self.case = dev.upload(s, params, first, state, device=device, hist=(mode == "verify"))
        self.out = torch.empty((n, s.B, s.T, s.H_v * s.d_v), device=device)
        self.host_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        self.abi_shape = self.case.abi_shape()
        self.kernel = gdn.gdn_kernel_variant(self.abi_shape, op)
        # kernels one call launches: the two-kernel chunked prefill launches two
        self.kernels_per_launch = 2 if (self.kernel or "").startswith("kda_chunked") else 1
        # dense products of the chunked form at the chunk length the kernel runs
        m = re.match(r"chunked<\d+,(\d+)>", self.kernel or "") if op == gdn.OP_PREFILL else None
        self.flops_per_launch = (prefill_flops(dataclasses.replace(s, chunk=int(m.group(1))))
                                 if m else 0.0)
        m = re.match(r"kda_chunked<(\d+)>", self.kernel or "") if op == gdn.OP_PREFILL else None
        if m:
            self.flops_per_launch = two_kernel_flops(s, int(m.group(1)))
        self.ws_bytes = gdn.gdn_prefill_workspace_bytes(self.abi_shape) if op == 2 else 0
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        self.h2d_bytes = sum(v[0].numel() * v.element_size() for v in self.dev_in.values())
        self.d2h_bytes = self.out[0].numel() * 4

    def _tensors(self, j):
        c = self.case
        return self.gdn.tensors_from_torch(
            qkv=self.dev_in["qkv"][j], f=self.dev_in["f"][j], beta=self.dev_in["beta"][j],
            z=self.dev_in["z"][j], conv_w=c.conv_w, A_log=c.A_log, dt_bias=c.dt_bias,
            norm_w=c.norm_w, conv_state=c.conv_state, state=c.state,
            out=None if self.mode == "commit" else self.out[j], state_hist=c.state_hist)

    def _launch(self, j):
        import torch
        st = torch.cuda.current_stream().cuda_stream
        g = self.gdn
        if self.mode == "decode":
            g.gdn_decode_step(self.abi_shape, self._tensors(j), st)
        elif self.mode == "commit":
            g.gdn_commit_accepted(self.abi_shape, self._tensors(j), None, st)
        elif self.op == g.OP_VERIFY:
            g.gdn_verify_T(self.abi_shape, self._tensors(j), st)
        else:
            g.gdn_prefill_chunked(self.abi_shape, self._tensors(j), self.ws.data_ptr(),
                                  self.ws_bytes, st)

    def step(self, i):
        self._launch(i % self.n)

    def e2e_step(self, i):
        j = i % self.n
        for k in self.dev_in:
            self.dev_in[k][j].copy_(self.host_in[k][j], non_blocking=True)
        self._launch(j)
        self.host_out[j].copy_(self.out[j], non_blocking=True)


class LayerDecode(Workload):
    """One KDA layer per step, projections included (gdn_layer_decode): the layer
    input x [B, d_model] bf16 -> q/k/v, f, beta, z rows -> the step -> x_out."""

    D_MODEL, RANK = 4096, 128

    def __init__(self, name, shape, device):
        import torch

        import linear_attention_decode_kda_gb300 as gdn
        from synth import device as dev
        self.gdn = gdn
        self.name = name
        s = dataclasses.replace(shape, bf16_in=False)  # fp32 rows between the launches
        self.shape = s
        D, R = self.D_MODEL, self.RANK
        params = synth.make_params(s)
        state = synth.make_state(s)
        W = synth.make_layer_weights(s, D, R)
        self.n = 4  # distinct inputs, cycled
        xs = np.stack([synth.make_layer_input(s, D, step=i) for i in range(self.n)])
        zero = synth.Inputs(np.zeros((s.B, 1, s.C), np.float32),
                            np.zeros((s.B, 1, s.H_v, s.d_k), np.float32),
                            np.zeros((s.B, 1, s.H_v), np.float32),
                            np.zeros((s.B, 1, s.H_v, s.d_v), np.float32))
        self.case = dev.upload(s, params, zero, state, device=device)
        self.abi_shape = self.case.abi_shape()
        self.w = {k: dev.to_torch(getattr(W, k), True, device) for k in W.FIELDS}
        self.weights = gdn.layer_weights_from_torch(D, R, **self.w)
        self.x = dev.to_torch(xs, True, device)
        self.host_x = dev.to_torch(xs, True, None).pin_memory()
        self.x_out = torch.empty((self.n, s.B, D), dtype=torch.float32, device=device)
        self.host_out = torch.empty(self.x_out.shape, dtype=torch.float32).pin_memory()
        self.ws_bytes = gdn.gdn_layer_workspace_bytes(self.abi_shape, self.weights)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        self.tensors = self.case.abi_tensors()
        self.kernel = "proj + " + (gdn.gdn_kernel_variant(self.abi_shape, gdn.OP_DECODE) or "?")
        self.launches_per_step = 1
        # in-projection, step, output projection; the gate pair is a launch of its own
        # unless the step runs on the column-slab kernel, which computes the gates itself
        step_kernel = gdn.gdn_kernel_variant(self.abi_shape, gdn.OP_DECODE) or ""
        self.kernels_per_launch = 3 if step_kernel.startswith("step<") else 4
        self.units_per_step = s.B
        wbytes = sum(int(v.numel()) * 2 for v in self.w.values())
        self.weight_bytes = wbytes
        self.bytes_per_launch = wbytes + s.B * D * (2 + 4) + algorithmic_bytes(s, "decode")
        self.h2d_bytes = s.B * D * 2
        self.d2h_bytes = s.B * D * 4

    def _launch(self, j):
        import torch
        self.gdn.gdn_layer_decode(self.abi_shape, self.weights, self.x[j], self.x_out[j],
                                  self.tensors, self.ws.data_ptr(), self.ws_bytes,
                                  torch.cuda.current_stream().cuda_stream)

    def step(self, i):
        self._launch(i % self.n)

    def e2e_step(self, i):
        j = i % self.n
        self.x[j].copy_(self.host_x[j], non_blocking=True)
        self._launch(j)
        self.host_out[j].copy_(self.x_out[j], non_blocking=True)


LAYER_WORKLOADS = {"kda_layer_decode_b1": 1, "kda_layer_decode_b64": 64}

# The 34-layer decode chain at a middle batch (8 sequences), 16 distinct tokens cycled.
MIDBATCH_WORKLOADS = {"kda_decode_b8_34layers": 8}

# The verify workload's two calls of a speculative step without per-token states:
# a verify that writes outputs only, then the in-place commit of the accepted tokens.
EXTRA_WORKLOADS = {"kda_verify_b32_t4_outputs_only": ("kda_verify_b32_t4", "verify_outputs"),
                   "kda_commit_b32_t4": ("kda_verify_b32_t4", "commit"),
                   # batched decode with the bounded per-channel gate and the sigmoid output gate
                   "kda_decode_b64_bounded_gate": ("kda_decode_b64", "decode"),
                   # the prefill at the same size with the per-channel decay, 32 qk heads
                   "kda_prefill_b4_t4096": ("gdn_prefill_b4_t4096", "prefill")}
EXTRA_SHAPES = {"kda_decode_b64_bounded_gate": dict(lb_gate=True, sigmoid_out=True),
                "kda_prefill_b4_t4096": dict(kda=True, H_qk=32)}
PREFILL_WORKLOADS = ("gdn_prefill_b4_t4096", "kda_prefill_b4_t4096")


def make_workload(name, device):
    import linear_attention_decode_kda_gb300 as gdn
    if name in LAYER_WORKLOADS:
        shape = dataclasses.replace(synth.WORKLOADS["kda_decode_b64"]["shape"], B=LAYER_WORKLOADS[name])
        return LayerDecode(name, shape, device)
    spec = synth.WORKLOADS.get(name)
    if name == "kda_decode_b1_34layers":
        return DecodeLayers(name, spec, device)
    if name in MIDBATCH_WORKLOADS:
        spec = dict(synth.WORKLOADS["kda_decode_b1_34layers"])
        spec["shape"] = dataclasses.replace(spec["shape"], B=MIDBATCH_WORKLOADS[name])
        return DecodeLayers(name, spec, device, tokens=16)
    if name in EXTRA_WORKLOADS:
        base, mode = EXTRA_WORKLOADS[name]
        spec = dict(synth.WORKLOADS[base])
        if name in EXTRA_SHAPES:
            spec["shape"] = dataclasses.replace(spec["shape"], **EXTRA_SHAPES[name])
        return SingleLaunch(name, spec, device, mode)
    mode = {"kda_decode_b64": "decode", "kda_verify_b32_t4": "verify",
            "gdn_prefill_b4_t4096": "prefill", "tiny_gdn_decode": "decode"}[name]
    return SingleLaunch(name, spec, device, mode)


# ---------------------------------------------------------------- ranks

def max_over_ranks(values, world: int, device=None) -> list:
    """Per-rank elapsed times (ms) -> their maximum over all ranks (every rank
    gets the same list).  One rank: unchanged.  Uses the default process group."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(units_per_step: int, steps: int, world: int, ms: float) -> float:
    """Units all ranks processed (each rank runs its own full workload: weak
    scaling) per second of the slowest rank's time."""
    return units_per_step * steps * world / (ms * 1e-3)


# ---------------------------------------------------------------- timing

def time_steps(fn, warmup, steps, flush):
    """Sum of per-step CUDA-event times (ms) on the current stream, L2 flushed before each."""
    import torch
    for i in range(warmup):
        flush.zero_()
        fn(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record()
        fn(warmup + i)
        ev[i][1].record()
    torch.cuda.synchronize()
    return float(sum(a.elapsed_time(b) for a, b in ev))


# Nominal HBM3e bandwidth of the part (about 8 TB/s).  The roofline fraction divides by
# the measured copy bandwidth; frac_nominal divides by this figure, the harder bar.
NOMINAL_HBM_GBS = 8000.0


def roofline(w: Workload, ms_per_step: float, peaks: dict) -> dict:
    per_launch_s = ms_per_step * 1e-3 / w.launches_per_step
    achieved = w.bytes_per_launch / per_launch_s / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": ncu_traffic(w.name), "kernel": w.kernel,
            "algorithmic_bytes_per_launch": w.bytes_per_launch,
            "peak_source": peaks["src"] + " copy bandwidth",
            "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "peak_nominal": NOMINAL_HBM_GBS}


def workload_entry(w: Workload, wms: float, peaks: dict) -> dict:
    """One workload's figures, short keys so the whole line stays a few KB:
    v layer-steps/s, us per call, frac of the measured copy peak achieved over the
    algorithmic bytes, fnom the same of the nominal 8 TB/s, tr ncu DRAM bytes per call
    (null when not taken on the current sources), k the kernel; prefill adds tc, the
    fraction of the bf16 tensor peak of the chunked form's dense products."""
    r = roofline(w, wms, peaks)
    e = {"v": round(w.units_per_step / (wms * 1e-3), 1), "us": round(wms * 1e3, 2),
         "frac": r["frac"], "fnom": r["frac_nominal"], "tr": r["traffic"], "k": w.kernel}
    if getattr(w, "flops_per_launch", 0):
        tf = w.flops_per_launch / (wms * 1e-3) / 1e12
        e["tc"] = round(tf / peaks["bf16_tflops"], 4)
    return e


# ---------------------------------------------------------------- CPU oracle legs

def oracle_decode_rate(name: str, tokens: int, nthreads: int, target_s: float = 12.0,
                       max_passes: int = 64) -> dict:
    """The fp64 oracle on a bounded sample of the workload: layer-steps/s.

    Every layer of the workload advances `tokens` tokens per pass (one oracle
    call per layer, threads over the (sequence, head) units); passes repeat,
    carrying the state, until about `target_s` seconds of oracle time.
    Generating the inputs is not timed.
    """
    import oracle
    spec = synth.WORKLOADS[name]
    s = spec["shape"]
    layers = spec["layers"]
    sT = dataclasses.replace(s, T=tokens)
    cases = []
    for l in range(layers):
        st = synth.make_state(s, layer=l)
        cases.append([synth.make_params(s, layer=l), synth.make_inputs(sT, layer=l),
                      st.conv, st.S])
    lib = oracle.load()
    dt, passes = 0.0, 0
    while passes < max_passes and (passes == 0 or dt < target_s):
        for c in cases:
            t0 = time.perf_counter()
            r = oracle.run(sT, c[0], c[1], c[2], c[3], nthreads=nthreads, lib=lib)
            dt += time.perf_counter() - t0
            c[2], c[3] = r["conv_state"], r["state"]
        passes += 1
    steps = passes * layers * s.B * tokens
    return {"value": round(steps / dt, 2), "unit": UNIT,
            "cores": min(nthreads, s.B * s.H_v), "kind": "oracle",
            "sample": f"{passes} passes x {layers} layers x {tokens} tokens, fp64 C, "
                      f"threads over units",
            "seconds": round(dt, 2)}


def cpu_baseline(name: str, tokens: int, nthreads: int) -> dict:
    """The oracle on every host core (about 12 s) and on one thread (about 6 s), with
    the effective GB/s over the same algorithmic bytes per layer-step as the GPU line."""
    multi = oracle_decode_rate(name, tokens, nthreads)
    single = oracle_decode_rate(name, tokens, 1, target_s=6.0)
    per_step = algorithmic_bytes(synth.WORKLOADS[name]["shape"]) / synth.WORKLOADS[name]["shape"].B
    multi["gbs"] = round(multi["value"] * per_step / 1e9, 2)
    multi["single_thread"] = {"value": single["value"], "unit": UNIT, "cores": 1,
                              "gbs": round(single["value"] * per_step / 1e9, 3),
                              "seconds": single["seconds"]}
    return multi


def run_reference(args):
    """--impl reference: the oracle timed as the reference arm, same workload and metric."""
    import ctypes

    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    name = args.workload
    spec = synth.WORKLOADS[name]
    s = spec["shape"]
    L = spec["layers"]
    lib = oracle.load()
    nthreads = os.cpu_count() or 1
    one = dataclasses.replace(s, T=1)
    sh = oracle.make_shape(one)
    tokens = min(spec["steps"], max(args.warmup + args.steps, 1))
    sT = dataclasses.replace(s, T=tokens)
    layers = []
    for l in range(L):
        p = synth.make_params(s, layer=l)
        i = synth.make_inputs(sT, layer=l)
        st = synth.make_state(s, layer=l)
        keep = dict(conv_w=np.ascontiguousarray(p.conv_w), A_log=np.ascontiguousarray(p.A_log),
                    dt_bias=np.ascontiguousarray(p.dt_bias),
                    norm_w=np.ascontiguousarray(p.norm_w),
                    cs=st.conv.astype(np.float64), S=st.S.astype(np.float64),
                    y=np.empty((s.B, 1, s.H_v, s.d_v)),
                    toks=[tuple(np.ascontiguousarray(getattr(i, n)[:, t:t + 1], np.float32)
                                for n in ("qkv", "f", "beta", "z")) for t in range(tokens)])
        layers.append(keep)
    P = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731

    def one_step(k):
        for d in layers:
            q, f, b, z = d["toks"][k % tokens]
            lib.gdn_oracle_run(ctypes.byref(sh), P(q), P(f), P(b), P(z), P(d["conv_w"]),
                               P(d["A_log"]), P(d["dt_bias"]), P(d["norm_w"]), P(d["cs"]),
                               P(d["S"]), P(d["y"]), None, None, nthreads)
    for k in range(args.warmup):
        one_step(k)
    t0 = time.perf_counter()
    for k in range(args.steps):
        one_step(args.warmup + k)
    dt = time.perf_counter() - t0
    value = L * s.B * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "B": s.B, "H": s.H_v, "d_k": s.d_k, "d_v": s.d_v,
                       "layers": L, "step": f"one token through {L} layers"},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "kind": "oracle",
                             "cores": min(nthreads, s.B * s.H_v),
                             "sample": f"{args.steps} steps of one token through {L} layers"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main (GPU arm)

def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    peaks = measured_peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    main = make_workload(args.workload, device)
    need = range(args.warmup + args.steps)
    main.capture(sorted({i % getattr(main, "tokens", 1) for i in need}))
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid

    if world > 1:
        dist.barrier()
    with ClockSampler(str(uuid) if uuid else None) as clk:
        ms = time_steps(main.step, args.warmup, args.steps, flush)
    ms_e2e = time_steps(main.e2e_step, args.warmup, args.steps, flush)
    graph_leg = getattr(main, "e2e_graph_step", None)
    ms_e2e_graph = time_steps(graph_leg, args.warmup, args.steps, flush) if graph_leg else 0.0
    ms, ms_e2e, ms_e2e_graph = max_over_ranks([ms, ms_e2e, ms_e2e_graph], world, device)
    if world > 1:
        dist.barrier()

    value = whole_job_rate(main.units_per_step, args.steps, world, ms)
    ms_step = ms / args.steps
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": main.name, "B": main.shape.B, "H": main.shape.H_v,
                       "d_k": main.shape.d_k, "d_v": main.shape.d_v,
                       "layers": main.launches_per_step if main.name.endswith("layers") else 1,
                       "gate": "per-channel (KDA)" if main.shape.kda else "per-head (GDN)",
                       "inputs": "bf16" if main.shape.bf16_in else "f32",
                       "state": "f32", "out": "f32",
                       "l2": f"{FLUSH_BYTES >> 20} MiB memset before each step",
                       "launch": "graph per token, PDL"
                       if isinstance(main, DecodeLayers) else "one ABI call per step",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline(main, ms_step, peaks),
            "e2e": {"value": round(whole_job_rate(main.units_per_step, args.steps, world,
                                                  ms_e2e), 2), "unit": UNIT,
                    "h2d_bytes_per_step": main.h2d_bytes, "d2h_bytes_per_step": main.d2h_bytes},
            "gpu_launches": main.launches_per_step * getattr(main, "kernels_per_launch", 1) * args.steps,
            "clocks": clk.summary()}
    if graph_leg:
        # the same copies and launches replayed from a CUDA graph captured per token
        line["e2e_graph"] = {"value": round(whole_job_rate(main.units_per_step, args.steps, world,
                                                           ms_e2e_graph), 2), "unit": UNIT}

    if rank == 0 and not args.no_workloads:
        extra = {}
        for name in ("kda_decode_b8_34layers", "kda_decode_b64", "kda_decode_b64_bounded_gate",
                     "kda_verify_b32_t4",
                     "kda_verify_b32_t4_outputs_only", "kda_commit_b32_t4", "gdn_prefill_b4_t4096",
                     "kda_prefill_b4_t4096", "kda_layer_decode_b1", "kda_layer_decode_b64"):
            if name == main.name:
                continue
            w = make_workload(name, device)
            k = args.aux_steps if name not in PREFILL_WORKLOADS else max(3, args.aux_steps // 10)
            w.capture(sorted({i % getattr(w, "tokens", 1) for i in range(3 + k)}))
            wms = time_steps(w.step, 3, k, flush) / k
            extra[name] = workload_entry(w, wms, peaks)
            del w
            torch.cuda.empty_cache()
        line["workloads"] = extra

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        name = main.name if isinstance(main, DecodeLayers) else DEFAULT_WORKLOAD
        line["cpu_baseline"] = cpu_baseline(name, args.cpu_tokens, os.cpu_count() or 1)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(list(synth.WORKLOADS) + list(EXTRA_WORKLOADS) +
                                   list(LAYER_WORKLOADS) + list(MIDBATCH_WORKLOADS)))
    ap.add_argument("--aux-steps", type=int, default=100)
    ap.add_argument("--cpu-tokens", type=int, default=64)
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
