"""The bench's host logic on CPU.

- The end-to-end input layout: one packed row per token holds every layer's qkv, f, beta
  and z rows, each segment on a 16-byte boundary. Slicing the row gives back exactly the
  arrays the layers were generated with.
- The DRAM-traffic figures: reported only for the kernel sources they were taken on.
"""

import dataclasses
import os
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.cpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


@pytest.mark.parametrize("B,kda,bf16", [(1, True, True), (3, False, True), (2, True, False)])
def test_packed_rows_round_trip(B, kda, bf16):
    shape = synth.Shape(B=B, T=1, H_qk=2, H_v=4, d_k=16, d_v=16, kda=kda, bf16_in=bf16)
    tokens, layers = 3, 2
    sT = dataclasses.replace(shape, T=tokens)
    ins = [synth.make_inputs(sT, seed=0, layer=l) for l in range(layers)]
    packed, seg = bench.pack_token_inputs(shape, ins, tokens)
    esz = 2 if bf16 else 4
    assert packed.shape[:2] == (tokens, layers)
    assert (packed.shape[2] * esz) % 16 == 0
    fw = shape.f_width if kda else 1
    widths = {"qkv": shape.C, "f": shape.H_v * fw, "beta": shape.H_v, "z": shape.H_v * shape.d_v}
    assert {k: w for k, (_, w) in seg.items()} == widths
    ends = []
    for k, (o, w) in seg.items():
        assert (o * esz) % 16 == 0, f"{k} segment starts off a 16-byte boundary"
        ends.append((o, o + B * w))
        for l in range(layers):
            ref = getattr(ins[l], k).reshape(B, tokens, w)
            for t in range(tokens):
                got = packed[t, l, o:o + B * w].reshape(B, w)
                np.testing.assert_array_equal(got, ref[:, t])
    ends.sort()
    for (a0, a1), (b0, _) in zip(ends, ends[1:]):
        assert a1 <= b0, "segments overlap"


def test_traffic_figures_only_for_unchanged_sources(tmp_path):
    """A DRAM-traffic figure is reported only while the sources of the workload's kernels
    hash to the value recorded with it; any other hash, or a missing entry, gives None."""
    import json
    w = "kda_decode_b64"
    good = bench.kernel_source_hash(bench.workload_sources(w))
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({w: {"dram_bytes_per_launch": 123, "source_sha256_16": good},
                             "kda_verify_b32_t4": {"dram_bytes_per_launch": 7,
                                                   "source_sha256_16": "0" * 16}}))
    assert bench.ncu_traffic(w, str(f)) == 123
    assert bench.ncu_traffic("kda_verify_b32_t4", str(f)) is None
    assert bench.ncu_traffic("kda_commit_b32_t4", str(f)) is None
    assert bench.ncu_traffic(w, str(tmp_path / "missing.json")) is None
    # each workload hashes the sources its kernels are built from
    assert "gdn_step.cu" in bench.workload_sources("kda_decode_b1_34layers")
    assert "gdn_stream.cu" in bench.workload_sources(w)
    assert "gdn_kda_prefill.cu" in bench.workload_sources("kda_prefill_b4_t4096")
    assert "gdn_proj.cu" in bench.workload_sources("kda_layer_decode_b1")
