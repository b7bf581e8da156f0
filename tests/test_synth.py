"""The seeded input generator: determinism, distributions, bf16 rounding."""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.cpu


def test_deterministic_and_distinct_streams():
    a = synth.normal(synth.stream_key(0, "qkv", 0, 0), 1000)
    b = synth.normal(synth.stream_key(0, "qkv", 0, 0), 1000)
    c = synth.normal(synth.stream_key(0, "qkv", 0, 1), 1000)
    assert np.array_equal(a, b)
    assert not np.allclose(a, c)
    # a prefix of a longer draw is the shorter draw (counter-based)
    d = synth.normal(synth.stream_key(0, "qkv", 0, 0), 1 << 23)
    assert np.array_equal(d[:1000], a)


def test_moments():
    x = synth.normal(synth.stream_key(5, "m"), 1 << 20)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    u = synth.uniform(synth.stream_key(5, "u"), 1 << 20, 0.0, np.log(16.0))
    assert u.min() > 0.0 and u.max() <= np.log(16.0)
    assert abs(u.mean() - np.log(16.0) / 2) < 5e-3


def test_bf16_round_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 1.0 + 2.0 ** -8 + 2.0 ** -20],
                 dtype=np.float32)
    r = synth.round_bf16(x)
    # halfway cases go to the even mantissa; above halfway rounds up
    assert r.tolist() == [1.0, 1.0, 1.0 + 2 * 2.0 ** -7, -2.5, 1.0 + 2.0 ** -7]
    assert synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0] == 0x3F80


def test_workload_shapes():
    s = synth.WORKLOADS["kda_decode_b64"]["shape"]
    assert s.C == 12288 and s.q_scale == np.float32(1 / np.sqrt(128))
    g = synth.WORKLOADS["gdn_prefill_b4_t4096"]["shape"]
    assert g.C == 8192 and g.f_width == 1
    t = synth.WORKLOADS["tiny_gdn_decode"]["shape"]
    assert t.C == 96
    inp = synth.make_inputs(s, seed=0)
    assert inp.qkv.shape == (64, 1, 12288)
    assert np.array_equal(synth.round_bf16(inp.qkv), inp.qkv)
