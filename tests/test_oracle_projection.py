"""Pins of the oracle's projections and of the layer composition around the
step ("Thirty tiny kernels per layer", the KDA decode budget: q/k/v, the
f_a/f_b and g_a/g_b low-rank gate chains, beta, and the output projection).

The projection is a library matmul; these pins fix its orientation (W is
[out][in], rows of x are tokens), the order of the low-rank chains, and that
the layer feeds the projected rows to the step unchanged."""

import dataclasses

import numpy as np

import oracle
import synth


def test_projection_selects_and_orients():
    # w[n][k] = 1 at (0, 3), (1, 0), (2, 4): y[:, 0] = x[:, 3], y[:, 1] = x[:, 0], ...
    x = np.arange(10, dtype=np.float64).reshape(2, 5) + 1.0
    w = np.zeros((3, 5))
    w[0, 3] = w[1, 0] = w[2, 4] = 1.0
    y = oracle.project(x, w)
    assert y.shape == (2, 3)
    assert np.array_equal(y, x[:, [3, 0, 4]])


def test_projection_brute_force_tiny():
    rng = np.random.default_rng(1)
    x, w = rng.standard_normal((3, 7)), rng.standard_normal((4, 7))
    y = oracle.project(x, w)
    for b in range(3):
        for n in range(4):
            assert abs(y[b, n] - sum(x[b, k] * w[n, k] for k in range(7))) < 1e-12


def _tiny():
    shape = synth.Shape(B=2, T=1, H_qk=2, H_v=2, d_k=4, d_v=4, kda=True, bf16_in=False)
    W = synth.make_layer_weights(shape, 16, 8, seed=3)
    x = synth.make_layer_input(shape, 16, seed=3)
    return shape, W, x


def test_low_rank_chains_compose_in_order():
    """f = f_b(f_a(x)) is x through the product w_fb w_fa; the reverse order has
    the wrong shape, and g uses its own pair."""
    shape, W, x = _tiny()
    p = synth.make_params(shape, seed=3)
    st = synth.make_state(shape, seed=3)
    out = oracle.layer_decode(shape, p, W, x, st.conv, st.S)
    f = out["rows"]["f"]
    assert np.allclose(f, x.astype(np.float64) @ (W.w_fb.astype(np.float64) @ W.w_fa).T,
                       rtol=1e-12, atol=1e-12)
    z = out["rows"]["z"]
    assert np.allclose(z, x.astype(np.float64) @ (W.w_gb.astype(np.float64) @ W.w_ga).T,
                       rtol=1e-12, atol=1e-12)
    assert not np.allclose(z, f)


def test_layer_runs_the_step_on_the_projected_rows():
    shape, W, x = _tiny()
    p = synth.make_params(shape, seed=4)
    st = synth.make_state(shape, seed=4)
    out = oracle.layer_decode(shape, p, W, x, st.conv, st.S)
    r = out["rows"]
    rows = synth.Inputs(r["qkv"].reshape(2, 1, -1), r["f"].reshape(2, 1, 2, 4),
                        r["beta"].reshape(2, 1, 2), r["z"].reshape(2, 1, 2, 4))
    ref = oracle.run(shape, p, rows, st.conv, st.S)
    assert np.array_equal(out["y"], ref["y"]) and np.array_equal(out["state"], ref["state"])
    # the output projection of the step's rows, per token
    yb = ref["y"].reshape(2, -1)
    for b in range(2):
        for n in range(16):
            assert abs(out["x_out"][b, n] - sum(yb[b, k] * W.w_o[n, k] for k in range(8))) < 1e-10


def test_layer_weights_give_unit_variance_rows():
    """N(0, 1/fan_in) weights keep the step's input distributions (rows ~ N(0, 1))."""
    shape = synth.Shape(B=64, T=1, H_qk=4, H_v=4, d_k=32, d_v=32, kda=True, bf16_in=False)
    W = synth.make_layer_weights(shape, 512, 64, seed=5)
    x = synth.make_layer_input(shape, 512, seed=5)
    q = oracle.project(x, W.w_qkv)
    f = oracle.project(oracle.project(x, W.w_fa), W.w_fb)
    assert 0.9 < q.std() < 1.1 and 0.9 < f.std() < 1.1
