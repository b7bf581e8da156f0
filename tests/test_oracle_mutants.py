"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is a textual edit of a copy of oracle/gdn_oracle.c, compiled on
the host into a temporary library; the oracle source itself is untouched.
Every edit keeps all memory accesses in bounds.
"""

import os

import pytest

import oracle
import oracle_pins

pytestmark = pytest.mark.cpu

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = {
    "decay_neighbour_channel": ("S[(size_t)i * d_v + j] *= alpha[i];",
                                "S[(size_t)i * d_v + j] *= alpha[(i + 1) % d_k];"),
    "beta_not_applied": ("u[j] = beta * (v[j] - kS);", "u[j] = (v[j] - kS);"),
    "delta_sign": ("u[j] = beta * (v[j] - kS);", "u[j] = beta * (v[j] + kS);"),
    "readout_with_k": ("acc += S[(size_t)i * d_v + j] * q[i];",
                       "acc += S[(size_t)i * d_v + j] * k[i];"),
    "conv_taps_reversed": ("(double)conv_w[c * s->K + j] *",
                           "(double)conv_w[c * s->K + (s->K - 1 - j)] *"),
    "q_scale_missing": ("gdn_oracle_l2norm(s->d_k, tmp, s->q_scale, s->eps_l2, q);",
                        "gdn_oracle_l2norm(s->d_k, tmp, 1.0, s->eps_l2, q);"),
    "gate_silu_missing": (": gdn_oracle_silu(z[j]));", ": z[j]);"),
    "sigmoid_gate_is_silu": ("(sigmoid_gate ? gdn_oracle_sigmoid(z[j])", "(sigmoid_gate ? gdn_oracle_silu(z[j])"),
    "lb_gate_sign": ("g[i] = lb * gdn_oracle_sigmoid(-a * f[i]);", "g[i] = lb * gdn_oracle_sigmoid(a * f[i]);"),
    "lb_gate_uses_exp_a": ("g[i] = lb * gdn_oracle_sigmoid(-a * f[i]);",
                           "g[i] = lb * gdn_oracle_sigmoid(-exp(a) * f[i]);"),
    "softplus_first_order": ("log1p(exp(-fabs(x)))", "exp(-fabs(x))"),
    "gva_head_map": ("int hq = h / group;", "int hq = h % s->H_qk;"),
    "conv_state_off_by_one": ("x_row(s, qkv, cs0, b, s->T + r, c)",
                              "x_row(s, qkv, cs0, b, s->T + r - 1, c)"),
    "rms_uses_sum": ("ms /= (double)n;", "ms /= 1.0;"),
    "A_log_sign": ("double a = exp(A_log);", "double a = exp(-A_log);"),
    "beta_head0": ("*beta = gdn_oracle_sigmoid((double)J->beta[bth]);",
                   "*beta = gdn_oracle_sigmoid((double)J->beta[bth - h]);"),
    "chunk_cumsum_skips_first": ("(t ? G[(t - 1) * dk + i] : 0.0)",
                                 "(t > 1 ? G[(t - 1) * dk + i] : 0.0)"),
    "chunk_state_decay_neighbour": ("double gl = G[(n - 1) * dk + i];",
                                    "double gl = G[(n - 1) * dk + (i + 1) % dk];"),
    "l2_eps_outside_root": ("double r = scale / sqrt(ss + eps);",
                            "double r = scale / (sqrt(ss) + eps);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert old in text, f"mutation anchor for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib_path = oracle.build(str(src), str(tmp_path / f"lib_{name}.so"))
    lib = oracle.load(lib_path)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
