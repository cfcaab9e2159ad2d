"""The oracle against its pins, and the pins against planted mistakes.

The mutation test copies ``oracle/oracle.c``, plants one plausible mistake
(a dropped term, a wrong sign or index, a transposed operand), compiles the
copy on the CPU and checks that at least one pin rejects it.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


CAUSAL_BODY = (
    "            update_state(S, z, fk, vi, P, Dv);\n"
    "            oracle_phi(qi, D, kind, W, m, fq);\n"
    "            readout(S, z, fq, out + (h * N + i) * Dv, P, Dv);\n"
)
CAUSAL_BODY_EXCLUSIVE = (
    "            oracle_phi(qi, D, kind, W, m, fq);\n"
    "            readout(S, z, fq, out + (h * N + i) * Dv, P, Dv);\n"
    "            update_state(S, z, fk, vi, P, Dv);\n"
)

MUTATIONS = {
    "elu_drops_plus_one": ("return x + 1.0;", "return x;"),
    "elu_wrong_sign": ("return exp(x);", "return exp(-x);"),
    "elu_wrong_branch": ("if (x > 0.0)", "if (x > 1.0)"),
    "prf_wx_sign": ("f[r] = exp(wx - 0.5 * sq)", "f[r] = exp(-wx - 0.5 * sq)"),
    "prf_drops_half": ("f[r] = exp(wx - 0.5 * sq)", "f[r] = exp(wx - sq)"),
    "prf_drops_norm": ("f[r] = exp(wx - 0.5 * sq)", "f[r] = exp(wx)"),
    "prf_scale_1_over_m": ("1.0 / sqrt((double)m)", "1.0 / (double)m"),
    "prf_transposed_W": ("W[(long)r * D + d]", "W[(long)d * m + r]"),
    "causal_exclusive": (CAUSAL_BODY, CAUSAL_BODY_EXCLUSIVE),
    "state_transposed": ("S[(long)a * Dv + c] += fk[a] * v[c];",
                         "S[(long)c * P + a] += fk[a] * v[c];"),
    "den_drops_phi_q": ("den += fq[a] * z[a];", "den += z[a];"),
    "num_wrong_index": ("num += fq[a] * S[(long)a * Dv + c];",
                        "num += fq[c % P] * S[(long)a * Dv + c];"),
    "noncausal_drops_last_key": ("for (long j = 0; j < N; j++) {\n            oracle_phi(k + (h * N + j)",
                                 "for (long j = 0; j < N - 1; j++) {\n            oracle_phi(k + (h * N + j)"),
    "step_wrong_v_offset": ("update_state(Sh, zh, f, v + h * Dv, P, Dv);",
                            "update_state(Sh, zh, f, v + h * D, P, Dv);"),
    "quadratic_strict_mask": ("long last = causal ? i : N - 1;",
                              "long last = causal ? i - 1 : N - 1;"),
    "z_not_accumulated": ("z[a] += fk[a];", "z[a] = fk[a];"),
    "bwd_dden_sign": ("dden[i] = -dot / den;", "dden[i] = dot / den;"),
    "bwd_dq_drops_dden": ("double s = z[a] * dden[i];", "double s = 0.0 * z[a] * dden[i];"),
    "bwd_dk_drops_r": ("double s = r[a];", "double s = 0.0 * r[a];"),
    "bwd_dv_uses_phi_q": ("s += R[(long)a * Dv + c] * f[a];", "s += R[(long)a * Dv + c] * g[a];"),
    "bwd_reverse_exclusive": ("accumulate_reverse(R, r, g, dnum + j * Dv, dden[j], P, Dv);\n            }\n            oracle_phi(kh + j * D, D, kind, W, m, f);",
                              "}\n            oracle_phi(kh + j * D, D, kind, W, m, f);"),
    "bwd_elu_vjp_branch": ("(x[d] > 0.0 ? 1.0 : exp(x[d]))", "(x[d] > 0.0 ? exp(x[d]) : 1.0)"),
    "bwd_prf_vjp_drops_x": ("dx[d] -= s * x[d];", "dx[d] -= 0.0 * s * x[d];"),
    "bwd_prf_vjp_transposed_W": ("dx[d] += c * W[(long)r * D + d];", "dx[d] += c * W[(long)d * m + r];"),
    "nprf_not_normalised": ("double scale = (kind == ORACLE_PHI_NPRF && sq > 0.0) ? 1.0 / sqrt(sq) : 1.0;",
                            "double scale = 1.0;"),
    "trf_sin_cos_swapped": ("f[r] = a * cos(wx);\n            f[m + r] = a * sin(wx);",
                            "f[r] = a * sin(wx);\n            f[m + r] = a * cos(wx);"),
    "trf_exponent_sign": ("double a = exp(0.5 * sq) * inv_sqrt_m;", "double a = exp(-0.5 * sq) * inv_sqrt_m;"),
    "bwd_nprf_no_projection": ("dx[d] = (dx[d] - dy_y * x[d] / n) / n;", "dx[d] = dx[d] / n;"),
    "bwd_trf_rotation_sign": ("double c = df[m + r] * f[r] - df[r] * f[m + r];",
                              "double c = df[r] * f[m + r] - df[m + r] * f[r];"),
    "rpe_offset_sign": ("a *= exp(bh[i - j + N - 1]);", "a *= exp(bh[j - i + N - 1]);"),
    "rpe_weight_on_num_only": ("                den += a;\n                for (int c = 0; c < Dv; c++)\n                    num[c] += a * v[(h * N + j) * Dv + c];",
                               "                den += a / exp(bh[i - j + N - 1]);\n                for (int c = 0; c < Dv; c++)\n                    num[c] += a * v[(h * N + j) * Dv + c];"),
    "prefix_u_not_rescaled": ("st[1] = st[1] * a + b;", "st[1] = st[1] + b;"),
    "prefix_no_running_max": ("double mn = s > m ? s : m;", "double mn = s;"),
    "prefix_w_drops_weight": ("st[2 + c] = st[2 + c] * a + b * v[c];", "st[2 + c] = st[2 + c] * a + v[c];"),
    "prefix_score_wrong_index": ("        s += q[d] * k[d];\n    double m = st[0];", "        s += q[d] * k[0];\n    double m = st[0];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found for {name}"
    mutated = src.replace(old, new)
    c_path = tmp_path / "oracle_mut.c"
    so_path = tmp_path / "liboracle_mut.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           str(c_path), "-o", str(so_path), "-lm"])
    lib = oracle.load(str(so_path))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, FloatingPointError, ValueError, ZeroDivisionError):
            caught.append(pin.__name__)
    assert caught, f"no pin rejects the planted mistake {name}"


def test_oracle_matches_exact_rational_fixture(oracle_lib):
    """The oracle against tests/golden/exact_elu1_causal.json: exact rational
    outputs of the causal form on positive integer inputs (phi(x) = x + 1
    there), written by tests/golden/make_exact_elu1.py without the oracle."""
    import json
    from fractions import Fraction

    import numpy as np

    doc = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "exact_elu1_causal.json")))
    q = np.array(doc["q"], dtype=np.float64)[None]
    k = np.array(doc["k"], dtype=np.float64)[None]
    v = np.array(doc["v"], dtype=np.float64)[None]
    got = oracle.forward(q, k, v, causal=True, lib=oracle_lib)[0]
    want = np.array([[[float(Fraction(x)) for x in row] for row in head] for head in doc["out"]])
    assert np.max(np.abs(got - want)) <= 1e-13 * np.max(np.abs(want))
