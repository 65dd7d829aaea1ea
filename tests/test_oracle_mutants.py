"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of oracle/kda_oracle.c -- a
flipped sign, a dropped term, a wrong index or operand, a shifted window --
builds it with gcc, and runs the pin suite (tests/test_oracle_pins.py) against
it in a child process.  Every mutant must fail at least one pin.  The frozen
regression values are left out of that run: they were written by the oracle
itself, so they would catch any change without saying anything about the
pages; the remaining pins come from the definition, closed forms, invariants,
hand-worked values and an independent dense numpy formulation.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

# name -> (text in kda_oracle.c, replacement); every mutant stays in bounds
MUTANTS = {
    "silu_sign": ("return y / (1.0 + exp(-y));", "return y / (1.0 + exp(y));"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "softplus_linear_branch": ("if (x > 20.0) return x;", "if (x > 20.0) return 20.0;"),
    "softplus_drops_one": ("return log1p(exp(x));", "return log(exp(x));"),
    "gate_sign": ("return -exp(A_log) * orc_softplus(a + dt_bias);",
                  "return exp(A_log) * orc_softplus(a + dt_bias);"),
    "gate_drops_dt_bias": ("return -exp(A_log) * orc_softplus(a + dt_bias);",
                           "return -exp(A_log) * orc_softplus(a);"),
    "safe_gate_unclamped": ("return a < 0.0 ? a : 0.0;", "return a;"),
    "conv_taps_reversed": ("acc += w[j] * xext[t + j];", "acc += w[W - 1 - j] * xext[t + j];"),
    "conv_state_reversed": ("xext[j] = cs[(size_t)c * (W - 1) + j];",
                            "xext[j] = cs[(size_t)c * (W - 1) + (W - 2 - j)];"),
    "l2norm_eps_outside_root": ("double inv = 1.0 / sqrt(ss + eps);",
                                "double inv = 1.0 / (sqrt(ss) + eps);"),
    "decay_dropped": ("for (int c = 0; c < V; ++c) S[(size_t)r * V + c] *= d;",
                      "for (int c = 0; c < V; ++c) S[(size_t)r * V + c] *= 1.0;"),
    "delta_sign": ("u[c] = v[c] - sk;", "u[c] = sk - v[c];"),
    "beta_dropped": ("S[(size_t)r * V + c] += beta * k[r] * u[c];",
                     "S[(size_t)r * V + c] += k[r] * u[c];"),
    "output_reads_k": ("for (int r = 0; r < K; ++r) sq += S[(size_t)r * V + c] * q[r];",
                       "for (int r = 0; r < K; ++r) sq += S[(size_t)r * V + c] * k[r];"),
    "output_unscaled": ("const double scale = 1.0 / sqrt((double)K);", "const double scale = 1.0;"),
    "gva_head_map": ("const int h = hv / G;", "const int h = hv % H;"),
    "k_reads_q_channels": ("kn[r] = yt[H * K + h * K + r];", "kn[r] = yt[h * K + r];"),
    "beta_not_sigmoid": ("const double beta = orc_sigmoid(b[(size_t)t * HV + hv]);",
                         "const double beta = b[(size_t)t * HV + hv];"),
    "snapshot_window_shift": ("snap[((size_t)t * dim + c) * (W - 1) + j] = xext[t + 1 + j];",
                              "snap[((size_t)t * dim + c) * (W - 1) + j] = xext[t + j];"),
    "rolled_state_shift": ("cs_new[(size_t)c * (W - 1) + j] = xext[T + j];",
                           "cs_new[(size_t)c * (W - 1) + j] = xext[T - 1 + j];"),
    "state_snapshot_is_S0": ("memcpy(inter + ((size_t)t * HV + hv) * K * V, S, sizeof(double) * (size_t)K * V);",
                             "memcpy(inter + ((size_t)t * HV + hv) * K * V, S0 + (size_t)hv * K * V,"
                             " sizeof(double) * (size_t)K * V);"),
    "commit_takes_first_token": ("memcpy(S_out, inter + (size_t)(acc - 1) * ns, sizeof(double) * ns);",
                                 "memcpy(S_out, inter, sizeof(double) * ns);"),
    "commit_conv_from_first_token": ("memcpy(cs_out, snap + (size_t)(acc - 1) * nc, sizeof(double) * nc);",
                                     "memcpy(cs_out, snap, sizeof(double) * nc);"),
    "q_not_normalised": ("      orc_l2norm(K, qn, eps);\n", ""),
    "conv_state_not_rolled": ("cs_new[(size_t)c * (W - 1) + j] = xext[T + j];",
                              "cs_new[(size_t)c * (W - 1) + j] = xext[j];"),
    "beta_from_qk_head": ("const double beta = orc_sigmoid(b[(size_t)t * HV + hv]);",
                          "const double beta = orc_sigmoid(b[(size_t)t * HV + h]);"),
    "gate_from_first_token": ("const double* at = a + ((size_t)t * HV + hv) * K;",
                              "const double* at = a + (size_t)hv * K;"),
    "silu_dropped": ("y[t] = orc_silu(acc);", "y[t] = acc;"),
    "k_not_normalised": ("      orc_l2norm(K, kn, eps);\n", ""),
    "l2norm_without_eps": ("double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / sqrt(ss);"),
    "rank1_update_uses_q": ("S[(size_t)r * V + c] += beta * k[r] * u[c];",
                            "S[(size_t)r * V + c] += beta * q[r] * u[c];"),
    "dt_bias_from_qk_head": ("dt_bias[(size_t)hv * K + r]", "dt_bias[(size_t)h * K + r]"),
    "A_log_from_qk_head": ("orc_gate_softplus(A_log[hv],", "orc_gate_softplus(A_log[h],"),
    "v_from_qk_head": ("const double* vt = yt + 2 * H * K + hv * V;", "const double* vt = yt + 2 * H * K + h * V;"),
    "decay_after_update": (
        "  /* S <- diag(exp g) S */\n"
        "  for (int r = 0; r < K; ++r) {\n"
        "    double d = exp(g[r]);\n"
        "    for (int c = 0; c < V; ++c) S[(size_t)r * V + c] *= d;\n"
        "  }\n"
        "  /* S <- S + beta k (v - S^T k)^T */\n"
        "  double* u = (double*)malloc(sizeof(double) * (size_t)V);\n"
        "  for (int c = 0; c < V; ++c) {\n"
        "    double sk = 0.0;\n"
        "    for (int r = 0; r < K; ++r) sk += S[(size_t)r * V + c] * k[r];\n"
        "    u[c] = v[c] - sk;\n"
        "  }\n"
        "  for (int r = 0; r < K; ++r)\n"
        "    for (int c = 0; c < V; ++c) S[(size_t)r * V + c] += beta * k[r] * u[c];\n",
        "  double* u = (double*)malloc(sizeof(double) * (size_t)V);\n"
        "  for (int c = 0; c < V; ++c) {\n"
        "    double sk = 0.0;\n"
        "    for (int r = 0; r < K; ++r) sk += S[(size_t)r * V + c] * k[r];\n"
        "    u[c] = v[c] - sk;\n"
        "  }\n"
        "  for (int r = 0; r < K; ++r)\n"
        "    for (int c = 0; c < V; ++c) S[(size_t)r * V + c] += beta * k[r] * u[c];\n"
        "  for (int r = 0; r < K; ++r) {\n"
        "    double d = exp(g[r]);\n"
        "    for (int c = 0; c < V; ++c) S[(size_t)r * V + c] *= d;\n"
        "  }\n"),
}


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"lib_{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib),
                    str(src), "-lm"], check=True)
    return str(lib)


def _run_pins(lib):
    # a child process loads the mutant build explicitly and runs the pins on it
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "mutant_pins_main.py"), lib],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unmutated_copy_passes_the_pins(tmp_path):
    rc, out = _run_pins(_build(tmp_path, "original", open(SRC).read()))
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not found once: {old}"
    rc, out = _run_pins(_build(tmp_path, name, text.replace(old, new)))
    assert rc == 1, f"mutant {name} passed every pin:\n{out}"
