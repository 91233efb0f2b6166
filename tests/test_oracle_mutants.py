"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is a copy of the oracle's C source with one plausible mistake
substituted in (a dropped term, a wrong sign or index, a transposed operand),
compiled on the CPU into a temporary library.  The pins in ``oracle_pins`` are
then run against it; a mutant that no pin catches means the pins leave that
part of the oracle unchecked.
"""
import os

import pytest

import oracle as oracle_pkg
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "gdn_oracle.c")

MUTANTS = {
    "no_decay": ("for (int i = 0; i < dv * dk; ++i) S[i] *= alpha;",
                 "for (int i = 0; i < dv * dk; ++i) S[i] *= 1.0;"),
    "alpha_is_g": ("double alpha = exp(g[t]);", "double alpha = g[t];"),
    "u_transposed": ("acc += S[(size_t)i * dk + j] * kt[j];", "acc += S[(size_t)j * dk + i] * kt[j];"),
    "delta_sign": ("double c = beta[t] * (vt[i] - u[i]);", "double c = beta[t] * (u[i] - vt[i]);"),
    "beta_dropped": ("double c = beta[t] * (vt[i] - u[i]);", "double c = (vt[i] - u[i]);"),
    "read_with_k": ("acc += S[(size_t)i * dk + j] * qt[j];", "acc += S[(size_t)i * dk + j] * kt[j];"),
    "conv_taps_reversed": ("acc += w[(size_t)c * W + j] * xv;", "acc += w[(size_t)c * W + (W - 1 - j)] * xv;"),
    "conv_buffer_not_advanced": ("int p = L - (W - 1) + i;", "int p = i - (W - 1);"),
    "silu_sign": ("return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    "gqa_modulo": ("int hk = h / r;", "int hk = h % hqk;"),
    "softplus_dropped": ("g[t] = -exp(A_log) * softplus_d(a[t] + dt_bias);", "g[t] = -exp(A_log) * (a[t] + dt_bias);"),
    "dt_bias_dropped": ("g[t] = -exp(A_log) * softplus_d(a[t] + dt_bias);", "g[t] = -exp(A_log) * softplus_d(a[t]);"),
    "A_log_not_exponentiated": ("g[t] = -exp(A_log) * softplus_d(a[t] + dt_bias);",
                                "g[t] = -A_log * softplus_d(a[t] + dt_bias);"),
    "beta_sign": ("beta[t] = sigmoid_d(b[t]);", "beta[t] = sigmoid_d(-b[t]);"),
    "l2_no_sqrt": ("double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / (ss + eps);"),
    "no_q_scale": ("qh[(size_t)(t0 + t) * Cq + i] *= qscale;", "qh[(size_t)(t0 + t) * Cq + i] *= 1.0;"),
    "rms_sum_not_mean": ("double inv = 1.0 / sqrt(ss / dv + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    "gate_z_not_silu": ("* w[i] * silu_d(z[(size_t)t * dv + i]);", "* w[i] * z[(size_t)t * dv + i];"),
    "norm_weight_dropped": ("* w[i] * silu_d(z[(size_t)t * dv + i]);", "* silu_d(z[(size_t)t * dv + i]);"),
    "v_head_uses_qk_index": ("vc + (size_t)(t0 + t) * Cv + (size_t)h * dv, sizeof(double) * dv);",
                             "vc + (size_t)(t0 + t) * Cv + (size_t)hk * dv, sizeof(double) * dv);"),
    "chunk_solve_sign": ("s -= A[(size_t)i * C + x] * T[(size_t)x * C + j];",
                         "s += A[(size_t)i * C + x] * T[(size_t)x * C + j];"),
    "chunk_decay_off_by_one": ("for (int t = j + 1; t <= i; ++t) sj += gc[t];",
                               "for (int t = j; t <= i; ++t) sj += gc[t];"),
    "chunk_no_state_read": ("Dl[(size_t)i * dv + r] = U[(size_t)i * dv + r] - s;",
                            "Dl[(size_t)i * dv + r] = U[(size_t)i * dv + r];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle_pkg.build(str(path), str(tmp_path / f"lib{name}.so"), openmp=False)
    mutant = oracle_pkg.load(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception as e:  # a crash in the pin also counts as a detection
            caught.append(f"{pin.__name__} ({type(e).__name__})")
    assert caught, f"mutant {name} passes every pin"
