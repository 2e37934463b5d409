"""The pins catch plausible mistakes: each mutant below is a copy of the oracle source with one
planted error (a dropped term, a wrong sign or index, a transposed operand), built on the CPU
into a temporary directory. Every mutant must fail at least one pin other than the matrix-form
cross-check, so the pins constrain the oracle independently of any second formulation."""
import os
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gr_oracle.c")

MUTANTS = {
    "drop_1/n_r_inside_silu": ("h[k] = silu(inv_nb * acc);", "h[k] = silu(acc);"),
    "drop_1/n_r_in_combine": ("x[c] = inv_nb * acc;", "x[c] = acc;"),
    "drop_2_in_s": ("s[i] = 2.0 * sigmoid(inv_nb * acc);", "s[i] = sigmoid(inv_nb * acc);"),
    "drop_1/n_r_in_s": ("s[i] = 2.0 * sigmoid(inv_nb * acc);", "s[i] = 2.0 * sigmoid(acc);"),
    "drop_gamma": ("Rh[(size_t)i * D + c] = Ri[c] * inv[i] * gamma[(size_t)i * D + c];",
                   "Rh[(size_t)i * D + c] = Ri[c] * inv[i];"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-a));", "return 1.0 / (1.0 + exp(a));"),
    "eps_outside_sqrt": ("inv[i] = 1.0 / sqrt(ms + eps);", "inv[i] = 1.0 / (sqrt(ms) + eps);"),
    "norm_over_all_branches": ("double ms = ss / (double)D;", "double ms = ss / (double)(D * nb);"),
    "transposed_w_up": ("acc += w[k] * h[k];", "acc += Wu[(size_t)k * K + j] * h[k];"),
    "write_uses_s0": ("const double si = s[(size_t)t * nb + i];",
                      "const double si = s[(size_t)t * nb];"),
    "silu_is_sigmoid": ("static double silu(double a) { return a * sigmoid(a); }",
                        "static double silu(double a) { return sigmoid(a); }"),
    "write_sign": ("R_out[e] = R[e] + si * y[(size_t)t * D + c];",
                   "R_out[e] = R[e] - si * y[(size_t)t * D + c];"),
    "vec_channel_major": ("Rh[(size_t)i * D + c] = Ri[c] * inv[i] * gamma[(size_t)i * D + c];",
                          "Rh[(size_t)c * nb + i] = Ri[c] * inv[i] * gamma[(size_t)i * D + c];"),
    "fixed_gate_no_1/n_r": ("x[(size_t)t * D + c] = acc / (double)nb;",
                            "x[(size_t)t * D + c] = acc;"),
    "gamma_wrong_branch": ("Rh[(size_t)i * D + c] = Ri[c] * inv[i] * gamma[(size_t)i * D + c];",
                           "Rh[(size_t)i * D + c] = Ri[c] * inv[i] * gamma[c];"),
    "bwd_drop_norm_term": ("inv[i] * dRh[j] * gamma[j] - i3 * Ri[c] * pr / (double)D;",
                           "inv[i] * dRh[j] * gamma[j];"),
    "bwd_silu_derivative": ("dz[k] = acc * sg * (1.0 + z[k] * (1.0 - sg));",
                            "dz[k] = acc * sg;"),
    "bwd_drop_sigmoid_derivative": ("dg[j] = dG * G[j] * (1.0 - G[j]);", "dg[j] = dG;"),
    "bwd_drop_1/n_r_in_dvec": ("dRh[j] += inv_nb * acc;", "dRh[j] += acc;"),
    "bwd_dgamma_without_inv": ("pg[j] += dRh[j] * Ri[c] * inv[i];", "pg[j] += dRh[j] * Ri[c];"),
    "bwd_write_ds_wrong_branch": ("acc += dRp[(size_t)t * K + (size_t)i * D + c] * y[(size_t)t * D + c];",
                                  "acc += dRp[(size_t)t * K + c] * y[(size_t)t * D + c];"),
    "fp8_scale_may_clip": ("    if (2.0 * f > 1.75)\n        e += 1;\n", ""),
    "fp8_truncating_rounding": ("double m = nearbyint(ldexp(a, 3 - E));",
                                "double m = floor(ldexp(a, 3 - E));"),
    "fp8_exponent_bias": ("ldexp(8.0 + m, E - 10)", "ldexp(8.0 + m, E - 9)"),
    "fp8_subnormal_step": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "fp8_scale_bias": ("scales[(size_t)t * nblk + k] = (uint8_t)(e + 127);",
                       "scales[(size_t)t * nblk + k] = (uint8_t)(e + 128);"),
    "fp8_amax_over_16": ("            for (int c = 0; c < 32; ++c)\n                if (fabs(vb[c]) > a)",
                         "            for (int c = 0; c < 16; ++c)\n                if (fabs(vb[c]) > a)"),
    "dec_drop_1/n_r": ("const double ai = inv_nb * G[j] * gamma[j] * inv[i] * su[i] * yu[c];",
                       "const double ai = G[j] * gamma[j] * inv[i] * su[i] * yu[c];"),
    "dec_s_of_branch0": ("const double ai = inv_nb * G[j] * gamma[j] * inv[i] * su[i] * yu[c];",
                         "const double ai = inv_nb * G[j] * gamma[j] * inv[i] * su[0] * yu[c];"),
    "dec_drop_inv": ("const double ai = inv_nb * G[j] * gamma[j] * inv[i] * su[i] * yu[c];",
                     "const double ai = inv_nb * G[j] * gamma[j] * su[i] * yu[c];"),
    "dec_norm_not_sqrt": ("norm[(size_t)t * U + u] = sqrt(sq);", "norm[(size_t)t * U + u] = sq;"),
    "dec_branch_norm_of_total": ("bq[i] += ai * ai;", "bq[i] += a * a;"),
    "dec_pi_unnormalised": ("total > 0.0 ? norm[(size_t)t * U + u] / total : 0.0;",
                            "total > 0.0 ? norm[(size_t)t * U + u] : 0.0;"),
    "dec_writer_token_transposed": ("const double *yu = Y + ((size_t)u * n + t) * D;",
                                    "const double *yu = Y + ((size_t)t * U + u) * D;"),
    "dec_a0_without_gate": ("a += inv_nb * G[j] * gamma[j] * inv[i] * R0t[j];",
                            "a += inv_nb * gamma[j] * inv[i] * R0t[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(oracle_mod, tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found once: {old}"
    mpath = tmp_path / "gr_oracle_mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(mpath), "-o",
                    str(so), "-lm"], check=True)
    caught = []
    with oracle.use_library(str(so)):
        for pin in pins.ALL_PINS:
            if pin is pins.pin_dense_bruteforce:
                continue
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every invariant pin"
