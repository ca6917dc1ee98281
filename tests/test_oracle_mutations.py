"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle.c (on the CPU, in a temporary
directory), builds it, and runs the pin suite against that copy in a child
process. The child must fail: a mutation that survives means some part of the
oracle is not pinned.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "drop_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "top_left_causal": ("int64_t n = i + (Sk - Sq) + 1;", "int64_t n = i + 1;"),
    "causal_off_by_one": ("int64_t n = i + (Sk - Sq) + 1;", "int64_t n = i + (Sk - Sq);"),
    "keys_as_values": ("const uint16_t *vj = vbh + (j0 + j) * d;\n        for (int64_t t = 0; t < d; ++t)\n            o[t] += s[j] * bf16_to_double(vj[t]);",
                       "const uint16_t *vj = kbh + (j0 + j) * d;\n        for (int64_t t = 0; t < d; ++t)\n            o[t] += s[j] * bf16_to_double(vj[t]);"),
    "no_max_subtraction": ("    /* pass 2: sum of exponentials under the max */",
                           "    m = 0.0;\n    /* pass 2: sum of exponentials under the max */"),
    "lse_without_max": ("    *lse = m + log(l);\n}", "    *lse = log(l);\n}"),
    "exp_sign_flipped": ("        l += exp(s[j] - m);\n    /* normalise",
                         "        l += exp(m - s[j]);\n    /* normalise"),
    "no_normalisation": ("        s[j] = exp(s[j] - m) / l;\n    /* o = P V */",
                         "        s[j] = exp(s[j] - m);\n    /* o = P V */"),
    "dot_skips_last_dim": ("        for (int64_t t = 0; t < d; ++t)\n            dot +=",
                           "        for (int64_t t = 0; t + 1 < d; ++t)\n            dot +="),
    "online_form1_no_correction": ("        for (int64_t t = 0; t < d; ++t)\n            acc[t] *= correction;",
                                   "        for (int64_t t = 0; t < d; ++t)\n            acc[t] *= 1.0;"),
    "online_form2_sum_uncorrected": ("        l = l * c_old + lb * c_blk;", "        l = l + lb * c_blk;"),
    "split_weights_unnormalised": ("                double w = exp(part_lse[c] - L);",
                                   "                double w = exp(part_lse[c] - M);"),
    "masked_ignores_mask": ("                if (vis[j])\n                    idx[n++] = j;",
                            "                if (vis[j] || 1)\n                    idx[n++] = j;"),
    "masked_drops_scale": ("                s[a] = sc * dot;", "                s[a] = dot;"),
    "backward_drops_D": ("                    const double ds = p[j] * (dp[j] - D);",
                         "                    const double ds = p[j] * dp[j];"),
    "backward_dk_unscaled": ("                        dkj[t] += sc * ds * bf16_to_double(qi[t]);",
                             "                        dkj[t] += ds * bf16_to_double(qi[t]);"),
    "backward_dv_uses_ds": ("                        dvj[t] += p[j] * bf16_to_double(doi[t]);",
                            "                        dvj[t] += ds * bf16_to_double(doi[t]);"),
    "combine_weights_unnormalised": ("            double w = exp(lse_parts[c * n_rows + r] - L);",
                                     "            double w = exp(lse_parts[c * n_rows + r] - M);"),
    "e4m3_bias_8": ("mag = ldexp(8.0 + m, e - 10);", "mag = ldexp(8.0 + m, e - 11);"),
    "e4m3_subnormal_step": ("mag = ldexp((double)m, -9);", "mag = ldexp((double)m, -10);"),
    "e4m3_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))",
                       "if (frac >= 0.5)"),
    "e4m3_truncates": ("if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))", "if (0)"),
    "fp8_drops_q_descale": ("dot += (dq * e4m3_to_double(qi[t]))", "dot += (e4m3_to_double(qi[t]))"),
    "fp8_drops_v_descale": ("o[t] += p * (dv * e4m3_to_double(vj[t]));",
                            "o[t] += p * e4m3_to_double(vj[t]);"),
    "fp8_reference_not_power_of_two": ("const double M = quantize_p ? ceil(mx) : mx;",
                                       "const double M = mx;"),
    "fp8_sum_after_rounding": ("        l += exp2(x[j] - M);",
                               "        l += quantize_p ? ldexp(e4m3_round(ldexp(exp2(x[j] - M), 7)), -7)"
                               " : exp2(x[j] - M);"),
    "fp8_lse_wrong_base": ("*lse = kLn2 * (M + log2(l));", "*lse = M + log(l);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found in oracle.c"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "oracle_mut.c"
    c_path.write_text(mutated)
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(c_path),
                    "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_backward_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_fp8_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {name} survived the oracle pins:\n{r.stdout[-2000:]}"
