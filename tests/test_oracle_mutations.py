"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pin suite rejects every one of them. The real oracle is never modified."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "alibi_oracle.c")

# (name, exact source text, replacement)
MUTANTS = [
    ("bias_sign", "double B = -m * D;", "double B = m * D;"),
    ("no_scale", "return s / sqrt((double)d);", "return s;"),
    ("scale_by_d", "return s / sqrt((double)d);", "return s / (double)d;"),
    ("q_dot_q", "content_score(qi, c->k + base + (size_t)j * c->d, c->d);\n        if (c->variant",
     "content_score(qi, c->q + base + (size_t)j * c->d, c->d);\n        if (c->variant"),
    ("mask_diagonal", "if (causal && j > i) return -INFINITY;", "if (causal && j >= i) return -INFINITY;"),
    ("value_row_i", "const float *vj = c->v + base + (size_t)j * c->d;",
     "const float *vj = c->v + base + (size_t)i * c->d;"),
    ("slope_exponent_h", "*num = 8 * (h + 1);", "*num = 8 * h + 4;"),
    ("appended_odd_entries", "*num = 8 * (2 * t + 1);", "*num = 8 * (2 * t + 2);"),
    ("lse_without_max", "if (c->lse) c->lse[r] = M + log(Z);", "if (c->lse) c->lse[r] = log(Z);"),
    ("decode_position", "const long pos = (long)c->L - 1;", "const long pos = (long)c->L;"),
    ("underflow_no_max", "double e = x[j] - M;", "double e = x[j];"),
    ("underflow_strict", "if (e <= c->tau) ++cnt;", "if (e < c->tau) ++cnt;"),
    ("band_strict", "if (fabs(e - c->tau) <= c->band) ++nr;", "if (fabs(e - c->tau) < c->band) ++nr;"),
    ("band_around_zero", "if (fabs(e - c->tau) <= c->band) ++nr;", "if (fabs(e) <= c->band) ++nr;"),
    ("band_in_log2_units", "if (fabs(e - c->tau) <= c->band) ++nr;",
     "if (fabs(e - c->tau) <= c->band * 0.6931471805599453) ++nr;"),
    ("band_below_only", "if (fabs(e - c->tau) <= c->band) ++nr;", "if (e - c->tau <= c->band) ++nr;"),
    ("threshold_127","t[2] = -126.0 * ln2;", "t[2] = -127.0 * ln2;"),
    ("softcap_no_z", "return z * tanh(a / z);", "return tanh(a / z);"),
    ("logdist_no_plus1", "D = log(D + 1.0);", "D = log(D);"),
    ("clamp_min", "if ((variant & ORACLE_CLAMP) && B < c_clamp) B = c_clamp;",
     "if ((variant & ORACLE_CLAMP) && B > c_clamp) B = c_clamp;"),
    ("noncausal_signed_distance", "double D = (double)(i >= j ? i - j : j - i);", "double D = (double)(i - j);"),
    ("explicit_arithmetic_spacing", "double delta = delta_first * pow(delta_last / delta_first, t);",
     "double delta = delta_first + (delta_last - delta_first) * t;"),
    ("explicit_log_ignored", "double dist = log_distance ? log(delta + 1.0) : delta;", "double dist = delta;"),
    ("prefill_one_slope", "const double m = c->m[h];", "const double m = c->m[0];"),
    ("decode_one_slope", "x[j] = a - c->m[h] * (double)(pos - j);", "x[j] = a - c->m[0] * (double)(pos - j);"),
    ("underflow_one_slope", "- c->m[h] * (double)(i - j);", "- c->m[0] * (double)(i - j);"),
    ("weights_unnormalised", "double wij = x[j] / Z;", "double wij = x[j];"),
    ("decode_unnormalised", "o[t] += (x[j] / Z) * (double)V", "o[t] += x[j] * (double)V"),
    # backward pass
    ("bwd_dq_no_rowdot", "double da = w * (bwd_g(c, bh, i, j) - c->rowdot[r]) * bwd_cap_factor(c, a);",
     "double da = w * bwd_g(c, bh, i, j) * bwd_cap_factor(c, a);"),
    ("bwd_dk_unscaled", "for (int t = 0; t < c->d; ++t) dk[t] /= sqrt((double)c->d);", ""),
    ("bwd_dv_uses_dx", "dv[t] += w * (double)oi[t];", "dv[t] += da * (double)oi[t];"),
    ("bwd_cap_factor_sign", "return 1.0 - t * t;", "return 1.0 + t * t;"),
    ("bwd_dk_with_k", "dk[t] += da * (double)qi[t];", "dk[t] += da * (double)c->k[base + (size_t)i * c->d + t];"),
    ("bwd_g_value_row_i", "(size_t)i * c->d, *vj = c->v + base + (size_t)j * c->d;",
     "(size_t)i * c->d, *vj = c->v + base + (size_t)i * c->d;"),
    ("bwd_rowdot_unweighted", "s += exp(x[j] - M) / Z * bwd_g(c, bh, i, j);", "s += bwd_g(c, bh, i, j);"),
    ("bwd_dq_uses_q", "const float *kj = c->k + base + (size_t)j * c->d;\n        for (int t = 0; t < c->d; ++t) dq",
     "const float *kj = c->q + base + (size_t)j * c->d;\n        for (int t = 0; t < c->d; ++t) dq"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    work = os.path.join(os.path.dirname(SRC), "_build", "mutants")  # git-ignored build folder
    os.makedirs(work, exist_ok=True)
    mut_c = os.path.join(work, f"{name}.c")
    with open(mut_c, "w") as f:
        f.write(src.replace(old, new))
    mut_so = os.path.join(work, f"{name}.so")
    oracle.compile_to(mut_c, mut_so)
    env = dict(os.environ, ALIBI_ORACLE_LIB=str(mut_so))
    pins = "test_oracle_bwd_pins.py" if name.startswith("bwd_") else "test_oracle_pins.py"
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, pins)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
