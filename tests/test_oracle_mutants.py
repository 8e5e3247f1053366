"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of oracle/path_oracle.c
(a dropped term, a wrong sign, an off-by-one, a misplaced scale), builds it,
and runs the pin suites (tests/test_oracle.py, tests/test_oracle_bwd.py)
against that build.  Every mutant must make at least one pin fail; a
surviving mutant means the pins do not constrain that part of the oracle.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "path_oracle.c")

MUTANTS = {
    "logit_after_transition": (
        "        logit[j] = scale * dot(k + j * d, u, d) + bias;\n"
        "        apply_transition(u, w + j * d, beta[j], d);\n",
        "        apply_transition(u, w + j * d, beta[j], d);\n"
        "        logit[j] = scale * dot(k + j * d, u, d) + bias;\n"),
    "reflection_sign": ("u[m] -= c * w[m];", "u[m] += c * w[m];"),
    "beta_dropped": ("double c = beta * dot(w, u, d);", "double c = dot(w, u, d);"),
    "bias_scaled": ("logit[j] = scale * dot(k + j * d, u, d) + bias;",
                    "logit[j] = scale * (dot(k + j * d, u, d) + bias);"),
    "bias_off_by_one": (
        "        logit[j] = scale * dot(k + j * d, u, d) + bias;\n"
        "        apply_transition(u, w + j * d, beta[j], d);\n"
        "        if (log_f)\n"
        "            bias += log_f[j];\n",
        "        if (log_f)\n"
        "            bias += log_f[j];\n"
        "        logit[j] = scale * dot(k + j * d, u, d) + bias;\n"
        "        apply_transition(u, w + j * d, beta[j], d);\n"),
    "lse_without_max": ("*lse = mx + log(sum);", "*lse = log(sum);"),
    "softmax_unnormalised": ("out[m] /= sum;", "out[m] /= 1.0;"),
    "decode_skips_last_key": ("for (int64_t j = 0; j < t; ++j)\n        apply_transition",
                              "for (int64_t j = 0; j + 1 < t; ++j)\n        apply_transition"),
    "decode_fox_bias_includes_own_gate": (
        "        logit[j] = scale * dot(kc + j * d, q_t, d) + bias;\n"
        "        if (lf)\n"
        "            bias += lf[j];\n",
        "        if (lf)\n"
        "            bias += lf[j];\n"
        "        logit[j] = scale * dot(kc + j * d, q_t, d) + bias;\n"),
    "kcache_sum_not_product": ("Mw[r] = dot(M + r * d, wh + j * d, d);", "Mw[r] = wh[j * d + r];"),
    "kcache_transposed_update": ("M[r * d + c] -= bb[j] * Mw[r] * wh[j * d + c];",
                                 "M[c * d + r] -= bb[j] * Mw[r] * wh[j * d + c];"),
    "boundary_q_one_short": ("for (int64_t s = i; s >= s0; --s)", "for (int64_t s = i; s > s0; --s)"),
    # backward
    "bwd_dlse_dropped": ("dl[j] -= p * (D - dlse_i);", "dl[j] -= p * D;"),
    "bwd_g_skips_transition": ("        apply_transition(g, w + s * d, beta[s], d);\n", ""),
    "bwd_dw_one_sided": ("(gamma * g[m] + alpha * bs[m])", "(2.0 * gamma * g[m])"),
    "bwd_dbeta_sign": ("dbeta[s] -= scale * alpha * gamma;", "dbeta[s] += scale * alpha * gamma;"),
    "bwd_fox_cum_inclusive": ("            dlog_f[s] += cum;\n        cum += dl[s];",
                              "            dlog_f[s] += cum + dl[s];\n        cum += dl[s];"),
    "bwd_dk_unscaled": ("dk[j * d + m] += scale * dl[j] * B[j * d + m];",
                        "dk[j * d + m] += dl[j] * B[j * d + m];"),
    "bwd_b_after_transition": (
        "        if (B)\n"
        "            memcpy(B + j * d, u, (size_t)d * sizeof(double));\n"
        "        logit[j] = scale * dot(k + j * d, u, d) + bias;\n"
        "        apply_transition(u, w + j * d, beta[j], d);\n",
        "        logit[j] = scale * dot(k + j * d, u, d) + bias;\n"
        "        apply_transition(u, w + j * d, beta[j], d);\n"
        "        if (B)\n"
        "            memcpy(B + j * d, u, (size_t)d * sizeof(double));\n"),
    "bwd_dq_before_own_key": (
        "    for (int64_t m = 0; m < d; ++m)\n        dq_i[m] = scale * g[m];",
        "    for (int64_t m = 0; m < d; ++m)\n        dq_i[m] = scale * (g[m] - dl[i] * k[i * d + m]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(before) == 1, "mutation site not found (oracle source changed?)"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(src.replace(before, after), encoding="utf-8")
    lib = oracle.build(str(mut_src), str(tmp_path / "libmutant.so"), force=True)
    env = dict(os.environ, PATH_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py"),
                        os.path.join(ROOT, "tests", "test_oracle_bwd.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])
