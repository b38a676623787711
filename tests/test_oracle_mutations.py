"""The oracle's pins must catch plausible mistakes in the oracle.

Each case edits one line of a copy of oracle.c (a swapped beta, a misplaced
eps, a wrong step count, a sum instead of a mean, ...), builds the copy in a
temporary directory, and runs the pin tests against it in a subprocess: the
pins must fail.  The unedited copy must pass.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "beta1_beta2_swapped_in_m": ("float m_old = m[i] * k.beta1;", "float m_old = m[i] * k.beta2;"),
    "one_minus_beta1_dropped": ("float m_new = k.one_minus_beta1 * g;", "float m_new = g;"),
    "v_uses_g_not_g2": ("float v_new = k.one_minus_beta2 * g2;", "float v_new = k.one_minus_beta2 * g;"),
    "eps_before_bias_correction": ("float den = root / k.bc2_sqrt;\n        den = den + k.eps;",
                                   "float den = root + k.eps;\n        den = den / k.bc2_sqrt;"),
    "eps_inside_sqrt": ("float root = sqrtf(vi);", "float root = sqrtf(vi + k.eps * k.eps * 100.0f);"),
    "bc2_dropped": ("float den = root / k.bc2_sqrt;", "float den = root;"),
    "bias_correction_t_minus_1": ("double bc1 = 1.0 - pow(b1, (double)t);", "double bc1 = 1.0 - pow(b1, (double)(t + 1));"),
    "decay_wrong_sign": ("out->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);",
                         "out->decay = (float)(1.0 + (double)hp->lr * (double)hp->weight_decay);"),
    "decay_not_scaled_by_lr": ("out->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);",
                               "out->decay = (float)(1.0 - (double)hp->weight_decay);"),
    "update_sign_flipped": ("th = th - delta;", "th = th + delta;"),
    "replica_sum_not_mean": ("s = s + oracle_bf16_to_f32(g[r][i]);\n        gm[i] = s / fr;",
                             "s = s + oracle_bf16_to_f32(g[r][i]);\n        gm[i] = s;"),
    "replica_index_stuck": ("s = s + oracle_bf16_to_f32(g[r][i]);", "s = s + oracle_bf16_to_f32(g[0][i]);"),
    "f32_replica_index_stuck": ("            s = s + g[r][i];", "            s = s + g[0][i];"),
    "f32_replica_sum_not_mean": ("        gm[i] = s / fr;\n    }\n}\n\n/* ---- a2", "        gm[i] = s;\n    }\n}\n\n/* ---- a2"),
    "clip_norm_without_sqrt": ("double norm = sqrt(sqnorm);", "double norm = sqnorm;"),
    "clip_not_clamped": ("if (c > 1.0)\n        c = 1.0;\n    return (float)c;", "return (float)c;"),
    "clip_coef_not_applied": ("float g = gm[i] * coef;", "float g = gm[i];"),
    "bf16_truncates": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (0)"),
    "bf16_ties_away": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (dropped >= 0x8000u)"),
}


def _build(tmp, text, name):
    c = os.path.join(tmp, name + ".c")
    with open(c, "w") as f:
        f.write(text)
    so = os.path.join(tmp, name + ".so")
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-I", os.path.join(ROOT, "oracle"), "-o", so, c, "-lm"], check=True)
    return so


def _run_pins(so):
    env = dict(os.environ, ORACLE_SO=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_unmutated_copy_passes(tmp_path):
    text = open(SRC).read()
    assert _run_pins(_build(str(tmp_path), text, "same")) == 0


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not found once: {name}"
    so = _build(str(tmp_path), text.replace(old, new), name)
    assert _run_pins(so) != 0, f"pins did not catch: {name}"
