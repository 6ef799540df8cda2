"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source to a temporary directory, plants one
mistake there (the committed oracle is never touched), compiles the copy and
runs the pin suite against it through ``ORACLE_LIB``: at least one pin must fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "rope_rotation_sign": ("v[m + half] = b * cs + a * sn;", "v[m + half] = b * cs - a * sn;"),
    "rope_frequency": ("pow(theta, -2.0 * (double)m / (double)head_dim)", "pow(theta, -1.0 * (double)m / (double)head_dim)"),
    "attention_scale": ("(float)(1.0 / sqrt((double)head_dim))", "(float)(1.0 / (double)head_dim)"),
    "rmsnorm_eps_outside_root": ("1.0 / sqrt(ss / (double)n + eps)", "1.0 / sqrt(ss / (double)n) + eps"),
    "rmsnorm_sum_not_mean": ("1.0 / sqrt(ss / (double)n + eps)", "1.0 / sqrt(ss + eps)"),
    "gqa_modulo_mapping": ("            int gi = i / grp;\n            orc_attend(q + i * hd, Kr",
                           "            int gi = i % kvh;\n            orc_attend(q + i * hd, Kr"),
    "cache_stores_q_for_k": ("kv_store(m, l, 0, i, p, k + i * hd);", "kv_store(m, l, 0, i, p, q + i * hd);"),
    "cache_reads_one_short": ("kv_load_rows(m, l, 0, i, L, Kr", "kv_load_rows(m, l, 0, i, L - (L > 1), Kr"),
    "penalty_sign_ignored": ("logits[i] = l > 0.0f ? l / penalty : l * penalty;", "logits[i] = l / penalty;"),
    "argmax_last_tie": ("if (logits[i] > logits[best]) best = i;", "if (logits[i] >= logits[best]) best = i;"),
    "migration_drops_last_row": ("for (int p = 0; p < m->pos; ++p)\n                    memcpy(nkv",
                                 "for (int p = 0; p < m->pos - 1; ++p)\n                    memcpy(nkv"),
    "dropped_attention_residual": ("matvec(c, W_(m, l, S_WO), h, qd, att, tmp);\n        for (int i = 0; i < h; ++i) x[i] = x[i] + tmp[i];",
                                   "matvec(c, W_(m, l, S_WO), h, qd, att, tmp);\n        for (int i = 0; i < h; ++i) x[i] = tmp[i];"),
    "silu_sign": ("gd / (1.0 + exp(-gd))", "gd / (1.0 + exp(gd))"),
    "bf16_truncation": ("u += 0x7fffu + lsb;", "u += 0u * lsb;"),
    "mrope_streams_h_w_swapped": ("--left[s];\n        s = (s + 1) % 3;", "--left[s];\n        s = (s + 2) % 3;"),
    "mrope_decode_restarts_at_cache_position": ("m->rope_delta = top + 1 - n;", "m->rope_delta = 0;"),
    "conv_taps_reversed": ("const int ts = t - (K - 1 - k) * dil;", "const int ts = t - k * dil;"),
    "transconv_one_frame_late": ("const int u = t * stride + k;", "const int u = (t + 1) * stride + k;"),
    "q8_scale_over_128": ("const float d = amax / 127.0f;", "const float d = amax / 128.0f;"),
    "q4k_nibbles_swapped": ("if (k & 1) o[16 + k / 2] |= (uint8_t)(q << 4);\n                    else o[16 + k / 2] = (uint8_t)q;",
                            "if (k & 1) o[16 + k / 2] |= (uint8_t)q;\n                    else o[16 + k / 2] = (uint8_t)(q << 4);"),
    "q4k_range_over_16": ("s[j] = (hi + mn[j]) / 15.0f;", "s[j] = (hi + mn[j]) / 16.0f;"),
    "q4k_min_added_in_gemv": ("(float)q - dm * (float)m[k / 32];", "(float)q + dm * (float)m[k / 32];"),
    # the same swap of gate and up in the cached step and in the full recompute, so
    # the two still agree with each other
    "gate_up_swapped": [("matvec(c, W_(m, l, S_WG), F, h, xn, g);\n        matvec(c, W_(m, l, S_WU), F, h, xn, u);",
                         "matvec(c, W_(m, l, S_WG), F, h, xn, u);\n        matvec(c, W_(m, l, S_WU), F, h, xn, g);"),
                        ("matvec(c, lw[S_WG], F, h, xn, g);\n            matvec(c, lw[S_WU], F, h, xn, u);",
                         "matvec(c, lw[S_WG], F, h, xn, u);\n            matvec(c, lw[S_WU], F, h, xn, g);")],
}
PIN_FILES = ("test_oracle_pins.py", "test_oracle_mrope.py", "test_oracle_codec_conv.py", "test_oracle_q8.py",
             "test_oracle_q4k.py")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    edits = MUTANTS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
        src = src.replace(old, new)
    d = tmp_path / "orc"
    d.mkdir()
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.h"), d / "oracle.h")
    (d / "oracle.c").write_text(src)
    lib = d / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           "-o", str(lib), str(d / "oracle.c"), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider"] +
                       [os.path.join(ROOT, "tests", f) for f in PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
