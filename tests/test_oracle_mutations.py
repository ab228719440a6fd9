"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of oracle/attn_oracle.c -- a dropped
scale, a wrong sign, an off-by-one in the causal mask, the other diagonal
alignment, a base-2 LSE, a transposed or mis-strided operand, a decoder slip,
a missing or mis-indexed descale, a NaN for empty rows, an ignored per-sequence
key length, an append one row off -- builds it, and runs the pin suite
(tests/test_oracle_pins.py) against that build.  Every mutant must be rejected
by at least one pin; the unmodified source must pass.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

MUTANTS = {
    "dropped_scale": ("s[j] = softmax_scale * acc;", "s[j] = acc;"),
    "scale_squared": ("s[j] = softmax_scale * acc;", "s[j] = softmax_scale * softmax_scale * acc;"),
    "wrong_sign_in_weights": ("double p = exp(s[j] - m) / l;", "double p = exp(m - s[j]) / l;"),
    "causal_off_by_one": ("(last + 1 < sk ? last + 1 : sk)", "(last < sk ? last : sk)"),
    "top_left_alignment": ("int64_t last = i + sk - sq;", "int64_t last = i;"),
    "lse_base2": ("lse_out[r] = m + log(l);", "lse_out[r] = m + log2(l);"),
    "lse_without_max": ("lse_out[r] = m + log(l);", "lse_out[r] = log(l);"),
    "max_over_first_half": ("for (int64_t j = 1; j < n_vis; ++j) if (s[j] > m) m = s[j];",
                            "for (int64_t j = 1; j < n_vis / 2; ++j) if (s[j] > m) m = s[j];"),
    "v_strided_by_d": ("int64_t v_off = ((k_row0 + j) * heads_k + hk) * (int64_t)dv;",
                       "int64_t v_off = ((k_row0 + j) * heads_k + hk) * (int64_t)d;"),
    "k_head_major": ("int64_t k_off = ((k_row0 + j) * heads_k + hk) * (int64_t)d;",
                     "int64_t k_off = ((int64_t)hk * (k_row0 + sk) + k_row0 + j) * (int64_t)d;"),
    "gqa_head_modulo": ("const int64_t hk = h / group;", "const int64_t hk = h % heads_k;"),
    "gqa_k_uses_query_head": ("int64_t k_off = ((k_row0 + j) * heads_k + hk) * (int64_t)d;",
                              "int64_t k_off = ((k_row0 + j) * heads_k + h % heads_k) * (int64_t)d;"),
    "q_row_ignores_batch": ("q_row = b * (int64_t)seqlen_q + i;", "q_row = i;"),
    "v_uses_k": ("o_row[c] += p * (orc_load(v, v_dtype, v_off + c) * vd);",
                 "o_row[c] += p * (orc_load(k, v_dtype, v_off + c) * vd);"),
    "k_descale_missing": ("(orc_load(k, k_dtype, k_off + c) * kd);", "(orc_load(k, k_dtype, k_off + c));"),
    "v_descale_missing": ("(orc_load(v, v_dtype, v_off + c) * vd);", "(orc_load(v, v_dtype, v_off + c));"),
    "v_decoded_as_k_type": ("orc_load(v, v_dtype, v_off + c)", "orc_load(v, k_dtype, v_off + c)"),
    "descale_per_query_head": ("const int64_t ds = b * descale_stride_b + hk * descale_stride_h;",
                               "const int64_t ds = b * descale_stride_b + (h % heads_k) * descale_stride_h;"),
    "descale_ignores_batch": ("const int64_t ds = b * descale_stride_b + hk * descale_stride_h;",
                              "const int64_t ds = hk * descale_stride_h;"),
    "v_descale_from_k": ("const double vd = v_descale ? v_descale[ds] : 1.0;",
                         "const double vd = k_descale ? k_descale[ds] : 1.0;"),
    "e5m2_bias": ("ldexp(1.0 + (double)m / 4.0, e - 15)", "ldexp(1.0 + (double)m / 4.0, e - 16)"),
    "e5m2_subnormal": ("ldexp((double)m / 4.0, -14)", "ldexp((double)m / 4.0, -15)"),
    "seqused_k_ignored": ("        if (seqused_k) sk = seqused_k[b];\n", ""),
    "append_one_row_late": ("seqlens[b] + i) * row_bytes", "seqlens[b] + i + 1) * row_bytes"),
    "empty_rows_nan": ("            lse_out[r] = -INFINITY;\n            continue;",
                       "            lse_out[r] = NAN;\n            continue;"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "bf16_shift": ("((uint32_t)bits) << 16;", "((uint32_t)bits) << 15;"),
}


def _build(src_text, out_dir, name):
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
                    "-ffp-contract=off", c, "-o", so, "-lm"], check=True, capture_output=True)
    return so


def _run_pins(so):
    env = dict(os.environ, FA_ORACLE_LIB_OVERRIDE=so)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-800:]


@pytest.fixture(scope="module")
def tmp():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmodified_oracle_passes_its_pins(tmp):
    so = _build(open(SRC).read(), tmp, "original")
    rc, out = _run_pins(so)
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    so = _build(src.replace(old, new), tmp, name)
    rc, out = _run_pins(so)
    assert rc != 0, f"mutant {name} passed every pin:\n{out}"
