"""Pin strength: a plausible mistake planted anywhere in the oracle must make at
least one pin fail.  Each mutant is a copy of the oracle source with one edit
(a dropped term, a wrong sign, index, group or rounding rule, a transposed
operand), built with gcc on the CPU; every mutant stays within its buffers."""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "wq_oracle.c")

MUTANTS = {
    "wq8_drop_scale": ("double wkn = (double)scales[(size_t)g * N + n] * (double)w[(size_t)k * N + n];",
                       "double wkn = (double)w[(size_t)k * N + n];"),
    "wq8_wrong_group": ("  for (int k = 0; k < K; ++k) {\n    int g = k / group;",
                        "  for (int k = 0; k < K; ++k) {\n    int g = (k / group + 1) % (K / group);"),
    "wq8_transposed_w": ("(double)w[(size_t)k * N + n]", "(double)w[(size_t)n * K + k]"),
    "wq3_zero_sign": ("double wkn = s * (double)wqo_code3(mat, N, k, n) - zero;",
                      "double wkn = s * (double)wqo_code3(mat, N, k, n) + zero;"),
    "wq3_drop_zero": ("double wkn = s * (double)wqo_code3(mat, N, k, n) - zero;",
                      "double wkn = s * (double)wqo_code3(mat, N, k, n);"),
    "wq3_straddle": ("if (off > 29) {", "if (off > 30) {"),
    "wq3_word_row": ("uint32_t lo = (uint32_t)mat[(size_t)(3 * block + word) * N + n];",
                     "uint32_t lo = (uint32_t)mat[(size_t)(3 * block) * N + n];"),
    "wq4_zero_sign": ("(double)(wqo_code4(qweight, N, k, n) - z)", "(double)(wqo_code4(qweight, N, k, n) + z)"),
    "wq4_ignore_gidx": ("int g = g_idx ? g_idx[k] : k / group;", "int g = k / group;"),
    "wq4_nibble_order": ("return (int)((word >> (4 * (k % 8))) & 15u);",
                         "return (int)((word >> (4 * (7 - k % 8))) & 15u);"),
    "wq4_zero_nibble": ("return (int)((word >> (4 * (n % 8))) & 15u);",
                        "return (int)((word >> (4 * (7 - n % 8))) & 15u);"),
    "wq4_scale_index": ("double s = dec(scales[(size_t)g * N + n]);",
                        "double s = dec(scales[(size_t)((g + 1) % (K / group)) * N + n]);"),
    "dq8_drop_scale": ("(double)srow[n] * (double)qrow[n]", "(double)qrow[n]"),
    "dq8_wrong_group": ("scales + (size_t)(k / group) * N;", "scales + (size_t)((k / group + 1) % (K / group)) * N;"),
    "dq3_zero_sign": ("s * (double)wqo_code3(mat, N, k, n) - wqo_f16_to_double(zeros[n]);",
                      "s * (double)wqo_code3(mat, N, k, n) + wqo_f16_to_double(zeros[n]);"),
    "dq4_zero_sign": ("(double)(q - zp)", "(double)(q + zp)"),
    "dq4_ignore_gidx": ("int grp = g_idx ? g_idx[k] : k / group;", "int grp = k / group;"),
    "smooth_multiply": ("xs[k] = (float)wqo_bf16_to_double(X[(size_t)m * K + k]) / smooth[k];",
                        "xs[k] = (float)wqo_bf16_to_double(X[(size_t)m * K + k]) * smooth[k];"),
    "smooth_ignored": ("xs[k] = (float)wqo_bf16_to_double(X[(size_t)m * K + k]) / smooth[k];",
                       "xs[k] = (float)wqo_bf16_to_double(X[(size_t)m * K + k]);"),
    "outlier_ge": ("if (fabs(wqo_bf16_to_double(X[(size_t)m * K + k])) > (double)threshold) is_outlier[k] = 1;",
                   "if (fabs(wqo_bf16_to_double(X[(size_t)m * K + k])) >= (double)threshold) is_outlier[k] = 1;"),
    "outlier_sign": ("        y[(size_t)r * N + n] += t;\n", "        y[(size_t)r * N + n] -= t;\n"),
    "outlier_drop_sw": ("double t = xv * ((double)Sw[n] * (double)W[(size_t)k * N + n]);",
                        "double t = xv * (double)W[(size_t)k * N + n];"),
    "w8a8_round_away": ("float rq = nearbyintf(r);", "float rq = roundf(r);"),
    "w8a8_scale_128": ("float sx = amax / 127.0f;", "float sx = amax / 128.0f;"),
    "w8a8_drop_term": ("        a[n] += p;\n", "        if (k > 0) a[n] += p;\n"),
    "w8a8_rescale_drop_sw": ("y[(size_t)r * N + n] = (double)Sx[m] * (double)a[n] * (double)Sw[n];",
                             "y[(size_t)r * N + n] = (double)Sx[m] * (double)a[n];"),
    "f16_exponent": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "bf16_precision": ("double r = round_to_format(a, 8, -126);", "double r = round_to_format(a, 9, -126);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = tmp_path / "mutant.so"
    hdr_dir = os.path.dirname(SRC)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", f"-I{hdr_dir}",
                    "-o", str(so), str(src), "-lm"], check=True)
    failed = []
    with oracle.using_library(str(so)):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
