"""Plant plausible mistakes in copies of the oracle and check a pin catches each.

Every mutant is a one-line edit of ``oracle/dsa_oracle.c`` compiled into a
temporary library; the pins of ``pins.py`` run against it and at least one
must fail.  The edits are memory-safe (no mutant reads outside its buffers).
"""
import os
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")

MUTANTS = {
    "decode_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 6);"),
    "decode_subnormal": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -8);"),
    "tie_to_odd": ("else c = (lo & 1) == 0 ? lo : hi;", "else c = (lo & 1) == 0 ? hi : lo;"),
    "saturate_wrong": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);\n  int lo",
                       "if (a >= 448.0) return (uint8_t)(sign | 0x7D);\n  int lo"),
    "sign_of_zero_lost": ("uint8_t sign = signbit(x) ? 0x80 : 0x00;\n  if (isnan(x)) return (uint8_t)(sign | 0x7F);\n  double a = fabs((double)x);\n  if (a >= 448.0) return (uint8_t)(sign | 0x7E);\n  int lo",
                          "uint8_t sign = (x < 0) ? 0x80 : 0x00;\n  if (isnan(x)) return (uint8_t)(sign | 0x7F);\n  double a = fabs((double)x);\n  if (a >= 448.0) return (uint8_t)(sign | 0x7E);\n  int lo"),
    "scale_divisor": ("  float s = amax / 448.0f;\n  for (int i = 0; i < ORACLE_GROUP; ++i) {",
                      "  float s = amax / 447.0f;\n  for (int i = 0; i < ORACLE_GROUP; ++i) {"),
    "writer_group_stride": ("oracle_bf16_to_float(x[g * ORACLE_GROUP + j]);", "oracle_bf16_to_float(x[g * 64 + j]);"),
    "scale_word_order": ("put_le_f32(row + 512 + 4 * g, sc);", "put_le_f32(row + 524 - 4 * g, sc);"),
    "scale_endianness": ("p[0] = (uint8_t)(u & 0xFF);", "p[3] = (uint8_t)(u & 0xFF);"),
    "read_group_mapping": ("le_f32(r + 512 + 4 * (d / ORACLE_GROUP))", "le_f32(r + 512 + 4 * (d % 4))"),
    "sm_scale_dropped": ("s[j] = J->sm_scale * dot;", "s[j] = dot;"),
    "lse_log2": ("double lse = m + log(l);", "double lse = m + log2(l);"),
    "page_offset": ("int64_t row = (int64_t)phys * J->page_size + off;", "int64_t row = (int64_t)phys + off;"),
    "token_seq_ignored": ("int seq = J->token_seq ? J->token_seq[t] : 0;", "int seq = 0;"),
    "all_masked_lse": ("      J->LSE[(int64_t)li * J->H + h] = -INFINITY;", "      J->LSE[(int64_t)li * J->H + h] = 0.0;"),
    "softmax_sign": ("l += exp(s[j] - m);", "l += exp(m - s[j]);"),
    "values_not_rows": ("o[d] += p * k[d];", "o[d] += p * q[d];"),
    "q8_scale_dropped": ("q[d] = oracle_e4m3_decode(q8[d]) * sc;", "q[d] = oracle_e4m3_decode(q8[d]);"),
    "q8_divisor": ("    float s = amax / 448.0f;\n    for (int j = 0; j < d; ++j)\n      q8",
                   "    float s = amax / 512.0f;\n    for (int j = 0; j < d; ++j)\n      q8"),
    "index_range_unchecked": ("if (page >= J->max_pages) { *err |= ORACLE_ERR_INDEX_RANGE; return -1; }",
                              "if (page >= J->max_pages) { return -1; }"),
    "reader_bf16_truncates": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;"),
    "reader_scale_group": ("const int g = d / ORACLE_GROUP;", "const int g = d % 4;"),
    "rope_ignored_in_keys": ("k[ORACLE_D + j] = (double)oracle_bf16_to_float((uint16_t)(r[528 + 2 * j] | (r[528 + 2 * j + 1] << 8)));",
                             "k[ORACLE_D + j] = 0.0;"),
    "rope_read_byte_order": ("(uint16_t)(r[528 + 2 * j] | (r[528 + 2 * j + 1] << 8))",
                             "(uint16_t)(r[528 + 2 * j + 1] | (r[528 + 2 * j] << 8))"),
    "rope_write_byte_order": ("row[528 + 2 * j] = (uint8_t)(b & 0xFF);", "row[528 + 2 * j] = (uint8_t)(b >> 8);"),
    "reader_index_not_remapped": ("idx_out[e] = (int32_t)e;\n        dequant_row_bf16",
                                  "idx_out[e] = topk[e];\n        dequant_row_bf16"),
    "reader_branch_boundary": ("const int full_pool = !(n_sel < pool_rows);", "const int full_pool = !(n_sel <= pool_rows);"),
    "reader_full_pool_keeps_entry": ("idx_out[e] = (int32_t)row;", "idx_out[e] = (int32_t)e;"),
    "reader_full_pool_short": ("for (int64_t r = 0; r < pool_rows; ++r) dequant_row_bf16",
                               "for (int64_t r = 0; r + 1 < pool_rows; ++r) dequant_row_bf16"),
    "reader_rows_bound_max": ("return n_selected < pool_rows ? n_selected : pool_rows;",
                              "return n_selected < pool_rows ? pool_rows : n_selected;"),
    "reader_rope_dropped": ("out[ORACLE_D + j] = (uint16_t)(((unsigned)r[528 + 2 * j + 1] << 8) | r[528 + 2 * j]);",
                            "out[ORACLE_D + j] = 0;"),
    "nan_sign_dropped": ("pthread_once(&g_table_once, build_table);\n  uint8_t sign = signbit(x) ? 0x80 : 0x00;\n  if (isnan(x)) return (uint8_t)(sign | 0x7F);",
                         "pthread_once(&g_table_once, build_table);\n  uint8_t sign = signbit(x) ? 0x80 : 0x00;\n  if (isnan(x)) return (uint8_t)0x7F;"),
    "scaled_nan_sign_from_quotient": ("q[i] = isnan(v[i]) ? oracle_e4m3_encode(v[i]) : oracle_e4m3_encode(v[i] / s);",
                                      "q[i] = oracle_e4m3_encode(isnan(v[i]) ? fabsf(v[i]) : v[i] / s);"),
    "q8_nan_sign_dropped": ("q8[i * d + j] = isnan(v[j]) ? oracle_e4m3_encode(v[j]) : oracle_e4m3_encode(v[j] / s);",
                            "q8[i * d + j] = isnan(v[j]) ? (uint8_t)0x7F : oracle_e4m3_encode(v[j] / s);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path, oracle_mod):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           str(src), "-o", str(so), "-lm", "-lpthread"])
    saved = oracle._lib
    oracle._lib = oracle.load(str(so))
    caught = None
    try:
        for pin in pins.ALL_PINS:
            try:
                pin()
            except AssertionError:
                caught = pin.__name__
                break
    finally:
        oracle._lib = saved
    assert caught is not None, f"no pin detects mutant {name}"
