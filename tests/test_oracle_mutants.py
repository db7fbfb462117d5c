"""Plant one plausible mistake at a time in a copy of the oracle and require a pin to fail.

This shows the pins are sharp enough: a dropped term, a wrong index, a wrong
sign, a transposed operand or a wrong rounding rule in ``oracle.c`` is caught.
The mutants are compiled from a temporary copy; the real oracle is untouched.
"""
import os

import pytest

import oracle
from tests import pins

MUTANTS = {
    "no_softmax_scale": [("s *= scale;", "s *= 1.0;")],
    "default_scale_1_over_D": [("1.0 / sqrt((double)D)", "1.0 / (double)D")],
    "kv_head_modulo": [("kvh = h / g;", "kvh = h % Hkv;")],
    "mask_excludes_new_token": [("int n = seq_lens[b] + j + 1;", "int n = seq_lens[b] + j;")],
    "mask_one_past": [("int n = seq_lens[b] + j + 1;", "int n = seq_lens[b] + j + 2;")],
    "multi_all_tokens_see_all": [("int n = seq_lens[b] + j + 1;", "int n = seq_lens[b] + T;")],
    "multi_tokens_see_first_only": [("int n = seq_lens[b] + j + 1;", "int n = seq_lens[b] + 1;")],
    "multi_append_one_row": [("const int L = seq_lens[b] + j; /* position of token j */",
                              "const int L = seq_lens[b]; /* position of token j */")],
    "multi_knew_ignores_token": [("size_t i = (((size_t)b * T + j) * Hkv + h) * D + d;",
                                  "size_t i = (((size_t)b * T) * Hkv + h) * D + d;")],
    "multi_token_index_swapped": [("j = (int)(bh / Hq % T)", "j = (int)(bh % T)")],
    "window_off_by_one": [("n - c->window : 0;", "n - c->window + 1 : 0;")],
    "window_ignored": [("int t_lo = (c->window > 0 && n > c->window) ? n - c->window : 0;", "int t_lo = 0;")],
    "no_k_bias": [("kf[d] = load_elem(k_new, c->qkv_dtype, i) + kb;",
                   "kf[d] = load_elem(k_new, c->qkv_dtype, i);")],
    "no_q_bias": [("qd[d] = (double)(load_elem(q, c->qkv_dtype, (size_t)bh * D + d) + qb);",
                   "qd[d] = (double)(load_elem(q, c->qkv_dtype, (size_t)bh * D + d));")],
    "v_bias_from_k_slot": [("(size_t)(Hq + Hkv + h) * D + d", "(size_t)(Hq + h) * D + d")],
    "bf16_truncates": [("u += 0x7fffu + lsb;", "u += 0u;")],
    "bf16_ties_away": [("u += 0x7fffu + lsb;", "u += 0x8000u;")],
    "i8_scale_128": [("amax / 127.0f", "amax / 128.0f")],
    "i8_truncates": [("float r = rintf(x[d] / s);", "float r = truncf(x[d] / s);")],
    "i8_zero_row_scale": [("*scale = 1.0f;", "*scale = 0.0f;")],
    "i8_abs_dropped": [("float a = fabsf(x[d]);", "float a = x[d];")],
    "no_max_subtraction": [("exp(s - m)", "exp(s)")],
    "no_normalisation": [("o[d] /= denom;", "o[d] /= 1.0;")],
    "v_reads_k": [("o[d] += w * dequant(c, v_cache, vs, b, kvh, t, d);",
                   "o[d] += w * dequant(c, k_cache, ks, b, kvh, t, d);")],
    "pv_uses_score_not_weight": [("o[d] += w * dequant(c, v_cache, vs, b, kvh, t, d);",
                                  "o[d] += s * dequant(c, v_cache, vs, b, kvh, t, d);")],
    "sign_flip_score": [("s += qd[d] * dequant(c, k_cache, ks, b, kvh, t, d);",
                         "s -= qd[d] * dequant(c, k_cache, ks, b, kvh, t, d);")],
    "transposed_cache_index": [("return (((size_t)b * c->Hkv + h) * c->Lmax + pos) * c->D + d;",
                                "return (((size_t)b * c->Hkv + h) * c->D + d) * c->Lmax + pos;")],
    "append_one_row_early": [("store_elem(k_cache, c->cache_dtype, cache_index(c, b, h, L, d), kf[d]);",
                              "store_elem(k_cache, c->cache_dtype, cache_index(c, b, h, L > 0 ? L - 1 : 0, d), kf[d]);")],
    "overflow_not_flagged": [("if (seq_lens[b] > Lmax - T) { overflow = 1; continue; }",
                              "if (seq_lens[b] > Lmax - T) { overflow = 0; continue; }")],
    "i8_dequant_ignores_scale": [("return s * (double)((const int8_t*)cache)[i];",
                                  "return (double)((const int8_t*)cache)[i];")],
    "i8_v_scale_from_k_plane": [("oracle_quant_i8(vf, D, code, &scales[plane + si]);",
                                 "oracle_quant_i8(vf, D, code, &scales[si]);")],
    "proj_weight_transposed": [("s += W[(size_t)f * K + k] * x[(size_t)t * K + k];",
                                "s += W[(size_t)k * F + f] * x[(size_t)t * K + k];")],
    "proj_reversed_k_of_x": [("s += W[(size_t)f * K + k] * x[(size_t)t * K + k];",
                              "s += W[(size_t)f * K + k] * x[(size_t)t * K + (K - 1 - k)];")],
    "proj_drops_last_k": [("for (int k = 0; k < K; ++k) s += W", "for (int k = 0; k < K - 1; ++k) s += W")],
    "proj_output_transposed": [("y[(size_t)t * F + f] = s;", "y[(size_t)f * n_tok + t] = s;")],
}


@pytest.fixture(scope="module")
def src_text():
    with open(oracle._SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, src_text, name):
    text = src_text
    for old, new in MUTANTS[name]:
        assert old in text, f"mutation anchor missing from oracle.c: {old!r}"
        text = text.replace(old, new)
    src = os.path.join(tmp_path, f"oracle_{name}.c")
    with open(src, "w") as f:
        f.write(text)
    lib = oracle.Oracle(oracle.build(src=src, out_dir=str(tmp_path)))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
        except (ValueError, FloatingPointError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
