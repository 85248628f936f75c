"""The oracle's pins are sensitive: each plausible mistake planted in a copy
of the oracle source (a dropped term, a wrong sign, index, operand order or
tie rule) must make at least one pin fail.  Runs on the CPU only; the
mutants are compiled into a temporary directory and never replace the real
oracle."""
import pytest

import oracle
from tests import test_oracle_formats as F
from tests import test_oracle_attention as A
from tests import test_oracle_gather as G
from tests import test_oracle_indexer_store as I
from tests import test_oracle_load as L
from tests import test_oracle_store as S

ALL_CHECKS = (F.CHECKS + S.CHECKS + G.CHECKS + L.CHECKS + I.CHECKS
              + A.CHECKS)

# (id, original text, planted mistake[, occurrence]) -- the mistake is
# planted at the given occurrence of the original (default: the only one)
MUTANTS = [
    ("scale_divides_by_g", "float sfv = (amax / 6.0f) * g;",
     "float sfv = (amax / 6.0f) / g;"),
    ("scale_drops_six", "float sfv = (amax / 6.0f) * g;",
     "float sfv = (amax / 4.0f) * g;"),
    ("ties_away_from_even", "return (c % 2 == 0) ? c : c + 1;",
     "return c + 1;"),
    ("ties_toward_zero", "return (c % 2 == 0) ? c : c + 1;", "return c;"),
    ("nibbles_swapped",
     "data8[k] = (uint8_t)(q[2 * k] | (q[2 * k + 1] << 4));",
     "data8[k] = (uint8_t)(q[2 * k + 1] | (q[2 * k] << 4));"),
    ("signed_amax", "float a = fabsf(xs[i]);", "float a = xs[i];"),
    ("ratio_without_g", "float r = g / (float)kvqo_e4m3_decode(sf);",
     "float r = 1.0f / (float)kvqo_e4m3_decode(sf);"),
    ("e4m3_subnormal_exponent", "ldexp((double)m / 8.0, 1 - 7)",
     "ldexp((double)m / 8.0, -7)"),
    ("e4m3_bias", "ldexp(1.0 + (double)m / 8.0, e - 7)",
     "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("e2m1_drops_sign",
     "return (uint8_t)((signbit(v) ? 0x8 : 0x0) | mag);",
     "return (uint8_t)(mag);"),
    ("saturates_one_code_low", "if (a >= vals[n - 1]) return n - 1;",
     "if (a >= vals[n - 1]) return n - 2;"),
    ("sf_zero_branch_missing", "if (sf == 0) {", "if (sf == 0xFF) {"),
    ("swizzle_row", "int row = (t / 4) * 4 + s / q;",
     "int row = (t / 4) * 4 + s % 4;"),
    ("swizzle_col", "int col = (s % q) * 4 + t % 4;",
     "int col = (s % q) * 4 + (t + 1) % 4;"),
    ("swizzles_k_not_v",
     "const int swizzle = (side == 1) || (flags & KVQO_F_SWIZZLE_K_SCALE);",
     "const int swizzle = (side == 0) || (flags & KVQO_F_SWIZZLE_K_SCALE);",
     0),
    ("load_swizzles_k_not_v",
     "const int swizzle = (side == 1) || (flags & KVQO_F_SWIZZLE_K_SCALE);",
     "const int swizzle = (side == 0) || (flags & KVQO_F_SWIZZLE_K_SCALE);",
     1),
    ("nhd_as_hnd", "dhs = data_dim;     dts = H * data_dim;",
     "dhs = B * data_dim; dts = data_dim;", 0),
    ("load_nhd_as_hnd", "dhs = data_dim;     dts = H * data_dim;",
     "dhs = B * data_dim; dts = data_dim;", 1),
    ("scale_region_offset",
     "uint8_t* scale_page = data_page + data_per_side;",
     "uint8_t* scale_page = data_page + data_per_side / 2;"),
    ("v_uses_k_scale",
     "const float g_side[2] = {1.0f / k_scale, 1.0f / v_scale};",
     "const float g_side[2] = {1.0f / k_scale, 1.0f / k_scale};"),
    ("skip_rule_includes_zero", "if (slot < 0) continue;",
     "if (slot <= 0) continue;", 0),
    ("ik_skip_rule_includes_zero", "if (slot < 0) continue;",
     "if (slot <= 0) continue;", 1),
    ("gather_offset", "const int64_t off = p % B;\n      if (blk < 0",
     "const int64_t off = (p + 1) % B;\n      if (blk < 0", 0),
    ("gather_scale_byte_order", "k_scale[row * 4 + k] = block[B * D + off * 4 + k];",
     "k_scale[row * 4 + k] = block[B * D + off * 4 + (3 - k)];"),
    ("f16_exponent_bias", "ldexp(1.0 + (double)m / 1024.0, e - 15)",
     "ldexp(1.0 + (double)m / 1024.0, e - 14)"),
    ("f16_subnormal_scale", "v = ldexp((double)m, -24);",
     "v = ldexp((double)m, -23);"),
    ("load_unswizzle_transposed",
     "sptr = scale_page + h * shs + (pos / S) * sts + pos % S;",
     "sptr = scale_page + h * shs + (pos % S) * sts + pos / S;", 0),
    ("load_k_uses_v_scale",
     "const float side_scale[2] = {k_scale, v_scale};",
     "const float side_scale[2] = {v_scale, v_scale};"),
    ("load_nibble_order",
     "(k % 2 == 0) ? (byte & 0xF) : (byte >> 4)",
     "(k % 2 == 0) ? (byte >> 4) : (byte & 0xF)", 0),
    ("attn_nibble_order",
     "(k % 2 == 0) ? (byte & 0xF) : (byte >> 4)",
     "(k % 2 == 0) ? (byte >> 4) : (byte & 0xF)", 1),
    ("bf16_cast_truncates",
     "return (uint16_t)((u + 0x7FFFu + lsb) >> 16);",
     "return (uint16_t)(u >> 16);"),
    ("load_divides_by_scale",
     "const float c = (float)kvqo_e4m3_decode(*sptr) * side_scale[side];",
     "const float c = (float)kvqo_e4m3_decode(*sptr) / side_scale[side];"),
    ("load_block_offset", "const int64_t off = p % B;\n      if (blk < 0",
     "const int64_t off = (p + 1) % B;\n      if (blk < 0", 1),
    ("ik_wrong_format_max", "const float scale = amax / 448.0f;",
     "const float scale = amax / 240.0f;"),
    ("ik_multiplies_by_scale", "kvqo_e4m3_encode(x / scale)",
     "kvqo_e4m3_encode(x * scale)"),
    ("ik_signed_amax", "if (fabsf(x) > amax) amax = fabsf(x);",
     "if (x > amax) amax = x;"),
    ("ik_scale_slot",
     "memcpy(cache + blk * block_stride + B * D + off * 4, &scale, 4);",
     "memcpy(cache + blk * block_stride + B * D + (off ^ 1) * 4, &scale, 4);"),
    ("ik_row_slot", "uint8_t* dst = cache + blk * block_stride + off * D;",
     "uint8_t* dst = cache + blk * block_stride + (off ^ 1) * D;"),
    ("gather_row_bytes", "k_fp8[row * D + d] = block[off * D + d];",
     "k_fp8[row * D + d] = block[off * D + (d ^ 1)];"),
    ("attn_kv_head_modulo", "const int64_t kh = h / G;",
     "const int64_t kh = h % Hkv;"),
    ("attn_sum_drops_last_token",
     "for (int64_t t = 0; t < L; ++t) l += exp(s[t] - m);",
     "for (int64_t t = 0; t < L - 1; ++t) l += exp(s[t] - m);"),
    ("attn_values_drop_last_token",
     "for (int64_t t = 0; t < L; ++t) {\n        const int64_t blk = "
     "block_table[b * bt_stride + t / B];\n        nvfp4_row_exact(value",
     "for (int64_t t = 0; t < L - 1; ++t) {\n        const int64_t blk = "
     "block_table[b * bt_stride + t / B];\n        nvfp4_row_exact(value"),
    ("attn_no_max_shift",
     "double m = s[0];\n      for (int64_t t = 1; t < L; ++t) "
     "if (s[t] > m) m = s[t];",
     "double m = 0.0;"),
    ("attn_drops_k_scale", "layout, k_swizzle, (double)k_scale, krow);",
     "layout, k_swizzle, 1.0, krow);"),
    ("attn_k_scales_always_swizzled",
     "layout, k_swizzle, (double)k_scale, krow);",
     "layout, 1, (double)k_scale, krow);"),
    ("attn_v_scales_linear", "layout, 1, (double)v_scale, vrow);",
     "layout, 0, (double)v_scale, vrow);"),
    ("attn_scale_squared", "s[t] = (double)scale * dot;",
     "s[t] = (double)scale * (double)scale * dot;"),
    ("attn_mag_signed", "mg[d] += p * fabs(vrow[d]);",
     "mg[d] += p * vrow[d];"),
    ("attn_token_offset",
     "nvfp4_row_exact(key_cache, page_stride, blk, t % B,",
     "nvfp4_row_exact(key_cache, page_stride, blk, (t + 1) % B,"),
    ("attn_query_head", "const uint16_t* q = query + b * q_stride0 + h * D;",
     "const uint16_t* q = query + b * q_stride0 + kh * D;"),
    ("attn_nhd_as_hnd", "dhs = data_dim;     dts = H * data_dim;",
     "dhs = B * data_dim; dts = data_dim;", 2),
    ("attn_unswizzle_transposed",
     "sptr = scale_page + h * shs + (pos / S) * sts + pos % S;",
     "sptr = scale_page + h * shs + (pos % S) * sts + pos / S;", 1),
]


def _plant(src, orig, mutant, occurrence):
    parts = src.split(orig)
    if occurrence is None:
        assert len(parts) == 2, "ambiguous original"
        occurrence = 0
    assert len(parts) > occurrence + 1, "occurrence not found"
    head = orig.join(parts[: occurrence + 1])
    tail = orig.join(parts[occurrence + 1:])
    return head + mutant + tail


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, mutant):
    mid, orig, planted = mutant[:3]
    occurrence = mutant[3] if len(mutant) > 3 else None
    src = open(oracle.SOURCE).read()
    path = tmp_path / f"kvq_oracle_{mid}.c"
    path.write_text(_plant(src, orig, planted, occurrence))
    so = oracle.compile_oracle(str(path), str(tmp_path / f"lib_{mid}.so"))
    o = oracle.Oracle(so)
    caught = None
    for check in ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError):
            caught = check.__name__
            break
    assert caught is not None, f"no pin caught mutant {mid}"
