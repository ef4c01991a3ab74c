"""Each oracle pin is shown to fail on the defect it guards.

The verification list of the bloomery pages ("bloomery early V4.1 README")
asks that a gate be seen failing on its defect before it is trusted.  Here a
plausible mistake is planted in a copy of oracle.c (on the CPU, in a temporary
directory; the committed oracle is never changed), the copy is compiled, and
the pins that guard that step must reject it.
"""
from __future__ import annotations

import os
import tempfile

import pytest

import oracle
from test_oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text to find, replacement, pins that must catch it)
MUTANTS = [
    ("fp16_exponent_bias", "expo - 15", "expo - 14", ["half_to_double", "q8_0_handbuilt"]),
    ("q8_0_unsigned", "if (q >= 128) q -= 256;", "", ["q8_0_handbuilt"]),
    ("q4k_nibbles_swapped", "int q = (j % 2 == 0) ? (byte & 15) : (byte >> 4)",
     "int q = (j % 2 == 1) ? (byte & 15) : (byte >> 4)", ["q4_k_handbuilt"]),
    ("q4k_min_dropped", "(double)q - dmin * (double)m;", "(double)q;", ["q4_k_handbuilt"]),
    ("q4k_min_sign", "(double)q - dmin * (double)m;", "(double)q + dmin * (double)m;", ["q4_k_handbuilt"]),
    ("q4k_scale_high_bits", "((S[j - 4] >> 6) << 4)", "((S[j] >> 6) << 4)", ["q4_k_handbuilt"]),
    ("q4k_min_high_bits", "((S[j] >> 6) << 4);", "((S[j - 4] >> 6) << 4);", ["q4_k_handbuilt"]),
    ("q4k_block_stride", "row + b * 144", "row + b * 128", ["q4_k_multiblock_rows"]),
    ("q5k_fifth_bit_index", "int hi = (QH[i] >> j) & 1;", "int hi = (QH[i] >> (j / 2)) & 1;",
     ["q5_k_handbuilt"]),
    ("q5k_fifth_bit_weight", "double qv = (double)(lo + 16 * hi);", "double qv = (double)(lo + 32 * hi);",
     ["q5_k_handbuilt"]),
    ("q5k_min_sign", "qv - dmin * (double)m;", "qv + dmin * (double)m;", ["q5_k_handbuilt"]),
    ("q5k_nibbles_swapped", "int lo = (j % 2 == 0) ? (byte & 15) : (byte >> 4);",
     "int lo = (j % 2 == 1) ? (byte & 15) : (byte >> 4);", ["q5_k_handbuilt"]),
    ("q5k_block_stride", "row + b * 176", "row + b * 160", ["kquant_multiblock_rows"]),
    ("q6k_offset", "int q = lo + 16 * hi - 32;", "int q = lo + 16 * hi - 31;", ["q6_k_handbuilt"]),
    ("q6k_quarter_nibble", "int lo = (r < 2) ? (byte & 15) : (byte >> 4);",
     "int lo = (r % 2 == 0) ? (byte & 15) : (byte >> 4);", ["q6_k_handbuilt"]),
    ("q6k_low_byte", "QL[64 * h + 32 * (r % 2) + l]", "QL[64 * h + 32 * (r / 2) + l]", ["q6_k_handbuilt"]),
    ("q6k_high_pair", "(QH[32 * h + l] >> (2 * r)) & 3", "(QH[32 * h + l] >> (2 * (3 - r))) & 3",
     ["q6_k_handbuilt"]),
    ("q6k_scale_unsigned", "if (sc >= 128) sc -= 256;", "", ["q6_k_handbuilt"]),
    ("q6k_scale_group", "(int)SC[i / 16]", "(int)SC[i / 32]", ["q6_k_handbuilt"]),
    ("q6k_d_first", "read_u16_le(blk + 208)", "read_u16_le(blk)", ["q6_k_handbuilt"]),
    ("q6k_block_stride", "row + b * 210", "row + b * 208", ["kquant_multiblock_rows"]),
    ("q3k_high_bit_sense", "int q = hbit ? lo : lo - 4;", "int q = hbit ? lo - 4 : lo;", ["q3_k_handbuilt"]),
    ("q3k_mask_bit", "(HM[l] >> (4 * h + r)) & 1", "(HM[l] >> (2 * h + r)) & 1", ["q3_k_handbuilt"]),
    ("q3k_scale_high_bits", "(S[8 + j % 4] >> (2 * (j / 4))) & 3", "(S[8 + j / 4] >> (2 * (j % 4))) & 3",
     ["q3_k_handbuilt"]),
    ("q3k_scale_nibbles", "(j < 8) ? (S[j] & 15) : (S[j - 8] >> 4)", "(j < 8) ? (S[j] >> 4) : (S[j - 8] & 15)",
     ["q3_k_handbuilt"]),
    ("q3k_scale_offset", "q3k_scale(S, i / 16) - 32", "q3k_scale(S, i / 16) - 31", ["q3_k_handbuilt"]),
    ("q3k_block_stride", "row + b * 110", "row + b * 108", ["kquant_multiblock_rows"]),
    ("q6k_row_bytes", "return K / 256 * 210;", "return K / 256 * 208;",
     ["kquant_multiblock_rows", "ffn_identity_kquants"]),
    ("e2m1_sign_ignored", "return sign ? -mag : mag;", "return mag;", ["e2m1", "mxfp4_handbuilt"]),
    ("e2m1_no_subnormal", "(expo == 0) ? 0.5 * (double)man :", "(expo == -1) ? 0.5 * (double)man :",
     ["e2m1", "mxfp4_handbuilt"]),
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * (double)man, expo - 1)", "ldexp(1.0 + 0.5 * (double)man, expo - 2)",
     ["e2m1"]),
    ("mxfp4_scale_bias", "ldexp(1.0, e - 127)", "ldexp(1.0, e - 128)", ["mxfp4_handbuilt"]),
    ("mxfp4_nibble_halves_swapped", "oracle_e2m1_to_double(blk[1 + j] & 15);\n            w[b * 32 + j + 16]",
     "oracle_e2m1_to_double(blk[1 + j] >> 4);\n            w[b * 32 + j + 16]", ["mxfp4_handbuilt"]),
    ("mxfp4_nan_scale_finite", "(e == 255) ? NAN :", "(e == 256) ? NAN :", ["mxfp4_handbuilt"]),
    ("mxfp4_block_stride", "row + b * 17;", "row + b * 16;", ["mxfp4_multiblock_rows"]),
    ("ffn_down_decoded_as_gate_type", "oracle_dequant_matrix(qtype_d, down", "oracle_dequant_matrix(qtype_gu, down",
     ["ffn_mixed_types", "layer_mixed_types"]),
    ("ffn_down_rows_of_gate_type", "rb_mid = row_bytes(qtype_d, I)", "rb_mid = row_bytes(qtype_gu, I)",
     ["ffn_mixed_types"]),
    ("layer_down_type_ignored", "oracle_expert_ffn_mixed(L->qtype, L->qtype_down,",
     "oracle_expert_ffn_mixed(L->qtype, L->qtype,", ["layer_mixed_types"]),
    ("router_transposed", "(double)Wr[(int64_t)e * H + h]", "(double)Wr[(int64_t)h * E + e]",
     ["router_integer"]),
    ("topk_smallest", "if (sa != sb) return sa > sb;", "if (sa != sb) return sa < sb;",
     ["softmax_topk_bruteforce", "sigmoid_group_bruteforce"]),
    ("softmax_no_renorm", "if (renormalize) for (int j = 0; j < k; ++j) denom",
     "if (0) for (int j = 0; j < k; ++j) denom", ["softmax_topk_bruteforce"]),
    ("sigmoid_gates_use_bias", "denom += s[top[j]];", "denom += sel[top[j]];",
     ["sigmoid_group_bruteforce"]),
    ("group_score_top1", "int take = per < 2 ? per : 2;", "int take = 1;",
     ["sigmoid_group_bruteforce", "sigmoid_group_special"]),
    ("permute_unstable", "for (int64_t p = 0; p < P; ++p) {\n        int32_t i = cursor[ids[p]]++;",
     "for (int64_t p = P - 1; p >= 0; --p) {\n        int32_t i = cursor[ids[p]]++;", ["permute_bruteforce"]),
    ("counts_reset_each_call", "counts[e] += n;", "counts[e] = n;", ["expert_counts"]),
    ("counts_off_by_one_expert", "if (ids[p] == e) n += 1;", "if (ids[p] == e + 1) n += 1;", ["expert_counts"]),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));", ["ffn_identity"]),
    ("gate_up_swapped_in_h", "h[i] = silu(g) * u;", "h[i] = g * silu(u);", ["ffn_identity"]),
    ("combine_drops_weights", "o[n] += w[(int64_t)t * k + j] * yp[n];", "o[n] += yp[n];",
     ["dense_masked_equals_sparse"]),
    ("shared_expert_dropped", "for (int n = 0; n < H; ++n) o[n] += ys[n];", "",
     ["dense_masked_equals_sparse"]),
    ("rmsnorm_no_mean", "sqrt(ss / H + eps)", "sqrt(ss + eps)", ["rmsnorm"]),
    ("bf16_truncates", "double r = nearbyint(scaled);", "double r = trunc(scaled);", ["round_bf16"]),
]


def _build_mutant(name, find, repl, tmp):
    src = open(SRC).read()
    assert src.count(find) == 1, f"mutation {name}: pattern must occur exactly once"
    mutated = src.replace(find, repl, 1)
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    return oracle.load(oracle.build(force=True, src=path, out=os.path.join(tmp, f"lib{name}.so")))


@pytest.mark.parametrize("name,find,repl,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_mutant(name, find, repl, pins):
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_mutant(name, find, repl, tmp)
        for pin in pins:
            with pytest.raises((AssertionError, ValueError)):
                PINS[pin](lib)


def test_unmutated_oracle_passes_all_pins(olib):
    for pin in PINS.values():
        pin(olib)
