"""Plant plausible mistakes in copies of the oracle and check a pin fails.

Each mutation rewrites one expression of pa_oracle.c (a dropped term, a wrong
sign, a wrong index, a swapped operand), compiles the copy into a temporary
directory on the CPU, and runs the pin battery against it.  A mutation that no
pin notices would mean the pins could not tell a broken oracle from a correct
one.
"""
import os

import pytest

import oracle
from pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTATIONS = {
    "drop_scale": ("weights[t] = scale * dot;", "weights[t] = dot;"),
    "softmax_sign": ("exp(weights[t] - max_score)", "exp(max_score - weights[t])"),
    "no_normalisation": ("double w = weights[t] / total;", "double w = weights[t];"),
    "offset_shift": ("int offset = t % block_size;", "int offset = (t + 1) % block_size;"),
    "logical_block": ("max_blocks_per_seq + t / block_size];",
                      "max_blocks_per_seq + (t / block_size) / 2];"),
    "k_from_v": ("K[(size_t)t * head_dim + d] = element_to_double(k_cache[at], dtype);",
                 "K[(size_t)t * head_dim + d] = element_to_double(v_cache[at], dtype);"),
    "q_wrong_head": ("qd[d] = element_to_double(q[(size_t)pair * head_dim + d], dtype);",
                     "qd[d] = element_to_double(q[(size_t)s * head_dim + d], dtype);"),
    "bf16_shift": ("uint32_t word = (uint32_t)bits << 16;", "uint32_t word = (uint32_t)bits << 15;"),
    "bf16_read_as_f16": ("return dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_half_to_double(bits);",
                         "return oracle_half_to_double(bits);"),
    "head_offset_transposed": ("size_t at = cache_index(phys, h, offset, d,",
                               "size_t at = cache_index(phys, offset % num_heads, h % block_size, d,"),
    "drop_last_token": ("weights[t] = exp(weights[t] - max_score);\n            total += weights[t];",
                        "weights[t] = (t + 1 < ctx) ? exp(weights[t] - max_score) : 0.0;\n            total += weights[t];"),
    "half_bias": ("exponent - 25);", "exponent - 24);"),
    "half_subnormal": ("ldexp((double)fraction, -24);", "ldexp((double)fraction, -25);"),
    "reshape_offset": ("int offset = slot % block_size;\n        for (int h = 0; h < num_heads; ++h) {",
                       "int offset = (slot + 1) % block_size;\n        for (int h = 0; h < num_heads; ++h) {"),
    "reshape_skips_zero": ("if (slot < 0)\n            continue;", "if (slot <= 0)\n            continue;"),
    "reshape_k_only": ("v_cache[dst] = v[src];", "v_cache[dst] = k[src];"),
    "prefill_not_causal": ("int pos = ctx - q_len + i;               /* this query's position */",
                           "int pos = ctx - 1;"),
    "prefill_position": ("int pos = ctx - q_len + i;               /* this query's position */",
                         "int pos = ctx - q_len + i - (i > 0);"),
    "copy_v_from_k": ("dst_v[to] = src_v[from];", "dst_v[to] = src_k[from];"),
    "copy_wrong_head": ("size_t to = cache_index(dst, h, t, d,", "size_t to = cache_index(dst, 0, t, d,"),
}


# Mutations of lines that appear in more than one function name the function
# whose copy they change.
IN_FUNCTION = {
    "drop_scale": "oracle_decode", "softmax_sign": "oracle_decode",
    "no_normalisation": "oracle_decode", "offset_shift": "oracle_decode",
    "logical_block": "oracle_decode", "k_from_v": "oracle_decode",
    "q_wrong_head": "oracle_decode", "head_offset_transposed": "oracle_decode",
    "prefill_drop_scale": "oracle_prefill", "prefill_softmax_sign": "oracle_prefill",
    "prefill_k_from_v": "oracle_prefill", "prefill_offset_shift": "oracle_prefill",
}
MUTATIONS.update({
    "prefill_drop_scale": ("weights[t] = scale * dot;", "weights[t] = dot;"),
    "prefill_softmax_sign": ("exp(weights[t] - max_score)", "exp(max_score - weights[t])"),
    "prefill_k_from_v": ("K[(size_t)t * head_dim + d] = element_to_double(k_cache[at], dtype);",
                         "K[(size_t)t * head_dim + d] = element_to_double(v_cache[at], dtype);"),
    "prefill_offset_shift": ("int offset = t % block_size;", "int offset = (t + 1) % block_size;"),
})


def function_span(text, name):
    start = text.index("\nint " + name + "(")
    end = text.index("\n}\n", start) + 3
    return start, end


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    text = open(SRC, encoding="utf-8").read()
    lo, hi = function_span(text, IN_FUNCTION[name]) if name in IN_FUNCTION else (0, len(text))
    body = text[lo:hi]
    assert body.count(old) == 1, f"mutation {name} no longer matches the oracle source"
    src = tmp_path / "mutant.c"
    src.write_text(text[:lo] + body.replace(old, new) + text[hi:], encoding="utf-8")
    lib = oracle.load(path=str(tmp_path / "libmutant.so"), src=str(src))
    caught = []
    for pin_name, fn in PINS:
        try:
            fn(lib)
        except (AssertionError, oracle.OracleError, FloatingPointError):
            caught.append(pin_name)
            break
    assert caught, f"no pin notices mutation {name}"
