"""Plant known mistakes in copies of the oracle source; the pins must catch each.

The mistakes are the ones the mojo-dllm page's check names ("swapping the
nibble halves or dropping the Q6_K zero point fails these tests", section
"Checks"), the dropped Q4_K min term, and the further slips listed in the
method's reading (scale index, d/dmin swap, quantizer rounding and division,
the 6-bit unpack of sub-blocks 4-7, the f16 exponent bias).  Each mutant is the
oracle source with one or two exact text substitutions, compiled with gcc to a
temporary directory; no mutant code lives in the oracle itself.
"""
import os

import pytest

import oracle
import pins

MUTANTS = {
    "swapped_nibble_halves": [
        ("return qs[32 * p + i] & 0x0F;", "return qs[32 * p + i] >> 4;"),
        ("return qs[32 * p + (i - 32)] >> 4;", "return qs[32 * p + (i - 32)] & 0x0F;"),
    ],
    "dropped_q4k_min_term": [
        ("acc += d * sc * dx * D - dmin * m * s;", "acc += d * sc * dx * D;"),
        ("return d * sc * q4k_nibble(blk + 16, e) - dmin * m;",
         "return d * sc * q4k_nibble(blk + 16, e);"),
    ],
    "dropped_q6k_zero_point": [
        ("D += (q6k_q(blk, 16 * g + i) - 32) * (int32_t)q[16 * g + i];",
         "D += q6k_q(blk, 16 * g + i) * (int32_t)q[16 * g + i];"),
        ("return d * q6k_scale(blk, e / 16) * (q6k_q(blk, e) - 32);",
         "return d * q6k_scale(blk, e / 16) * q6k_q(blk, e);"),
        ("int w = qtype == ORACLE_Q4_K ? q4k_nibble(blk + 16, e) : q6k_q(blk, e) - 32;",
         "int w = qtype == ORACLE_Q4_K ? q4k_nibble(blk + 16, e) : q6k_q(blk, e);"),
    ],
    "high_scales_as_low_6_bits": [
        ("*sc = (scales[j + 4] & 0x0F) | ((scales[j - 4] >> 6) << 4);", "*sc = scales[j] & 63;"),
    ],
    "d_dmin_swapped": [
        ("double d = half_to_double(load_u16(blk));\n                double dmin = half_to_double(load_u16(blk + 2));",
         "double d = half_to_double(load_u16(blk + 2));\n                double dmin = half_to_double(load_u16(blk));"),
    ],
    "subblock_scale_index_off_by_one": [
        ("q4k_scale_min(blk + 4, j, &sc, &m);", "q4k_scale_min(blk + 4, (j + 1) % 8, &sc, &m);"),
    ],
    "q6k_scale_per_32": [
        ("acc += d * q6k_scale(blk, g) * dx * D;", "acc += d * q6k_scale(blk, g / 2) * dx * D;"),
    ],
    "q6k_activation_scale_index": [
        ("double dx = xds[2 * (t * nb32 + b * 8 + g / 2) + 0];",
         "double dx = xds[2 * (t * nb32 + b * 8 + g % 8) + 0];"),
    ],
    "quantize_floor": [("q = (int)nearbyintf(r);", "q = (int)floorf(r);")],
    "quantize_round_half_away": [("q = (int)nearbyintf(r);", "q = (int)roundf(r);")],
    "quantize_times_reciprocal": [("float r = xb[i] / d;", "float r = xb[i] * (1.0f / d);")],
    "quantize_scale_128": [("float d = amax / 127.0f;", "float d = amax / 128.0f;")],
    "sum_without_scale": [("xds[2 * (t * nb + b) + 1] = d * (float)sum;",
                           "xds[2 * (t * nb + b) + 1] = (float)sum;")],
    "f16_exponent_bias": [("v = ldexp((double)(1024 + m), e - 25);",
                           "v = ldexp((double)(1024 + m), e - 24);")],
    "q6k_high_bits_order": [("int hi = (H[l] >> (2 * quad)) & 3;", "int hi = (H[l] >> (6 - 2 * quad)) & 3;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = oracle.source_text()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
        src = src.replace(old, new)
    lib_path = oracle.compile_variant(src, os.path.join(str(tmp_path), f"mut_{name}.so"))
    o = oracle.Oracle(oracle.load(lib_path))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the mutant {name}"
