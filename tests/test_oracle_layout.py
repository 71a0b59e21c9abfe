"""The layout accounting against the numbers printed on the pages (tests/golden/pages_numbers.json).

Bits per KV element of one request of T tokens: (T - 320)(2 + 32/g) + 320*16, over T.
The printed 2.28 (128K), 2.38 (32K), 2.25 (history only) and 4.25 (INT4 with the same
scale/zero) are all reproduced only with groups of 128 and a bf16 scale and zero per group.
"""
import json
import os

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def test_bits_per_element_at_128k():
    e = GOLD["oscar_bits_per_element"]
    v = oracle.bits_per_element(e["context_tokens"], e["group"])
    assert abs(v - e["value"]) < e["rounding"]


def test_bits_per_element_at_32k():
    e = GOLD["oscar_bits_per_element_32k"]
    v = oracle.bits_per_element(e["context_tokens"], e["group"])
    assert abs(v - e["value"]) < e["rounding"]


def test_history_only_bits():
    e = GOLD["history_only_int2_bits"]
    assert abs(oracle.bits_per_element(10 ** 9, e["group"], 0, 0) - e["value"]) < e["rounding"]


def test_int4_same_scale_zero_accounting():
    # 4-bit codes with the same bf16 scale and zero per group of 128: 4 + 32/128.
    e = GOLD["int4_bits"]
    assert abs(e["code_bits"] + 32.0 / e["group"] - e["value"]) < e["rounding"]


def test_other_groups_miss_the_printed_numbers():
    for g in (32, 64):
        assert abs(oracle.bits_per_element(131072, g) - 2.28) > 0.005


def test_bf16_window_share():
    e = GOLD["bf16_window_share_128k"]
    share = 100.0 * (e["sink"] + e["recent"]) / e["context_tokens"]
    assert abs(share - e["value_percent"]) < e["rounding_percent"]


def test_constants_match_pages():
    assert oracle.SINK == GOLD["sink_tokens"]["value"]
    assert oracle.RECENT == GOLD["recent_tokens"]["value"]
    assert oracle.C_K == GOLD["clip_ratio_key"]["value"]
    assert oracle.C_V == GOLD["clip_ratio_value"]["value"]
    assert 16 // 2 == GOLD["history_memory_reduction"]["value"]
    assert 8 // 2 == GOLD["codes_per_byte"]["value"]
    assert 2 ** 2 == GOLD["int2_levels"]["value"]
