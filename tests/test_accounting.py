"""Byte accounting of the bench against the figures the pages print."""
import os

import pytest

from mla_decode_attention_run_gb300 import accounting as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_byte_accounting.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v, *_ = line.split()
            vals[k] = float(v)
    return vals


def test_full_pool_cast_matches_page_figures():
    g = _golden()
    assert g["kv_lora_rank"] + g["qk_rope_head_dim"] == g["row_elements"] == A.D_QK
    el = A.full_pool_cast_elements(int(g["pool_slots"]))
    assert el == 495552 * 576 == 285_437_952
    # the prose's 285.6 M elements is within its own rounding of the shape
    assert abs(el / 1e6 - g["prose_elements_millions"]) / g["prose_elements_millions"] < 1e-3
    mb = A.full_pool_cast_bytes(int(g["pool_slots"])) / 1e6
    assert abs(mb - g["prose_cast_mb_per_layer"]) / g["prose_cast_mb_per_layer"] < 1e-3
    gb = A.full_pool_cast_bytes(int(g["pool_slots"])) * int(g["layers"]) / 1e9
    assert round(gb, 1) == g["prose_cast_gb_per_step"]


def test_gather_of_500_tokens():
    g = _golden()
    n = int(g["gather_tokens"])
    assert n * A.D_QK == int(g["gather_elements"])
    assert A.gather_cast_bytes(n, n) == int(g["gather_elements"]) * 3 + 4 * n


def test_decode_call_bytes_terms():
    lens = [17, 33]
    b = A.decode_call_bytes(lens, heads=4, page_size=1)
    assert b == 50 * 576 + 50 * 4 + 2 * 4 * 576 * 2 + 2 * 4 * 512 * 2 + 2 * 4 * 4 + 5 * 4
    assert A.decode_call_kv_bytes(lens) == 28_800
    assert A.decode_call_flops([1], heads=16) == 16 * 2176
    assert A.pages_of([1, 64, 65], 64) == 1 + 1 + 2


def test_extend_counts():
    # one new token per request is decode
    assert A.extend_call_flops([17, 33], [1, 1], 4) == A.decode_call_flops([17, 33], 4)
    # a 3-token prefill sees 1 + 2 + 3 tokens; 2 new tokens on a 5-token context see 4 + 5
    assert A.extend_visible_tokens([3, 5], [3, 2]) == 6 + 9
    # a request without new tokens moves nothing
    b = A.extend_call_bytes([10, 7], [0, 2], heads=2, page_size=1)
    assert b == 7 * 576 + 7 * 4 + 2 * 2 * (576 * 2 + 512 * 2 + 4) + (3 * 2 + 2) * 4
