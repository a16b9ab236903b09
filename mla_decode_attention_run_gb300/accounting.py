"""Algorithmic byte and flop counts of the decode path (the roofline
numerators).  Only bytes the method must move are counted: split-KV partials
and padding are implementation overhead and never enter these figures.

Reference figures: the full-pool cast moves every FP8 byte in and a BF16 copy
out, 3 bytes per element ("The KV Cache Cast Bottleneck", section "The
Context": [495552, 1, 576] per layer, 78 layers); a gather-then-cast touches
only the active rows ("The Gather-Then-Cast Pivot", section "Assumptions and
Potential Mistakes": 500 tokens x 576 elements).
"""
from __future__ import annotations

import numpy as np

D_CKV, D_KPE = 512, 64
D_QK = D_CKV + D_KPE


def pages_of(seq_lens, page_size: int) -> int:
    lens = np.asarray(seq_lens, np.int64)
    return int(((lens + page_size - 1) // page_size).sum())


def decode_call_bytes(seq_lens, heads: int, page_size: int, kv_elem_bytes: int = 1) -> int:
    """Bytes one decode call must move: every active KV row once (576
    elements), the page-table entries, q, o, lse, kv_indptr and seq_lens."""
    lens = np.asarray(seq_lens, np.int64)
    B = lens.size
    return int(lens.sum() * D_QK * kv_elem_bytes + pages_of(lens, page_size) * 4
               + B * heads * D_QK * 2 + B * heads * D_CKV * 2 + B * heads * 4 + (2 * B + 1) * 4)


def decode_call_kv_bytes(seq_lens) -> int:
    """The FP8 cache bytes alone (the dominant term)."""
    return int(np.asarray(seq_lens, np.int64).sum() * D_QK)


def decode_call_flops(seq_lens, heads: int) -> int:
    """2 flops per multiply-add: 576 for the score and 512 for the output,
    per token and head."""
    return int(np.asarray(seq_lens, np.int64).sum() * heads * 2 * (D_QK + D_CKV))


def extend_visible_tokens(seq_lens, q_lens) -> int:
    """Sum over new tokens of the tokens each sees: new token i of a request
    with context L and q new tokens sees L - q + i + 1 of them."""
    total = 0
    for L, q in zip(np.asarray(seq_lens, np.int64), np.asarray(q_lens, np.int64)):
        total += int(q * (L - q) + q * (q + 1) // 2)
    return total


def extend_call_bytes(seq_lens, q_lens, heads: int, page_size: int) -> int:
    """Bytes one extend call must move: every KV row of every request with new
    tokens once, its page-table entries, q, o and lse of every new token, and
    qo_indptr, kv_indptr and seq_lens."""
    lens = np.asarray(seq_lens, np.int64)
    ql = np.asarray(q_lens, np.int64)
    act = lens[ql > 0]
    n_q = int(ql.sum())
    B = lens.size
    return int(act.sum() * D_QK + pages_of(act, page_size) * 4 + n_q * heads * (D_QK * 2 + D_CKV * 2 + 4)
               + (3 * B + 2) * 4)


def extend_call_flops(seq_lens, q_lens, heads: int) -> int:
    """2 flops per multiply-add over the causally visible tokens of every new
    token and head (576 for the score, 512 for the output)."""
    return int(extend_visible_tokens(seq_lens, q_lens) * heads * 2 * (D_QK + D_CKV))


def kv_proj_bytes(n_tokens: int, d_model: int) -> int:
    """Fused projection + store: the weights [576, d_model] and the hidden
    states [n, d_model] in BF16, the E4M3 rows and the slots out."""
    return int(D_QK * d_model * 2 + n_tokens * d_model * 2 + n_tokens * (D_QK + 8))


def store_bytes(n_tokens: int) -> int:
    """Quantize-on-store: BF16 rows in (2 B/element), E4M3 rows out, slots."""
    return int(n_tokens * (D_QK * 2 + D_QK + 8))


def full_pool_cast_elements(num_slots: int) -> int:
    return int(num_slots * D_QK)


def full_pool_cast_bytes(num_slots: int) -> int:
    """FP8 in + BF16 out over the whole pool."""
    return full_pool_cast_elements(num_slots) * 3


def gather_cast_bytes(n_rows: int, n_pages: int) -> int:
    """Active FP8 rows in, BF16 rows out, page indices."""
    return int(n_rows * D_QK * 3 + n_pages * 4)
