"""Seeded synthetic workloads for paged MLA decode over an FP8 KV cache.

This module only draws inputs: shapes, seeds, random latents, queries and page
tables.  It holds none of the method's arithmetic (no encoding, no attention)
so that both the CPU oracle and the CUDA library can be fed from it.

Shapes follow the web pages: cache rows of 576 = 512 (c_kv) + 64 (k_pe) and a
pool of 495,552 slots ("The KV Cache Cast Bottleneck", section "The
Context"), 78 layers (same section), page size 1 ("The Gather-Then-Cast
Pivot", section "The Knowledge Required"), concurrency 40 and 16 query heads
per KV head ("When a Faster Kernel Doesn't Speed Up Serving", section
"Setup": the qh16 / gqaratio16 kernel).  The pages measure live serving of
proprietary models; these seeded draws with the same shapes stand in for
that traffic.

Recipe (all draws with torch.Generator(seed = 1000 + the workload's number), CPU):
  * latents c_kv / k_pe: normal with the config's std, drawn in fp32 and
    rounded to BF16; k_scale = absmax(latents) / 448 in fp32, except the tiny
    config (std 1, k_scale 1.0);
  * q: BF16 from N(0, 1), shape [B, H, 576];
  * slots: the first N_tok entries of a random permutation of the pool
    (page size 1), or a random permutation of the page ids (page size 64);
  * context lengths: fixed, or integers uniform in [1024, 8192] inclusive;
  * extend steps: the context counts the request's new tokens (they are
    stored before attention); their queries, [n_new, H, 576], are drawn with
    the generator seeded 7919 above the workload's seed;
  * softmax_scale = 1/sqrt(192);
  * unused pool rows: random bytes other than the two NaN codes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

D_CKV, D_KPE = 512, 64
D_ALL = D_CKV + D_KPE
POOL_SLOTS = 495_552
NUM_LAYERS = 78
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)


@dataclass
class Workload:
    name: str
    batch: int
    heads: int
    page_size: int
    num_slots: int            # pool rows (slots)
    seq_lens: np.ndarray      # int32 [B]
    kv_indptr: np.ndarray     # int32 [B+1] (pages)
    kv_indices: np.ndarray    # int32 [n_pages]
    q_bf16: np.ndarray        # uint16 [B, H, 576] (BF16 bits)
    latent_bf16: np.ndarray   # uint16 [n_active_slots, 576]: rows to store
    latent_slots: np.ndarray  # int64 [n_active_slots]: their slots
    k_scale: float
    softmax_scale: float = SOFTMAX_SCALE
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        return int(self.seq_lens.sum())


# name -> (workload number (seed offset), B, H, contexts, page_size, latent std)
CONFIGS = {
    "tiny": dict(number=1, batch=2, heads=4, lens=[17, 33], page_size=1, pool=128, std=1.0),
    "single": dict(number=2, batch=1, heads=16, lens=[4096], page_size=1, pool=POOL_SLOTS,
                   std=0.5),
    "concurrency": dict(number=3, batch=40, heads=16, lens="uniform", page_size=1,
                        pool=POOL_SLOTS, std=0.5),
    "large_head": dict(number=4, batch=128, heads=128, lens=[32768] * 128, page_size=64,
                       pool=None, std=0.5),
}


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns to float32 (no rounding involved)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def random_fill_bytes(gen: np.random.Generator, shape) -> np.ndarray:
    """Random E4M3 bytes for unused pool rows, avoiding the NaN codes."""
    b = gen.integers(0, 256, size=shape, dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x3C
    return b


def make_workload(name: str, *, batch: int | None = None, heads: int | None = None,
                  lens=None, page_size: int | None = None, num_slots: int | None = None,
                  seed: int | None = None, std: float | None = None,
                  k_scale: float | None = None, latent_requests=None) -> Workload:
    """Build one seeded workload.  Keyword overrides give smaller variants of
    a named config (same recipe, other sizes).  latent_requests, if given,
    limits the drawn latents to those requests' slots (the other active
    slots are left to the caller, e.g. random bytes): the H=128 long-context
    pool holds 2.4 G latents, and a parity check needs only a sample."""
    cfg = dict(CONFIGS[name])
    B = batch if batch is not None else cfg["batch"]
    H = heads if heads is not None else cfg["heads"]
    ps = page_size if page_size is not None else cfg["page_size"]
    sd = std if std is not None else cfg["std"]
    seed = seed if seed is not None else 1000 + cfg["number"]
    g = torch.Generator().manual_seed(seed)

    if lens is None:
        lens = cfg["lens"]
    if isinstance(lens, str) and lens == "uniform":
        seq = torch.randint(1024, 8193, (B,), generator=g).numpy().astype(np.int32)
    else:
        seq = np.asarray(list(lens)[:B] if len(list(lens)) >= B else
                         (list(lens) * B)[:B], np.int32)
    pages_per = (seq.astype(np.int64) + ps - 1) // ps
    n_pages = int(pages_per.sum())
    if num_slots is None:
        num_slots = cfg["pool"] if cfg["pool"] is not None else n_pages * ps
    pool_pages = num_slots // ps
    if n_pages > pool_pages:
        raise ValueError(f"{name}: {n_pages} pages do not fit a pool of {pool_pages} pages")
    perm = torch.randperm(pool_pages, generator=g).numpy().astype(np.int32)
    kv_indices = perm[:n_pages].copy()
    kv_indptr = np.zeros(B + 1, np.int32)
    kv_indptr[1:] = np.cumsum(pages_per)

    # slots actually holding tokens (every row of every listed page that a
    # token of the request covers)
    slot_list = []
    chosen = range(B) if latent_requests is None else sorted(set(latent_requests))
    for b in chosen:
        pg = kv_indices[kv_indptr[b]:kv_indptr[b + 1]].astype(np.int64)
        t = np.arange(seq[b], dtype=np.int64)
        slot_list.append(pg[t // ps] * ps + t % ps)
    slots = np.concatenate(slot_list) if slot_list else np.zeros(0, np.int64)

    lat = torch.randn((slots.shape[0], D_ALL), generator=g, dtype=torch.float32) * sd
    lat_bf16 = lat.to(torch.bfloat16)
    if k_scale is None:
        if (cfg["number"] == 1 and std is None) or slots.shape[0] == 0:   # no latents drawn
            k_scale = 1.0
        else:
            k_scale = float(lat_bf16.float().abs().max().item()) / 448.0
            k_scale = float(np.float32(k_scale))
    q = torch.randn((B, H, D_ALL), generator=g, dtype=torch.float32)
    return Workload(name=name, batch=B, heads=H, page_size=ps, num_slots=int(num_slots),
                    seq_lens=seq, kv_indptr=kv_indptr, kv_indices=kv_indices,
                    q_bf16=_bf16_bits(q), latent_bf16=_bf16_bits(lat_bf16), latent_slots=slots,
                    k_scale=float(k_scale), seed=seed)


# name -> (workload number (seed offset), B, H, contexts, new tokens per request): extend
# steps.  The pages time the extend path's cast of the whole history (once
# per layer and extend step) but give no chunk size; the readings here are a
# prefill chunk of 256 new tokens over the decode workload's history law, and
# 4 speculative tokens per request at the decode concurrency.
EXTEND_CONFIGS = {
    "extend_chunk": dict(base="concurrency", number=6, batch=8, q_len=256),
    "spec_decode": dict(base="concurrency", number=7, batch=40, q_len=4),
}


def make_extend_workload(name: str, q_lens=None, **overrides) -> Workload:
    """A seeded extend step: make_workload's page table and latents with
    contexts that end in each request's new tokens, plus their queries.
    name is an EXTEND_CONFIGS entry (its base config, batch and new-token
    count) or a make_workload config (q_lens then required).  q_lens: one
    count per request (or one for all), each <= its context.  Returns the
    Workload with q_bf16 [n_new, H, 576] and extra["qo_indptr"] (int32 [B+1])."""
    if name in EXTEND_CONFIGS:
        ec = EXTEND_CONFIGS[name]
        overrides.setdefault("batch", ec["batch"])
        overrides.setdefault("seed", 1000 + ec["number"])
        if q_lens is None:
            q_lens = ec["q_len"]
        name = ec["base"]
    w = make_workload(name, **overrides)
    B = w.batch
    ql = np.broadcast_to(np.asarray(q_lens, np.int64), (B,)).astype(np.int32)
    if np.any(ql < 0) or np.any(ql > w.seq_lens):
        raise ValueError("each request's new tokens must fit in its context")
    qo = np.zeros(B + 1, np.int32)
    qo[1:] = np.cumsum(ql)
    g = torch.Generator().manual_seed(w.seed + 7919)
    q = torch.randn((int(qo[-1]), w.heads, D_ALL), generator=g, dtype=torch.float32)
    w.q_bf16 = _bf16_bits(q)
    w.extra["qo_indptr"] = qo
    return w


def decode_step_workload(batch: int, layers: int = NUM_LAYERS, seed: int = 1005,
                         with_latents: bool = False):
    """The full decode step: per layer the same page table, a new token per
    request appended into a random free slot (so each context grows by one),
    and per-layer latents / queries.  Returns the base workload (contexts
    before the append), the new slots [B] and the number of layers."""
    lens = [4096] if batch == 1 else "uniform"
    w = make_workload("single" if batch == 1 else "concurrency", batch=batch, lens=lens,
                      seed=seed, latent_requests=None if with_latents else [])
    g = np.random.default_rng(seed)
    used = np.zeros(w.num_slots, bool)
    used[w.kv_indices] = True                      # page size 1: pages are slots
    free = np.flatnonzero(~used)
    new_slots = g.choice(free, size=batch, replace=False).astype(np.int64)
    return w, new_slots, layers


def append_tokens(w: Workload, new_slots: np.ndarray):
    """Page table (page size 1) after appending one token per request at
    new_slots: returns (kv_indptr, kv_indices, seq_lens)."""
    assert w.page_size == 1
    B = w.batch
    seq = w.seq_lens + 1
    indptr = np.zeros(B + 1, np.int32)
    indptr[1:] = np.cumsum(seq)
    idx = np.empty(int(indptr[-1]), np.int32)
    for b in range(B):
        old = w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        idx[indptr[b]:indptr[b + 1] - 1] = old
        idx[indptr[b + 1] - 1] = new_slots[b]
    return indptr, idx, seq.astype(np.int32)
