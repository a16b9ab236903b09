"""Helpers shared by the GPU tests: oracle-made pools, device copies, one
call through the C ABI, and the attention tolerance check.

Every expected value comes from the CPU oracle; the CUDA path only receives
the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import mla_decode_attention_run_gb300 as M
import oracle
import workloads as W

ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3


def oracle_pool(w: W.Workload, fill_seed: int = 0) -> np.ndarray:
    """uint8 [num_slots, 576]: random non-NaN bytes, with the workload's
    latents encoded by the oracle into their slots."""
    pool = W.random_fill_bytes(np.random.default_rng(fill_seed), (w.num_slots, 576))
    if w.latent_slots.shape[0]:
        bad = oracle.kv_store_fp8(w.latent_bf16[:, :512], w.latent_bf16[:, 512:],
                                  w.latent_slots, w.k_scale, pool[:, :512], pool[:, 512:])
        assert bad == 0
    return pool


def dev_i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)


def dev_bf16(bits: np.ndarray, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_decode(w: W.Workload, ckv, kpe, *, kv_dtype=M.MLA_KV_FP8_E4M3, q=None, k_scale=None,
               kv_indptr=None, kv_indices=None, seq_lens=None, num_slots=None, plan=None):
    """Plan + run through the C ABI; returns (out bf16, lse fp32, plan)."""
    dev = ckv.device
    indptr = w.kv_indptr if kv_indptr is None else kv_indptr
    indices = w.kv_indices if kv_indices is None else kv_indices
    lens = w.seq_lens if seq_lens is None else seq_lens
    plan = M.mla_decode_plan(indptr, lens, w.batch, w.heads, w.page_size, kv_dtype, plan=plan)
    if q is None:
        q = dev_bf16(w.q_bf16, dev)
    out = torch.full((w.batch, w.heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.batch, w.heads), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    M.mla_decode_run(plan, q, ckv, kpe, ckv.shape[0] if num_slots is None else num_slots,
                     dev_i32(indptr, dev), dev_i32(indices, dev), dev_i32(lens, dev),
                     w.k_scale if k_scale is None else k_scale, w.softmax_scale, out, lse, ws)
    return out, lse, plan


def check_attention(out: torch.Tensor, lse: torch.Tensor, o_ref: np.ndarray,
                    lse_ref: np.ndarray, where: str = ""):
    """|o - ref| <= 1e-2 + 1e-2 |ref| elementwise; |lse - ref| <= 1e-3."""
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy().astype(np.float64)
    assert o.shape == o_ref.shape
    excess = np.abs(o - o_ref) - (ATOL + RTOL * np.abs(o_ref))
    worst = np.unravel_index(np.argmax(excess), excess.shape) if excess.size else None
    assert np.all(np.isfinite(o)), f"{where}: non-finite output"
    assert excess.max(initial=-1) <= 0, (
        f"{where}: output error {np.abs(o - o_ref)[worst]:.3e} at {worst} "
        f"(ref {o_ref[worst]:.4f}, got {o[worst]:.4f})")
    both_inf = np.isneginf(l) & np.isneginf(lse_ref)
    dl = np.abs(np.where(both_inf, 0.0, l) - np.where(both_inf, 0.0, lse_ref))
    assert np.all(dl <= LSE_TOL), f"{where}: lse error {np.nanmax(dl):.3e}"
    return float(np.abs(o - o_ref).max(initial=0)), float(dl.max(initial=0))
