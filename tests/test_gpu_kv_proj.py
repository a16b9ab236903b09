"""GPU parity of the fused KV projection + FP8 store (kv_proj_store_fp8)
against the CPU oracle.

The projection accumulates in fp32 on the tensor cores, so its BF16 latent
may differ from the exactly rounded one by the accumulation error: each
latent must lie within 2^-8 |exact| + d * 2^-24 * sum_k |x_k w_k| of the
exact dot product (one BF16 rounding plus the standard fp32 summation
bound).  The quantization is then decided on identical inputs: the pool
bytes must equal the oracle's store of the kernel's own BF16 latent, bit
for bit, and every row not written must be untouched."""
import math

import numpy as np
import pytest
import torch

import mla_decode_attention_run_gb300 as M
import oracle
import workloads as W
from gpu_util import bf16_bits, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    M.mla_get_last_error()


def _inputs(seed, n, d, pool_slots, x_std=1.0):
    g = torch.Generator().manual_seed(seed)
    x = bf16_bits((torch.randn(n, d, generator=g) * x_std).to(torch.bfloat16))
    w = bf16_bits((torch.randn(576, d, generator=g) / math.sqrt(d)).to(torch.bfloat16))
    rng = np.random.default_rng(seed)
    slots = rng.permutation(pool_slots)[:n].astype(np.int64)
    pool = W.random_fill_bytes(rng, (pool_slots, 576))
    return x, w, slots, pool


def _check(x, w, slots, pool0, k_scale, got_pool, got_lat, where):
    d = x.shape[1]
    xf = W.bf16_bits_to_float(x).astype(np.float64)
    wf = W.bf16_bits_to_float(w).astype(np.float64)
    exact = xf @ wf.T
    bound = 2.0 ** -8 * np.abs(exact) + d * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T)
    lat = W.bf16_bits_to_float(got_lat).astype(np.float64)
    err = np.abs(lat - exact) - bound
    assert err.max() <= 0, f"{where}: latent off by {np.abs(lat - exact).flat[np.argmax(err)]:.3e}"
    ref_pool = pool0.copy()
    bad = oracle.kv_store_fp8(got_lat[:, :512], got_lat[:, 512:], slots, k_scale,
                              ref_pool[:, :512], ref_pool[:, 512:])
    assert bad == 0
    diff = np.argwhere(got_pool != ref_pool)
    assert diff.size == 0, f"{where}: {diff.shape[0]} pool bytes differ, first {diff[:3]}"
    # how often fp32 accumulation moved a latent off the exactly rounded value
    ref_lat, _ = oracle.kv_proj_fp8(x, w, slots, k_scale, pool0.copy()[:, :512],
                                    pool0.copy()[:, 512:])
    return float(np.mean(ref_lat != got_lat))


@pytest.mark.parametrize("n,d", [(40, 7168), (1, 64), (130, 512), (300, 1024), (5, 192)])
def test_kv_proj_matches_oracle(n, d):
    P = 2 * n + 16
    x, w, slots, pool0 = _inputs(n * 31 + d, n, d, P)
    k_scale = 3.5 / 448.0
    pool = torch.from_numpy(pool0).cuda()
    lat = torch.full((n, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.kv_proj_store_fp8(dev_bf16(x), dev_bf16(w), torch.from_numpy(slots).cuda(), k_scale,
                        pool[:, :512], pool[:, 512:], latent_out=lat)
    assert M.mla_get_last_error() == 0
    moved = _check(x, w, slots, pool0, k_scale, pool.cpu().numpy(), bf16_bits(lat),
                   f"n={n} d={d}")
    assert moved < 0.05


def test_kv_proj_without_latent_and_padded_pools_and_strided_x():
    n, d = 70, 256
    x_full, w, slots, pool0 = _inputs(7, n, d + 64, 200)
    x = np.ascontiguousarray(x_full[:, :d])
    w = np.ascontiguousarray(w[:, :d])
    k_scale = 0.011
    ckv0 = W.random_fill_bytes(np.random.default_rng(1), (200, 544))
    kpe0 = W.random_fill_bytes(np.random.default_rng(2), (200, 80))
    ckv, kpe = torch.from_numpy(ckv0).cuda(), torch.from_numpy(kpe0).cuda()
    xd = dev_bf16(x_full)[:, :d]                 # row stride d + 64 elements
    M.kv_proj_store_fp8(xd, dev_bf16(w), torch.from_numpy(slots).cuda(), k_scale,
                        ckv[:, :512], kpe[:, :64])
    lat = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    ckv2, kpe2 = torch.from_numpy(ckv0).cuda(), torch.from_numpy(kpe0).cuda()
    M.kv_proj_store_fp8(xd, dev_bf16(w), torch.from_numpy(slots).cuda(), k_scale,
                        ckv2[:, :512], kpe2[:, :64], latent_out=lat)
    assert M.mla_get_last_error() == 0
    assert torch.equal(ckv, ckv2) and torch.equal(kpe, kpe2)
    got = bf16_bits(lat)
    ref_ckv, ref_kpe = ckv0.copy(), kpe0.copy()
    oracle.kv_store_fp8(got[:, :512], got[:, 512:], slots, k_scale, ref_ckv[:, :512],
                        ref_kpe[:, :64])
    assert np.array_equal(ckv.cpu().numpy(), ref_ckv)
    assert np.array_equal(kpe.cpu().numpy(), ref_kpe)


def test_kv_proj_out_of_range_slot_is_skipped_and_flagged():
    n, d = 9, 128
    x, w, slots, pool0 = _inputs(3, n, d, 40)
    slots[4] = 40                                     # == num_pool_slots
    pool = torch.from_numpy(pool0).cuda()
    lat = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    M.kv_proj_store_fp8(dev_bf16(x), dev_bf16(w), torch.from_numpy(slots).cuda(), 0.02,
                        pool[:, :512], pool[:, 512:], latent_out=lat)
    assert M.mla_get_last_error() == M.FLAG_INDEX_OOB
    got = bf16_bits(lat)
    ref = pool0.copy()
    bad = oracle.kv_store_fp8(got[:, :512], got[:, 512:], slots, 0.02, ref[:, :512], ref[:, 512:])
    assert bad == 1
    assert np.array_equal(pool.cpu().numpy(), ref)


def test_kv_proj_then_decode_equals_store_then_decode():
    """The fused write feeds the decode exactly like kv_store_fp8 of the same
    BF16 latents."""
    n, d, P = 24, 512, 512
    x, w, slots, pool0 = _inputs(11, n, d, P)
    k_scale = 2.0 / 448.0
    fused = torch.from_numpy(pool0).cuda()
    lat = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    M.kv_proj_store_fp8(dev_bf16(x), dev_bf16(w), torch.from_numpy(slots).cuda(), k_scale,
                        fused[:, :512], fused[:, 512:], latent_out=lat)
    plain = torch.from_numpy(pool0).cuda()
    M.kv_store_fp8(lat[:, :512].contiguous(), lat[:, 512:].contiguous(),
                   torch.from_numpy(slots).cuda(), k_scale, plain[:, :512], plain[:, 512:])
    assert torch.equal(fused, plain)
