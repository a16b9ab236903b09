"""Benchmark: paged MLA decode over an FP8 E4M3 KV cache on GB300.

Workload (seeded, synthetic; stands in for the pages' live serving traffic):
the full decode step at batch 40 -- 78 layers, each with its own pool of
495,552 x 576 E4M3 slots, 16 heads, contexts uniform in [1024, 8192] plus the
token appended this step (page size 1).  Per layer: kv_store_fp8 of the new
token's latent, then mla_decode_run.  All 78 pools (22.3 GB) stay resident;
one step touches ~8.4 GB of cache, far more than L2, so every layer's rows
come from HBM.

Reported (one JSON line from rank 0):
  value         microseconds per MLA FP8 decode call (mla_decode_run over one
                layer, batch 40), from K passes over the 78 layers
  ms_per_step   the whole decode step (host plan + 78 x (store + decode))
  roofline      the decode call's algorithmic bytes / its time vs measured HBM
  e2e           the same per-call time with the step's inputs copied from
                pinned host memory and the outputs read back, per layer-call
  baselines     per decode step: full-pool cast + BF16 decode, and
                gather-then-cast + BF16 decode
  cpu_baseline  the CPU oracle on one layer's call, all host cores
`--impl reference` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402
from mla_decode_attention_run_gb300 import accounting as A  # noqa: E402

METRIC = "MLA FP8 decode µs/call & achieved HBM GB/s vs ~8 TB/s peak; decode step ms"
HEADS, PAGE = 16, 1
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ["decode_tc.cu", "decode_params.h", "plan.h", "tc.cuh", "common.cuh"]   # the tcgen05 decode kernel's sources


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist=None, device=None) -> float:
    """Max of a float over all ranks (the slowest replica sets the time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist=None):
    if dist is not None:
        dist.barrier()


def whole_job_us_per_call(max_ms: float, steps: int, calls_per_step: int, world: int) -> float:
    """Replicas: every rank runs the same calls, the slowest rank's time
    covers all of them, so the job's time per call is divided by world."""
    return max_ms * 1e3 / (steps * calls_per_step * world)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def decode_source_hash() -> str:
    """Hash of the tcgen05 decode kernel's code: its sources with comments
    and blank lines removed, so that an edit of a comment keeps the recorded
    traffic valid and any change of code voids it."""
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "mla_decode_attention_run_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, only if
    it was taken on the current decode kernel source."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_sha") != decode_source_hash() or d.get("workload") != workload:
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            # nvidia-smi takes a while to start: the region begins once it samples
            t0 = time.time()
            while time.time() - t0 < 5 and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- the workload

def step_page_table(batch: int, seed: int = 1005):
    """Contexts after this step's append: (indptr, indices, seq_lens, new_slots)."""
    w, new_slots, _ = W.decode_step_workload(batch, seed=seed)
    indptr, idx, lens = W.append_tokens(w, new_slots)
    return w, indptr, idx, lens, new_slots


def fill_pools(torch, M, pools, active_slots_d, layers, seed):
    """Random non-NaN bytes everywhere; the active slots get N(0, 0.5) BF16
    latents quantized by kv_store_fp8 with k_scale = absmax / 448."""
    k_scales = []
    n_active = active_slots_d.shape[0]
    for l in range(layers):
        g = torch.Generator(device=pools.device).manual_seed(seed * 1000 + l)
        pool = pools[l]
        pool.random_(0, 256, generator=g)
        pool[(pool & 0x7F) == 0x7F] = 0x3C
        lat = (torch.randn(n_active, 576, generator=g, device=pools.device) * 0.5).to(
            torch.bfloat16)
        ks = float(np.float32(lat.float().abs().max().item() / 448.0))
        M.kv_store_fp8(lat[:, :512].contiguous(), lat[:, 512:].contiguous(), active_slots_d, ks,
                       pool[:, :512], pool[:, 512:])
        k_scales.append(ks)
        del lat
    return k_scales


# k_scale of the timing pools below: absmax / 448 for N(0, 0.5) latents
# (the largest of ~10^9 draws is about 6.3 sigma)
TIMING_K_SCALE = float(np.float32(0.5 * 6.3 / 448.0))


def latent_pool_(torch, pool, seed, k_scale=TIMING_K_SCALE, rows_per_chunk=1 << 20):
    """Fills a uint8 [slots, 576] pool in place with E4M3 bytes of N(0, 0.5)
    latents at k_scale (torch's float8 cast, clamped to +-448): the score
    distribution the attention sees in service, so the online softmax
    rescales as rarely as it does there.  Input preparation only."""
    g = torch.Generator(device=pool.device).manual_seed(seed)
    for r0 in range(0, pool.shape[0], rows_per_chunk):
        r1 = min(pool.shape[0], r0 + rows_per_chunk)
        x = torch.randn(r1 - r0, pool.shape[1], generator=g, device=pool.device)
        x.mul_(0.5 / k_scale).clamp_(-448.0, 448.0)
        pool[r0:r1] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        del x
    return k_scale


def run_ours(args, rank, world, local):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import mla_decode_attention_run_gb300 as M

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    L, P = args.layers, W.POOL_SLOTS

    # ---- resident state: 78 pools with latents in the headline batch's
    # active slots (per-layer k_scale = absmax / 448 of those latents)
    pools = torch.empty(L, P, 576, dtype=torch.uint8, device=dev)
    w = step_page_table(args.batch)[0]
    active_d = torch.from_numpy(w.kv_indices.astype(np.int64)).to(dev)
    k_scales = fill_pools(torch, M, pools, active_d, L, seed=5)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    result = measure_step(torch, M, args, args.batch, pools, k_scales, stream, dist, world, local,
                          headline=True)
    # the single-stream step: the same 78 pools, latents stored into its own
    # active slots with each layer's k_scale
    if args.batch != 1 and not args.no_batch1:
        w1 = step_page_table(1)[0]
        g1 = torch.Generator(device=dev).manual_seed(4097)
        slots1 = torch.from_numpy(w1.kv_indices.astype(np.int64)).to(dev)
        for l in range(L):
            lat = (torch.randn(slots1.numel(), 576, generator=g1, device=dev) * 0.5).to(torch.bfloat16)
            M.kv_store_fp8(lat[:, :512].contiguous(), lat[:, 512:].contiguous(), slots1,
                           k_scales[l], pools[l, :, :512], pools[l, :, 512:])
        torch.cuda.synchronize()
        result["decode_step_b1"] = measure_step(torch, M, args, 1, pools, k_scales, stream, dist,
                                                world, local, headline=False)

    # ---- the other configurations' decode call, timed alone (rank 0)
    if rank == 0 and not args.no_configs:
        result["configs"] = measure_configs(torch, M, dev, stream)
        result["extend"] = measure_extend(torch, M, dev, stream)
        result["kv_proj"] = measure_kv_proj(torch, M, dev, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.no_configs:
        result["cpu_oracle_configs"] = oracle_timings()
    return result


def measure_step(torch, M, args, B, pools, k_scales, stream, dist, world, local, headline):
    """The full decode step at batch B over the resident pools: host plan +
    a CUDA graph of 78 x (kv_store_fp8 of the new token, mla_decode_run);
    the 78 decode calls alone (value: us per call); the same through host
    buffers (e2e); the two cast baselines and the category ledger; the CPU
    oracle on one layer's call.  headline: the benchmark line's own keys
    (and its launch count); otherwise the same figures as a sub-dict."""
    dev = pools.device
    L, P = args.layers, W.POOL_SLOTS
    rank = dist.get_rank() if dist is not None else 0
    w, indptr, idx, lens, new_slots = step_page_table(B)
    n_tok = int(lens.sum())
    gq = torch.Generator(device=dev).manual_seed(77 if headline else 77 + 1000 + B)
    q = torch.randn(L, B, HEADS, 576, generator=gq, device=dev).to(torch.bfloat16)
    new_ckv = (torch.randn(L, B, 512, generator=gq, device=dev) * 0.5).to(torch.bfloat16)
    new_kpe = (torch.randn(L, B, 64, generator=gq, device=dev) * 0.5).to(torch.bfloat16)
    out = torch.empty(L, B, HEADS, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(L, B, HEADS, dtype=torch.float32, device=dev)
    indptr_d = torch.from_numpy(indptr).to(dev)
    idx_d = torch.from_numpy(idx).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    slots_d = torch.from_numpy(new_slots).to(dev)
    sm_scale = W.SOFTMAX_SCALE

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        plan = M.mla_decode_plan(indptr, lens, B, HEADS, PAGE, M.MLA_KV_FP8_E4M3, stream=stream)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    info = M.mla_decode_plan_info(plan)
    # per call: the tensor-core path (FP8, H <= 16) runs a q
    # split and the decode, the mma.sync path the decode alone; both add the
    # merge kernel when requests are split
    tc_path = M.mla_decode_schedule(indptr, lens, B, HEADS, PAGE, M.MLA_KV_FP8_E4M3)[1]["kernel"] == 1
    launches_per_call = (2 if tc_path else 1) + (1 if info["num_partials"] > 0 else 0)

    def store(l, s):
        M.kv_store_fp8(new_ckv[l], new_kpe[l], slots_d, k_scales[l], pools[l, :, :512],
                       pools[l, :, 512:], stream=s)

    def decode(l, s, pl=plan, ck=None, kp=None, ix=None, kscale=None):
        M.mla_decode_run(pl, q[l], pools[l, :, :512] if ck is None else ck,
                         pools[l, :, 512:] if kp is None else kp,
                         P if ck is None else ck.shape[0], indptr_d,
                         idx_d if ix is None else ix, lens_d,
                         k_scales[l] if kscale is None else kscale, sm_scale, out[l], lse[l], ws,
                         stream=s)

    def capture(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body(torch.cuda.current_stream())
        return g

    # one eager pass first (checks every call returns OK), then graphs
    with torch.cuda.stream(stream):
        for l in range(L):
            store(l, stream)
            decode(l, stream)
    torch.cuda.synchronize()
    flags = M.mla_get_last_error(stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x} after the eager pass")

    g_step = capture(lambda s: [(store(l, s), decode(l, s)) for l in range(L)])
    g_decode = capture(lambda s: [decode(l, s) for l in range(L)])

    def plan_step():
        M.mla_decode_plan(indptr, lens, B, HEADS, PAGE, M.MLA_KV_FP8_E4M3, stream=stream,
                          plan=plan)

    def timed(fn, steps):
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        return e0.elapsed_time(e1)                     # ms

    def full_step():
        plan_step()
        g_step.replay()

    # ---- warm-up, then the K timed decode steps and K decode-only passes
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            full_step()
            g_decode.replay()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            t_step = timed(full_step, args.steps)
            t_dec = timed(g_decode.replay, args.steps)
    clocks = clk.summary()
    t_step = reduce_max(t_step, dist, dev)
    t_dec = reduce_max(t_dec, dist, dev)
    if M.mla_get_last_error(stream):
        raise RuntimeError("device flags set during the timed region")

    ms_per_step = t_step / args.steps
    us_per_call = whole_job_us_per_call(t_dec, args.steps, L, world)
    call_bytes = A.decode_call_bytes(lens, HEADS, PAGE)
    achieved = call_bytes / (t_dec * 1e-3 / (args.steps * L)) / 1e9
    peak, peak_src = measured_peaks()
    workload_name = f"decode_step_b{B}_h{HEADS}_l{L}"

    result = {} if not headline else {"metric": METRIC}
    result.update({
        "value": round(us_per_call, 3), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 mma (q as three e4m3 terms, p as two) / f32 accumulate",
        "data": "synthetic (seeded N(0,0.5) latents, N(0,1) q; no model weights)",
        "config": {"workload": workload_name, "batch": B, "heads": HEADS, "layers": L,
                   "page_size": PAGE, "pool_slots": P, "tokens_per_call": n_tok,
                   "contexts": ("4096" if B == 1 else "uniform[1024,8192]") + " + 1 appended",
                   "parallelism": "replicas",
                   "l2": "inputs larger than L2 (78 pools, %.2f GB touched per step)" % (
                       L * n_tok * 576 / 1e9),
                   "graphs": "CUDA graph per step; plan rebuilt on the host each step"},
        "decode_step_ms": round(ms_per_step, 4),
        "tokens_per_s": round(B * world / (ms_per_step * 1e-3), 1),
        # our kernels in the two timed regions: K steps of 78 x (store + decode
        # [+ merge]) and K decode-only passes of 78 x (decode [+ merge])
        "gpu_launches": int(args.steps * L * (1 + 2 * launches_per_call)),
        "plan": info,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": committed_traffic(workload_name),
                     "kernel": "mla_decode_run: q split + tcgen05 decode + split-KV merge, timed together",
                     "traffic_of": "mla_decode_tc_kernel (ncu, profiles/decode_traffic.json)",
                     "algorithmic_bytes_per_launch": call_bytes,
                     "peak_source": f"{peak_src} HBM copy bandwidth"},
    })
    if not headline:
        for k in ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                  "vs_baseline", "dtype", "data", "gpu_launches"):
            result.pop(k, None)
        if L * n_tok * 576 < 3 * 129e6:
            result["config"]["l2"] = ("%d layers x %.1f MB of active rows per step (%.2f GB): "
                                      "about L2's size, so part of each call's rows may still be "
                                      "in L2 from the previous step" % (L, n_tok * 576 / 1e6,
                                                                        L * n_tok * 576 / 1e9))

    # ---- e2e through the public API from pinned host buffers
    h_q = torch.empty_like(q, device="cpu").pin_memory()
    h_q.copy_(q.cpu())
    h_ckv = new_ckv.cpu().pin_memory()
    h_kpe = new_kpe.cpu().pin_memory()
    h_pt = [torch.from_numpy(a).pin_memory() for a in (indptr, idx, lens)]
    h_slots = torch.from_numpy(new_slots).pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    # The step's inputs go up and its outputs come back a chunk of layers at a
    # time on two copy streams, so that each chunk's copies overlap the
    # neighbouring chunks' store + decode (every byte still crosses within the
    # timed step); small chunks at both ends (the first upload and the last
    # download are not hidden), large ones in the middle.  The copies, the
    # stores and the decode calls of a step are captured together as one CUDA
    # graph on three streams joined by events, so that a step costs the host
    # one plan and one replay.
    ramp = [2, 4, 8]
    sizes = ramp + [max(1, (L - 2 * sum(ramp)) // 3)] * 3 + ramp[::-1]
    if sum(sizes) > L or L < 2 * sum(ramp) + 3:
        sizes = [L]
    sizes[len(sizes) // 2] += L - sum(sizes)
    bounds = [0]
    for z in sizes:
        bounds.append(bounds[-1] + z)
    spans = list(zip(bounds[:-1], bounds[1:]))
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_start, ev_out = torch.cuda.Event(), torch.cuda.Event()
    ev_in = [torch.cuda.Event() for _ in spans]
    ev_done = [torch.cuda.Event() for _ in spans]

    def e2e_body(s):
        ev_start.record(s)
        up_s.wait_event(ev_start)
        down_s.wait_event(ev_start)
        with torch.cuda.stream(up_s):
            for d, h in zip((indptr_d, idx_d, lens_d), h_pt):
                d.copy_(h, non_blocking=True)
            slots_d.copy_(h_slots, non_blocking=True)
            for c, (a, b) in enumerate(spans):
                q[a:b].copy_(h_q[a:b], non_blocking=True)
                new_ckv[a:b].copy_(h_ckv[a:b], non_blocking=True)
                new_kpe[a:b].copy_(h_kpe[a:b], non_blocking=True)
                ev_in[c].record(up_s)
        for c, (a, b) in enumerate(spans):
            s.wait_event(ev_in[c])
            for l in range(a, b):
                store(l, s)
                decode(l, s)
            ev_done[c].record(s)
            down_s.wait_event(ev_done[c])
            with torch.cuda.stream(down_s):
                h_out[a:b].copy_(out[a:b], non_blocking=True)
                h_lse[a:b].copy_(lse[a:b], non_blocking=True)
        ev_out.record(down_s)
        s.wait_event(ev_out)

    g_e2e = capture(e2e_body)

    def e2e_step():
        plan_step()
        g_e2e.replay()

    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_step()
        k_e2e = max(3, min(args.steps, 10))
        t_e2e = reduce_max(timed(e2e_step, k_e2e), dist, dev)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_ckv, h_kpe, *h_pt, h_slots))
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    result["e2e"] = {"value": round(whole_job_us_per_call(t_e2e, k_e2e, L, world), 3),
                     "unit": "us/call",
                     "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                     "per": "layer-call incl. store and host copies",
                     "overlap": f"inputs up and outputs down per chunk of layers {sizes} on two copy "
                                "streams, overlapping compute; copies, stores and decode calls of a step "
                                "in one CUDA graph, the plan on the host before it"}

    # ---- the two baselines the pages describe, per decode step
    if not args.no_baselines:
        base = run_baselines(torch, M, args, B, stream, pools, q, out, lse, ws, k_scales, store,
                             indptr, idx, lens, timed, dist, dev)
        ledger = base.pop("ledger")
        # the fused step's graph (store + decode per layer) without the host plan
        with torch.cuda.stream(stream):
            t_graph = reduce_max(timed(g_step.replay, args.steps), dist, dev) / args.steps
        ledger["fused_fp8"] = category_ledger(t_graph, {"store": base.pop("store_ms"),
                                                        "attention": t_dec / args.steps})
        result["baselines"] = base
        result["ledger"] = ledger

    # ---- CPU oracle baseline (rank 0, one GPU): one layer's call of this step
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_from_device(pools[0], q[0], indptr, idx, lens,
                                                          k_scales[0], B)
    del g_step, g_decode, g_e2e
    M.mla_decode_plan_destroy(plan)
    return result


def measure_configs(torch, M, dev, stream, names=("single", "large_head"), batch=None):
    """The single-stream (1 x 4,096 tokens) and 128-head (128 x 32,768 tokens,
    page size 64, 2.4 GB pool) decode calls, each timed as a CUDA graph of
    back-to-back calls on pools of quantized N(0, 0.5) latents.  The
    128-head call is also set against the measured BF16 tensor peak: it does
    2,176 flops per token and head."""
    peak, peak_src = measured_peaks()
    tflops_peak = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            tflops_peak = float(json.load(f).get("bf16_tflops", 0)) or None
    res = {}
    for name, reps in (("single", 50), ("large_head", 4)):
        if name not in names:
            continue
        # batch: fewer requests of the same shape (a smaller case for profilers)
        w = W.make_workload(name, latent_requests=[], **({"batch": batch} if batch else {}))
        B, H, ps = w.batch, w.heads, w.page_size
        pool = torch.empty((w.num_slots, W.D_ALL), dtype=torch.uint8, device=dev)
        k_scale = latent_pool_(torch, pool, seed=11)
        q = torch.randn(B, H, W.D_ALL, device=dev).to(torch.bfloat16)
        out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, H, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            plan = M.mla_decode_plan(w.kv_indptr, w.seq_lens, B, H, ps, stream=stream)
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
        ip, ix, ln = (torch.from_numpy(a).to(dev) for a in (w.kv_indptr, w.kv_indices, w.seq_lens))
        kernel = M.mla_decode_schedule(w.kv_indptr, w.seq_lens, B, H, ps)[1]["kernel"]

        def call(s):
            M.mla_decode_run(plan, q, pool[:, :512], pool[:, 512:], w.num_slots, ip, ix, ln,
                             k_scale, W.SOFTMAX_SCALE, out, lse, ws, stream=s)
        with torch.cuda.stream(stream):
            for _ in range(3):
                call(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                call(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(3):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (3 * reps)
        nbytes = A.decode_call_bytes(w.seq_lens, H, ps)
        flops = A.decode_call_flops(w.seq_lens, H)
        r = {"batch": B, "heads": H, "page_size": ps, "tokens": int(w.seq_lens.sum()),
             "kernel": "tcgen05" if kernel == 1 else "mma.sync",
             "token_ranges": M.mla_decode_plan_info(plan)["num_ctas"], "us_per_call": round(us, 3),
             "achieved_gbs": round(nbytes / us / 1e3, 1), "hbm_frac": round(nbytes / us / 1e3 / peak, 4),
             "tflops": round(flops / us / 1e6, 2),
             "l2": "the whole call fits in L2 (latency-bound)" if nbytes < 64e6 else "inputs larger than L2"}
        if tflops_peak and name == "large_head":
            r["tensor_frac"] = round(flops / us / 1e6 / tflops_peak, 4)
            r["tensor_peak"] = "measured cuBLAS bf16 burst " + str(tflops_peak) + " TFLOP/s"
        res[name] = r
        M.mla_decode_plan_destroy(plan)
        del pool, q, out, lse, ws, g
        torch.cuda.empty_cache()
    return res


def measure_extend(torch, M, dev, stream, n_pools=8):
    """Causal extend calls (several new tokens per request over a cached
    history), each timed as a CUDA graph of calls rotating over n_pools
    pools of quantized N(0, 0.5) latents (one per layer; together larger than
    L2).  Beside each:
    the gather-then-cast of the same pages, the least a BF16 prefill kernel
    would need before it runs, which the FP8-native extend does not do."""
    peak, _ = measured_peaks()
    tflops_peak = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            tflops_peak = float(json.load(f).get("bf16_tflops", 0)) or None
    res = {}
    P = W.POOL_SLOTS
    pools = torch.empty((n_pools, P, W.D_ALL), dtype=torch.uint8, device=dev)
    for l in range(n_pools):
        k_scale = latent_pool_(torch, pools[l], seed=100 + l)
    for name in ("spec_decode", "extend_chunk"):
        w = W.make_extend_workload(name, latent_requests=[])
        qo = w.extra["qo_indptr"]
        q_lens = np.diff(qo)
        B, H, ps, n_q = w.batch, w.heads, w.page_size, int(qo[-1])
        q = torch.randn(n_pools, n_q, H, W.D_ALL, device=dev).to(torch.bfloat16)
        out = torch.empty(n_pools, n_q, H, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(n_pools, n_q, H, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            plan = M.mla_extend_plan(qo, w.kv_indptr, w.seq_lens, B, H, ps, stream=stream)
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
        ip, ix, ln = (torch.from_numpy(a).to(dev) for a in (w.kv_indptr, w.kv_indices, w.seq_lens))
        rows = int(ix.numel()) * ps
        ckv_c = torch.empty(rows, 512, dtype=torch.bfloat16, device=dev)
        kpe_c = torch.empty(rows, 64, dtype=torch.bfloat16, device=dev)
        info = M.mla_extend_schedule(qo, w.kv_indptr, w.seq_lens, B, H, ps)[2]

        def extend(l, s):
            M.mla_extend_run(plan, q[l], pools[l, :, :512], pools[l, :, 512:], P, ip, ix, ln,
                             k_scale, W.SOFTMAX_SCALE, out[l], lse[l], ws, stream=s)

        def gather(l, s):
            M.kv_gather_cast(pools[l, :, :512], pools[l, :, 512:], ix, ps, 1.0, ckv_c, kpe_c,
                             stream=s)

        def time_graph(fn):
            with torch.cuda.stream(stream):
                for l in range(n_pools):
                    fn(l, stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for l in range(n_pools):
                    fn(l, torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(3):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / (3 * n_pools)

        us = time_graph(extend)
        us_cast = time_graph(gather)
        nbytes = A.extend_call_bytes(w.seq_lens, q_lens, H, ps)
        flops = A.extend_call_flops(w.seq_lens, q_lens, H)
        r = {"batch": B, "heads": H, "page_size": ps, "new_tokens_per_request": int(q_lens[0]),
             "context_tokens": int(w.seq_lens.sum()), "visible_tokens":
             A.extend_visible_tokens(w.seq_lens, q_lens), "block_rows": info["block_rows"],
             "blocks": info["num_blocks"], "us_per_call": round(us, 3),
             "achieved_gbs": round(nbytes / us / 1e3, 1), "hbm_frac": round(nbytes / us / 1e3 / peak, 4),
             "tflops": round(flops / us / 1e6, 2),
             "gather_cast_us": round(us_cast, 3),
             "gather_cast_note": "kv_gather_cast of the same pages to BF16 (not part of the FP8 extend)"}
        if tflops_peak:
            r["tensor_frac"] = round(flops / us / 1e6 / tflops_peak, 4)
        res[name] = r
        M.mla_decode_plan_destroy(plan)
        del q, out, lse, ws, ckv_c, kpe_c
    del pools
    torch.cuda.empty_cache()
    return res


# Hidden size of the projection's input.  The pages do not give it; this is
# the hidden size of the DeepSeek-V3 family that Kimi-K2.5 belongs to.
PROJ_D_MODEL = 7168


def measure_kv_proj(torch, M, dev, stream, batch=40, layers=W.NUM_LAYERS, d_model=PROJ_D_MODEL):
    """The decode step's KV write with the projection: per layer, batch new
    tokens' hidden states [batch, d_model] times that layer's weights
    [576, d_model] into the latent, stored as E4M3 into the pool.  Fused:
    kv_proj_store_fp8 (one kernel).  Unfused: cuBLAS BF16 GEMMs (torch.matmul)
    to the BF16 c_kv and k_pe latents, then kv_store_fp8.  Each is a CUDA graph over all
    layers (the layers' weights, 0.64 GB, are far larger than L2)."""
    peak, _ = measured_peaks()
    g = torch.Generator(device=dev).manual_seed(77)
    P = W.POOL_SLOTS
    pool = torch.empty((P, W.D_ALL), dtype=torch.uint8, device=dev)
    k_scale = latent_pool_(torch, pool, seed=78)
    x = torch.randn(layers, batch, d_model, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(layers, W.D_ALL, d_model, generator=g, device=dev) / math.sqrt(d_model)).to(
        torch.bfloat16)
    slots = torch.randperm(P, generator=g, device=dev)[:batch].to(torch.int64)
    lat_ckv = torch.empty(layers, batch, 512, dtype=torch.bfloat16, device=dev)
    lat_kpe = torch.empty(layers, batch, 64, dtype=torch.bfloat16, device=dev)

    def fused(l, s):
        M.kv_proj_store_fp8(x[l], w[l], slots, k_scale, pool[:, :512], pool[:, 512:], stream=s)

    def unfused(l, s):
        # the store takes c_kv and k_pe as separate contiguous arrays
        torch.matmul(x[l], w[l, :512].t(), out=lat_ckv[l])
        torch.matmul(x[l], w[l, 512:].t(), out=lat_kpe[l])
        M.kv_store_fp8(lat_ckv[l], lat_kpe[l], slots, k_scale, pool[:, :512], pool[:, 512:],
                       stream=s)

    def time_graph(fn):
        with torch.cuda.stream(stream):
            for l in range(layers):
                fn(l, stream)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for l in range(layers):
                fn(l, torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            gr.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                gr.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (5 * layers)

    us_fused = time_graph(fused)
    us_unfused = time_graph(unfused)
    nbytes = A.kv_proj_bytes(batch, d_model)
    res = {"batch": batch, "d_model": d_model, "layers": layers,
           "fused_us_per_layer": round(us_fused, 3), "unfused_us_per_layer": round(us_unfused, 3),
           "unfused": "cuBLAS BF16 GEMMs (torch.matmul: c_kv and k_pe outputs) + kv_store_fp8",
           "achieved_gbs": round(nbytes / us_fused / 1e3, 1),
           "hbm_frac": round(nbytes / us_fused / 1e3 / peak, 4),
           "bytes_per_layer": nbytes, "d_model_source": "DeepSeek-V3 family hidden size (not on the pages)"}
    del pool, x, w, lat_ckv, lat_kpe
    torch.cuda.empty_cache()
    return res


def category_ledger(step_ms, parts):
    """Per-step category ledger: each category's time (a graph of only that
    category's launches over the step's layers), its share of the step, and
    the step time if that category cost nothing.  Tags follow the launching
    call: kv_store_fp8 -> store, the PyTorch full-pool .to(bfloat16) -> cast,
    kv_gather_cast -> gather, mla_decode_run (q split, decode, merge) ->
    attention.  'other' is what the categories alone do not account for
    (gaps between launches, overlap)."""
    out = {"step_ms": round(step_ms, 4), "categories": {}}
    for k, v in parts.items():
        out["categories"][k] = {"ms": round(v, 4), "share": round(v / step_ms, 4),
                                "step_ms_if_free": round(max(step_ms - v, 0.0), 4)}
    out["other_ms"] = round(step_ms - sum(parts.values()), 4)
    return out


def run_baselines(torch, M, args, B, stream, pools, q, out, lse, ws, k_scales, store, indptr, idx,
                  lens, timed, dist, dev):
    L, P = args.layers, W.POOL_SLOTS
    n = idx.size
    idx_d = torch.from_numpy(idx).to(dev)
    indptr_d = torch.from_numpy(indptr).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    seq_d = torch.arange(n, dtype=torch.int32, device=dev)
    full = torch.empty(P, 576, dtype=torch.bfloat16, device=dev)
    compact = torch.empty(n, 576, dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(stream):
        plan_bf16 = M.mla_decode_plan(indptr, lens, B, HEADS, PAGE, M.MLA_KV_BF16, stream=stream)
    ws_b = torch.empty(max(plan_bf16.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    sm = W.SOFTMAX_SCALE

    def cast_layer(l, s):      # the pages' full-pool .to(bfloat16), then BF16 attention
        full.copy_(pools[l].view(torch.float8_e4m3fn))
        M.mla_decode_run(plan_bf16, q[l], full[:, :512], full[:, 512:], P, indptr_d, idx_d,
                         lens_d, k_scales[l], sm, out[l], lse[l], ws_b, stream=s)

    def gather_layer(l, s):    # gather-then-cast of the active slots, replan 0..n-1
        M.kv_gather_cast(pools[l, :, :512], pools[l, :, 512:], idx_d, 1, 1.0, compact[:, :512],
                         compact[:, 512:], stream=s)
        M.mla_decode_run(plan_bf16, q[l], compact[:, :512], compact[:, 512:], n, indptr_d, seq_d,
                         lens_d, k_scales[l], sm, out[l], lse[l], ws_b, stream=s)

    def cast_only(l, s):
        full.copy_(pools[l].view(torch.float8_e4m3fn))

    def gather_only(l, s):
        M.kv_gather_cast(pools[l, :, :512], pools[l, :, 512:], idx_d, 1, 1.0, compact[:, :512],
                         compact[:, 512:], stream=s)

    def cast_attention(l, s):
        M.mla_decode_run(plan_bf16, q[l], full[:, :512], full[:, 512:], P, indptr_d, idx_d,
                         lens_d, k_scales[l], sm, out[l], lse[l], ws_b, stream=s)

    def gather_attention(l, s):
        M.mla_decode_run(plan_bf16, q[l], compact[:, :512], compact[:, 512:], n, indptr_d, seq_d,
                         lens_d, k_scales[l], sm, out[l], lse[l], ws_b, stream=s)

    def step_ms(*layer_fns):
        """ms per step of a graph of L layers, each running layer_fns in order."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            s = torch.cuda.current_stream()
            for l in range(L):
                for fn in layer_fns:
                    fn(l, s)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            k = max(3, min(args.steps, 5))
            t = reduce_max(timed(g.replay, k), dist, dev)
        del g
        return t / k

    res, ledger = {}, {}
    store_ms = step_ms(store)
    for name, layer_fn, tag, only, attention in (
            ("full_pool_cast_then_bf16_decode", cast_layer, "cast", cast_only, cast_attention),
            ("gather_then_cast_then_bf16_decode", gather_layer, "gather", gather_only, gather_attention)):
        t = step_ms(store, layer_fn)
        res[name] = {"decode_step_ms": round(t, 3)}
        ledger[name] = category_ledger(t, {"store": store_ms, tag: step_ms(only),
                                           "attention": step_ms(attention)})
    res["ledger"] = ledger
    res["store_ms"] = store_ms
    cast_bytes = A.full_pool_cast_bytes(P) * L
    gather_bytes = A.gather_cast_bytes(n, n) * L
    res["full_pool_cast_then_bf16_decode"]["cast_bytes_per_step"] = cast_bytes
    res["gather_then_cast_then_bf16_decode"]["cast_bytes_per_step"] = gather_bytes
    M.mla_decode_plan_destroy(plan_bf16)
    return res


def oracle_call(pool_np, q_bits, indptr, idx, lens, k_scale, nthreads=0):
    import oracle
    t0 = time.perf_counter()
    oracle.decode_fp8(q_bits, pool_np[:, :512], pool_np[:, 512:], indptr, idx, lens, PAGE,
                      k_scale, W.SOFTMAX_SCALE, nthreads=nthreads)
    return time.perf_counter() - t0


def oracle_timings():
    """The oracle beside each measured configuration, on this host's cores
    (random pool bytes: timing does not depend on the values).  Small cases
    single-threaded and on all cores; the 128-head call on one of its 128
    requests, the 4-token extend on 4 of its 40 requests, both scaled
    linearly by the work (labelled extrapolated); the projection store of
    one layer in full."""
    import oracle
    rng = np.random.default_rng(3)
    # taken before any call: a call with nthreads = 1 sets OpenMP's default
    cores = oracle.max_threads()
    res = {"cores": cores}

    def timed_call(fn):
        t0 = time.perf_counter()
        fn()
        return (time.perf_counter() - t0) * 1e6

    def decode_case(name, requests=None, threads=(1, None)):
        w = W.make_workload(name, latent_requests=[])
        B = w.batch
        keep = list(range(B)) if requests is None else requests
        lens = w.seq_lens[keep]
        ps = w.page_size
        pages = [w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]] for b in keep]
        indptr = np.zeros(len(keep) + 1, np.int32)
        indptr[1:] = np.cumsum([len(x) for x in pages])
        idx = np.concatenate(pages).astype(np.int32)
        pool = W.random_fill_bytes(rng, (w.num_slots, W.D_ALL))
        q = w.q_bf16[keep]
        out = {}
        for t in threads:
            nt = cores if t is None else t
            us = timed_call(lambda: oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, idx,
                                                      lens, ps, w.k_scale, W.SOFTMAX_SCALE,
                                                      nthreads=nt))
            scale = float(w.seq_lens.sum()) / float(lens.sum())
            out["us_per_call_" + ("1_thread" if t == 1 else "all_cores")] = round(us * scale, 1)
        if requests is not None:
            out["extrapolated"] = f"timed on {len(keep)} of {B} requests, scaled by tokens"
        return out

    res["tiny"] = decode_case("tiny")
    res["single"] = decode_case("single")
    res["concurrency"] = decode_case("concurrency", threads=(None,))
    res["large_head"] = decode_case("large_head", requests=[0], threads=(None,))

    w = W.make_extend_workload("spec_decode", latent_requests=[])
    keep = [0, 1, 2, 3]
    qo = w.extra["qo_indptr"]
    sub_qo = np.zeros(len(keep) + 1, np.int32)
    sub_qo[1:] = np.cumsum([qo[b + 1] - qo[b] for b in keep])
    pages = [w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]] for b in keep]
    sub_ip = np.zeros(len(keep) + 1, np.int32)
    sub_ip[1:] = np.cumsum([len(x) for x in pages])
    sub_q = np.concatenate([w.q_bf16[qo[b]:qo[b + 1]] for b in keep])
    pool = W.random_fill_bytes(rng, (w.num_slots, W.D_ALL))
    us = timed_call(lambda: oracle.extend_fp8(sub_q, pool[:, :512], pool[:, 512:], sub_qo, sub_ip,
                                              np.concatenate(pages).astype(np.int32),
                                              w.seq_lens[keep], 1, w.k_scale, W.SOFTMAX_SCALE,
                                              nthreads=cores))
    ql = np.diff(qo)
    scale = A.extend_visible_tokens(w.seq_lens, ql) / A.extend_visible_tokens(w.seq_lens[keep], ql[keep])
    res["spec_decode"] = {"us_per_call_all_cores": round(us * scale, 1),
                          "extrapolated": f"timed on {len(keep)} of {w.batch} requests, scaled by "
                                          "visible tokens"}

    n, d = 40, PROJ_D_MODEL
    x = rng.integers(0, 1 << 16, size=(n, d), dtype=np.uint16) & 0xBFFF   # finite BF16 bit patterns
    wts = rng.integers(0, 1 << 16, size=(W.D_ALL, d), dtype=np.uint16) & 0xBFFF
    slots = rng.permutation(4096)[:n].astype(np.int64)
    ppool = np.zeros((4096, W.D_ALL), np.uint8)
    us = timed_call(lambda: oracle.kv_proj_fp8(x, wts, slots, 0.01, ppool[:, :512], ppool[:, 512:]))
    res["kv_proj"] = {"us_per_layer_all_cores": round(us, 1)}
    return res


def cpu_baseline_from_device(pool_d, q_d, indptr, idx, lens, k_scale, batch):
    import oracle
    import torch
    pool_np = pool_d.cpu().numpy()
    q_bits = q_d.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    threads = oracle.max_threads()
    dt = oracle_call(pool_np, q_bits, indptr, idx, lens, k_scale)
    return {"value": round(dt * 1e6, 1), "unit": "us/call", "cores": threads, "kind": "oracle",
            "sample": f"one layer's full decode call (batch {batch}, 16 heads, all contexts), "
                      "C fp64 oracle with OpenMP over (request, head)"}


def run_reference(args, rank, world, local):
    """The reference arm: the CPU oracle, as it stands, on the same decode
    call (one layer of the batch-40 step), each step one full call."""
    if rank != 0:
        return None
    import oracle
    w, indptr, idx, lens, new_slots = step_page_table(args.batch)
    wl = W.make_workload("concurrency", batch=args.batch, seed=1005)   # same page table
    pool = W.random_fill_bytes(np.random.default_rng(5), (W.POOL_SLOTS, 576))
    oracle.kv_store_fp8(wl.latent_bf16[:, :512], wl.latent_bf16[:, 512:], wl.latent_slots,
                        wl.k_scale, pool[:, :512], pool[:, 512:])
    new = W.make_workload("concurrency", batch=args.batch, lens=[1] * args.batch, seed=99)
    oracle.kv_store_fp8(new.latent_bf16[:, :512], new.latent_bf16[:, 512:], new_slots,
                        wl.k_scale, pool[:, :512], pool[:, 512:])
    q_bits = wl.q_bf16
    for _ in range(args.warmup):
        oracle_call(pool, q_bits, indptr, idx, lens, wl.k_scale)
    times = [oracle_call(pool, q_bits, indptr, idx, lens, wl.k_scale) for _ in range(args.steps)]
    us = float(np.mean(times)) * 1e6
    cores = oracle.max_threads()
    sample = ("one layer's full decode call per step (batch 40, 16 heads, contexts "
              "uniform[1024,8192]+1), C fp64 oracle, OpenMP over (request, head)")
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/call",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(us / 1e3, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"decode_step_b{args.batch}_h{HEADS}_l{args.layers}",
                       "batch": args.batch, "heads": HEADS, "page_size": PAGE,
                       "tokens_per_call": int(lens.sum()), "parallelism": "replicas"},
            "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=40)
    ap.add_argument("--layers", type=int, default=W.NUM_LAYERS)
    ap.add_argument("--no-baselines", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--no-batch1", action="store_true",
                    help="skip the batch-1 (single-stream) decode step")
    ap.add_argument("--extend-only", action="store_true",
                    help="time only the extend workloads and print their JSON (a diagnostic, "
                         "not the benchmark line)")
    ap.add_argument("--proj-only", action="store_true",
                    help="time only the fused KV projection store against cuBLAS + store and "
                         "print its JSON (a diagnostic)")
    ap.add_argument("--config", choices=["single", "large_head"],
                    help="time only that decode configuration and print its JSON (a diagnostic)")
    ap.add_argument("--config-batch", type=int, default=None,
                    help="with --config: that many requests of the configuration's shape (a smaller "
                         "case for profilers)")
    ap.add_argument("--pools", type=int, default=8,
                    help="pools the extend timing rotates over (--extend-only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.proj_only:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        import mla_decode_attention_run_gb300 as M
        torch.cuda.set_device(local)
        stream = torch.cuda.Stream()
        res = measure_kv_proj(torch, M, torch.device("cuda", local), stream, layers=args.layers)
        if rank == 0:
            print(json.dumps({"kv_proj": res}), flush=True)
        return
    if args.config:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        import mla_decode_attention_run_gb300 as M
        torch.cuda.set_device(local)
        stream = torch.cuda.Stream()
        res = measure_configs(torch, M, torch.device("cuda", local), stream, names=(args.config,),
                              batch=args.config_batch)
        if rank == 0:
            print(json.dumps({"configs": res}), flush=True)
        return
    if args.extend_only:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        import mla_decode_attention_run_gb300 as M
        torch.cuda.set_device(local)
        stream = torch.cuda.Stream()
        res = measure_extend(torch, M, torch.device("cuda", local), stream, n_pools=args.pools)
        if rank == 0:
            print(json.dumps({"extend": res}), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world, local)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
