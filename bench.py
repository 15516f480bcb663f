#!/usr/bin/env python3
"""Benchmark of paged draft-block attention (one call = split kernel + combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line on rank 0.  ``value`` is the algorithmic KV-read
bandwidth of the whole job in GB/s (K and V rows each read once per call,
summed over ranks, divided by the slowest rank's device time); ``us_per_call``
is the mean device time of one call.  Inputs are resident in HBM when the
timed region starts and L2 is flushed (a 512 MiB write) before every timed
call, outside its CUDA-event pair.

Workloads (``--workload``): ``tiny``, ``minimax_B{B}_K{K}_L{L}`` (16/1 heads,
D=128, W=4096, page 64), ``adp_B{B}_K{K}_L{L}`` (64/4 heads, 1 % key outliers),
``longctx_{8|12}x2_B{B}_L{L}`` (D=64, page 32, unwindowed),
``ragged_B{B}`` (64/16 heads, contexts uniform in [1K, 128K]); a suffix
``_r{R}`` turns any of them into the causal block with a right window of R
block keys.  The default is the ragged stress batch at its largest point,
B=256 requests of 64/16 heads with contexts uniform in [1K, 128K] (about 69 GB
of K/V per call): the largest configuration that fits one GPU, and the one
whose contexts reach the long-context range.  ``us_per_call`` and ``value``
use the median call time; the mean and the 90th percentile are reported
beside it.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores (the slow baseline arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft-block attention µs/call and KV-read HBM GB/s (% of GB300 peak)"
DEFAULT_WORKLOAD = "ragged_B256"
L2_FLUSH_BYTES = 512 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def workload_spec(name: str, seed_offset: int = 0):
    import dataclasses

    m = re.fullmatch(r"(.+)_r(\d+)", name)
    if m:
        base = workload_spec(m[1], seed_offset)
        return dataclasses.replace(base, name=name, future_keys=0, right_window=int(m[2]))
    from speculative_decoding_draft_paged_gb300 import workloads as W

    if name == "tiny":
        return W.tiny(seed=1001 + seed_offset)
    m = re.fullmatch(r"minimax_B(\d+)_K(\d+)_L(\d+)", name)
    if m:
        return W.minimax(B=int(m[1]), K=int(m[2]), L=int(m[3]), seed=1002 + seed_offset)
    m = re.fullmatch(r"adp_B(\d+)_K(\d+)_L(\d+)", name)
    if m:
        return W.adp(B=int(m[1]), K=int(m[2]), L=int(m[3]), seed=1003 + seed_offset)
    m = re.fullmatch(r"longctx_(\d+)x2_B(\d+)_L(\d+)", name)
    if m:
        return W.longctx(B=int(m[2]), L=int(m[3]), Hq=int(m[1]), seed=1004 + seed_offset)
    m = re.fullmatch(r"ragged_B(\d+)", name)
    if m:
        return W.ragged(B=int(m[1]), seed=1005 + seed_offset)
    raise SystemExit(f"unknown workload {name!r}")


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_sha() -> str:
    from speculative_decoding_draft_paged_gb300 import build as B

    h = hashlib.sha256()
    for p in sorted(B._deps()):
        if p.endswith("build.py"):
            continue
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources are unchanged since it was taken."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def reduce_over_ranks(times, nbytes, device):
    """Slowest rank's times (MAX) and the job's bytes (SUM); identity on one rank."""
    import torch
    import torch.distributed as dist

    vals = torch.tensor(list(times) + [float(nbytes)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = vals[:-1].clone()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        b = vals[-1:].clone()
        dist.all_reduce(b, op=dist.ReduceOp.SUM)
        vals = torch.cat([t, b])
    out = [float(x) for x in vals.tolist()]
    return out[:-1], out[-1]


def time_oracle_sample(spec, budget_s: float = 15.0, device_inputs=None, fp8: bool = False):
    """Run the oracle on a bounded sample of the workload's requests (the
    fp8-context form over E4M3 casts of the same pages when ``fp8``).

    Returns (kv_bytes_per_s, seconds, n_requests, threads, description)."""
    import numpy as np
    import torch

    import oracle
    from speculative_decoding_draft_paged_gb300 import workloads as W

    threads = os.cpu_count() or 1
    # Estimated oracle cost: ~4 flops per (row, key, dim) at ~2.5 GFLOP/s per
    # core (measured on a 16-core Arm host: 127 GFLOP of ragged_B256 requests
    # in 3.1 s), so that the sample takes about budget_s seconds.
    per_req = [spec.Hq * spec.K * (spec.visible_ctx(L) + spec.K) * spec.D * 4 for L in spec.ctx_lens]
    rate = 2.5e9 * threads
    ids, cost = [], 0.0
    for b in range(spec.B):
        if ids and cost + per_req[b] / rate > budget_s:
            break
        ids.append(b)
        cost += per_req[b] / rate
    sub = W.CaseSpec(spec.name + "_sample", B=len(ids), Hq=spec.Hq, Hkv=spec.Hkv, D=spec.D, K=spec.K,
                     P=spec.P, window=spec.window, future_keys=spec.future_keys,
                     right_window=spec.right_window,
                     ctx_lens=[spec.ctx_lens[b] for b in ids], sigma=spec.sigma,
                     outlier_frac=spec.outlier_frac, seed=spec.seed)
    inp = W.make_inputs(sub, "cpu")

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    kw = dict(block_size=sub.K, window=sub.window, future_keys=sub.future_keys,
              right_window=sub.right_window, scale=sub.softmax_scale, nthreads=threads)
    if fp8:
        codes = {k: inp[k].float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                 for k in ("k_pages", "v_pages")}
        shape = (sub.B, sub.K, sub.Hkv, sub.D)
        g = torch.Generator().manual_seed(sub.seed)
        kb = bits(torch.randn(shape, generator=g).to(torch.bfloat16))
        vb = bits(torch.randn(shape, generator=g).to(torch.bfloat16))
        t0 = time.perf_counter()
        oracle.block_attn_fp8(bits(inp["q"]), codes["k_pages"], codes["v_pages"], inp["page_table"].numpy(),
                              inp["ctx_lens"].numpy(), k_scale=0.0431, v_scale=1.73, k_block=kb,
                              v_block=vb, **kw)
        dt = time.perf_counter() - t0
        nbytes = sub.kv_bytes(1)
    else:
        t0 = time.perf_counter()
        oracle.block_attn(bits(inp["q"]), bits(inp["k_pages"]), bits(inp["v_pages"]),
                          inp["page_table"].numpy(), inp["ctx_lens"].numpy(), **kw)
        dt = time.perf_counter() - t0
        nbytes = sub.kv_bytes()
    desc = (f"{len(ids)} of {spec.B} requests (same shapes and lengths), fp64, {threads} threads" +
            (", fp8-context form" if fp8 else ""))
    return nbytes / dt, dt, len(ids), threads, desc


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    spec = workload_spec(args.workload)
    # About 90 s of oracle work for the whole run, at least 1 s per step.
    budget = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    vals, times = [], []
    cores = None
    desc = ""
    for i in range(args.warmup + args.steps):
        v, dt, n, cores, desc = time_oracle_sample(spec, budget_s=budget)
        if i >= args.warmup:
            vals.append(v)
            times.append(dt)
    gbs = sum(vals) / len(vals) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(spec.describe(), parallelism="replicas"),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fused-append", action="store_true",
                    help="time dflash_block_attn_append: the block's K/V append to the pages "
                         "followed by the attention in one launch sequence")
    ap.add_argument("--dense-suffix", action="store_true",
                    help="time dflash_block_attn_dense_suffix: the block's K/V from dense "
                         "tensors, the context from the pages")
    ap.add_argument("--fp8-context", action="store_true",
                    help="time dflash_block_attn_fp8_context: the dense-suffix form over E4M3 "
                         "context pages (the seeded bf16 pages cast to fp8) with per-tensor scales")
    args = ap.parse_args()
    if args.fp8_context:
        args.dense_suffix = True
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import speculative_decoding_draft_paged_gb300 as dflash
    from speculative_decoding_draft_paged_gb300 import build as B
    from speculative_decoding_draft_paged_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.build()

    # Weak scaling: every rank runs the same-sized workload on its own GPU with
    # its own seed; the attention has no cross-request exchange.
    spec = workload_spec(args.workload, seed_offset=100 * rank)
    inp = W.make_inputs(spec, dev)
    p = dflash.params_for(inp["q"], inp["k_pages"], inp["page_table"], block_size=spec.K,
                          window=spec.window, future_keys=spec.future_keys,
                          scale=spec.softmax_scale, max_ctx_len=spec.max_ctx_len,
                          right_window=spec.right_window,
                          kv_dtype=dflash.KV_FP8_E4M3 if args.fp8_context else dflash.KV_BF16)
    plan = dflash.plan(p)
    ws_bytes = dflash.workspace_size(p)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(inp["q"])
    lse = torch.empty(inp["q"].shape[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    if args.fused_append or args.dense_suffix:
        # The block's own K/V rows (already in the pages from the input
        # recipe): re-appending them each call leaves the pools unchanged,
        # and the dense-suffix form reads the same values from these tensors.
        kb = torch.empty((spec.B, spec.K, spec.Hkv, spec.D), dtype=torch.bfloat16, device=dev)
        vb = torch.empty_like(kb)
        tab = inp["page_table"].cpu()
        for b, L in enumerate(spec.ctx_lens):
            for j in range(spec.K):
                pg, off = int(tab[b, (L + j) // spec.P]), (L + j) % spec.P
                kb[b, j] = inp["k_pages"][pg, :, off, :]
                vb[b, j] = inp["v_pages"][pg, :, off, :]

    if args.fp8_context:
        # E4M3 codes of the same seeded values, with per-tensor scales.
        kp8 = inp["k_pages"].float().to(torch.float8_e4m3fn).view(torch.uint8)
        vp8 = inp["v_pages"].float().to(torch.float8_e4m3fn).view(torch.uint8)
        k_scale, v_scale = 0.0431, 1.73

    def call():
        if args.fp8_context:
            rc = dflash.block_attn_fp8_context_raw(
                p, inp["q"].data_ptr(), kb.data_ptr(), vb.data_ptr(), kp8.data_ptr(), vp8.data_ptr(),
                k_scale, v_scale, inp["page_table"].data_ptr(), inp["ctx_lens"].data_ptr(),
                out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws_bytes,
                torch.cuda.current_stream().cuda_stream)
        elif args.dense_suffix:
            rc = dflash.block_attn_dense_suffix_raw(
                p, inp["q"].data_ptr(), kb.data_ptr(), vb.data_ptr(), inp["k_pages"].data_ptr(),
                inp["v_pages"].data_ptr(), inp["page_table"].data_ptr(), inp["ctx_lens"].data_ptr(),
                out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws_bytes,
                torch.cuda.current_stream().cuda_stream)
        elif args.fused_append:
            rc = dflash.block_attn_append_raw(
                p, inp["q"].data_ptr(), kb.data_ptr(), vb.data_ptr(), inp["k_pages"].data_ptr(),
                inp["v_pages"].data_ptr(), inp["page_table"].data_ptr(), inp["ctx_lens"].data_ptr(),
                out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws_bytes,
                torch.cuda.current_stream().cuda_stream)
        else:
            rc = dflash.block_attn_raw(p, inp["q"].data_ptr(), inp["k_pages"].data_ptr(),
                                       inp["v_pages"].data_ptr(), inp["page_table"].data_ptr(),
                                       inp["ctx_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       ws.data_ptr(), ws_bytes,
                                       torch.cuda.current_stream().cuda_stream)
        if rc != 0:
            raise dflash.DflashError(rc)

    # Capture one call in a CUDA graph (the grid depends on the parameters only).
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()

    for _ in range(args.warmup):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize()
    if dflash.read_device_status(ws) != 0:
        raise SystemExit("device status flags set during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        starts[k].record(stream)
        graph.replay()
        ends[k].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    call_ms = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    mean_ms = sum(call_ms) / len(call_ms)
    p90_ms = call_ms[min(len(call_ms) - 1, int(math.ceil(0.9 * len(call_ms))) - 1)]
    ms = call_ms[len(call_ms) // 2] if len(call_ms) % 2 else \
        0.5 * (call_ms[len(call_ms) // 2 - 1] + call_ms[len(call_ms) // 2])

    # Split-kernel duration (the dominant kernel) with events on its stream.
    k_ms, c_ms = [], []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)   # torch creates the CUDA events on first record
    e1.record(stream)
    for k in range(max(3, min(args.steps, 20))):
        flush.fill_(k & 0xFF)
        if args.fp8_context:
            rc = dflash.block_attn_fp8_context_timed_raw(
                p, inp["q"].data_ptr(), kb.data_ptr(), vb.data_ptr(), kp8.data_ptr(), vp8.data_ptr(),
                k_scale, v_scale, inp["page_table"].data_ptr(), inp["ctx_lens"].data_ptr(),
                out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws_bytes, stream.cuda_stream, e0, e1)
        else:
            rc = dflash.block_attn_timed_raw(p, inp["q"].data_ptr(), inp["k_pages"].data_ptr(),
                                             inp["v_pages"].data_ptr(), inp["page_table"].data_ptr(),
                                             inp["ctx_lens"].data_ptr(), out.data_ptr(), lse.data_ptr(),
                                             ws.data_ptr(), ws_bytes, stream.cuda_stream, e0, e1)
        if rc != 0:
            raise dflash.DflashError(rc)
        e2.record(stream)
        e2.synchronize()
        k_ms.append(e0.elapsed_time(e1))
        c_ms.append(e1.elapsed_time(e2))
    # CUDA-event timestamps here come in steps of ~2 us: the interquartile mean
    # of the samples resolves below that step where a median cannot.
    def iq_mean(v):
        v = sorted(v)
        q = len(v) // 4
        mid = v[q:len(v) - q] or v
        return sum(mid) / len(mid)

    split_ms = iq_mean(k_ms)
    combine_ms = iq_mean(c_ms)

    # End to end through the public API: per step, copy q / page table /
    # lengths from pinned host memory, run the call, read out and lse2 back.
    h_q = inp["q"].cpu().pin_memory()
    h_tab = inp["page_table"].cpu().pin_memory()
    h_len = inp["ctx_lens"].cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = h_q.numel() * 2 + h_tab.numel() * 4 + h_len.numel() * 4
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for k in range(args.warmup + args.steps):
        flush.fill_(k & 0xFF)
        if k >= args.warmup:
            ee[k - args.warmup][0].record(stream)
        inp["q"].copy_(h_q, non_blocking=True)
        inp["page_table"].copy_(h_tab, non_blocking=True)
        inp["ctx_lens"].copy_(h_len, non_blocking=True)
        call()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
        if k >= args.warmup:
            ee[k - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in ee) / len(ee)

    # Max over ranks (time) and sum (bytes) for the whole-job figures.
    kv_bytes = spec.kv_bytes(1 if args.fp8_context else 2)
    (ms, mean_ms, p90_ms, split_ms, e2e_ms), total_bytes = reduce_over_ranks(
        [ms, mean_ms, p90_ms, split_ms, e2e_ms], kv_bytes, dev)

    peaks = measured_peaks()
    gbs = total_bytes / (ms * 1e-3) / 1e9
    split_gbs = kv_bytes / (split_ms * 1e-3) / 1e9
    kernel = "split_tc" if plan["path"] == dflash.PATH_TCGEN05 else "split_mma"
    traffic = stored_traffic(spec.name, kernel + ("_fp8" if args.fp8_context else ""))

    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "us_per_call": ms * 1e3,
        "call_us": {"median": ms * 1e3, "mean": mean_ms * 1e3, "p90": p90_ms * 1e3,
                    "samples": args.steps},
        "pct_of_peak_hbm": 100.0 * gbs / world / peaks["hbm_gbs"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": f"synthetic (seeded N(0,{spec.sigma:g}) bf16 pages, random page permutation)",
        "config": dict(spec.describe(), parallelism=f"replicas{world}",
                       l2="flushed before every timed call (512 MiB write)" +
                       ("; K/V larger than L2" if kv_bytes > (129 << 20) else ""),
                       kv_bytes_per_call=kv_bytes, path=kernel, split_tiles=plan["split_tiles"],
                       max_splits=plan["max_splits"], ctas=plan["units"], cuda_graph=True,
                       fused_append=bool(args.fused_append), dense_suffix=bool(args.dense_suffix),
                       fp8_context=bool(args.fp8_context)),
        "roofline": {"bound": "hbm", "achieved": split_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": split_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": kernel, "kernel_us": split_ms * 1e3,
                     "combine_kernel_us": combine_ms * 1e3,
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"
                     if peaks["source"] == "measured" else "fallback 6.8 TB/s"},
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "us_per_call": e2e_ms * 1e3, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        # Per call: [append] + split kernel + combine (tcgen05 path, or several
        # units per request on the mma path).
        "gpu_launches": args.steps * (int(bool(args.fused_append)) + 1 +
                                      int(kernel == "split_tc" or plan["max_splits"] > 1)),
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, n, cores, desc = time_oracle_sample(spec, fp8=bool(args.fp8_context))
        line["cpu_baseline"] = {"value": v / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
