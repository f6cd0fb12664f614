#!/usr/bin/env python
"""Benchmark of attention over a paged KV cache on GB300.

Headline: the 7B-like paged decode step (batch 16, 32 heads x head_dim 128, fp16,
block_size 16, contexts uniform in [1024, 8192], pages shuffled over a pool 1.2x the
pages needed). One step = attend one query per sequence to its whole paged context
(split-KV kernel + merge) and append the new token's K/V. Reported metric: K/V bytes
read per step / step time (GB/s), next to the decode call's roofline fraction.

Secondary lines (in "extra"): the block-size sweep 8..512 (32 x 4096 tokens, fp16),
the mixed serving batch (64 lognormal contexts, GQA 32/8, bf16, fragmented pool) and,
when the prefill kernel is available, the long causal prefill (4 x 8192, bf16, 512-token
chunks, append then attend).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run; every rank is an independent replica with
its own pool (the path has no exchange step), value = sum over ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV-read GB/s (% of HBM peak); prefill attn TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
PROFILES = os.path.join(ROOT, "profiles")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--profile-batch", type=int, default=1,
                    help="prefill / prefill_fp8 profile cases: sequences of the 4 x 8192 prompt set (4 = the bench's occupancy)")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-full", action="store_true",
                    help="time the oracle on every workload in full (the long prefill: minutes), not on bounded "
                         "samples")
    ap.add_argument("--only", default="", help="comma list of extra workloads (bs_sweep,mixed,prefix,fp8,mqa,mixed_call,prefill,prefill_fp8)")
    ap.add_argument("--profile", choices=["decode", "append", "prefill", "decode_mixed", "decode_prefix", "decode_fp8",
                                          "prefill_fp8", "decode_mqa", "prefill_d256", "append_chunk"],
                    default=None,
                    help="small case for ncu captures: W + K launches of one kernel, nothing else timed")
    return ap.parse_args()


def profile_case(args):
    """A few GB at most on the device, a few launches: the case ncu --set full captures."""
    import torch
    from paged_kv_flash_cache_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    if args.profile in ("decode", "append"):
        # 7B-like decode at batch 4: ~0.3 GB of K/V (above L2), same shapes otherwise
        p = W.decode_7b(batch=4, pool_init="none", device="cuda")
        cache = torch.zeros((p.num_blocks, 2, 32, 16, 128), dtype=torch.float16, device="cuda")
        k, v, cu, bt = p.k_ctx.cuda(), p.v_ctx.cuda(), p.cu_ctx_lens.cuda(), p.block_tables.cuda()
        zeros = torch.zeros(p.batch, dtype=torch.int32, device="cuda")
        pkv.kv_cache_append(cache, k, v, cu, zeros, bt)
        q, ctx = p.q.cuda(), p.context_lens.cuda()
        out = torch.empty((p.batch, 32, 128), dtype=torch.float16, device="cuda")
        step = W.append_step(p, seed=7)  # the decode step's token, as the bench's step appends it
        bt_step, k_step, v_step = step["block_tables"].cuda(), step["k_new"].cuda(), step["v_new"].cuda()
        for _ in range(args.warmup + args.steps):
            if args.profile == "decode":
                pkv.paged_attn_decode_step(cache, q, bt_step, ctx, k_step, v_step, scale=p.scale, out=out)
            else:
                pkv.kv_cache_append(cache, k, v, cu, zeros, bt)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    elif args.profile == "decode_mixed":
        # the mixed serving batch itself: 0.62 GB of K/V in a 1.2 GB pool
        p = W.mixed_serving(pool_init="none", device="cuda")
        cache = torch.zeros((p.num_blocks, 2, 8, 32, 128), dtype=torch.bfloat16, device="cuda")
        bt = p.block_tables.cuda()
        pkv.kv_cache_append(cache, p.k_ctx.cuda(), p.v_ctx.cuda(), p.cu_ctx_lens.cuda(),
                            torch.zeros(p.batch, dtype=torch.int32, device="cuda"), bt)
        q, ctx = p.q.cuda(), p.context_lens.cuda()
        out = torch.empty((p.batch, 32, 128), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup + args.steps):
            pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, out=out)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    elif args.profile == "decode_fp8":
        # 7B-like decode at batch 4 on an FP8 cache: 0.2 GB of codes + scales (above L2)
        p = W.decode_7b(batch=4, pool_init="none", device="cuda", kv_format="fp8")
        shape = (p.num_blocks, 2, 32, 16, 128)
        codes = torch.zeros(shape, dtype=torch.uint8, device="cuda")
        scales = torch.zeros(shape[:4], dtype=torch.float32, device="cuda")
        bt = p.block_tables.cuda()
        pkv.kv_cache_append(codes, p.k_ctx, p.v_ctx, p.cu_ctx_lens.cuda(),
                            torch.zeros(p.batch, dtype=torch.int32, device="cuda"), bt, scales=scales)
        q, ctx = p.q.cuda(), p.context_lens.cuda()
        out = torch.empty((p.batch, 32, 128), dtype=torch.float16, device="cuda")
        for _ in range(args.warmup + args.steps):
            pkv.paged_attn_decode(codes, q, bt, ctx, scale=p.scale, out=out, scales=scales)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    elif args.profile == "decode_mqa":
        # the MQA batch itself: 0.30 GB of K/V (above L2)
        p = mqa_problem(torch)
        cache = device_problem(p, torch)
        q, bt, ctx = p.q.cuda(), p.block_tables.cuda(), p.context_lens.cuda()
        out = torch.empty((p.batch, 32, 128), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup + args.steps):
            pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, out=out)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    elif args.profile == "decode_prefix":
        # the shared-prompt decode batch itself: 0.37 GB of unique K/V, 1.38 GB read per call
        p = W.prefix_shared(pool_init="none", device="cuda")
        cache = torch.zeros((p.num_blocks, 2, 32, 16, 128), dtype=torch.float16, device="cuda")
        for ap_ in (W.shared_append(p), W.private_append(p)):
            pkv.kv_cache_append(cache, ap_["k_new"].cuda(), ap_["v_new"].cuda(), ap_["cu_new_lens"].cuda(),
                                ap_["ctx_before"].cuda(), ap_["block_tables"].cuda())
        q, ctx, bt = p.q.cuda(), p.context_lens.cuda(), p.block_tables.cuda()
        out = torch.empty((p.batch, 32, 128), dtype=torch.float16, device="cuda")
        for _ in range(args.warmup + args.steps):
            pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, out=out)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    elif args.profile == "append_chunk":
        # one chunk's append of the long prefill pass: 4 sequences x 512 new tokens, 32 KV heads x 128,
        # bf16 (33.5 MB of K/V in, the same out into their pages)
        p = W.prefill_long(device="cuda")
        shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
        cache = torch.zeros(shape, dtype=p.q.dtype, device="cuda")
        bt = p.block_tables.cuda()
        v = W.prefill_chunk_view(p, 15)
        rows = v["rows"].cuda()
        k, vv = p.k_ctx[rows].contiguous(), p.v_ctx[rows].contiguous()
        cu, before = v["cu_q_lens"].cuda(), v["ctx_before"].cuda()
        for _ in range(args.warmup + args.steps):
            pkv.kv_cache_append(cache, k, vv, cu, before, bt)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    elif args.profile == "prefill_d256":
        # the head_dim 256 prefill of the bench line: 4 x 4096 tokens, 16 query / 8 KV heads, one
        # causal call (0.13 GB of K/V)
        gen = torch.Generator().manual_seed(1256)
        nb = 4 * 4096 // 16
        order = torch.randperm(nb, generator=gen).tolist()
        p = W.make_problem("d256", batch=4, num_q_heads=16, num_kv_heads=8, head_dim=256, block_size=16,
                           context_lens=[4096] * 4, q_lens=[4096] * 4, dtype=W.BF16, causal=True, seed=1257,
                           num_blocks=nb, free_order=order, pool_init="none", device="cuda")
        cache = device_problem(p, torch)
        q, cu, ctx, bt = p.q.cuda(), p.cu_q_lens.cuda(), p.context_lens.cuda(), p.block_tables.cuda()
        for _ in range(args.warmup + args.steps):
            pkv.paged_attn_prefill(cache, q, cu, ctx, bt, max_q_len=4096, scale=p.scale, causal=True)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    else:
        fp8 = args.profile == "prefill_fp8"
        p = W.prefill_long(batch=args.profile_batch, device="cuda")
        shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
        if fp8:
            cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
            scales = torch.zeros(shape[:4], dtype=torch.float32, device="cuda")
        else:
            cache = torch.zeros(shape, dtype=p.q.dtype, device="cuda")
            scales = None
        bt = p.block_tables.cuda()
        pkv.kv_cache_append(cache, p.k_ctx.cuda(), p.v_ctx.cuda(), p.cu_ctx_lens.cuda(),
                            torch.zeros(p.batch, dtype=torch.int32, device="cuda"), bt, scales=scales)
        v = W.prefill_chunk_view(p, 15)
        q = p.q[v["rows"]].cuda()
        cu, ctx = v["cu_q_lens"].cuda(), v["context_lens"].cuda()
        for _ in range(args.warmup + args.steps):
            pkv.paged_attn_prefill(cache, q, cu, ctx, bt, max_q_len=512, scale=p.scale, causal=True, scales=scales)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
    print("profile case done:", args.profile)


# ------------------------------------------------------------------------------------------------
# distributed plumbing (barrier + max of the timing only; no data-path collective)
# ------------------------------------------------------------------------------------------------

class Dist:
    def __init__(self):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.torch = torch
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = self.torch.tensor([x], dtype=self.torch.float64,
                              device="cuda" if self.torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        t = self.torch.tensor([x], dtype=self.torch.float64,
                              device="cuda" if self.torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------------------------------------
# clocks: nvidia-smi sampled in the background, kept for the timed window
# ------------------------------------------------------------------------------------------------

class NvmlClocks:
    """Read-only, in-process NVML (the driver's libnvidia-ml) reads of one GPU's SM clock and its
    clock event reasons, cheap enough to take while timed work is executing. Nothing is set."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        import ctypes
        self.lib = None
        self.samples = []
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(handle)) != 0:
                return
            self.ct, self.lib, self.handle = ctypes, lib, handle
            mx = ctypes.c_uint()
            self.max_mhz = mx.value if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0 else None
            name = "nvmlDeviceGetCurrentClocksEventReasons"
            self.reasons_fn = getattr(lib, name, None) or getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            self.lib = None

    def probe(self):
        if not self.lib:
            return
        ct = self.ct
        mhz, reasons = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(mhz)) == 0 and \
                self.reasons_fn(self.handle, ct.byref(reasons)) == 0:
            self.samples.append((mhz.value, reasons.value))

    def summary(self):
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median([m for m, _ in self.samples]), "sm_max_mhz": self.max_mhz,
                "reasons": sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit}),
                "samples": len(self.samples),
                "window": "timed: in-process NVML reads while the timed steps execute (after half and after all "
                          "of them are enqueued, before the closing synchronize)"}

    def close(self):
        if self.lib:
            self.lib.nvmlShutdown()


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            # timed region shorter than the sampling period: nearest samples around it
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:3]
            inside = [s for _, s in near]
            window = "nearest to timed region (region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        mhz = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if len(s) > 5 + i and s[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------------------------------------
# measured peaks and committed ncu traffic figures
# ------------------------------------------------------------------------------------------------

def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "paged_kv_flash_cache_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(summary_name: str, files) -> float | None:
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on the current source."""
    p = os.path.join(PROFILES, summary_name)
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256_16") != kernel_source_hash(files):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------------------------
# workloads on the device
# ------------------------------------------------------------------------------------------------

def device_problem(p, torch):
    """Move a generated problem to the GPU: pool allocated, context appended by the library."""
    import paged_kv_flash_cache_gb300 as pkv
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    cache = torch.zeros(shape, dtype=p.k_ctx.dtype, device="cuda")
    pkv.kv_cache_append(cache, p.k_ctx.cuda(), p.v_ctx.cuda(), p.cu_ctx_lens.cuda(),
                        torch.zeros(p.batch, dtype=torch.int32, device="cuda"), p.block_tables.cuda())
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    return cache


def decode_bytes(p, appended=False) -> dict:
    """Algorithmic bytes of one decode call: K/V of every cached token once per KV head, q in,
    output out, the block-table entries and context lengths read; with `appended` (a decode step),
    also the new token's K and V rows read and written."""
    kv = p.kv_bytes_read()
    qo = 2 * p.batch * p.num_q_heads * p.head_dim * 2
    pages = sum((int(L) + p.block_size - 1) // p.block_size for L in p.context_lens.tolist())
    table = pages * 4 + p.batch * 4
    app = 2 * 2 * p.batch * p.num_kv_heads * p.head_dim * 2 if appended else 0
    return {"kv": kv, "append": app, "total": kv + qo + table + app}


def time_loop(torch, fn, steps, stream, inner_events=None):
    """K calls of fn between two events on `stream`; returns total ms."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end)


def bench_decode(torch, p, steps, warmup, dist, want_clocks=True):
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    cache = device_problem(p, torch)
    q = p.q.cuda()
    ctx = p.context_lens.cuda()
    step_in = W.append_step(p, seed=7)
    bt = step_in["block_tables"].cuda()
    k_new, v_new = step_in["k_new"].cuda(), step_in["v_new"].cuda()
    mb = bt.shape[1]
    ws_bytes = pkv.decode_workspace_size(p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.block_size, mb)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((p.batch, p.num_q_heads, p.head_dim), dtype=q.dtype, device="cuda")
    stream = torch.cuda.current_stream()

    # one decode step: attend each sequence's context, append its new token at position
    # context_lens[b] (one call: the split kernel writes the new rows, then the merge). The step is
    # that one call, so the call's average duration is the timed loop's time per step; events
    # around each call would also stop each step's first kernel from overlapping the previous
    # step's tail (programmatic dependent launch), which a serving loop does not do.
    def step(i):
        pkv.paged_attn_decode_step(cache, q, bt, ctx, k_new, v_new, scale=p.scale, workspace=ws, out=out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    sampler = ClockSampler(torch.cuda.current_device()) if want_clocks else None
    nvml = NvmlClocks(torch.cuda.current_device()) if want_clocks else None
    if nvml:
        nvml.probe()  # the first read is slow (library set-up): take it before the timed region
        nvml.samples.clear()
    if sampler:
        time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()

    def timed_step(i):
        step(i)
        if nvml and (i == steps // 2 or i == steps - 1):
            nvml.probe()  # the GPU is executing the steps enqueued before this one

    ms = time_loop(torch, timed_step, steps, stream)
    torch.cuda.synchronize()
    t1 = time.time()
    dist.barrier()
    decode_ms = ms / steps  # the step is the one call
    clocks = None
    if sampler:
        time.sleep(0.25)
        sampler.stop()
        clocks = sampler.summary(t0, t1)
        in_region = nvml.summary() if nvml else None
        if in_region:
            # the in-process reads are of the timed region itself; the sampled ones stay beside them
            in_region["nvidia_smi"] = clocks
            clocks = in_region
    if nvml:
        nvml.close()
    assert pkv.get_device_error() == 0
    res = {"ms_total": ms, "ms_per_step": ms / steps, "decode_ms": decode_ms, "clocks": clocks,
           "launches_per_step": 2, "bytes": decode_bytes(p, appended=True)}
    # end to end through the public API: inputs copied from pinned host memory every step, the
    # step's output read back. The step's inputs (q, the new K/V, the tables and lengths) sit in one
    # pinned host buffer, 16-byte aligned pieces, and go to the device in one transfer a step; the
    # call takes device views of its pieces. Copies run on streams of their own (the copy engines),
    # two slots deep: step i's inputs upload while step i - 1 computes, and step i's output is read
    # back while step i + 1 computes. Every step's transfers lie inside the timed region, which
    # ends when the last read-back has landed.
    host_parts = [p.q.cpu(), step_in["k_new"], step_in["v_new"], step_in["block_tables"], p.context_lens]
    offs, total = [], 0
    for t in host_parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 15) // 16 * 16
    h_stage = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(host_parts, offs):
        nb = t.numel() * t.element_size()
        h_stage[o:o + nb].copy_(t.contiguous().flatten().view(torch.uint8))
    d_stage, views = [], []
    for _ in range(2):
        d = torch.empty(total, dtype=torch.uint8, device="cuda")
        d_stage.append(d)
        views.append([d[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                      for t, o in zip(host_parts, offs)])
    outs = [torch.empty_like(out) for _ in range(2)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_parts)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # slot's inputs on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # slot's step computed
    ev_back = [torch.cuda.Event() for _ in range(2)]   # slot's output read back

    def e2e_step(i):
        j = i & 1
        up.wait_event(ev_done[j])       # the slot's previous step has read its inputs
        with torch.cuda.stream(up):
            d_stage[j].copy_(h_stage, non_blocking=True)
        ev_in[j].record(up)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_back[j])   # the slot's previous output has been read back
        d_q, d_k, d_v, d_bt, d_ctx = views[j]
        pkv.paged_attn_decode_step(cache, d_q, d_bt, d_ctx, d_k, d_v, scale=p.scale, workspace=ws, out=outs[j])
        ev_done[j].record(stream)
        down.wait_event(ev_done[j])
        with torch.cuda.stream(down):
            h_outs[j].copy_(outs[j], non_blocking=True)
        ev_back[j].record(down)

    def e2e_loop(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        up.wait_stream(stream)
        down.wait_stream(stream)
        for i in range(n):
            e2e_step(i)
        stream.wait_stream(down)
        stream.wait_stream(up)
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end)

    e2e_loop(max(warmup, 1))
    torch.cuda.synchronize()
    # the same inputs as the device-resident steps: the read-back output is theirs, bit for bit
    assert torch.equal(h_outs[(max(warmup, 1) - 1) & 1], out.cpu()), "end-to-end step output differs"
    dist.barrier()
    e2e_ms = e2e_loop(steps)
    torch.cuda.synchronize()
    dist.barrier()
    assert pkv.get_device_error() == 0
    res.update(e2e_ms_per_step=e2e_ms / steps, h2d=h2d, d2h=d2h)
    del cache
    torch.cuda.empty_cache()
    return res


def cpu_baseline_decode(p, budget_s=8.0):
    """The oracle as it stands, all host cores, on the same decode workload (whole batch,
    repeated until `budget_s` of wall time is spent)."""
    import oracle
    oracle.build()
    t_build = time.time()
    cache = oracle.build_cache(p)
    t_build = time.time() - t_build
    cores = os.cpu_count() or 1
    reps, t = 0, 0.0
    while t < budget_s and reps < 50:
        t0 = time.time()
        oracle.attention_of(p, cache, nthreads=cores)
        t += time.time() - t0
        reps += 1
    gbs = p.kv_bytes_read() * reps / t / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "whole decode batch (%d sequences x %d heads, %d cached tokens), %d repetition(s), %.1f s; "
                      "fp64 token walk + two-pass softmax; cache build %.1f s not timed"
                      % (p.batch, p.num_q_heads, int(p.context_lens.sum()), reps, t, t_build)}


def cpu_model() -> str:
    """The host CPU's name as the OS reports it."""
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":", 1)[0].strip().lower()
            if key in ("model name", "cpu model", "hardware"):
                return line.split(":", 1)[1].strip()
        # Arm: no model name line; the part number identifies the core
        parts = {line.split(":", 1)[1].strip() for line in open("/proc/cpuinfo") if line.startswith("CPU part")}
        impl = {line.split(":", 1)[1].strip() for line in open("/proc/cpuinfo") if line.startswith("CPU implementer")}
        if parts:
            names = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd0c": "Neoverse N1", "0xd49": "Neoverse N2",
                     "0xd8e": "Neoverse N3", "0xd83": "Neoverse V3"}
            known = ", ".join(sorted({names[p] for p in parts if p in names}))
            return "Arm %s(implementer %s, part %s)" % (known + " " if known else "", ",".join(sorted(impl)),
                                                         ",".join(sorted(parts)))
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_seconds(fn, budget_s):
    """Seconds per call of fn: repeated until budget_s of wall time (at least once)."""
    reps, t = 0, 0.0
    while reps == 0 or (t < budget_s and reps < 20):
        t0 = time.time()
        fn()
        t += time.time() - t0
        reps += 1
    return t / reps, reps


def cpu_baseline_breadth(torch, p7b, full=False, budget_s=2.5):
    """The oracle as it stands, at one thread and at all host cores, on the workloads of the GPU
    lines (same generators and seeds). Decode workloads run in full; the long prefill (2.2 TFLOP in
    fp64) on a seeded sample of its query rows: 1/16 at all cores and 1/256 at one thread, or with
    full all rows and 1/16 (about a minute each on 16 cores). Returns {workload: {threads: {...}}};
    values in the GPU line's unit."""
    import numpy as np

    import oracle
    from paged_kv_flash_cache_gb300 import workloads as W
    oracle.build()
    cores = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    res = {}

    def decode_case(name, p, note):
        cache = oracle.build_cache(p)
        ent = {}
        for thr in (1, cores):
            sec, reps = oracle_seconds(lambda: oracle.attention_of(p, cache, nthreads=thr), budget_s)
            ent["%d_thread%s" % (thr, "" if thr == 1 else "s")] = {
                "value": round(p.kv_bytes_read() / sec / 1e9, 3), "unit": "GB/s of K/V", "threads": thr,
                "seconds_per_call": round(sec, 3), "calls": reps, "sample": "whole batch: " + note}
        del cache
        res[name] = ent

    dec, pre = W.tiny()
    decode_case("tiny_decode", dec, "2 sequences (37, 100 tokens), 4 heads x 64, fp16, bs 16")
    decode_case("decode_7b", p7b, "16 sequences U[1024, 8192], 32 heads x 128, fp16, bs 16")
    decode_case("bs_sweep_16", W.bs_sweep(16, kv_data=W.bs_sweep_kv(device=dev), pool_init="none", device=dev),
                "32 x 4096 tokens, 32 heads x 128, fp16, bs 16 (one page size of the sweep)")
    decode_case("mixed", W.mixed_serving(pool_init="none", device=dev),
                "64 lognormal contexts, 32 q / 8 kv heads x 128, bf16, bs 32")
    # long causal prefill: TFLOP/s over the sampled rows (4 D Hq per row and key it sees)
    p = W.prefill_long(device=dev)
    cache = oracle.build_cache(p)
    total_rows = int(p.q_lens.sum())
    gen = np.random.default_rng(3)
    ent = {}
    for thr, frac in ((cores, 1 if full else 16), (1, 16 if full else 256)):
        rows = np.sort(gen.choice(total_rows, total_rows // frac, replace=False))
        pos = rows % 8192                              # absolute position: row r sees keys 0 .. pos
        flops = float(np.sum(pos + 1)) * 4 * p.head_dim * p.num_q_heads
        sec, reps = oracle_seconds(
            lambda: oracle.paged_attention(p.dtype, cache, p.q, p.num_q_heads, p.cu_q_lens, p.context_lens,
                                           p.block_tables, p.scale, True, rows=rows, nthreads=thr), 0.0)
        ent["%d_thread%s" % (thr, "" if thr == 1 else "s")] = {
            "value": round(flops / sec / 1e12, 6), "unit": "TFLOP/s (causal)", "threads": thr,
            "seconds_per_call": round(sec, 3), "calls": reps,
            "sample": "%s of the 4 x 8192 query rows (%d rows, seeded), all 32 heads, bf16, bs 16 pages"
                      % ("all" if frac == 1 else "1/%d" % frac, rows.size)}
    del cache
    res["prefill_long"] = ent
    return res


def bench_bs_sweep(torch, steps, warmup):
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    kv = W.bs_sweep_kv(device="cuda")
    out = {}
    pk = peaks()
    for bs in (8, 16, 32, 64, 128, 512):
        p = W.bs_sweep(bs, kv_data=kv, pool_init="none", device="cuda")
        cache = device_problem(p, torch)
        q, bt, ctx = p.q.cuda(), p.block_tables.cuda(), p.context_lens.cuda()
        ws = torch.empty(max(16, pkv.decode_workspace_size(p.batch, 32, 32, 128, bs, bt.shape[1])),
                         dtype=torch.uint8, device="cuda")
        o = torch.empty((p.batch, 32, 128), dtype=q.dtype, device="cuda")
        fn = lambda i: pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, workspace=ws, out=o)
        for i in range(warmup):
            fn(i)
        ms = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
        b = decode_bytes(p)
        out[str(bs)] = {"ms": round(ms, 4), "kv_gbs": round(b["kv"] / ms / 1e6, 1),
                        "frac_of_hbm": round(b["total"] / ms / 1e6 / pk["hbm_gbs"], 3)}
        del cache
        torch.cuda.empty_cache()
    vals = [out[k]["kv_gbs"] for k in ("16", "32", "64", "128")]
    return {"workload": "32 seqs x 4096 ctx, 32 heads x 128, fp16, identical K/V data per block size, "
                        "pool = pages needed, randomly permuted", "per_block_size": out,
            "flatness_16_128": round(min(vals) / max(vals), 3)}


def bench_mixed(torch, steps, warmup):
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    p = W.mixed_serving(pool_init="none", device="cuda")
    cache = device_problem(p, torch)
    q, bt, ctx = p.q.cuda(), p.block_tables.cuda(), p.context_lens.cuda()
    ws = torch.empty(max(16, pkv.decode_workspace_size(p.batch, 32, 8, 128, 32, bt.shape[1])), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((p.batch, 32, 128), dtype=q.dtype, device="cuda")
    fn = lambda i: pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, workspace=ws, out=o)
    for i in range(warmup):
        fn(i)
    ms = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
    b = decode_bytes(p)
    del cache
    torch.cuda.empty_cache()
    return {"workload": "64 seqs, lognormal ctx (median 2048, sigma 1, [16, 32768]), GQA 32/8, 128, bf16, "
                        "bs 32, fragmented pool 2x", "total_ctx_tokens": int(p.context_lens.sum()),
            "ms": round(ms, 4), "kv_gbs": round(b["kv"] / ms / 1e6, 1),
            "frac_of_hbm": round(b["total"] / ms / 1e6 / peaks()["hbm_gbs"], 3),
            "tokens_per_s": round(p.batch / ms * 1e3, 1)}


def bench_prefix(torch, steps, warmup):
    """Decode over a batch whose block tables share a cached prompt's pages (prefix caching),
    against the same contexts with private copies of those pages."""
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    p = W.prefix_shared(pool_init="none", device="cuda")
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    cache = torch.zeros(shape, dtype=p.k_ctx.dtype, device="cuda")
    for a in (W.shared_append(p), W.private_append(p)):
        pkv.kv_cache_append(cache, a["k_new"].cuda(), a["v_new"].cuda(), a["cu_new_lens"].cuda(),
                            a["ctx_before"].cuda(), a["block_tables"].cuda())
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    lens = p.context_lens.tolist()
    flat = W.make_problem("prefix_unshared", batch=p.batch, num_q_heads=32, num_kv_heads=32, head_dim=128,
                          block_size=16, context_lens=lens, q_lens=[1] * p.batch, dtype=p.dtype, causal=False,
                          seed=5, pool_init="none", kv_data=(p.k_ctx, p.v_ctx), device="cuda")
    res = {}
    for name, prob, c in (("shared", p, cache), ("unshared", flat, None)):
        if c is None:
            c = device_problem(prob, torch)
        q, bt, ctx = p.q.cuda(), prob.block_tables.cuda(), prob.context_lens.cuda()
        ws = torch.empty(max(16, pkv.decode_workspace_size(p.batch, 32, 32, 128, 16, bt.shape[1])),
                         dtype=torch.uint8, device="cuda")
        o = torch.empty((p.batch, 32, 128), dtype=q.dtype, device="cuda")
        fn = lambda i: pkv.paged_attn_decode(c, q, bt, ctx, scale=p.scale, workspace=ws, out=o)
        for i in range(warmup):
            fn(i)
        res[name] = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
        del c
    del cache
    torch.cuda.empty_cache()
    logical = p.kv_bytes_read()
    s_tok = p.meta["shared_tokens"]
    unique = (s_tok + sum(L - s_tok for L in lens)) * p.num_kv_heads * p.head_dim * 2 * 2
    ms = res["shared"]
    return {"workload": "16 requests sharing a 4096-token prompt (256 shared pages of 16) + 256..2048 own tokens "
                        "each, 32 heads x 128, fp16; decode; same contexts with private pages for comparison",
            "ms": round(ms, 4), "unshared_ms": round(res["unshared"], 4),
            "logical_kv_gbs": round(logical / ms / 1e6, 1), "unique_kv_bytes": unique, "logical_kv_bytes": logical,
            "unique_kv_gbs": round(unique / ms / 1e6, 1),
            "unshared_frac_of_hbm": round(decode_bytes(flat)["total"] / res["unshared"] / 1e6 / peaks()["hbm_gbs"], 3),
            "tokens_per_s": round(p.batch / ms * 1e3, 1)}


def bench_fp8(torch, steps, warmup, fp16_ms=None):
    """The 7B-like decode batch with the cache in FP8 (E4M3 codes + one FP32 scale per row)."""
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    p = W.decode_7b(pool_init="none", device="cuda", kv_format="fp8")
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    codes = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(shape[:4], dtype=torch.float32, device="cuda")
    pkv.kv_cache_append(codes, p.k_ctx, p.v_ctx, p.cu_ctx_lens.cuda(), torch.zeros(p.batch, dtype=torch.int32,
                        device="cuda"), p.block_tables.cuda(), scales=scales)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    q, bt, ctx = p.q.cuda(), p.block_tables.cuda(), p.context_lens.cuda()
    ws = torch.empty(max(16, pkv.decode_workspace_size(p.batch, 32, 32, 128, 16, bt.shape[1])), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((p.batch, 32, 128), dtype=q.dtype, device="cuda")
    fn = lambda i: pkv.paged_attn_decode(codes, q, bt, ctx, scale=p.scale, workspace=ws, out=o, scales=scales)
    for i in range(warmup):
        fn(i)
    ms = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
    tokens = int(p.context_lens.sum())
    kv = tokens * p.num_kv_heads * 2 * (p.head_dim + 4)          # codes + one FP32 scale per row
    qo = 2 * p.batch * p.num_q_heads * p.head_dim * 2
    table = sum((int(L) + 15) // 16 for L in p.context_lens.tolist()) * 4 + p.batch * 4
    del codes, scales
    torch.cuda.empty_cache()
    r = {"workload": "7B-like decode batch (16 x U[1024, 8192] contexts, 32 heads x 128, bs 16) with an FP8 "
                     "E4M3 cache, one FP32 scale per (page, K/V, head, token) row; fp16 q and output",
         "ms": round(ms, 4), "kv_bytes": kv, "kv_gbs": round(kv / ms / 1e6, 1),
         "frac_of_hbm": round((kv + qo + table) / ms / 1e6 / peaks()["hbm_gbs"], 3),
         "tokens_per_s": round(p.batch / ms * 1e3, 1)}
    if fp16_ms:
        r["speedup_vs_fp16_cache"] = round(fp16_ms / ms, 3)
    return r


def mqa_problem(torch):
    """128 sequences, contexts U[1024, 8192], 32 query heads sharing one KV head of 128, bf16, bs 16:
    0.30 GB of K/V in a pool of exactly the pages needed, shuffled."""
    from paged_kv_flash_cache_gb300 import workloads as W
    gen = torch.Generator().manual_seed(1241)
    lens = torch.randint(1024, 8193, (128,), generator=gen).tolist()
    nb = sum((L + 15) // 16 for L in lens)
    order = torch.randperm(nb, generator=gen).tolist()
    return W.make_problem("mqa", batch=128, num_q_heads=32, num_kv_heads=1, head_dim=128, block_size=16,
                          context_lens=lens, q_lens=[1] * 128, dtype=W.BF16, causal=False, seed=1242, num_blocks=nb,
                          free_order=order, pool_init="none", device="cuda")


def bench_mqa(torch, steps, warmup):
    """Multi-query decode: 128 sequences, 32 query heads sharing one KV head."""
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    p = mqa_problem(torch)
    cache = device_problem(p, torch)
    q, bt, ctx = p.q.cuda(), p.block_tables.cuda(), p.context_lens.cuda()
    ws = torch.empty(max(16, pkv.decode_workspace_size(p.batch, 32, 1, 128, 16, bt.shape[1])), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((p.batch, 32, 128), dtype=q.dtype, device="cuda")
    fn = lambda i: pkv.paged_attn_decode(cache, q, bt, ctx, scale=p.scale, workspace=ws, out=o)
    for i in range(warmup):
        fn(i)
    ms = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
    b = decode_bytes(p)
    del cache
    torch.cuda.empty_cache()
    return {"workload": "MQA decode: 128 seqs, contexts U[1024, 8192], 32 query heads / 1 KV head x 128, bf16, "
                        "bs 16 (the 32 query heads are one tensor-core unit over the shared pages)",
            "ms": round(ms, 4), "kv_gbs": round(b["kv"] / ms / 1e6, 1),
            "frac_of_hbm": round(b["total"] / ms / 1e6 / peaks()["hbm_gbs"], 3),
            "tokens_per_s": round(p.batch / ms * 1e3, 1)}


def bench_head_dim_256(torch, steps, warmup):
    """head_dim 256: a causal prefill of 4 prompts x 4096 tokens (16 query heads on 8 KV heads, bf16,
    bs 16) as one call, and the decode of a token per sequence over the same 4 x 4096 context with
    the same heads (the tcgen05 decode, units of 2 query heads)."""
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    gen = torch.Generator().manual_seed(1256)
    lens = [4096] * 4
    nb = sum((L + 15) // 16 for L in lens)
    order = torch.randperm(nb, generator=gen).tolist()
    p = W.make_problem("d256", batch=4, num_q_heads=16, num_kv_heads=8, head_dim=256, block_size=16,
                       context_lens=lens, q_lens=lens, dtype=W.BF16, causal=True, seed=1257, num_blocks=nb,
                       free_order=order, pool_init="none", device="cuda")
    cache = device_problem(p, torch)
    q, cu, ctx, bt = p.q.cuda(), p.cu_q_lens.cuda(), p.context_lens.cuda(), p.block_tables.cuda()
    out = torch.empty_like(q)
    fn = lambda i: pkv.paged_attn_prefill(cache, q, cu, ctx, bt, max_q_len=4096, scale=p.scale, causal=True,
                                          out=out)
    for i in range(warmup):
        fn(i)
    ms = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
    flops = p.causal_flops()
    # decode: the last token of each prompt against its whole context
    qd = q[cu[1:].long() - 1].contiguous()
    od = torch.empty_like(qd)
    ws = torch.empty(max(16, pkv.decode_workspace_size(4, 16, 8, 256, 16, bt.shape[1])), dtype=torch.uint8,
                     device="cuda")
    fd = lambda i: pkv.paged_attn_decode(cache, qd, bt, ctx, scale=p.scale, workspace=ws, out=od)
    for i in range(warmup):
        fd(i)
    ms_d = time_loop(torch, fd, steps, torch.cuda.current_stream()) / steps
    kv = 4 * 4096 * 8 * 256 * 2 * 2
    pk = peaks()
    del cache
    torch.cuda.empty_cache()
    return {"workload": "head_dim 256, bf16, bs 16, 16 query heads on 8 KV heads, 4 x 4096 tokens",
            "prefill": {"ms": round(ms, 3), "tflops": round(flops / ms / 1e9, 1),
                        "frac_of_dense_bf16": round(flops / ms / 1e9 / pk["bf16_tflops"], 3),
                        "kernel": "prefill_wide_kernel (causal, one call)"},
            "decode": {"ms": round(ms_d, 4), "kv_gbs": round(kv / ms_d / 1e6, 1),
                       "frac_of_hbm": round(kv / ms_d / 1e6 / pk["hbm_gbs"], 3),
                       "kernel": "decode_tc_kernel<256> + combine"}}


def bench_mixed_call(torch, steps, warmup):
    """One paged_attn_mixed call over 64 decode sequences and 4 prefill chunks, against the same
    work as a decode call plus a prefill call."""
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    gen = torch.Generator().manual_seed(1243)
    dec_lens = torch.randint(1024, 8193, (64,), generator=gen).tolist()
    chunk_lens = [2048, 4096, 6144, 8192]
    lens = dec_lens + chunk_lens
    q_lens = [1] * 64 + [512] * 4
    nb = sum((L + 15) // 16 for L in lens)
    order = torch.randperm(nb, generator=gen).tolist()
    p = W.make_problem("mixed_call", batch=len(lens), num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
                       context_lens=lens, q_lens=q_lens, dtype=W.BF16, causal=True, seed=1244, num_blocks=nb,
                       free_order=order, pool_init="none", device="cuda")
    cache = device_problem(p, torch)
    q, bt, ctx, cu = p.q.cuda(), p.block_tables.cuda(), p.context_lens.cuda(), p.cu_q_lens.cuda()
    ws = torch.empty(max(16, pkv.decode_workspace_size(p.batch, 32, 32, 128, 16, bt.shape[1])), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(q)
    mixed = lambda i: pkv.paged_attn_mixed(cache, q, cu, ctx, bt, max_q_len=512, scale=p.scale, workspace=ws, out=out)
    qd, qp = q[:64].contiguous(), q[64:].contiguous()
    bt_d, bt_p = bt[:64].contiguous(), bt[64:].contiguous()
    ctx_d, ctx_p = ctx[:64].contiguous(), ctx[64:].contiguous()
    cu_p = torch.tensor([0, 512, 1024, 1536, 2048], dtype=torch.int32, device="cuda")
    od, op = torch.empty_like(qd), torch.empty_like(qp)
    ws_d = torch.empty(max(16, pkv.decode_workspace_size(64, 32, 32, 128, 16, bt.shape[1])), dtype=torch.uint8,
                       device="cuda")

    def separate(i):
        pkv.paged_attn_decode(cache, qd, bt_d, ctx_d, scale=p.scale, workspace=ws_d, out=od)
        pkv.paged_attn_prefill(cache, qp, cu_p, ctx_p, bt_p, max_q_len=512, scale=p.scale, causal=True, out=op)

    res = {}
    for name, fn in (("mixed", mixed), ("separate", separate)):
        for i in range(warmup):
            fn(i)
        res[name] = time_loop(torch, fn, steps, torch.cuda.current_stream()) / steps
    kv_dec = sum(dec_lens) * 32 * 128 * 2 * 2
    flops = 4 * 128 * 32 * (sum(dec_lens) + sum(512 * (L - 512) + 512 * 513 // 2 for L in chunk_lens))
    del cache
    torch.cuda.empty_cache()
    return {"workload": "one call: 64 decode sequences (contexts U[1024, 8192]) + 4 prefill chunks of 512 "
                        "(contexts 2k-8k), 32 heads x 128, bf16, bs 16",
            "ms": round(res["mixed"], 4), "separate_calls_ms": round(res["separate"], 4),
            "decode_kv_bytes": kv_dec, "flops": flops, "tflops": round(flops / res["mixed"] / 1e9, 1),
            "rows_per_s": round((64 + 2048) / res["mixed"] * 1e3, 1)}


def bench_prefill(torch, steps, warmup, fp8=False):
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    p = W.prefill_long(device="cuda")
    shape = (p.num_blocks, 2, p.num_kv_heads, p.block_size, p.head_dim)
    if fp8:  # the same prompt tokens quantised into an FP8 cache (codes + one FP32 scale per row)
        cache = torch.zeros(shape, dtype=torch.uint8, device="cuda")
        scales = torch.zeros(shape[:4], dtype=torch.float32, device="cuda")
    else:
        cache = torch.zeros(shape, dtype=p.q.dtype, device="cuda")
        scales = None
    bt = p.block_tables.cuda()
    chunks = []
    for c in range(8192 // p.meta["chunk"]):
        v = W.prefill_chunk_view(p, c)
        rows = v["rows"].cuda()
        chunks.append(dict(q=p.q[rows].contiguous(), k=p.k_ctx[rows].contiguous(), v=p.v_ctx[rows].contiguous(),
                           cu=v["cu_q_lens"].cuda(), ctx=v["context_lens"].cuda(), before=v["ctx_before"].cuda(),
                           out=torch.empty_like(p.q[rows]), ql=int(v["q_lens"][0])))

    n_chunks = len(chunks)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_chunks)]
    stream = torch.cuda.current_stream()

    def step(i, timed=False):
        for c, ch in enumerate(chunks):
            if timed:
                ev[c][0].record(stream)
            pkv.kv_cache_append(cache, ch["k"], ch["v"], ch["cu"], ch["before"], bt, scales=scales)
            if timed:
                ev[c][1].record(stream)
            pkv.paged_attn_prefill(cache, ch["q"], ch["cu"], ch["ctx"], bt, max_q_len=ch["ql"], scale=p.scale,
                                   causal=True, out=ch["out"], scales=scales)
            if timed:
                ev[c][2].record(stream)

    step(0)
    torch.cuda.synchronize()
    for i in range(warmup):
        step(i)
    # whole passes back to back (no events between the calls, so launches overlap as in use)
    ms = time_loop(torch, step, steps, stream) / steps
    # the same passes with an event around every call: splits appends from attention
    app_ms = attn_ms = 0.0
    for i in range(steps):
        time_loop(torch, lambda k: step(k, True), 1, stream)
        app_ms += sum(e[0].elapsed_time(e[1]) for e in ev)
        attn_ms += sum(e[1].elapsed_time(e[2]) for e in ev)
    app_ms, attn_ms = app_ms / steps, attn_ms / steps
    flops = p.causal_flops()
    # append moves every prompt token's K and V row-set once in, once out (FP8: out as codes + scales)
    rows_kv = 2 * p.batch * 8192 * p.num_kv_heads
    app_bytes = rows_kv * p.head_dim * 2 + (rows_kv * (p.head_dim + 4) if fp8 else rows_kv * p.head_dim * 2)
    pk = peaks()
    del cache, scales
    torch.cuda.empty_cache()
    return {"workload": "4 x 8192 causal prefill, 32 heads x 128, bf16, bs 16 pages, 16 chunks of 512 "
                        "(append chunk, then attend)" + ("; FP8 E4M3 cache, products in f16" if fp8 else ""),
            "ms_per_pass": round(ms, 3),
            "tflops": round(flops / ms / 1e9, 1), "frac_of_dense_bf16": round(flops / ms / 1e9 / pk["bf16_tflops"], 3),
            "attention_only": {"ms": round(attn_ms, 3), "tflops": round(flops / attn_ms / 1e9, 1),
                               "frac_of_dense_bf16": round(flops / attn_ms / 1e9 / pk["bf16_tflops"], 3),
                               "kernel": "prefill_kernel, 16 launches per pass", "launches": n_chunks},
            "append": {"ms": round(app_ms, 3), "gbs": round(app_bytes / app_ms / 1e6, 1),
                       "frac_of_hbm": round(app_bytes / app_ms / 1e6 / pk["hbm_gbs"], 3),
                       "bytes": app_bytes, "launches": n_chunks},
            "causal_flops": flops, "prompt_tokens_per_s": round(4 * 8192 / ms * 1e3, 1)}


# ------------------------------------------------------------------------------------------------

def main():
    args = parse()
    if args.profile:
        profile_case(args)
        return
    import torch
    dist = Dist()
    workload_cfg = {"workload": "7B-like paged decode step: batch 16, 32 heads x head_dim 128, fp16, block_size 16, "
                                "contexts uniform in [1024, 8192] (seeded), pages shuffled over a pool 1.2x the "
                                "pages needed",
                    "step": "paged_attn_decode_step: attention over each context (split-KV kernel, whose merge "
                            "warps also append the step's new token at position context_lens[b], 16 tokens) + "
                            "merge kernel",
                    "l2": "inputs larger than L2: %.2f GB of K/V read per step vs 129 MB L2" % 0,
                    "parallelism": "replicas" if args.gpus > 1 else "single GPU"}
    if args.impl == "reference":
        # The oracle is the reference arm: rank 0 only, on the host cores.
        if dist.rank != 0:
            dist.close()
            return
        from paged_kv_flash_cache_gb300 import workloads as W
        p = W.decode_7b(pool_init="none", device="cuda" if torch.cuda.is_available() else "cpu")
        workload_cfg["l2"] = "n/a (CPU)"
        import oracle
        oracle.build()
        cache = oracle.build_cache(p)
        cores = os.cpu_count() or 1
        for _ in range(args.warmup):
            oracle.attention_of(p, cache, nthreads=cores)
        t0 = time.time()
        for _ in range(args.steps):
            oracle.attention_of(p, cache, nthreads=cores)
        dt = (time.time() - t0) / args.steps
        v = p.kv_bytes_read() / dt / 1e9
        line = {"metric": METRIC, "value": round(v, 3), "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload_cfg,
                "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": "whole decode batch per step (16 seqs x 32 heads, %d cached tokens)"
                                           % int(p.context_lens.sum())},
                "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        dist.close()
        return

    from paged_kv_flash_cache_gb300 import build as pkv_build
    pkv_build.build()
    import paged_kv_flash_cache_gb300 as pkv
    from paged_kv_flash_cache_gb300 import workloads as W
    torch.cuda.set_device(dist.local)
    pk = peaks()
    p = W.decode_7b(seed=1236 + 100 * dist.rank, pool_init="none", device="cuda")
    r = bench_decode(torch, p, args.steps, args.warmup, dist)
    kv_gb = r["bytes"]["kv"] / 1e9
    workload_cfg["l2"] = "inputs larger than L2: %.2f GB of K/V read per step vs 129 MB L2" % kv_gb
    ms = dist.max(r["ms_per_step"])
    total_kv = dist.sum(r["bytes"]["kv"])
    value = total_kv / (ms * 1e-3) / 1e9
    e2e_ms = dist.max(r["e2e_ms_per_step"])
    achieved = r["bytes"]["total"] / (r["decode_ms"] * 1e-3) / 1e9
    files = ["decode.cu", "decode_common.cuh", "pkv_device.cuh", "pkv_internal.h"]
    roofline = {"bound": "hbm", "kernel": "paged_attn_decode_step call (decode_split_kernel, which also writes the "
                "step's new K/V rows, + combine_kernel)",
                "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 3), "peak_source": pk["source"],
                "traffic": ncu_traffic("decode_split_7b_ncu.txt", files),
                "traffic_of": "decode_split_kernel (ncu, scaled from a batch-4 capture by cached tokens)",
                "algorithmic_bytes_per_launch": r["bytes"]["total"], "avg_launch_ms": round(r["decode_ms"], 4)}
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": workload_cfg,
            "roofline": roofline,
            "e2e": {"value": round(total_kv / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": r["launches_per_step"] * args.steps, "clocks": r["clocks"],
            "tokens_per_s": round(args.gpus * p.batch / (ms * 1e-3), 1)}
    if dist.rank == 0 and not args.no_extra:
        extra = {}
        only = set(filter(None, args.only.split(",")))
        for name, fn in (("bs_sweep", bench_bs_sweep), ("mixed", bench_mixed), ("prefix", bench_prefix),
                         ("fp8", lambda t, k, w: bench_fp8(t, k, w, r["decode_ms"])), ("mqa", bench_mqa),
                         ("mixed_call", bench_mixed_call), ("head_dim_256", bench_head_dim_256),
                         ("prefill", bench_prefill),
                         ("prefill_fp8", lambda t, k, w: bench_prefill(t, k, w, fp8=True))):
            if only and name not in only:
                continue
            try:
                extra[name] = fn(torch, max(3, args.steps // 4), 3)
            except Exception as e:  # a secondary workload must not hide the headline line
                extra[name] = {"error": "%s: %s" % (type(e).__name__, str(e)[:200])}
        line["extra"] = extra
    if dist.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(p)
        line["cpu_baseline"]["cpu_model"] = cpu_model()
        try:
            breadth = cpu_baseline_breadth(torch, p, full=args.cpu_full)
            line["cpu_baseline"]["by_workload"] = breadth
            # beside each GPU line: the oracle on the same workload
            for name, key in (("bs_sweep", "bs_sweep_16"), ("mixed", "mixed"), ("prefill", "prefill_long")):
                if isinstance(line.get("extra", {}).get(name), dict) and key in breadth:
                    line["extra"][name]["oracle"] = breadth[key]
        except Exception as e:  # the baseline's breadth must not hide the headline line
            line["cpu_baseline"]["by_workload"] = {"error": "%s: %s" % (type(e).__name__, str(e)[:200])}
    if dist.rank == 0:
        print(json.dumps(line))
    dist.close()


if __name__ == "__main__":
    main()
