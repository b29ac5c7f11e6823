#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on GB300.

One decode step of the long-context workload (write the new token of every
sequence through slot_mapping, then paged decode with split-KV over 16K-40K
cached keys; batch 8, GQA 16/8, head_dim 128, block 256, bf16) is the headline
(decode KV GB/s); the same run also measures one chunked-prefill step of the
varlen workload (write 16 requests' new tokens, then causal varlen prefill over
cached + new keys; TFLOP/s of the visible query-key pairs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  With torchrun (N > 1) every rank runs its own replica of
the workload on its own GPU (no collective on the data path; "replicas only"),
and timing is the max over ranks.  ``--impl reference`` times the CPU oracle (the
reference arm of this build) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s & % HBM peak; varlen prefill TFLOP/s & % bf16 peak"
DECODE_CFG, PREFILL_CFG = 3, 4


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", choices=["all", "decode", "prefill", "copy", "shared", "mixed"],
                   default="all",
                   help="measure one half only (profiling runs)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# algorithmic work of the workloads
# ---------------------------------------------------------------------------
def decode_kernel_bytes(step) -> int:
    """Bytes paged_decode must move: K and V of every visible key, q, out,
    the block-table entries of every page touched, and cache_seqlens."""
    L = step.cache_seqlens.astype(np.int64)
    kv = int(L.sum()) * step.kv_dim * step.elt * 2
    qo = 2 * step.n_decode * step.hq * step.d * step.elt
    table = int(np.sum(-(-L // step.block_size))) * 4
    return kv + qo + table + step.n_decode * 4


def write_bytes(step) -> int:
    """slot_mapping build (token_seq, token_pos read, slot written) and the
    K/V rows of every non-padding token read and written once."""
    n_rows = len(step.token_seq)
    n_real = int((step.token_seq >= 0).sum())
    return n_rows * 12 + n_real * 4 + n_real * step.kv_dim * step.elt * 2 * 2 + n_rows * 4


def prefill_pairs(step) -> int:
    q = np.diff(step.cu_q).astype(np.int64)
    k = np.diff(step.cu_k).astype(np.int64)
    tot = 0
    for qq, kk in zip(q, k):
        i = np.arange(qq)
        tot += int(np.clip(i + kk - qq + 1, 0, kk).sum()) if step.causal else int(qq * kk)
    return tot


def prefill_flops(step) -> int:
    return 4 * step.d * step.hq * prefill_pairs(step)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# device-side workload
# ---------------------------------------------------------------------------
def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pinned(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory()


class DeviceStep:
    """Device-resident copy of a synthetic step and the calls of one pass."""

    def __init__(self, step, pkv):
        self.s, self.pkv = step, pkv
        self.table = to_dev(step.table)
        self.k_cache = to_dev(step.k_cache)
        self.v_cache = to_dev(step.v_cache)
        self.new_k, self.new_v = to_dev(step.new_k), to_dev(step.new_v)
        self.token_seq, self.token_pos = to_dev(step.token_seq), to_dev(step.token_pos)
        self.slots = torch.empty(len(step.token_seq), dtype=torch.int32, device="cuda")
        if step.n_decode:
            self.q = to_dev(step.q_decode)
            self.seqlens = to_dev(step.cache_seqlens)
            self.dtable = self.table[: step.n_decode].contiguous()
            self.out = torch.empty_like(self.q)
            self.ws = torch.empty(max(1, pkv.paged_decode_workspace_size(
                step.n_decode, step.hq, self.k_cache)), dtype=torch.uint8, device="cuda")
        if step.n_prefill:
            self.q = to_dev(step.q_prefill)
            self.cu_q, self.cu_k = to_dev(step.cu_q), to_dev(step.cu_k)
            self.ptable = self.table[step.n_decode:].contiguous()
            self.out = torch.empty_like(self.q)
            need = pkv.paged_varlen_prefill_workspace_size(step.n_prefill, step.max_seqlen_q,
                                                          step.hq, self.k_cache)
            self.ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None

    def write(self):
        pkv, s = self.pkv, self.s
        pkv.paged_build_slot_mapping(self.table, self.token_seq, self.token_pos, s.block_size,
                                     out=self.slots)
        pkv.paged_kv_write(self.new_k, self.new_v, self.slots, self.k_cache, self.v_cache)

    def attend(self):
        pkv, s = self.pkv, self.s
        if s.n_decode:
            pkv.paged_decode(self.q, self.k_cache, self.v_cache, self.dtable, self.seqlens,
                             s.scale, out=self.out, workspace=self.ws)
        else:
            pkv.paged_varlen_prefill(self.q, self.k_cache, self.v_cache, self.cu_q, self.cu_k,
                                     s.max_seqlen_q, s.max_seqlen_k, self.ptable,
                                     causal=s.causal, scale=s.scale, out=self.out,
                                     workspace=self.ws)


def soak(dev: DeviceStep, seconds: float = 0.5):
    """Keep running the same pass (untimed) so the clock sampler sees the GPU
    under this load for longer than the timed region itself lasts."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(20):
            dev.write()
            dev.attend()
        torch.cuda.synchronize()


def time_steps(dev: DeviceStep, steps: int, warmup: int, flush: torch.Tensor | None, world: int):
    """Warm up, then time `steps` passes (write + attend) with CUDA events on
    the current stream.  Returns (total ms of the passes, mean ms of attend)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        dev.write()
        dev.attend()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xff)  # evict the previous pass from L2 (not timed)
        starts[i].record(stream)
        dev.write()
        mids[i].record(stream)
        dev.attend()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    total = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    attend = [m.elapsed_time(e) for m, e in zip(mids, ends)]
    return total, float(np.mean(attend)), float(np.median(attend))


def time_e2e(step, dev: DeviceStep, steps: int, warmup: int, world: int, keep_out=None):
    """The same pass through the public API from pinned HOST buffers.  Every
    step copies its inputs host->device and reads the output back.  The step's
    inputs sit in one pinned host buffer (each at a 256-byte aligned offset),
    as a serving engine stages a step's inputs, and go over in one transfer
    into one device buffer whose slices are the tensors the calls read."""
    s = step
    host_in = {"new_k": pinned(s.new_k), "new_v": pinned(s.new_v),
               "token_seq": pinned(s.token_seq), "token_pos": pinned(s.token_pos),
               "table": pinned(s.table)}
    if s.n_decode:
        host_in.update(q=pinned(s.q_decode), seqlens=pinned(s.cache_seqlens))
    else:
        host_in.update(q=pinned(s.q_prefill), cu_q=pinned(s.cu_q), cu_k=pinned(s.cu_k))
    offs, total = {}, 0
    for name, t in host_in.items():
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = {}
    for name, t in host_in.items():
        nb = t.numel() * t.element_size()
        host_buf[offs[name]:offs[name] + nb].copy_(t.reshape(-1).view(torch.uint8))
        views[name] = dev_buf[offs[name]:offs[name] + nb].view(t.dtype).view(t.shape)
    host_out = torch.empty(dev.out.shape, dtype=dev.out.dtype).pin_memory()
    h2d = total
    d2h = host_out.numel() * host_out.element_size()

    # the calls read the slices of the staged buffer (restored afterwards)
    saved = dict(vars(dev))
    dev.new_k, dev.new_v = views["new_k"], views["new_v"]
    dev.token_seq, dev.token_pos = views["token_seq"], views["token_pos"]
    dev.table, dev.q = views["table"], views["q"]
    if s.n_decode:
        dev.seqlens = views["seqlens"]
        dev.dtable = views["table"][: s.n_decode]
    else:
        dev.cu_q, dev.cu_k = views["cu_q"], views["cu_k"]
        dev.ptable = views["table"][s.n_decode:]

    # Two copy streams: a step's upload may run while the previous step's
    # output is read back (the link carries both directions at once), but the
    # step's kernels start only when its inputs have arrived and the previous
    # output has left the device, and the upload starts only once the previous
    # step's kernels are done with the inputs.
    cur = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in, ev_done, ev_out = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    ev_done.record(cur)
    ev_out.record(cur)

    def one():
        up.wait_event(ev_done)
        with torch.cuda.stream(up):
            dev_buf.copy_(host_buf, non_blocking=True)
        ev_in.record(up)
        cur.wait_event(ev_in)
        cur.wait_event(ev_out)
        dev.write()
        dev.attend()
        ev_done.record(cur)
        down.wait_event(ev_done)
        with torch.cuda.stream(down):
            host_out.copy_(dev.out, non_blocking=True)
        ev_out.record(down)

    try:
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        barrier(world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(cur)
        ev_done.record(cur)
        ev_out.record(cur)
        for _ in range(steps):
            one()
        cur.wait_event(ev_out)
        t1.record(cur)
        torch.cuda.synchronize()
    finally:
        vars(dev).update(saved)
    if keep_out is not None:
        keep_out.append(host_out.clone())
    ms = max_over_ranks(t0.elapsed_time(t1), world) / steps
    return ms, h2d, d2h


def traffic_of(kernel: str):
    """DRAM bytes per launch from the committed ncu capture of `kernel`, or None
    when the kernel's source has changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec["dram_bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def oracle_decode_sample(step, n_seqs: int):
    """Oracle decode of the first n_seqs sequences; returns (seconds, bytes)."""
    import oracle
    sub = np.arange(n_seqs, dtype=np.int32)
    t = time.perf_counter()
    oracle.decode(step.q_decode, step.k_cache, step.v_cache, step.decode_table,
                  step.cache_seqlens, step.scale, seq_subset=sub)
    dt = time.perf_counter() - t
    L = step.cache_seqlens[:n_seqs].astype(np.int64)
    return dt, int(L.sum()) * step.kv_dim * step.elt * 2


def oracle_prefill_sample(step, every: int):
    """Oracle prefill of every `every`-th query row; returns (seconds, flops)."""
    import oracle
    rows = np.arange(0, int(step.cu_q[-1]), every, dtype=np.int32)
    t = time.perf_counter()
    oracle.prefill(step.q_prefill, step.k_cache, step.v_cache, step.cu_q, step.cu_k, step.scale,
                   causal=step.causal, block_table=step.prefill_table,
                   block_size=step.block_size, row_subset=rows)
    dt = time.perf_counter() - t
    q = np.diff(step.cu_q)
    k = np.diff(step.cu_k)
    req = np.searchsorted(step.cu_q, rows, side="right") - 1
    i = rows - step.cu_q[req]
    vis = np.clip(i + k[req] - q[req] + 1, 0, k[req]).astype(np.int64)
    return dt, int(4 * step.d * step.hq * vis.sum())


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on a bounded sample of the decode workload."""
    from paged_kv_cache_70_gb300 import workloads as W
    import oracle
    if rank != 0:
        return
    step = W.config(DECODE_CFG)
    n_seqs = step.n_decode  # each step: the whole decode workload
    for _ in range(args.warmup):
        oracle_decode_sample(step, n_seqs)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, nbytes = oracle_decode_sample(step, n_seqs)
        times.append(dt)
    sec = sum(times) / len(times)
    value = nbytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": W.CONFIG_NAMES[DECODE_CFG],
                   "sample": f"all {n_seqs} sequences per step (decode only, no write)",
                   "seed": 1000 + DECODE_CFG},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"fp64 oracle decode of all {n_seqs} sequences x 16 heads "
                                   f"({int(step.cache_seqlens.sum())} keys) per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    args = parse_args()
    world, rank = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import paged_kv_cache_70_gb300 as pkv
    from paged_kv_cache_70_gb300 import workloads as W
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()

    line = {"metric": METRIC, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "gpu_launches": 0,
            "error_flags": 0}
    dstep = None
    if args.only in ("all", "decode"):
        dstep = run_decode(args, world, pkv, W, hbm_peak, peak_src, line)
    if args.only in ("all", "prefill"):
        run_prefill(args, world, pkv, W, bf16_peak, peak_src, line)
    if args.only in ("all", "copy"):
        run_copy(args, world, pkv, hbm_peak, peak_src, line)
    if args.only in ("all", "shared"):
        run_shared_prefix(args, world, pkv, W, hbm_peak, peak_src, line)
    if args.only in ("all", "mixed"):
        run_mixed_step(args, world, pkv, W, hbm_peak, peak_src, line)
    if args.only == "prefill":  # headline comes from the prefill half
        line["metric"] = "varlen prefill TFLOP/s"
        line["value"], line["unit"] = line["prefill"].get("value"), "TFLOP/s"
        line["ms_per_step"] = line["prefill"].get("ms_per_step")
    if args.only == "mixed":
        line["metric"] = line["mixed_step"]["metric"]
        line["value"] = line["mixed_step"]["value"]
        line["ms_per_step"] = line["mixed_step"]["ms_per_step"]
    if args.only == "shared":
        line["metric"] = line["decode_shared_prefix"]["metric"]
        line["value"] = line["decode_shared_prefix"]["value"]
        line["ms_per_step"] = line["decode_shared_prefix"]["ms_per_step"]
    if args.only == "copy":
        line["metric"] = line["copy_blocks"]["metric"]
        line["value"] = line["copy_blocks"]["value"]
        line["ms_per_step"] = line["copy_blocks"]["ms_per_step"]
    cpu_baseline(args, world, rank, W, dstep, line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_decode(args, world, pkv, W, hbm_peak, peak_src, line):
    dstep = W.config(DECODE_CFG)
    ddev = DeviceStep(dstep, pkv)
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()  # warm-up + timed region + a short untimed soak of the same step
    total_ms, dec_mean, dec_med = time_steps(ddev, args.steps, args.warmup, None, world)
    soak(ddev)
    clk = clocks.stop()
    clk["window"] = "warm-up, timed region, then 0.5 s more of the same step (untimed)"
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    dbytes = decode_kernel_bytes(dstep)
    wbytes = write_bytes(dstep)
    step_bytes = dbytes + wbytes
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    # workspace traffic of the split (partials written and read back)
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    part = (ctas + dstep.n_decode) * dstep.hq * (dstep.d + 2) * 4 * 2
    achieved = dbytes / (dec_mean * 1e-3) / 1e9
    line.update({
        "value": round(value, 2), "ms_per_step": round(ms_step, 5),
        "config": {"workload": W.CONFIG_NAMES[DECODE_CFG] + "; step = slot_mapping build + "
                               "new-token write + paged decode (split-KV + combine)",
                   "batch": dstep.n_decode, "seq_lens_total": int(dstep.cache_seqlens.sum()),
                   "block_size": dstep.block_size, "num_heads": dstep.hq,
                   "num_kv_heads": dstep.hkv, "head_dim": dstep.d, "seed": 1000 + DECODE_CFG,
                   "bytes_per_step": step_bytes,
                   "l2": "inputs larger than L2 (%.0f MB of K/V per step)" % (dbytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": "paged_decode (split kernel + combine)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": peak_src,
                     "traffic": traffic_of("decode_split_kernel"),
                     "algorithmic_bytes_per_launch": dbytes,
                     "workspace_bytes_per_launch": part,
                     "mean_ms": round(dec_mean, 5), "median_ms": round(dec_med, 5)},
        "clocks": clk,
    })
    line["gpu_launches"] += 4 * args.steps
    run_decode_append(args, world, pkv, dstep, ddev, step_bytes, hbm_peak, peak_src, line)
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(dstep, ddev, args.steps, args.warmup, world)
        line["e2e"] = {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    line["error_flags"] |= pkv.paged_error_flags()
    del ddev
    torch.cuda.empty_cache()
    return dstep


W_NAME_PACKED = ("causal varlen prefill over packed K/V: the chunked-prefill workload's 16 "
                 "requests (q~U[1,2048], cached~U[0,2048]) with each request's keys "
                 "contiguous; L2 flushed between steps")
COPY_PAIRS, COPY_GEOM = 8192, (16, 8, 128)  # block pairs; B, Hkv, d (bf16)


def run_decode_append(args, world, pkv, dstep, ddev, step_bytes, hbm_peak, peak_src, line):
    """The same decode step in one call: paged_decode_append writes the new
    token's K/V and attends over the cached keys plus the new one (split +
    combine, two launches instead of four)."""
    before = to_dev((dstep.cache_seqlens - 1).astype(np.int32))
    out = torch.empty_like(ddev.q)
    call = lambda: pkv.paged_decode_append(ddev.q, ddev.new_k, ddev.new_v, ddev.k_cache,
                                           ddev.v_cache, ddev.dtable, before, dstep.scale,
                                           out=out, workspace=ddev.ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean = max_over_ranks(float(np.mean(ms)), world)
    gbs = step_bytes / (mean * 1e-3) / 1e9
    line["decode_append"] = {
        "metric": "decode KV GB/s, step as one call with the in-place append", "unit": "GB/s",
        "value": round(world * gbs, 2), "ms_per_step": round(mean, 5),
        "workload": "the headline long-context decode step (same bytes per step)",
        "roofline": {"bound": "hbm", "kernel": "paged_decode_append (split + combine with the "
                     "appended key and its cache write)", "achieved": round(gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": None, "mean_ms": round(mean, 5),
                     "median_ms": round(float(np.median(ms)), 5)}}
    line["gpu_launches"] += 2 * args.steps


def run_copy(args, world, pkv, hbm_peak, peak_src, line):
    """paged_copy_blocks: the copies of copy-on-write.  8192 block pairs of a
    B=16, Hkv=8, d=128 bf16 pool (32 KiB per block per pool): 512 MiB read and
    512 MiB written per launch, far beyond L2."""
    B, hkv, d = COPY_GEOM
    nb = 2 * COPY_PAIRS + 16
    g = torch.Generator().manual_seed(1099)
    k = torch.randint(-32768, 32767, (nb, B, hkv, d), generator=g, dtype=torch.int16)
    k_cache = k.view(torch.bfloat16).cuda()
    v_cache = torch.roll(k, 1, 0).view(torch.bfloat16).cuda()
    perm = torch.randperm(nb, generator=g)
    src = perm[:COPY_PAIRS].to(torch.int32).cuda()
    dst = perm[COPY_PAIRS: 2 * COPY_PAIRS].to(torch.int32).cuda()
    block_bytes = B * hkv * d * 2
    nbytes = COPY_PAIRS * block_bytes * 2 * 2  # K and V, read and written
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        pkv.paged_copy_blocks(k_cache, v_cache, src, dst)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        pkv.paged_copy_blocks(k_cache, v_cache, src, dst)
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean = max_over_ranks(float(np.mean(ms)), world)
    gbs = nbytes / (mean * 1e-3) / 1e9
    line["copy_blocks"] = {
        "metric": "copy-on-write block copies GB/s", "unit": "GB/s",
        "value": round(world * gbs, 1), "ms_per_step": round(mean, 5),
        "workload": f"{COPY_PAIRS} block pairs, B={B}, Hkv={hkv}, d={d}, bf16 "
                    f"({block_bytes // 1024} KiB per block per pool); step = one paged_copy_blocks",
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel", "achieved": round(gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": traffic_of("copy_blocks_kernel"),
                     "algorithmic_bytes_per_launch": nbytes, "mean_ms": round(mean, 5),
                     "median_ms": round(float(np.median(ms)), 5)},
        "l2": "inputs larger than L2 (512 MiB read per launch)"}
    line["gpu_launches"] += args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del k_cache, v_cache
    torch.cuda.empty_cache()


def run_shared_prefix(args, world, pkv, W, hbm_peak, peak_src, line):
    """Decode half of the continuous-batching workload: 256 sequences in 8
    groups of 32 that share a 2048-token prefix (128 blocks of 16), suffixes
    U[0,512] plus the new token.  Shared-prefix decode (each prefix block read
    once per group) against plain paged decode of the same step.  The roofline
    counts UNIQUE bytes: the prefixes once, every suffix, q and out."""
    s = W.config(5)
    nd = s.n_decode
    dev = lambda a: to_dev(a)
    k_cache, v_cache = dev(s.k_cache), dev(s.v_cache)
    q, table, lens = dev(s.q_decode), dev(s.decode_table.copy()), dev(s.cache_seqlens)
    groups = 8
    gcu = dev(np.arange(0, nd + 1, nd // groups, dtype=np.int32))
    plen = dev(np.full(groups, 2048, np.int32))
    out = torch.empty_like(q)
    row = s.hkv * s.d * 2 * 2  # K + V bytes per key
    unique = (groups * 2048 + int((s.cache_seqlens - 2048).sum())) * row + 2 * q.numel() * 2
    logical = int(s.cache_seqlens.sum()) * row + 2 * q.numel() * 2
    ws = torch.empty(pkv._binding.load_library().paged_decode_shared_prefix_workspace_size(
        nd, ctypes.byref(pkv.geom_of(k_cache, s.hq))), dtype=torch.uint8, device="cuda")
    wsp = torch.empty(max(1, pkv.paged_decode_workspace_size(nd, s.hq, k_cache)),
                      dtype=torch.uint8, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    shared = lambda: pkv.paged_decode_shared_prefix(q, k_cache, v_cache, table, lens, gcu, plen,
                                                    nd // groups, s.scale, out=out, workspace=ws)
    plain = lambda: pkv.paged_decode(q, k_cache, v_cache, table, lens, s.scale, out=out,
                                     workspace=wsp)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i, (a, b) in enumerate(ev):
            flush.fill_(i & 0xff)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms = [a.elapsed_time(b) for a, b in ev]
        return max_over_ranks(float(np.mean(ms)), world), float(np.median(ms))

    sh_ms, sh_med = timed(shared)
    pl_ms, _ = timed(plain)
    gbs = unique / (sh_ms * 1e-3) / 1e9
    line["decode_shared_prefix"] = {
        "metric": "shared-prefix decode GB/s of unique K/V", "unit": "GB/s",
        "value": round(world * gbs, 1), "ms_per_step": round(sh_ms, 5),
        "workload": "decode half of the continuous-batching step: 256 sequences, 8 groups of "
                    "32 sharing a 2048-token prefix (B=16), suffixes U[0,512]+1, GQA 16/8, "
                    "d=128, bf16; L2 flushed between steps",
        "unique_bytes": unique, "logical_bytes": logical,
        "roofline": {"bound": "hbm", "kernel": "paged_decode_shared_prefix (prefix on the "
                     "tensor cores + suffix split + combine)", "achieved": round(gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": None, "mean_ms": round(sh_ms, 5),
                     "median_ms": round(sh_med, 5)},
        "plain_decode_same_step": {"ms": round(pl_ms, 5),
                                   "logical_GBps": round(logical / (pl_ms * 1e-3) / 1e9, 1),
                                   "speedup_of_shared": round(pl_ms / sh_ms, 3)}}
    line["gpu_launches"] += 3 * args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del k_cache, v_cache, ws, wsp, flush
    torch.cuda.empty_cache()


def run_mixed_step(args, world, pkv, W, hbm_peak, peak_src, line):
    """The whole continuous-batching step in one paged_mixed_step call: 2304
    new rows (+5 % padding) written, causal prefill of 4 x 512 tokens, and
    the in-place append + shared-prefix decode of 256 sequences.  Bytes
    counted once each: K/V of every key read (shared prefixes once), the new
    rows read and written, q and out."""
    s = W.config(5)
    nd = s.n_decode
    is_dec = (s.token_seq >= 0) & (s.token_seq < nd)
    dec_rows = np.where(is_dec)[0]
    dec_rows = dec_rows[np.argsort(s.token_seq[dec_rows])]
    pf_rows = np.where(~is_dec)[0]
    B = s.block_size
    seq = s.token_seq
    slots = np.full(len(seq), -1, np.int32)
    ok = seq >= 0
    slots[ok] = s.table[seq[ok], s.token_pos[ok] // B] * B + s.token_pos[ok] % B
    kc, vc = to_dev(s.k_cache), to_dev(s.v_cache)
    decode = dict(q=to_dev(s.q_decode), k_new=to_dev(s.new_k[dec_rows]),
                  v_new=to_dev(s.new_v[dec_rows]), table=to_dev(s.decode_table.copy()),
                  seqlens=to_dev(s.cache_seqlens - 1),
                  group_cu=to_dev(np.arange(0, nd + 1, nd // 8, dtype=np.int32)),
                  group_prefix_len=to_dev(np.full(8, 2048, np.int32)), max_group_size=nd // 8,
                  out=torch.empty(s.q_decode.shape, dtype=torch.bfloat16, device="cuda"))
    prefill = dict(k_new=to_dev(s.new_k[pf_rows]), v_new=to_dev(s.new_v[pf_rows]),
                   slots=to_dev(slots[pf_rows]), q=to_dev(s.q_prefill), cu_q=to_dev(s.cu_q),
                   cu_k=to_dev(s.cu_k), max_q=s.max_seqlen_q, max_k=s.max_seqlen_k,
                   table=to_dev(s.prefill_table.copy()),
                   out=torch.empty(s.q_prefill.shape, dtype=torch.bfloat16, device="cuda"))
    ws = torch.empty(pkv._binding.load_library().paged_mixed_step_workspace_size(
        nd, ctypes.byref(pkv.geom_of(kc, s.hq))), dtype=torch.uint8, device="cuda")
    row = s.hkv * s.d * 2 * 2
    n_new = int((s.token_seq >= 0).sum())
    nbytes = ((8 * 2048 + int((s.cache_seqlens - 1 - 2048).sum())) * row  # decode keys once
              + int(s.cu_k[-1]) * row                                    # prefill keys
              + 2 * n_new * row                                           # new rows r + w
              + 2 * (s.q_decode.size + s.q_prefill.size) * 2)             # q and out
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    call = lambda: pkv.paged_mixed_step(kc, vc, s.scale, prefill=prefill, decode=decode,
                                        workspace=ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i, (a, b) in enumerate(ev):
        flush.fill_(i & 0xff)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean = max_over_ranks(float(np.mean(ms)), world)
    gbs = nbytes / (mean * 1e-3) / 1e9
    line["mixed_step"] = {
        "metric": "continuous-batching step GB/s of unique bytes", "unit": "GB/s",
        "value": round(world * gbs, 1), "ms_per_step": round(mean, 5),
        "workload": W.CONFIG_NAMES[5] + "; one paged_mixed_step call; L2 flushed between steps",
        "unique_bytes": nbytes,
        "roofline": {"bound": "hbm", "kernel": "paged_mixed_step (write, prefill, shared-prefix "
                     "pass, split, combine with append)", "achieved": round(gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": None, "mean_ms": round(mean, 5),
                     "median_ms": round(float(np.median(ms)), 5)}}
    line["gpu_launches"] += 5 * args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del kc, vc, ws, flush
    torch.cuda.empty_cache()


def run_prefill(args, world, pkv, W, bf16_peak, peak_src, line):
    pstep = W.config(PREFILL_CFG)
    pdev = DeviceStep(pstep, pkv)
    try:
        pdev.attend()
        ok = True
    except pkv.PagedKVError as e:
        ok = False
        line["prefill"] = {"unavailable": str(e)}
    if ok:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        clocks = Clocks(torch.cuda.current_device())
        clocks.start()
        ptotal, pmean, pmed = time_steps(pdev, args.steps, args.warmup, flush, world)
        soak(pdev)
        pclk = clocks.stop()
        pclk["window"] = "warm-up, timed region, then 0.5 s more of the same step (untimed)"
        ptotal = max_over_ranks(ptotal, world)
        flops = prefill_flops(pstep)
        p_ms = ptotal / args.steps
        tflops = flops / (pmean * 1e-3) / 1e12
        line["prefill"] = {
            "metric": "varlen prefill TFLOP/s", "workload": W.CONFIG_NAMES[PREFILL_CFG],
            "value": round(world * flops / (p_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(p_ms, 5),
            "step": "slot_mapping build + write of 16 requests' new K/V + causal varlen "
                    "prefill (L2 flushed between steps, not timed)",
            "flops_per_step": flops, "visible_pairs": prefill_pairs(pstep),
            "roofline": {"bound": "tensor", "kernel": "paged_varlen_prefill",
                         "achieved": round(tflops, 1), "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": round(tflops / bf16_peak, 4),
                         "peak_source": peak_src + " (bf16 burst)",
                         "traffic": traffic_of("prefill_tc_kernel"),
                         "mean_ms": round(pmean, 5), "median_ms": round(pmed, 5)},
            "clocks": pclk,
        }
        if not args.no_e2e:
            pe2e_ms, ph2d, pd2h = time_e2e(pstep, pdev, args.steps, args.warmup, world)
            line["prefill"]["e2e"] = {
                "value": round(world * flops / (pe2e_ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(pe2e_ms, 5),
                "h2d_bytes_per_step": ph2d, "d2h_bytes_per_step": pd2h}
        line["gpu_launches"] += 3 * args.steps
        line["error_flags"] |= pkv.paged_error_flags()
        run_prefill_packed(args, world, pkv, pstep, pdev, flops, flush, bf16_peak, peak_src,
                           line)
    del pdev
    torch.cuda.empty_cache()


def run_prefill_packed(args, world, pkv, pstep, pdev, flops, flush, bf16_peak, peak_src, line):
    """The same attention with packed K/V (block_table = NULL): each request's
    keys gathered once (untimed) into contiguous [total_k, Hkv, d] arrays."""
    s = pstep
    B = s.block_size
    rows = []
    for r in range(s.n_prefill):
        kl = int(s.cu_k[r + 1] - s.cu_k[r])
        p = np.arange(kl)
        rows.append(s.prefill_table[r][p // B].astype(np.int64) * B + p % B)
    idx = torch.from_numpy(np.concatenate(rows)).cuda()
    kp = pdev.k_cache.view(-1, s.hkv, s.d)[idx].contiguous()
    vp = pdev.v_cache.view(-1, s.hkv, s.d)[idx].contiguous()
    call = lambda: pkv.paged_varlen_prefill(pdev.q, kp, vp, pdev.cu_q, pdev.cu_k,
                                            s.max_seqlen_q, s.max_seqlen_k, None,
                                            causal=s.causal, scale=s.scale, out=pdev.out)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i, (a, b) in enumerate(ev):
        flush.fill_(i & 0xff)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean = max_over_ranks(float(np.mean(ms)), world)
    tf = flops / (mean * 1e-3) / 1e12
    line["prefill_contiguous"] = {
        "metric": "varlen prefill TFLOP/s (packed K/V, block_table = NULL)",
        "workload": W_NAME_PACKED, "value": round(world * tf, 2), "unit": "TFLOP/s",
        "ms_per_step": round(mean, 5), "flops_per_step": flops,
        "roofline": {"bound": "tensor", "kernel": "paged_varlen_prefill (packed)",
                     "achieved": round(tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(tf / bf16_peak, 4), "peak_source": peak_src + " (bf16 burst)",
                     "traffic": None, "mean_ms": round(mean, 5),
                     "median_ms": round(float(np.median(ms)), 5)}}
    line["gpu_launches"] += args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del kp, vp


def cpu_baseline(args, world, rank, W, dstep, line):
    """The oracle as it stands, on the host cores (rank 0, N=1 only)."""
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n_seqs = 8
        if dstep is None:
            dstep = W.config(DECODE_CFG)
        dt, nb, reps = 0.0, 0, 0
        while dt < 5.0 and reps < 1000:  # the whole decode workload, repeated for >= 5 s
            t, b = oracle_decode_sample(dstep, n_seqs)
            dt, nb, reps = dt + t, nb + b, reps + 1
        line["cpu_baseline"] = {
            "value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle decode of the whole decode workload (8 sequences x 16 "
                      f"heads), {reps} times ({dt:.1f} s)"}
        if "prefill" in line and "value" in line["prefill"]:
            pstep = W.config(PREFILL_CFG)
            dt, fl = oracle_prefill_sample(pstep, 1)
            line["prefill"]["cpu_baseline"] = {
                "value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s",
                "cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"fp64 oracle prefill of every query row of the prefill workload "
                          f"({dt:.1f} s)"}


if __name__ == "__main__":
    main()
