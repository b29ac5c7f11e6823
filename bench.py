#!/usr/bin/env python
"""Benchmark of the paged KV-cache hot path on GB300.

The headline is one decode step of the long-context workload (batch 8,
16K-40K cached keys, GQA 16/8, head_dim 128, block 256, bf16): every
sequence's new token is written into the cache and attended to together with
the cached keys in one paged_decode_append call (the kvcache call of "Sayfalı
dikkat"), reported as decode KV GB/s.  The same run measures, each as a
sub-object of the JSON line:

  decode_qwen3            the Qwen3-0.6B-shaped decode (batch 64, L~U[128,4096],
                          block 16), the same one-call step;
  decode_separate_write   the headline step as slot_mapping build + write +
                          paged_decode (four launches);
  kv_write                the slot_mapping write of the chunked-prefill
                          workload's 17,928 new rows (paged_kv_write alone);
  prefill                 one chunked-prefill step (write the new rows, then
                          causal varlen prefill; TFLOP/s of visible pairs), and
  prefill_contiguous      the same attention over packed K/V;
  copy_blocks             the copy-on-write block copies;
  decode_shared_prefix    the decode half of the continuous-batching workload;
  mixed_step              the whole continuous-batching step in one call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  With torchrun (N > 1) every rank runs its own replica of
the workload on its own GPU (no collective on the data path; "replicas only"),
and timing is the max over ranks.  ``--impl reference`` times the CPU oracle (the
reference arm) on a bounded sample of the same workload.

Between timed steps L2 is flushed (untimed): a 256 MiB buffer is written and
then a 1 GiB buffer is read, so that the dirty lines of the write go back to
HBM before the next timed step starts instead of inside it.
"""
from __future__ import annotations

import argparse
import ctypes
import json
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
DECODE_CFG, QWEN_CFG, PREFILL_CFG, MIXED_CFG = 3, 2, 4, 5
PARTS = ("all", "decode", "qwen3", "shapes", "write", "prefill", "copy", "shared", "mixed")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--only", choices=PARTS, default="all",
                   help="measure one part only (profiling runs)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end passes")
    p.add_argument("--no-soak", action="store_true",
                   help="skip the untimed clock-sampling passes (a fixed launch count for ncu)")
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


def decode_append_bytes(step) -> int:
    """Bytes paged_decode_append must move: K and V of every cached key, the
    new token's K and V rows read and written once, q, out, the block-table
    entries of every page touched, and cache_seqlens."""
    L = step.cache_seqlens.astype(np.int64) - 1  # keys cached before the step
    row = step.kv_dim * step.elt * 2              # K + V of one key
    qo = 2 * step.n_decode * step.hq * step.d * step.elt
    table = int(np.sum(-(-(L + 1) // step.block_size))) * 4
    return int(L.sum()) * row + 2 * step.n_decode * row + qo + table + step.n_decode * 4


def slot_build_bytes(step) -> int:
    """paged_build_slot_mapping: token_seq, token_pos and one table entry read,
    the slot written, per row."""
    return len(step.token_seq) * 16


def write_bytes(step) -> int:
    """paged_kv_write: the slot of every row read; K and V of every non-padding
    row read once and written once."""
    n_rows = len(step.token_seq)
    n_real = int((step.token_seq >= 0).sum())
    return n_rows * 4 + n_real * step.kv_dim * step.elt * 2 * 2


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
# device-side workloads
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


class L2Flush:
    """Evicts the previous step from L2 (untimed): writes a 256 MiB buffer,
    then reads a 1 GiB buffer.  The read pushes every dirty line of the write
    back to HBM before the timed step starts: after a write alone (or a write
    followed by a read of 256 MiB) the next step would pay for those
    write-backs (measured: +15 us and +7 us on the long-context decode, whose
    time with this flush equals its time with no flush at all)."""

    def __init__(self):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones((1 << 30) // 8, dtype=torch.int64, device="cuda")
        self.sink = torch.empty((), dtype=torch.int64, device="cuda")

    def __call__(self, i: int):
        self.w.fill_(i & 0xff)
        torch.sum(self.r, dim=0, out=self.sink)


class DecodeStep:
    """A decode step with the in-place append, resident on the device: every
    sequence's new token (k_new/v_new row b) is written at position
    cache_seqlens[b] - 1 and attended to together with the cached keys in one
    paged_decode_append call (split kernel + combine)."""

    launches = 2

    def __init__(self, step, pkv):
        s = step
        nd = s.n_decode
        # the workloads put decode sequence b's new row first, in order
        assert np.array_equal(s.token_seq[:nd], np.arange(nd))
        assert np.array_equal(s.token_pos[:nd], s.cache_seqlens - 1)
        self.s, self.pkv = s, pkv
        self.host = {"q": s.q_decode, "k_new": s.new_k[:nd], "v_new": s.new_v[:nd],
                     "table": s.decode_table, "seqlens": (s.cache_seqlens - 1).astype(np.int32)}
        self.dev = {k: to_dev(v) for k, v in self.host.items()}
        self.k_cache, self.v_cache = to_dev(s.k_cache), to_dev(s.v_cache)
        self.out = torch.empty_like(self.dev["q"])
        self.ws = torch.empty(max(1, pkv.paged_decode_workspace_size(nd, s.hq, self.k_cache)),
                              dtype=torch.uint8, device="cuda")

    def run(self, t=None):
        t = self.dev if t is None else t
        self.pkv.paged_decode_append(t["q"], t["k_new"], t["v_new"], self.k_cache, self.v_cache,
                                     t["table"], t["seqlens"], self.s.scale, out=self.out,
                                     workspace=self.ws)


class WriteDecodeStep:
    """The same decode step as three calls: slot_mapping build, paged_kv_write
    of the new rows, paged_decode over the cached keys including the new one."""

    def __init__(self, step, pkv):
        s = step
        self.s, self.pkv = s, pkv
        self.table = to_dev(s.table)
        self.dtable = self.table[: s.n_decode].contiguous()
        self.k_cache, self.v_cache = to_dev(s.k_cache), to_dev(s.v_cache)
        self.new_k, self.new_v = to_dev(s.new_k), to_dev(s.new_v)
        self.token_seq, self.token_pos = to_dev(s.token_seq), to_dev(s.token_pos)
        self.slots = torch.empty(len(s.token_seq), dtype=torch.int32, device="cuda")
        self.q, self.seqlens = to_dev(s.q_decode), to_dev(s.cache_seqlens)
        self.out = torch.empty_like(self.q)
        self.ws = torch.empty(max(1, pkv.paged_decode_workspace_size(s.n_decode, s.hq,
                                                                     self.k_cache)),
                              dtype=torch.uint8, device="cuda")

    def write(self):
        self.pkv.paged_build_slot_mapping(self.table, self.token_seq, self.token_pos,
                                          self.s.block_size, out=self.slots)
        self.pkv.paged_kv_write(self.new_k, self.new_v, self.slots, self.k_cache, self.v_cache)

    def attend(self):
        self.pkv.paged_decode(self.q, self.k_cache, self.v_cache, self.dtable, self.seqlens,
                              self.s.scale, out=self.out, workspace=self.ws)


class PrefillStep:
    """A chunked-prefill step resident on the device: slot_mapping build and
    write of the requests' new rows (one paged_kv_write_positions launch, which
    also stores the slot mapping for other layers), then causal varlen prefill
    over cached + new keys through the block table."""

    launches = 2

    def __init__(self, step, pkv):
        s = step
        assert s.n_decode == 0
        self.s, self.pkv = s, pkv
        self.host = {"new_k": s.new_k, "new_v": s.new_v, "token_seq": s.token_seq,
                     "token_pos": s.token_pos, "table": s.prefill_table, "q": s.q_prefill,
                     "cu_q": s.cu_q, "cu_k": s.cu_k}
        self.dev = {k: to_dev(v) for k, v in self.host.items()}
        self.k_cache, self.v_cache = to_dev(s.k_cache), to_dev(s.v_cache)
        self.slots = torch.empty(len(s.token_seq), dtype=torch.int32, device="cuda")
        self.out = torch.empty_like(self.dev["q"])
        need = pkv.paged_varlen_prefill_workspace_size(s.n_prefill, s.max_seqlen_q, s.hq,
                                                      self.k_cache)
        self.ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None

    def slot_build(self, t=None):
        t = self.dev if t is None else t
        self.pkv.paged_build_slot_mapping(t["table"], t["token_seq"], t["token_pos"],
                                          self.s.block_size, out=self.slots)

    def write(self, t=None):
        t = self.dev if t is None else t
        self.pkv.paged_kv_write(t["new_k"], t["new_v"], self.slots, self.k_cache, self.v_cache)

    def write_pos(self, t=None):
        t = self.dev if t is None else t
        self.pkv.paged_kv_write_positions(t["new_k"], t["new_v"], t["table"], t["token_seq"],
                                          t["token_pos"], self.k_cache, self.v_cache,
                                          slot_mapping_out=self.slots)

    def attend(self, t=None):
        t = self.dev if t is None else t
        s = self.s
        self.pkv.paged_varlen_prefill(t["q"], self.k_cache, self.v_cache, t["cu_q"], t["cu_k"],
                                      s.max_seqlen_q, s.max_seqlen_k, t["table"],
                                      causal=s.causal, scale=s.scale, out=self.out,
                                      workspace=self.ws)

    def run(self, t=None):
        self.write_pos(t)
        self.attend(t)


def time_parts(parts, steps: int, warmup: int, world: int, flush=None):
    """Warm up, then time `steps` passes of the callables in `parts` (run in
    order) with CUDA events on the current stream, an event between
    consecutive parts.  Returns (mean ms of a pass, [(mean, median) per part])
    with the pass mean taken as the max over ranks."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for f in parts:
            f()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)]
           for _ in range(steps)]
    # Keep the GPU busy while the first timed pass is enqueued, so that no
    # host launch latency lands inside a timed region (later passes are
    # queued behind the previous ones).
    if flush is not None:
        flush(steps)
    else:
        torch.cuda._sleep(2_000_000)
    for i in range(steps):
        if flush is not None:
            flush(i)
        evs[i][0].record(stream)
        for j, f in enumerate(parts):
            f()
            evs[i][j + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    steps_ms = [e[0].elapsed_time(e[-1]) for e in evs]
    total = max_over_ranks(float(np.mean(steps_ms)), world)
    print("steps (us):", " ".join(f"{1e3 * x:.1f}" for x in steps_ms), file=sys.stderr, flush=True)
    per = []
    for j in range(len(parts)):
        ms = [e[j].elapsed_time(e[j + 1]) for e in evs]
        per.append((max_over_ranks(float(np.mean(ms)), world), float(np.median(ms))))
    return total, per


def soak(fn, seconds: float = 0.5):
    """Keep running the same pass (untimed) so the clock sampler sees the GPU
    under this load for longer than the timed region itself lasts."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(20):
            fn()
        torch.cuda.synchronize()


def time_e2e(dstep, steps: int, warmup: int, world: int):
    """The step through the public API from pinned HOST buffers.  Every step
    copies its inputs host->device and reads the output back.  The step's
    inputs sit in one pinned host buffer (each at a 256-byte aligned offset),
    as a serving engine stages a step's inputs, and go over in one transfer
    into one device buffer whose slices are the tensors the calls read.
    Returns (ms per step, h2d bytes, d2h bytes)."""
    host_in = {k: pinned(v) for k, v in dstep.host.items()}
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
    host_out = torch.empty(dstep.out.shape, dtype=dstep.out.dtype).pin_memory()
    h2d = total
    d2h = host_out.numel() * host_out.element_size()

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
        dstep.run(views)
        ev_done.record(cur)
        down.wait_event(ev_done)
        with torch.cuda.stream(down):
            host_out.copy_(dstep.out, non_blocking=True)
        ev_out.record(down)

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
    ms = max_over_ranks(t0.elapsed_time(t1), world) / steps
    return ms, h2d, d2h


def traffic_of(key: str):
    """DRAM bytes per call from the committed ncu capture of workload `key`
    (the sum over the call's kernels), or None when a kernel's source file has
    changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(key)
    if not rec:
        return None
    for src, h in rec["sources"].items():
        path = os.path.join(ROOT, src)
        if not os.path.exists(path):
            return None
        if hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] != h:
            return None
    return rec["dram_bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def hbm_roofline(kernel, nbytes, mean, med, peak, src, traffic_key):
    gbs = nbytes / (mean * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(gbs, 1), "peak": peak,
            "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": src,
            "traffic": traffic_of(traffic_key), "algorithmic_bytes_per_launch": nbytes,
            "mean_ms": round(mean, 5), "median_ms": round(med, 5)}


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
    peaks = load_peaks()
    flush = L2Flush()

    line = {"metric": METRIC, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "gpu_launches": 0,
            "error_flags": 0}
    dstep = None
    only = args.only
    if only in ("all", "decode"):
        dstep = run_decode(args, world, pkv, W, peaks, flush, line)
    if only in ("all", "qwen3"):
        run_qwen3(args, world, pkv, W, peaks, flush, line)
    if only in ("all", "shapes"):
        run_shapes(args, world, pkv, W, peaks, flush, line)
    if only in ("all", "write"):
        run_write(args, world, pkv, W, peaks, flush, line)
    if only in ("all", "prefill"):
        run_prefill(args, world, pkv, W, peaks, flush, line)
    if only in ("all", "copy"):
        run_copy(args, world, pkv, peaks, line)
    if only in ("all", "shared"):
        run_shared_prefix(args, world, pkv, W, peaks, flush, line)
    if only in ("all", "mixed"):
        run_mixed_step(args, world, pkv, W, peaks, flush, line)
    sub = {"qwen3": "decode_qwen3", "write": "kv_write", "prefill": "prefill",
           "copy": "copy_blocks", "shared": "decode_shared_prefix", "mixed": "mixed_step"}
    if only in sub and "value" in line.get(sub[only], {}):
        part = line[sub[only]]
        line["metric"], line["value"] = part["metric"], part["value"]
        line["unit"], line["ms_per_step"] = part["unit"], part["ms_per_step"]
    cpu_baseline(args, world, rank, W, dstep, line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_decode(args, world, pkv, W, peaks, flush, line):
    """Headline: the long-context decode step in one paged_decode_append call."""
    hbm_peak, _, _, peak_src = peaks
    dstep = W.config(DECODE_CFG)
    ddev = DecodeStep(dstep, pkv)
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()  # warm-up + timed region + a short untimed soak of the same step
    ms_step, per = time_parts([ddev.run], args.steps, args.warmup, world, flush)
    if not args.no_soak:
        soak(ddev.run)
    clk = clocks.stop()
    clk["window"] = "warm-up, timed region, then 0.5 s more of the same step (untimed)"
    nbytes = decode_append_bytes(dstep)
    value = world * nbytes / (ms_step * 1e-3) / 1e9
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    part = (ctas + dstep.n_decode) * dstep.hq * (dstep.d + 2) * 4 * 2
    line.update({
        "value": round(value, 2), "ms_per_step": round(ms_step, 5),
        "config": {"workload": W.CONFIG_NAMES[DECODE_CFG] + "; step = one paged_decode_append "
                               "call: the new token of every sequence written into the cache "
                               "and attended to with the cached keys (split-KV + combine)",
                   "batch": dstep.n_decode, "seq_lens_total": int(dstep.cache_seqlens.sum()),
                   "block_size": dstep.block_size, "num_heads": dstep.hq,
                   "num_kv_heads": dstep.hkv, "head_dim": dstep.d, "seed": 1000 + DECODE_CFG,
                   "bytes_per_step": nbytes,
                   "l2": "flushed between steps (256 MiB written, then 1 GiB read; untimed); "
                         "K/V per step %.0f MB, larger than L2" % (nbytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": hbm_roofline("paged_decode_append (split kernel + combine)", nbytes,
                                 per[0][0], per[0][1], hbm_peak, peak_src,
                                 "long_context_decode"),
        "clocks": clk,
    })
    line["roofline"]["workspace_bytes_per_launch"] = part
    line["gpu_launches"] += DecodeStep.launches * args.steps
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(ddev, args.steps, args.warmup, world)
        line["e2e"] = {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        line["gpu_launches"] += DecodeStep.launches * args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del ddev
    torch.cuda.empty_cache()
    run_separate_write(args, world, pkv, W, dstep, peaks, flush, line)
    return dstep


def run_separate_write(args, world, pkv, W, dstep, peaks, flush, line):
    """The headline step as slot_mapping build + paged_kv_write + paged_decode."""
    hbm_peak, _, _, peak_src = peaks
    dev = WriteDecodeStep(dstep, pkv)
    ms_step, per = time_parts([dev.write, dev.attend], args.steps, args.warmup, world, flush)
    dbytes = decode_kernel_bytes(dstep)
    nbytes = dbytes + slot_build_bytes(dstep) + write_bytes(dstep)
    line["decode_separate_write"] = {
        "metric": "decode KV GB/s, step as slot_mapping build + write + paged_decode",
        "unit": "GB/s", "value": round(world * nbytes / (ms_step * 1e-3) / 1e9, 2),
        "ms_per_step": round(ms_step, 5), "bytes_per_step": nbytes,
        "workload": W.CONFIG_NAMES[DECODE_CFG] + "; L2 flushed between steps",
        "write_ms": round(per[0][0], 5),
        "roofline": hbm_roofline("paged_decode (split kernel + combine)", dbytes, per[1][0],
                                 per[1][1], hbm_peak, peak_src, "long_context_decode_plain")}
    line["gpu_launches"] += 4 * args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del dev
    torch.cuda.empty_cache()


def run_qwen3(args, world, pkv, W, peaks, flush, line):
    """The Qwen3-0.6B-shaped decode (batch 64, L~U[128,4096], block 16): the
    same one-call step as the headline."""
    hbm_peak, _, _, peak_src = peaks
    s = W.config(QWEN_CFG)
    dev = DecodeStep(s, pkv)
    ms_step, per = time_parts([dev.run], args.steps, args.warmup, world, flush)
    nbytes = decode_append_bytes(s)
    part = {
        "metric": "decode KV GB/s (Qwen3-0.6B-shaped decode)", "unit": "GB/s",
        "value": round(world * nbytes / (ms_step * 1e-3) / 1e9, 2),
        "ms_per_step": round(ms_step, 5), "bytes_per_step": nbytes,
        "workload": W.CONFIG_NAMES[QWEN_CFG] + "; step = one paged_decode_append call; "
                    "L2 flushed between steps",
        "seq_lens_total": int(s.cache_seqlens.sum()),
        "roofline": hbm_roofline("paged_decode_append (split kernel + combine)", nbytes,
                                 per[0][0], per[0][1], hbm_peak, peak_src, "qwen3_decode")}
    line["gpu_launches"] += DecodeStep.launches * args.steps
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(dev, args.steps, args.warmup, world)
        part["e2e"] = {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        line["gpu_launches"] += DecodeStep.launches * args.steps
    line["decode_qwen3"] = part
    line["error_flags"] |= pkv.paged_error_flags()
    del dev
    torch.cuda.empty_cache()


# Decode shapes beyond the workloads: the long-context lengths (8 sequences,
# U[16384, 40960] keys, block 256) with GQA groups of 4, 8 and 16, head_dim 64,
# and 4 KV heads.  bf16 groups of 4 and more attend through the tensor-core
# pass (two launches: that pass and the combine; no split).
SHAPES = {"gqa4_32q_8kv_d128": (32, 8, 128), "d64_16q_8kv": (16, 8, 64),
          "16q_4kv_d128": (16, 4, 128), "gqa8_64q_8kv_d128": (64, 8, 128),
          "gqa16_128q_8kv_d128": (128, 8, 128)}


def run_shapes(args, world, pkv, W, peaks, flush, line):
    hbm_peak, _, _, peak_src = peaks
    lens = np.random.default_rng(1003 + 7_000_000).integers(16384, 40960, size=8, endpoint=True)
    out = {}
    for i, (name, (hq, hkv, d)) in enumerate(SHAPES.items()):
        s = W.make_step(name=name, dtype="bf16", hq=hq, hkv=hkv, d=d, block_size=256,
                        decode_lens=lens, seed=1200 + i)
        dev = DecodeStep(s, pkv)
        ms_step, per = time_parts([dev.run], args.steps, args.warmup, world, flush)
        nbytes = decode_append_bytes(s)
        tc = hq // hkv >= 4
        kernels = ("paged_decode_append (tensor-core pass + combine)" if tc else
                   "paged_decode_append (split kernel + combine)")
        out[name] = {"value": round(world * nbytes / (ms_step * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "ms_per_step": round(ms_step, 5), "bytes_per_step": nbytes,
                     "path": "tensor cores" if tc else "CUDA cores",
                     "roofline": hbm_roofline(kernels, nbytes, per[0][0], per[0][1], hbm_peak,
                                              peak_src, "decode_" + name)}
        line["gpu_launches"] += DecodeStep.launches * args.steps
        del dev
        torch.cuda.empty_cache()
    line["decode_shapes"] = {
        "metric": "decode KV GB/s at shapes beyond the workloads", "unit": "GB/s",
        "workload": "8 sequences, L~U[16384,40960], B=256, bf16, one paged_decode_append call; "
                    "L2 flushed between steps", "shapes": out}
    line["error_flags"] |= pkv.paged_error_flags()


def run_write(args, world, pkv, W, peaks, flush, line):
    """The slot_mapping write of the chunked-prefill workload's new rows
    (17,928 rows of 2 KiB each for K and V): slot build and paged_kv_write
    timed separately, the write against the HBM roofline."""
    hbm_peak, _, _, peak_src = peaks
    s = W.config(PREFILL_CFG)
    dev = PrefillStep(s, pkv)
    ms_step, per = time_parts([dev.slot_build, dev.write], args.steps, args.warmup, world,
                              flush)
    wb, sb = write_bytes(s), slot_build_bytes(s)
    line["kv_write"] = {
        "metric": "slot_mapping KV-cache write GB/s", "unit": "GB/s",
        "value": round(world * (wb + sb) / (ms_step * 1e-3) / 1e9, 2),
        "ms_per_step": round(ms_step, 5), "bytes_per_step": wb + sb,
        "workload": f"the chunked-prefill workload's {len(s.token_seq)} new rows "
                    f"(Hkv=8, d=128, bf16, B=256); step = paged_build_slot_mapping + "
                    f"paged_kv_write; L2 flushed between steps",
        "slot_build_ms": round(per[0][0], 5),
        "roofline": hbm_roofline("kv_write_copy_kernel (paged_kv_write)", wb, per[1][0],
                                 per[1][1], hbm_peak, peak_src, "kv_write")}
    line["gpu_launches"] += 2 * args.steps
    # the same rows through paged_kv_write_positions: slot build and write in
    # one launch (the slot mapping stored for other layers)
    ms_pos, per_pos = time_parts([dev.write_pos], args.steps, args.warmup, world, flush)
    line["kv_write"]["write_positions"] = {
        "value": round(world * (wb + sb) / (ms_pos * 1e-3) / 1e9, 2), "unit": "GB/s",
        "ms_per_step": round(ms_pos, 5), "bytes_per_step": wb + sb,
        "roofline": hbm_roofline("kv_write_copy_kernel<slots from positions> "
                                 "(paged_kv_write_positions)", wb + sb, per_pos[0][0],
                                 per_pos[0][1], hbm_peak, peak_src, "kv_write_positions")}
    line["gpu_launches"] += args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del dev
    torch.cuda.empty_cache()


W_NAME_PACKED = ("causal varlen prefill over packed K/V: the chunked-prefill workload's 16 "
                 "requests (q~U[1,2048], cached~U[0,2048]) with each request's keys "
                 "contiguous; L2 flushed between steps")
COPY_PAIRS, COPY_GEOM = 8192, (16, 8, 128)  # block pairs; B, Hkv, d (bf16)


def run_prefill(args, world, pkv, W, peaks, flush, line):
    _, bf16_peak, _, peak_src = peaks
    pstep = W.config(PREFILL_CFG)
    pdev = PrefillStep(pstep, pkv)
    try:
        pdev.attend()
    except pkv.PagedKVError as e:
        line["prefill"] = {"unavailable": str(e)}
        return
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    p_ms, per = time_parts([pdev.write_pos, pdev.attend], args.steps, args.warmup, world, flush)
    if not args.no_soak:
        soak(pdev.run)
    pclk = clocks.stop()
    pclk["window"] = "warm-up, timed region, then 0.5 s more of the same step (untimed)"
    flops = prefill_flops(pstep)
    pmean, pmed = per[1]
    tflops = flops / (pmean * 1e-3) / 1e12
    line["prefill"] = {
        "metric": "varlen prefill TFLOP/s", "workload": W.CONFIG_NAMES[PREFILL_CFG],
        "value": round(world * flops / (p_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_step": round(p_ms, 5),
        "step": "slot_mapping build and write of 16 requests' new K/V in one launch "
                "(paged_kv_write_positions) + causal varlen prefill (L2 flushed between "
                "steps, not timed)",
        "write_ms": round(per[0][0], 5),
        "flops_per_step": flops, "visible_pairs": prefill_pairs(pstep),
        "roofline": {"bound": "tensor", "kernel": "paged_varlen_prefill",
                     "achieved": round(tflops, 1), "peak": bf16_peak,
                     "unit": "TFLOP/s", "frac": round(tflops / bf16_peak, 4),
                     "peak_source": peak_src + " (bf16 burst)",
                     "traffic": traffic_of("chunked_prefill"),
                     "mean_ms": round(pmean, 5), "median_ms": round(pmed, 5)},
        "clocks": pclk,
    }
    line["gpu_launches"] += PrefillStep.launches * args.steps
    if not args.no_e2e:
        pe2e_ms, ph2d, pd2h = time_e2e(pdev, args.steps, args.warmup, world)
        line["prefill"]["e2e"] = {
            "value": round(world * flops / (pe2e_ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(pe2e_ms, 5),
            "h2d_bytes_per_step": ph2d, "d2h_bytes_per_step": pd2h}
        line["gpu_launches"] += PrefillStep.launches * args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    run_prefill_packed(args, world, pkv, pstep, pdev, flops, flush, bf16_peak, peak_src, line)
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
    t = pdev.dev
    call = lambda: pkv.paged_varlen_prefill(t["q"], kp, vp, t["cu_q"], t["cu_k"],
                                            s.max_seqlen_q, s.max_seqlen_k, None,
                                            causal=s.causal, scale=s.scale, out=pdev.out)
    _, per = time_parts([call], args.steps, args.warmup, world, flush)
    mean, med = per[0]
    tf = flops / (mean * 1e-3) / 1e12
    line["prefill_contiguous"] = {
        "metric": "varlen prefill TFLOP/s (packed K/V, block_table = NULL)",
        "workload": W_NAME_PACKED, "value": round(world * tf, 2), "unit": "TFLOP/s",
        "ms_per_step": round(mean, 5), "flops_per_step": flops,
        "roofline": {"bound": "tensor", "kernel": "paged_varlen_prefill (packed)",
                     "achieved": round(tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(tf / bf16_peak, 4), "peak_source": peak_src + " (bf16 burst)",
                     "traffic": traffic_of("chunked_prefill_packed"), "mean_ms": round(mean, 5),
                     "median_ms": round(med, 5)}}
    line["gpu_launches"] += args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del kp, vp


def run_copy(args, world, pkv, peaks, line):
    """paged_copy_blocks: the copies of copy-on-write.  8192 block pairs of a
    B=16, Hkv=8, d=128 bf16 pool (32 KiB per block per pool): 512 MiB read and
    512 MiB written per launch, far beyond L2."""
    hbm_peak, _, _, peak_src = peaks
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
    call = lambda: pkv.paged_copy_blocks(k_cache, v_cache, src, dst)
    _, per = time_parts([call], args.steps, args.warmup, world)
    mean, med = per[0]
    gbs = nbytes / (mean * 1e-3) / 1e9
    line["copy_blocks"] = {
        "metric": "copy-on-write block copies GB/s", "unit": "GB/s",
        "value": round(world * gbs, 1), "ms_per_step": round(mean, 5),
        "workload": f"{COPY_PAIRS} block pairs, B={B}, Hkv={hkv}, d={d}, bf16 "
                    f"({block_bytes // 1024} KiB per block per pool); step = one paged_copy_blocks",
        "roofline": hbm_roofline("copy_blocks_kernel", nbytes, mean, med, hbm_peak, peak_src,
                                 "copy_blocks"),
        "l2": "inputs larger than L2 (512 MiB read per launch)"}
    line["gpu_launches"] += args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del k_cache, v_cache
    torch.cuda.empty_cache()


def run_shared_prefix(args, world, pkv, W, peaks, flush, line):
    """Decode half of the continuous-batching workload: 256 sequences in 8
    groups of 32 that share a 2048-token prefix (128 blocks of 16), suffixes
    U[0,512] plus the new token.  Shared-prefix decode (each prefix block read
    once per group) against plain paged decode of the same step.  The roofline
    counts UNIQUE bytes: the prefixes once, every suffix, q and out."""
    hbm_peak, _, _, peak_src = peaks
    s = W.config(MIXED_CFG)
    nd = s.n_decode
    k_cache, v_cache = to_dev(s.k_cache), to_dev(s.v_cache)
    q, table, lens = to_dev(s.q_decode), to_dev(s.decode_table.copy()), to_dev(s.cache_seqlens)
    groups = 8
    gcu = to_dev(np.arange(0, nd + 1, nd // groups, dtype=np.int32))
    plen = to_dev(np.full(groups, 2048, np.int32))
    out = torch.empty_like(q)
    row = s.hkv * s.d * 2 * 2  # K + V bytes per key
    unique = (groups * 2048 + int((s.cache_seqlens - 2048).sum())) * row + 2 * q.numel() * 2
    logical = int(s.cache_seqlens.sum()) * row + 2 * q.numel() * 2
    ws = torch.empty(pkv._binding.load_library().paged_decode_shared_prefix_workspace_size(
        nd, ctypes.byref(pkv.geom_of(k_cache, s.hq))), dtype=torch.uint8, device="cuda")
    wsp = torch.empty(max(1, pkv.paged_decode_workspace_size(nd, s.hq, k_cache)),
                      dtype=torch.uint8, device="cuda")
    shared = lambda: pkv.paged_decode_shared_prefix(q, k_cache, v_cache, table, lens, gcu, plen,
                                                    nd // groups, s.scale, out=out, workspace=ws)
    plain = lambda: pkv.paged_decode(q, k_cache, v_cache, table, lens, s.scale, out=out,
                                     workspace=wsp)
    _, per = time_parts([shared], args.steps, args.warmup, world, flush)
    sh_ms, sh_med = per[0]
    _, per = time_parts([plain], args.steps, args.warmup, world, flush)
    pl_ms = per[0][0]
    gbs = unique / (sh_ms * 1e-3) / 1e9
    line["decode_shared_prefix"] = {
        "metric": "shared-prefix decode GB/s of unique K/V", "unit": "GB/s",
        "value": round(world * gbs, 1), "ms_per_step": round(sh_ms, 5),
        "workload": "decode half of the continuous-batching step: 256 sequences, 8 groups of "
                    "32 sharing a 2048-token prefix (B=16), suffixes U[0,512]+1, GQA 16/8, "
                    "d=128, bf16; L2 flushed between steps",
        "unique_bytes": unique, "logical_bytes": logical,
        "roofline": hbm_roofline("paged_decode_shared_prefix (every kernel of the call)", unique,
                                 sh_ms, sh_med, hbm_peak, peak_src, "shared_prefix_decode"),
        "plain_decode_same_step": {"ms": round(pl_ms, 5),
                                   "logical_GBps": round(logical / (pl_ms * 1e-3) / 1e9, 1),
                                   "speedup_of_shared": round(pl_ms / sh_ms, 3)}}
    line["gpu_launches"] += 5 * args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del k_cache, v_cache, ws, wsp
    torch.cuda.empty_cache()


def run_mixed_step(args, world, pkv, W, peaks, flush, line):
    """The whole continuous-batching step in one paged_mixed_step call: 2304
    new rows (+5 % padding) written, causal prefill of 4 x 512 tokens, and
    the in-place append + shared-prefix decode of 256 sequences.  Bytes
    counted once each: K/V of every key read (shared prefixes once), the new
    rows read and written, q and out."""
    hbm_peak, _, _, peak_src = peaks
    s = W.config(MIXED_CFG)
    nd = s.n_decode
    is_dec = (s.token_seq >= 0) & (s.token_seq < nd)
    dec_rows = np.where(is_dec)[0]
    dec_rows = dec_rows[np.argsort(s.token_seq[dec_rows])]
    pf_rows = np.where(~is_dec)[0]
    kc, vc = to_dev(s.k_cache), to_dev(s.v_cache)
    # the prefill rows' slots, built by the library (set-up, not timed)
    slots = pkv.paged_build_slot_mapping(to_dev(s.table), to_dev(s.token_seq),
                                         to_dev(s.token_pos), s.block_size)
    pf_idx = torch.from_numpy(pf_rows).cuda()
    decode = dict(q=to_dev(s.q_decode), k_new=to_dev(s.new_k[dec_rows]),
                  v_new=to_dev(s.new_v[dec_rows]), table=to_dev(s.decode_table.copy()),
                  seqlens=to_dev(s.cache_seqlens - 1),
                  group_cu=to_dev(np.arange(0, nd + 1, nd // 8, dtype=np.int32)),
                  group_prefix_len=to_dev(np.full(8, 2048, np.int32)), max_group_size=nd // 8,
                  out=torch.empty(s.q_decode.shape, dtype=torch.bfloat16, device="cuda"))
    prefill = dict(k_new=to_dev(s.new_k[pf_rows]), v_new=to_dev(s.new_v[pf_rows]),
                   slots=slots[pf_idx].contiguous(), q=to_dev(s.q_prefill), cu_q=to_dev(s.cu_q),
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
    call = lambda: pkv.paged_mixed_step(kc, vc, s.scale, prefill=prefill, decode=decode,
                                        workspace=ws)
    _, per = time_parts([call], args.steps, args.warmup, world, flush)
    mean, med = per[0]
    gbs = nbytes / (mean * 1e-3) / 1e9
    line["mixed_step"] = {
        "metric": "continuous-batching step GB/s of unique bytes", "unit": "GB/s",
        "value": round(world * gbs, 1), "ms_per_step": round(mean, 5),
        "workload": W.CONFIG_NAMES[MIXED_CFG] + "; one paged_mixed_step call; L2 flushed "
                    "between steps",
        "unique_bytes": nbytes,
        "roofline": hbm_roofline("paged_mixed_step (every kernel of the call)", nbytes, mean,
                                 med, hbm_peak, peak_src, "mixed_step")}
    line["gpu_launches"] += 4 * args.steps  # write, tensor-core launch, split, combine
    # the same step as ONE kernel launch (paged_mixed_step_one_launch)
    call1 = lambda: pkv.paged_mixed_step(kc, vc, s.scale, prefill=prefill, decode=decode,
                                         workspace=ws, one_launch=True)
    _, per1 = time_parts([call1], args.steps, args.warmup, world, flush)
    mean1, med1 = per1[0]
    gbs1 = nbytes / (mean1 * 1e-3) / 1e9
    line["mixed_step"]["one_launch"] = {
        "value": round(world * gbs1, 1), "unit": "GB/s", "ms_per_step": round(mean1, 5),
        "call": "paged_mixed_step_one_launch (one kernel: write, tensor-core items, split and "
                "combine as CTAs of one grid)",
        "roofline": hbm_roofline("step_one_kernel", nbytes, mean1, med1, hbm_peak, peak_src,
                                 "mixed_step_one_launch")}
    line["gpu_launches"] += args.steps
    line["error_flags"] |= pkv.paged_error_flags()
    del kc, vc, ws
    torch.cuda.empty_cache()


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
