"""paged_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (a plugin whose host framework owns every device
allocation, or a serving loop that must not call cudaMalloc because it can
synchronise the device), through the C ABI.

Its scratch is one process-wide array inside the library that every call
reuses.  The checks therefore run several calls in a row on that array: the
Qwen3-shaped decode, a small step with a different length mix, then the
Qwen3-shaped decode again, which must reproduce its first result bit for bit
(a larger problem after a smaller one: every scratch byte read must have been
written by the same call).  Each result is compared with paged_decode and
with the CPU oracle.

The file name sorts last on purpose: the array is shared by the whole
process, so a failure here may leave it in any state; collected last, a run
that stops at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep, assert_close, widen

pytestmark = pytest.mark.gpu


def _noalloc(lib, dev, out, batch=None):
    s = dev.s
    g = pkv.geom_of(dev.k_cache, s.hq)
    st = lib.paged_decode_noalloc(
        ctypes.c_void_p(dev.q_decode.data_ptr()), ctypes.c_void_p(dev.k_cache.data_ptr()),
        ctypes.c_void_p(dev.v_cache.data_ptr()), ctypes.c_void_p(dev.decode_table.data_ptr()),
        dev.decode_table.shape[1], ctypes.c_void_p(dev.cache_seqlens.data_ptr()),
        s.n_decode if batch is None else batch, s.scale, ctypes.c_void_p(out.data_ptr()),
        ctypes.byref(g), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_paged_decode_and_oracle_on_calls_in_a_row():
    lib = pkv.load_library()
    big = W.config(2)
    small = W.make_step(name="mix", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                        decode_lens=[0, 5000, 17, 300, 1], seed=12)
    devs = {"big": DevStep(big), "small": DevStep(small)}
    # set-up call (batch 0): resolves the scratch array, launches nothing
    probe = torch.empty_like(devs["small"].q_decode)
    assert _noalloc(lib, devs["small"], probe, batch=0) == 0
    first = None
    for name in ("big", "small", "big"):
        dev = devs[name]
        s = dev.s
        want_gpu = dev.decode()
        out = torch.full_like(dev.q_decode, float("nan"))
        assert _noalloc(lib, dev, out) == 0
        torch.cuda.synchronize()
        assert_close(widen(out), widen(want_gpu), s.dtype, f"{name} vs paged_decode")
        want = oracle.decode(s.q_decode, s.k_cache, s.v_cache, s.decode_table, s.cache_seqlens,
                             s.scale)
        assert_close(widen(out), want, s.dtype, f"{name} vs oracle")
        if name == "big":
            if first is None:
                first = out.clone()
            else:  # the same problem again after a smaller one: identical bits
                assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert pkv.paged_error_flags() == 0


def test_noalloc_rejects_problems_beyond_the_scratch():
    lib = pkv.load_library()
    step = W.make_step(name="big", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                       decode_lens=[1] * 3000, seed=13)
    dev = DevStep(step)
    need = pkv.paged_decode_workspace_size(step.n_decode, step.hq, dev.k_cache)
    assert need > (8 << 20)
    out = torch.zeros_like(dev.q_decode)
    assert _noalloc(lib, dev, out) == -3
    assert torch.count_nonzero(out) == 0
