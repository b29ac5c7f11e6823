"""paged_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (a plugin whose host framework owns every device
allocation, or a serving loop that must not call cudaMalloc), against
paged_decode on the same inputs.  It runs through the C ABI and must match on
two calls in a row: the second call reuses the built-in scratch array the first
one left behind.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep, assert_close, widen

pytestmark = pytest.mark.gpu


def _noalloc(lib, dev, out):
    s = dev.s
    g = pkv.geom_of(dev.k_cache, s.hq)
    st = lib.paged_decode_noalloc(
        ctypes.c_void_p(dev.q_decode.data_ptr()), ctypes.c_void_p(dev.k_cache.data_ptr()),
        ctypes.c_void_p(dev.v_cache.data_ptr()), ctypes.c_void_p(dev.decode_table.data_ptr()),
        dev.decode_table.shape[1], ctypes.c_void_p(dev.cache_seqlens.data_ptr()), s.n_decode,
        s.scale, ctypes.c_void_p(out.data_ptr()), ctypes.byref(g),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_paged_decode_twice():
    lib = pkv.load_library()
    steps = [W.config(2), W.make_step(name="mix", dtype="bf16", hq=16, hkv=8, d=128,
                                      block_size=16, decode_lens=[0, 5000, 17, 300, 1],
                                      seed=12)]
    for step in steps:  # two calls in a row, different length mixes
        dev = DevStep(step)
        want = dev.decode()
        out = torch.full_like(dev.q_decode, float("nan"))
        assert _noalloc(lib, dev, out) == 0
        torch.cuda.synchronize()
        assert_close(widen(out), widen(want), step.dtype, step.name)
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
