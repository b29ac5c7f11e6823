"""A decode whose pipeline wait runs out, on a test-only build of the split
kernel: its producer issues no copy and every wait gives up after 1 ms.  The
consumers' first wait then times out with nothing in flight (decode uses no
TMEM).  The call must return, the kernels must finish, and the device error
word of that build must carry PKV_FLAG_TIMEOUT.  With two KV heads the eight
consumer warps share heads and merge through time-limited barriers, which must
not hold any warp after the timeout.

The build compiles step.cu (the unit that holds the decode kernels) with the
two test defines into its own library (_build/test_wait_timeout/); the default
library is not changed."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import build as B
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep

pytestmark = pytest.mark.gpu

DEFINES = ("-DPKV_WAIT_LIMIT_NS=1000000ull", "-DPKV_TEST_SPLIT_PRODUCER_IDLE")


@pytest.fixture(scope="module")
def timeout_lib():
    return pkv.load_library(B.build_variant("test_wait_timeout", DEFINES, ("step.cu",)))


def _flags(lib, clear=1):
    v = ctypes.c_uint32(0)
    assert lib.paged_error_flags(ctypes.byref(v), clear) == 0
    return v.value


@pytest.mark.parametrize("hq,hkv", [(16, 8), (4, 2)])
def test_decode_wait_timeout_sets_flag_and_returns(timeout_lib, hq, hkv):
    lib = timeout_lib
    step = W.make_step(name="timeout", dtype="bf16", hq=hq, hkv=hkv, d=128, block_size=16,
                       decode_lens=[100, 37, 500, 2000], seed=5)
    dev = DevStep(step)
    g = pkv.geom_of(dev.k_cache, step.hq)
    need = lib.paged_decode_workspace_size(step.n_decode, ctypes.byref(g))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.full_like(dev.q_decode, float("nan"))
    torch.cuda.synchronize()
    _flags(lib)  # clear the timeout library's error word
    pkv.paged_error_flags()  # and the default library's
    st = lib.paged_decode(
        ctypes.c_void_p(dev.q_decode.data_ptr()), ctypes.c_void_p(dev.k_cache.data_ptr()),
        ctypes.c_void_p(dev.v_cache.data_ptr()), ctypes.c_void_p(dev.decode_table.data_ptr()),
        dev.decode_table.shape[1], ctypes.c_void_p(dev.cache_seqlens.data_ptr()), step.n_decode,
        step.scale, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), need,
        ctypes.byref(g), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()  # the kernels finished: every wait gave up after 1 ms
    assert _flags(lib) & pkv.PKV_FLAG_TIMEOUT
    assert pkv.paged_error_flags() == 0  # the default library saw nothing
    # (the output of a call whose wait ran out is unspecified: only the flag
    # says so)
    # the default library still decodes correctly on the same inputs
    want = dev.decode()
    torch.cuda.synchronize()
    assert np.isfinite(want.float().cpu().numpy()).all()
    assert pkv.paged_error_flags() == 0
