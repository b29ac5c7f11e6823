"""The C-ABI library builds, loads and exports every entry point that
include/pagedkv.h declares; host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s+(\w+)\s*\(", text,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pkv.load_library()


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("paged_kv_write", "paged_decode", "paged_varlen_prefill",
              "paged_build_slot_mapping"):
        assert n in names
    assert set(names) == set(pkv.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.paged_status_string(0) == b"ok"
    assert lib.paged_status_string(-1) == b"invalid argument"
    assert lib.paged_status_string(-3) == b"workspace missing or too small"


def test_host_side_argument_checks(lib):
    """Checks that fail before any CUDA call (no GPU needed)."""
    g = pkv.Geom(16, 8, 128, 16, 100, pkv.PKV_BF16)
    assert lib.paged_kv_write(None, None, 1, None, 1, None, None, None, None) == -1
    bad = pkv.Geom(16, 6, 128, 16, 100, pkv.PKV_BF16)  # Hq % Hkv != 0
    assert lib.paged_kv_write(None, None, 1, None, 1, None, None, ctypes.byref(bad), None) == -1
    assert lib.paged_kv_write(None, None, 1, None, 0, None, None, ctypes.byref(g), None) == 0
    assert lib.paged_decode(None, None, None, None, 4, None, 0, 1.0, None, None, 0,
                            ctypes.byref(g), None) == 0  # empty batch
    assert lib.paged_decode(None, None, None, None, 4, None, 2, 1.0, None, None, 0,
                            ctypes.byref(g), None) == -1
    assert lib.paged_build_slot_mapping(None, 4, 1, None, None, -1, 16, None, None) == -1
    assert lib.paged_varlen_prefill_workspace_size(4, 100, None) == 0
    huge = pkv.Geom(16, 8, 128, 256, 1 << 24, pkv.PKV_BF16)  # 2^32 slots > int32
    assert lib.paged_kv_write(None, None, 1, None, 1, None, None, ctypes.byref(huge), None) == -2


def test_host_side_checks_of_the_step_calls(lib):
    """Shared-prefix decode, decode with append, prefill, the mixed step and
    the block copies reject bad arguments (-1) and unsupported combinations
    (-2) before any CUDA call, and accept empty work (0).  Pointer arguments
    are a non-null dummy: the host checks never dereference them."""
    g = ctypes.byref(pkv.Geom(16, 8, 128, 16, 100, pkv.PKV_BF16))
    f32 = ctypes.byref(pkv.Geom(16, 8, 128, 16, 100, pkv.PKV_F32))
    d96 = ctypes.byref(pkv.Geom(16, 8, 96, 16, 100, pkv.PKV_BF16))
    p = ctypes.c_void_p(256)
    shared = lib.paged_decode_shared_prefix
    assert shared(p, p, p, p, 4, p, 2, p, p, 0, 1, 1.0, p, p, 0, g, None) == -1  # no groups
    assert shared(None, p, p, p, 4, p, 2, p, p, 1, 2, 1.0, p, p, 0, g, None) == -1  # q null
    assert shared(p, p, p, p, 4, p, 2, p, p, 1, 2, 1.0, p, p, 0, f32, None) == -2  # bf16 only
    assert shared(None, None, None, None, 4, None, 0, None, None, 0, 0, 1.0, None, None, 0, g,
                  None) == 0  # empty batch
    append = lib.paged_decode_append
    assert append(None, p, p, p, p, p, 4, p, 2, 1.0, p, p, 0, g, None) == -1
    assert append(None, None, None, None, None, None, 4, None, 0, 1.0, None, None, 0, g, None) == 0
    prefill = lib.paged_varlen_prefill
    assert prefill(None, p, p, p, p, 2, 4, 4, p, 4, 1, 1.0, p, None, 0, g, None) == -1
    assert prefill(p, p, p, p, p, 2, 4, 4, p, 4, 1, 1.0, p, None, 0, f32, None) == -2
    assert prefill(p, p, p, p, p, 2, 4, 4, p, 4, 1, 1.0, p, None, 0, d96, None) == -2
    assert prefill(None, None, None, None, None, 0, 0, 0, None, 4, 1, 1.0, None, None, 0, g,
                   None) == 0
    assert lib.paged_mixed_step(None, p, p, None, 0, g, None) == -1
    assert lib.paged_copy_blocks(p, p, p, p, -1, g, None) == -1
    assert lib.paged_copy_blocks(p, p, None, p, 3, g, None) == -1
    assert lib.paged_copy_blocks(p, p, p, p, 70000, g, None) == -2
    assert lib.paged_copy_blocks(None, None, None, None, 0, g, None) == 0
    # batch 0 is paged_decode_noalloc's set-up call (it resolves the built-in
    # scratch array on the current device), so it needs a device
    import torch
    want = 0 if torch.cuda.is_available() else -4
    assert lib.paged_decode_noalloc(None, None, None, None, 4, None, 0, 1.0, None, g, None) == want


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        pkv.load_library(str(tmp_path / "missing.so"))


def test_every_source_is_compiled_once():
    """Every csrc/*.cu is either a translation unit of its own or included by
    step.cu (which compiles decode.cu, write.cu and prefill.cu together), never
    both: a source compiled twice would define its kernels twice."""
    csrc = build.CSRC
    step = open(os.path.join(csrc, "step.cu")).read()
    included = set(re.findall(r'^#include "(\w+\.cu)"', step, flags=re.M))
    assert included == set(build.INCLUDED)
    units = {os.path.basename(p) for p in build.sources()}
    every = {f for f in os.listdir(csrc) if f.endswith(".cu")}
    assert units | included == every
    assert not units & included
