"""CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (``paged_kv_cache_70_gb300``) never imports, links or runs it, and this
package imports nothing from the product.

The arithmetic lives in ``pagedkv_oracle.c`` (plain C, IEEE double, OpenMP over
independent (row, head) pairs); this module compiles it with gcc and wraps it
with ctypes over numpy arrays.  bf16 arrays are passed as ``uint16`` bit
patterns.  See the C file's header for the pages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .sizing import (  # noqa: F401  (re-exported)
    blocks_per_layer,
    kv_bytes_per_token,
    pool_blocks,
    pool_bytes,
    tokens_in_last_block,
)

F32, BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False, extra_flags: tuple[str, ...] = (), out_path: str | None = None) -> str:
    """Compile the oracle C file into a shared library; return its path.

    ``extra_flags`` / ``out_path`` let tests compile variants (for example with
    a planted mistake) without touching the default build.
    """
    out = out_path or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and out_path is None and os.path.exists(out) and \
            os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           *extra_flags, _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.ora_num_threads.restype = ctypes.c_int
        lib.ora_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.ora_f32_to_bf16.restype = ctypes.c_uint16
        lib.ora_slot_id.argtypes = [vp, i32, i64]
        lib.ora_slot_id.restype = i64
        lib.ora_element_offset.argtypes = [vp, i32, i64, i64]
        lib.ora_element_offset.restype = i64
        lib.ora_build_slot_mapping.argtypes = [vp, i32, vp, vp, i64, i32, vp]
        lib.ora_kv_write.argtypes = [vp, vp, ctypes.c_int, vp, i64, i64, vp, vp, ctypes.c_int]
        lib.ora_decode.argtypes = [vp, vp, vp, ctypes.c_int, vp, i32, vp, i32, i32, i32, i32,
                                   i32, dbl, vp, i32, vp]
        lib.ora_prefill.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, i32, vp, i32, i32,
                                    ctypes.c_int, i32, i32, i32, dbl, vp, i64, vp]
        lib.ora_request_index.argtypes = [vp, i32, vp]
        lib.ora_online_softmax_trace.argtypes = [vp, i64, vp, vp]
        lib.ora_online_attention.argtypes = [vp, vp, vp, i64, i32, dbl, vp, i64, vp, vp, vp]
        lib.ora_flash_tiles.argtypes = [vp, vp, vp, i64, i32, i64, i64, dbl, vp, vp, vp, vp]
        if path is None:
            _lib = lib
        return lib


# ---------------------------------------------------------------------------
# numpy-level wrappers
# ---------------------------------------------------------------------------

def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {a.dtype}")


def _c(a, dtype=None):
    return np.ascontiguousarray(a, dtype=dtype) if a is not None else None


def num_threads(lib=None) -> int:
    return int((lib or load()).ora_num_threads())


def f32_to_bf16(x: np.ndarray, lib=None) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (nearest, ties to even)."""
    lib = lib or load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.ora_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def widen(x: np.ndarray) -> np.ndarray:
    """Exact widening of float32 or bf16-bit arrays to float64."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def slot_id(table_row, block_size: int, pos: int, lib=None) -> int:
    lib = lib or load()
    t = _c(table_row, np.int32)
    return int(lib.ora_slot_id(_p(t), block_size, pos))


def element_offset(table_row, block_size: int, kv_dim: int, pos: int, lib=None) -> int:
    lib = lib or load()
    t = _c(table_row, np.int32)
    return int(lib.ora_element_offset(_p(t), block_size, kv_dim, pos))


def build_slot_mapping(block_table, token_seq, token_pos, block_size: int, lib=None) -> np.ndarray:
    """Slot id of every new-token row (-1 for padding rows with token_seq < 0)."""
    lib = lib or load()
    bt = _c(block_table, np.int32)
    ts = _c(token_seq, np.int32)
    tp = _c(token_pos, np.int32)
    out = np.full(ts.shape[0], -7, dtype=np.int32)
    lib.ora_build_slot_mapping(_p(bt), bt.shape[1], _p(ts), _p(tp), ts.shape[0], block_size,
                               _p(out))
    return out


def kv_write(k, v, slot_mapping, k_cache, v_cache, lib=None) -> None:
    """In-place slot_mapping write into numpy caches (float32 or bf16 bits)."""
    lib = lib or load()
    k = _c(k)
    v = _c(v)
    sm = _c(slot_mapping, np.int32)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    n = sm.shape[0]
    kv_dim = k.size // max(n, 1) if n else 0
    lib.ora_kv_write(_p(k), _p(v), _dtype_code(k), _p(sm), n, kv_dim, _p(k_cache), _p(v_cache),
                     _dtype_code(k_cache))


def decode(q, k_cache, v_cache, block_table, cache_seqlens, scale: float, seq_subset=None,
           lib=None) -> np.ndarray:
    """fp64 paged decode.  q [batch, Hq, d]; caches [num_blocks, B, Hkv, d]."""
    lib = lib or load()
    q = _c(q)
    bt = _c(block_table, np.int32)
    cs = _c(cache_seqlens, np.int32)
    batch, hq, d = q.shape
    _, bs, hkv, d2 = k_cache.shape
    assert d2 == d
    sub = _c(seq_subset, np.int32) if seq_subset is not None else None
    n_out = len(sub) if sub is not None else batch
    out = np.empty((n_out, hq, d), dtype=np.float64)
    lib.ora_decode(_p(q), _p(k_cache), _p(v_cache), _dtype_code(q), _p(bt), bt.shape[1], _p(cs),
                   batch, hq, hkv, d, bs, float(scale), _p(sub), n_out if sub is not None else 0,
                   _p(out))
    return out


def prefill(q, k_src, v_src, cu_q, cu_k, scale: float, causal: bool = True, block_table=None,
            block_size: int = 0, row_subset=None, lib=None) -> np.ndarray:
    """fp64 varlen prefill.  q [total_q, Hq, d].  With ``block_table`` the K/V
    sources are paged caches [num_blocks, B, Hkv, d]; without one they are the
    packed [total_k, Hkv, d] tensors."""
    lib = lib or load()
    q = _c(q)
    cq = _c(cu_q, np.int32)
    ck = _c(cu_k, np.int32)
    total_q, hq, d = q.shape
    if block_table is not None:
        _, bs, hkv, _ = k_src.shape
        bt = _c(block_table, np.int32)
        mb = bt.shape[1]
    else:
        _, hkv, _ = k_src.shape
        bt, mb, bs = None, 0, 0
    sub = _c(row_subset, np.int32) if row_subset is not None else None
    n_rows = len(sub) if sub is not None else total_q
    out = np.empty((n_rows, hq, d), dtype=np.float64)
    lib.ora_prefill(_p(q), _p(k_src), _p(v_src), _dtype_code(q), _p(cq), _p(ck), len(cq) - 1,
                    _p(bt), mb, bs, 1 if causal else 0, hq, hkv, d, float(scale), _p(sub),
                    n_rows if sub is not None else 0, _p(out))
    return out


def request_index(cu, lib=None) -> np.ndarray:
    lib = lib or load()
    c = _c(cu, np.int32)
    out = np.full(int(c[-1]), -1, dtype=np.int32)
    lib.ora_request_index(_p(c), len(c) - 1, _p(out))
    return out


def online_softmax_trace(x, lib=None):
    lib = lib or load()
    x = _c(x, np.float64)
    m = np.empty_like(x)
    l = np.empty_like(x)
    lib.ora_online_softmax_trace(_p(x), x.size, _p(m), _p(l))
    return m, l


def online_attention(q, K, V, scale: float, chunk_lens, lib=None):
    """Block-wise online attention of one query over dense K/V [n, d]."""
    lib = lib or load()
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    cl = _c(chunk_lens, np.int64)
    n, d = K.shape
    out = np.empty(d, dtype=np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    lib.ora_online_attention(_p(q), _p(K), _p(V), n, d, float(scale), _p(cl), cl.size, _p(out),
                             ctypes.byref(m), ctypes.byref(l))
    return out, m.value, l.value


def flash_tiles(Q, K, V, Br: int, Bc: int, scale: float, lib=None):
    """FlashAttention Q-outer / K-inner tiling; returns O and per-step history."""
    lib = lib or load()
    Q = _c(Q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    N, d = Q.shape
    nq, nk = -(-N // Br), -(-N // Bc)
    O = np.empty((N, d), dtype=np.float64)
    mh = np.full((nq, nk, Br), np.nan)
    lh = np.full((nq, nk, Br), np.nan)
    ch = np.full((nq, nk, Br), np.nan)
    lib.ora_flash_tiles(_p(Q), _p(K), _p(V), N, d, Br, Bc, float(scale), _p(O), _p(mh), _p(lh),
                        _p(ch))
    return O, mh, lh, ch
