"""ctypes binding of libpagedkv.so (include/pagedkv.h).

Argument marshalling only: shapes and dtypes are read from torch tensors,
device pointers and the current CUDA stream are passed to the C ABI, and a
non-zero status raises :class:`PagedKVError`.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback path.  PyTorch is used
for device memory and streams.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpagedkv.so")

PKV_F32, PKV_BF16 = 0, 1
PKV_FLAG_BAD_BLOCK = 1 << 0
PKV_FLAG_BAD_SLOT = 1 << 1
PKV_FLAG_BAD_LENGTH = 1 << 2
PKV_FLAG_BAD_SEQ = 1 << 3
PKV_FLAG_TIMEOUT = 1 << 4

# every extern "C" entry point of include/pagedkv.h
EXPORTED = (
    "paged_build_slot_mapping",
    "paged_kv_write",
    "paged_kv_write_positions",
    "paged_decode_workspace_size",
    "paged_decode",
    "paged_varlen_prefill_workspace_size",
    "paged_varlen_prefill",
    "paged_error_flags",
    "paged_status_string",
    "paged_decode_noalloc",
    "paged_bm_create",
    "paged_bm_destroy",
    "paged_bm_allocate",
    "paged_bm_fork",
    "paged_bm_append",
    "paged_bm_free",
    "paged_bm_block_table",
    "paged_bm_seq_len",
    "paged_bm_ref_count",
    "paged_bm_free_blocks",
    "paged_copy_blocks",
    "paged_decode_shared_prefix_workspace_size",
    "paged_decode_shared_prefix",
    "paged_decode_append",
    "paged_mixed_step_workspace_size",
    "paged_mixed_step",
    "paged_mixed_step_one_launch",
)
PKV_ERR_NO_SPACE = -5


class PagedKVError(RuntimeError):
    def __init__(self, func: str, status: int, msg: str):
        super().__init__(f"{func} failed with status {status}: {msg}")
        self.status = status


class Geom(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
    ]


class MixedStep(ctypes.Structure):
    """pkv_mixed_step of include/pagedkv.h"""
    _fields_ = [
        ("prefill_k_new", ctypes.c_void_p), ("prefill_v_new", ctypes.c_void_p),
        ("prefill_slots", ctypes.c_void_p), ("prefill_new_tokens", ctypes.c_int64),
        ("prefill_q", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p), ("prefill_batch", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32), ("max_seqlen_k", ctypes.c_int32),
        ("prefill_table", ctypes.c_void_p), ("prefill_max_blocks", ctypes.c_int32),
        ("prefill_out", ctypes.c_void_p),
        ("decode_q", ctypes.c_void_p), ("decode_k_new", ctypes.c_void_p),
        ("decode_v_new", ctypes.c_void_p), ("decode_table", ctypes.c_void_p),
        ("decode_max_blocks", ctypes.c_int32), ("decode_seqlens", ctypes.c_void_p),
        ("decode_batch", ctypes.c_int32), ("group_cu", ctypes.c_void_p),
        ("group_prefix_len", ctypes.c_void_p), ("n_groups", ctypes.c_int32),
        ("max_group_size", ctypes.c_int32), ("decode_out", ctypes.c_void_p),
        ("scale", ctypes.c_float),
    ]


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None):
    """Load libpagedkv.so (built in-tree by ``paged_kv_cache_70_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libpagedkv.so not found at {p}; build it with "
                "`python -m paged_kv_cache_70_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(p)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        gp = ctypes.POINTER(Geom)
        lib.paged_build_slot_mapping.argtypes = [vp, i32, i32, vp, vp, i64, i32, vp, vp]
        lib.paged_build_slot_mapping.restype = ctypes.c_int
        lib.paged_kv_write.argtypes = [vp, vp, i32, vp, i64, vp, vp, gp, vp]
        lib.paged_kv_write.restype = ctypes.c_int
        lib.paged_kv_write_positions.argtypes = [vp, vp, i32, vp, i32, i32, vp, vp, i64, vp, vp,
                                                 vp, gp, vp]
        lib.paged_kv_write_positions.restype = ctypes.c_int
        lib.paged_decode_workspace_size.argtypes = [i32, gp]
        lib.paged_decode_workspace_size.restype = sz
        lib.paged_decode.argtypes = [vp, vp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp, sz,
                                     gp, vp]
        lib.paged_decode.restype = ctypes.c_int
        lib.paged_varlen_prefill_workspace_size.argtypes = [i32, i32, gp]
        lib.paged_varlen_prefill_workspace_size.restype = sz
        lib.paged_varlen_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, i32, i32,
                                             ctypes.c_float, vp, vp, sz, gp, vp]
        lib.paged_varlen_prefill.restype = ctypes.c_int
        lib.paged_decode_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, i32, ctypes.c_float, vp,
                                             gp, vp]
        lib.paged_decode_noalloc.restype = ctypes.c_int
        lib.paged_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.paged_error_flags.restype = ctypes.c_int
        pp, i64p, i32p = ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i32)
        lib.paged_bm_create.argtypes = [i64, i32, pp]
        lib.paged_bm_destroy.argtypes = [vp]
        lib.paged_bm_allocate.argtypes = [vp, vp, i64, i64p, i64p]
        lib.paged_bm_fork.argtypes = [vp, i64, i64p]
        lib.paged_bm_append.argtypes = [vp, i64, i64, i32p, i32p]
        lib.paged_bm_free.argtypes = [vp, i64]
        lib.paged_bm_block_table.argtypes = [vp, i64, vp, i32, i32p]
        lib.paged_bm_seq_len.argtypes = [vp, i64, i64p]
        lib.paged_bm_ref_count.argtypes = [vp, i32, i32p]
        lib.paged_bm_free_blocks.argtypes = [vp, vp, i64, i64p]
        for f in ("create", "destroy", "allocate", "fork", "append", "free", "block_table",
                  "seq_len", "ref_count", "free_blocks"):
            getattr(lib, "paged_bm_" + f).restype = ctypes.c_int
        lib.paged_decode_shared_prefix_workspace_size.argtypes = [i32, gp]
        lib.paged_decode_shared_prefix_workspace_size.restype = sz
        lib.paged_decode_shared_prefix.argtypes = [vp, vp, vp, vp, i32, vp, i32, vp, vp, i32, i32,
                                                   ctypes.c_float, vp, vp, sz, gp, vp]
        lib.paged_decode_shared_prefix.restype = ctypes.c_int
        lib.paged_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, ctypes.c_float,
                                            vp, vp, sz, gp, vp]
        lib.paged_decode_append.restype = ctypes.c_int
        lib.paged_mixed_step_workspace_size.argtypes = [i32, gp]
        lib.paged_mixed_step_workspace_size.restype = sz
        lib.paged_mixed_step.argtypes = [ctypes.POINTER(MixedStep), vp, vp, vp, sz, gp, vp]
        lib.paged_mixed_step.restype = ctypes.c_int
        lib.paged_mixed_step_one_launch.argtypes = [ctypes.POINTER(MixedStep), vp, vp, vp, sz, gp,
                                                    vp]
        lib.paged_mixed_step_one_launch.restype = ctypes.c_int
        lib.paged_copy_blocks.argtypes = [vp, vp, vp, vp, i32, gp, vp]
        lib.paged_copy_blocks.restype = ctypes.c_int
        lib.paged_status_string.argtypes = [ctypes.c_int]
        lib.paged_status_string.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _check(func: str, status: int) -> None:
    if status != 0:
        msg = load_library().paged_status_string(status).decode()
        raise PagedKVError(func, status, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _cuda_contig(name: str, t: torch.Tensor, dtype=None) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def geom_of(k_cache: torch.Tensor, num_heads: int) -> Geom:
    """pkv_geom of a pool [num_blocks, block_size, num_kv_heads, head_dim]."""
    nb, bs, hkv, d = k_cache.shape
    return Geom(num_heads, hkv, d, bs, nb, _dtype_code(k_cache))


def paged_build_slot_mapping(block_table: torch.Tensor, token_seq: torch.Tensor,
                             token_pos: torch.Tensor, block_size: int,
                             out: torch.Tensor | None = None) -> torch.Tensor:
    """slot_mapping[n] = table[s][p // B] * B + p % B (-1 where token_seq < 0)."""
    for n, t in (("block_table", block_table), ("token_seq", token_seq), ("token_pos", token_pos)):
        _cuda_contig(n, t, torch.int32)
    n_tok = token_seq.numel()
    if out is None:
        out = torch.empty(n_tok, dtype=torch.int32, device=token_seq.device)
    _cuda_contig("out", out, torch.int32)
    rows, width = block_table.shape
    st = load_library().paged_build_slot_mapping(
        _ptr(block_table), width, rows, _ptr(token_seq), _ptr(token_pos), n_tok, block_size,
        _ptr(out), _stream(token_seq))
    _check("paged_build_slot_mapping", st)
    return out


def paged_kv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """In-place write of k/v [N, Hkv, d] rows into the pools at slot_mapping."""
    _cuda_contig("k", k)
    _cuda_contig("v", v, k.dtype)
    _cuda_contig("slot_mapping", slot_mapping, torch.int32)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    if k.shape != v.shape or k.shape[1:] != k_cache.shape[2:] or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between k/v rows and the pools")
    if slot_mapping.numel() != k.shape[0]:
        raise ValueError("slot_mapping must have one entry per token row")
    g = geom_of(k_cache, k_cache.shape[2])
    st = load_library().paged_kv_write(_ptr(k), _ptr(v), _dtype_code(k), _ptr(slot_mapping),
                                       k.shape[0], _ptr(k_cache), _ptr(v_cache),
                                       ctypes.byref(g), _stream(k))
    _check("paged_kv_write", st)


def paged_kv_write_positions(k: torch.Tensor, v: torch.Tensor, block_table: torch.Tensor,
                             token_seq: torch.Tensor, token_pos: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor,
                             slot_mapping_out: torch.Tensor | None = None) -> None:
    """paged_build_slot_mapping and paged_kv_write in one launch; the slots go
    to slot_mapping_out when given."""
    _cuda_contig("k", k)
    _cuda_contig("v", v, k.dtype)
    for n, t in (("block_table", block_table), ("token_seq", token_seq), ("token_pos", token_pos)):
        _cuda_contig(n, t, torch.int32)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    if k.shape != v.shape or k.shape[1:] != k_cache.shape[2:] or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between k/v rows and the pools")
    n_tok = k.shape[0]
    if token_seq.numel() != n_tok or token_pos.numel() != n_tok:
        raise ValueError("token_seq and token_pos must have one entry per token row")
    if slot_mapping_out is not None:
        _cuda_contig("slot_mapping_out", slot_mapping_out, torch.int32)
        if slot_mapping_out.numel() != n_tok:
            raise ValueError("slot_mapping_out must have one entry per token row")
    rows, width = block_table.shape
    g = geom_of(k_cache, k_cache.shape[2])
    st = load_library().paged_kv_write_positions(
        _ptr(k), _ptr(v), _dtype_code(k), _ptr(block_table), width, rows, _ptr(token_seq),
        _ptr(token_pos), n_tok, _ptr(slot_mapping_out),
        _ptr(k_cache), _ptr(v_cache), ctypes.byref(g), _stream(k))
    _check("paged_kv_write_positions", st)


def paged_decode_workspace_size(batch: int, q_heads: int, k_cache: torch.Tensor) -> int:
    g = geom_of(k_cache, q_heads)
    with torch.cuda.device(k_cache.device):
        return int(load_library().paged_decode_workspace_size(batch, ctypes.byref(g)))


def paged_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_table: torch.Tensor, cache_seqlens: torch.Tensor,
                 scale: float | None = None, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One query token per sequence over its cache_seqlens[b] cached keys."""
    _cuda_contig("q", q, k_cache.dtype)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("cache_seqlens", cache_seqlens, torch.int32)
    batch, hq, d = q.shape
    if d != k_cache.shape[3] or block_table.shape[0] < batch or cache_seqlens.numel() < batch:
        raise ValueError("shape mismatch")
    g = geom_of(k_cache, hq)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = int(lib.paged_decode_workspace_size(batch, ctypes.byref(g)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = lib.paged_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                              block_table.shape[1], _ptr(cache_seqlens), batch, scale, _ptr(out),
                              _ptr(workspace), workspace.numel(), ctypes.byref(g), _stream(q))
    _check("paged_decode", st)
    return out


def paged_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_table: torch.Tensor, cache_seqlens: torch.Tensor,
                         scale: float | None = None,
                         out: torch.Tensor | None = None) -> torch.Tensor:
    """paged_decode without a workspace, for callers that cannot allocate
    device memory: the library's built-in scratch array is used instead (see
    include/pagedkv.h; calls that overlap on the GPU race on that array)."""
    _cuda_contig("q", q, k_cache.dtype)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("cache_seqlens", cache_seqlens, torch.int32)
    batch, hq, d = q.shape
    g = geom_of(k_cache, hq)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = load_library().paged_decode_noalloc(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
            _ptr(cache_seqlens), batch, scale, _ptr(out), ctypes.byref(g), _stream(q))
    _check("paged_decode_noalloc", st)
    return out


def paged_decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                        cache_seqlens: torch.Tensor, scale: float | None = None,
                        out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Decode with the in-place append: k_new/v_new [batch, Hkv, d] are written
    at position cache_seqlens[b] (keys cached before the step) and attended to
    together with the cached keys."""
    _cuda_contig("q", q, k_cache.dtype)
    _cuda_contig("k_new", k_new, k_cache.dtype)
    _cuda_contig("v_new", v_new, k_cache.dtype)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("cache_seqlens", cache_seqlens, torch.int32)
    batch, hq, d = q.shape
    if k_new.shape != (batch,) + tuple(k_cache.shape[2:]) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [batch, Hkv, d]")
    g = geom_of(k_cache, hq)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = int(lib.paged_decode_workspace_size(batch, ctypes.byref(g)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = lib.paged_decode_append(
            _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
            block_table.shape[1], _ptr(cache_seqlens), batch, scale, _ptr(out), _ptr(workspace),
            workspace.numel(), ctypes.byref(g), _stream(q))
    _check("paged_decode_append", st)
    return out


def paged_decode_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_table: torch.Tensor, cache_seqlens: torch.Tensor,
                               group_cu: torch.Tensor, group_prefix_len: torch.Tensor,
                               max_group_size: int, scale: float | None = None,
                               out: torch.Tensor | None = None,
                               workspace: torch.Tensor | None = None) -> torch.Tensor:
    """paged_decode for a batch ordered by groups (sequences group_cu[g] ..
    group_cu[g+1]-1) whose first group_prefix_len[g] keys sit in shared blocks:
    each shared block is read once per group."""
    _cuda_contig("q", q, k_cache.dtype)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    _cuda_contig("block_table", block_table, torch.int32)
    _cuda_contig("cache_seqlens", cache_seqlens, torch.int32)
    _cuda_contig("group_cu", group_cu, torch.int32)
    _cuda_contig("group_prefix_len", group_prefix_len, torch.int32)
    batch, hq, d = q.shape
    n_groups = group_cu.numel() - 1
    if group_prefix_len.numel() < n_groups or block_table.shape[0] < batch:
        raise ValueError("shape mismatch")
    g = geom_of(k_cache, hq)
    lib = load_library()
    with torch.cuda.device(q.device):
        need = int(lib.paged_decode_shared_prefix_workspace_size(batch, ctypes.byref(g)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = lib.paged_decode_shared_prefix(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
            _ptr(cache_seqlens), batch, _ptr(group_cu), _ptr(group_prefix_len), n_groups,
            int(max_group_size), scale, _ptr(out), _ptr(workspace), workspace.numel(),
            ctypes.byref(g), _stream(q))
    _check("paged_decode_shared_prefix", st)
    return out


def paged_varlen_prefill_workspace_size(batch: int, max_seqlen_q: int, q_heads: int,
                                        k_cache: torch.Tensor) -> int:
    g = geom_of(k_cache, q_heads)
    return int(load_library().paged_varlen_prefill_workspace_size(batch, max_seqlen_q,
                                                                 ctypes.byref(g)))


def paged_varlen_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                         max_seqlen_q: int, max_seqlen_k: int, block_table: torch.Tensor | None,
                         causal: bool = True, scale: float | None = None,
                         out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Causal varlen prefill of q [total_q, Hq, d] over the paged cache, or
    (block_table None) over packed K/V [total_k, Hkv, d] whose request r holds
    rows cu_seqlens_k[r] .. cu_seqlens_k[r+1]-1."""
    _cuda_contig("q", q, k_cache.dtype)
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    _cuda_contig("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _cuda_contig("cu_seqlens_k", cu_seqlens_k, torch.int32)
    batch = cu_seqlens_q.numel() - 1
    total_q, hq, d = q.shape
    if block_table is None:
        if k_cache.dim() != 3 or v_cache.shape != k_cache.shape:
            raise ValueError("packed K/V must be [total_k, Hkv, d]")
        rows, hkv, dk = k_cache.shape
        g = Geom(hq, hkv, dk, 1, rows, _dtype_code(k_cache))
    else:
        _cuda_contig("block_table", block_table, torch.int32)
        g = geom_of(k_cache, hq)
    lib = load_library()
    need = int(lib.paged_varlen_prefill_workspace_size(batch, max_seqlen_q, ctypes.byref(g)))
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _cuda_contig("out", out, q.dtype)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = lib.paged_varlen_prefill(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch,
            int(max_seqlen_q), int(max_seqlen_k), _ptr(block_table),
            0 if block_table is None else block_table.shape[1],
            1 if causal else 0, scale, _ptr(out), _ptr(workspace),
            0 if workspace is None else workspace.numel(), ctypes.byref(g), _stream(q))
    _check("paged_varlen_prefill", st)
    return out


def paged_error_flags(clear: bool = True) -> int:
    """Device error word of the current device (PKV_FLAG_* bits)."""
    v = ctypes.c_uint32(0)
    _check("paged_error_flags", load_library().paged_error_flags(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


class BlockManager:
    """Host-side block manager of one pool (reference counts, free stack,
    prefix sharing of full blocks, copy-on-write), a handle on the library's
    native manager (include/pagedkv.h, paged_bm_*)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check("paged_bm_create", self._lib.paged_bm_create(num_blocks, block_size,
                                                            ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self) -> None:
        if self._h:
            self._lib.paged_bm_destroy(self._h)
            self._h = None

    def __del__(self):  # pragma: no cover - interpreter shutdown order
        try:
            self.close()
        except Exception:
            pass

    def allocate(self, tokens) -> tuple[int, int]:
        """New sequence; returns (sequence id, tokens already cached)."""
        arr = (ctypes.c_int64 * max(1, len(tokens)))(*[int(t) for t in tokens])
        sid, cached = ctypes.c_int64(), ctypes.c_int64()
        _check("paged_bm_allocate", self._lib.paged_bm_allocate(
            self._h, ctypes.cast(arr, ctypes.c_void_p), len(tokens), ctypes.byref(sid),
            ctypes.byref(cached)))
        return sid.value, cached.value

    def fork(self, seq: int) -> int:
        c = ctypes.c_int64()
        _check("paged_bm_fork", self._lib.paged_bm_fork(self._h, seq, ctypes.byref(c)))
        return c.value

    def append(self, seq: int, token: int) -> tuple[int, int]:
        """Returns the (src, dst) block copy the write needs first, or (-1, -1)."""
        s, d = ctypes.c_int32(), ctypes.c_int32()
        _check("paged_bm_append", self._lib.paged_bm_append(self._h, seq, int(token),
                                                            ctypes.byref(s), ctypes.byref(d)))
        return s.value, d.value

    def free(self, seq: int) -> None:
        _check("paged_bm_free", self._lib.paged_bm_free(self._h, seq))

    def table(self, seq: int) -> list[int]:
        n = ctypes.c_int32()
        self._lib.paged_bm_block_table(self._h, seq, None, 0, ctypes.byref(n))
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check("paged_bm_block_table", self._lib.paged_bm_block_table(
            self._h, seq, ctypes.cast(buf, ctypes.c_void_p), n.value, ctypes.byref(n)))
        return list(buf[: n.value])

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int64()
        _check("paged_bm_seq_len", self._lib.paged_bm_seq_len(self._h, seq, ctypes.byref(n)))
        return n.value

    def ref_count(self, block: int) -> int:
        r = ctypes.c_int32()
        _check("paged_bm_ref_count", self._lib.paged_bm_ref_count(self._h, block,
                                                                  ctypes.byref(r)))
        return r.value

    def free_stack(self) -> list[int]:
        """Free blocks, bottom of the stack first."""
        n = ctypes.c_int64()
        _check("paged_bm_free_blocks", self._lib.paged_bm_free_blocks(self._h, None, 0,
                                                                      ctypes.byref(n)))
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check("paged_bm_free_blocks", self._lib.paged_bm_free_blocks(
            self._h, ctypes.cast(buf, ctypes.c_void_p), n.value, ctypes.byref(n)))
        return list(buf[: n.value])

    def num_free(self) -> int:
        n = ctypes.c_int64()
        _check("paged_bm_free_blocks", self._lib.paged_bm_free_blocks(self._h, None, 0,
                                                                      ctypes.byref(n)))
        return n.value


def paged_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src: torch.Tensor,
                      dst: torch.Tensor) -> None:
    """Block dst[i] of both pools becomes a copy of block src[i] (int32 CUDA
    tensors): the copies a copy-on-write needs."""
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    _cuda_contig("src", src, torch.int32)
    _cuda_contig("dst", dst, torch.int32)
    if src.numel() != dst.numel() or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    g = geom_of(k_cache, k_cache.shape[2])
    with torch.cuda.device(k_cache.device):
        st = load_library().paged_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src), _ptr(dst),
                                              src.numel(), ctypes.byref(g), _stream(k_cache))
    _check("paged_copy_blocks", st)


def paged_mixed_step(k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float,
                     prefill: dict | None = None, decode: dict | None = None,
                     workspace: torch.Tensor | None = None, one_launch: bool = False):
    """One continuous-batching step (include/pagedkv.h, paged_mixed_step;
    paged_mixed_step_one_launch with one_launch=True).

    prefill: k_new, v_new [N, Hkv, d] and slots [N] (the requests' new rows,
    negative slots skipped), q [total_q, Hq, d], cu_q, cu_k, max_q, max_k,
    table; decode: q [batch, Hq, d], k_new, v_new [batch, Hkv, d], table,
    seqlens (keys cached before the step), optionally group_cu,
    group_prefix_len, max_group_size.  Returns (prefill_out, decode_out)."""
    _cuda_contig("k_cache", k_cache)
    _cuda_contig("v_cache", v_cache, k_cache.dtype)
    st = MixedStep()
    st.scale = float(scale)
    keep = []
    pout = dout = None
    hq = None
    if prefill:
        for n in ("k_new", "v_new", "q"):
            _cuda_contig("prefill " + n, prefill[n], k_cache.dtype)
        for n in ("slots", "cu_q", "cu_k", "table"):
            _cuda_contig("prefill " + n, prefill[n], torch.int32)
        pout = prefill.get("out")
        if pout is None:
            pout = torch.empty_like(prefill["q"])
        hq = prefill["q"].shape[1]
        st.prefill_k_new, st.prefill_v_new = prefill["k_new"].data_ptr(), prefill["v_new"].data_ptr()
        st.prefill_slots = prefill["slots"].data_ptr()
        st.prefill_new_tokens = prefill["slots"].numel()
        st.prefill_q, st.prefill_out = prefill["q"].data_ptr(), pout.data_ptr()
        st.cu_seqlens_q, st.cu_seqlens_k = prefill["cu_q"].data_ptr(), prefill["cu_k"].data_ptr()
        st.prefill_batch = prefill["cu_q"].numel() - 1
        st.max_seqlen_q, st.max_seqlen_k = int(prefill["max_q"]), int(prefill["max_k"])
        st.prefill_table = prefill["table"].data_ptr()
        st.prefill_max_blocks = prefill["table"].shape[1]
    if decode:
        for n in ("q", "k_new", "v_new"):
            _cuda_contig("decode " + n, decode[n], k_cache.dtype)
        for n in ("table", "seqlens"):
            _cuda_contig("decode " + n, decode[n], torch.int32)
        dout = decode.get("out")
        if dout is None:
            dout = torch.empty_like(decode["q"])
        hq = decode["q"].shape[1]
        st.decode_q, st.decode_out = decode["q"].data_ptr(), dout.data_ptr()
        st.decode_k_new, st.decode_v_new = decode["k_new"].data_ptr(), decode["v_new"].data_ptr()
        st.decode_table = decode["table"].data_ptr()
        st.decode_max_blocks = decode["table"].shape[1]
        st.decode_seqlens = decode["seqlens"].data_ptr()
        st.decode_batch = decode["q"].shape[0]
        if decode.get("group_cu") is not None:
            _cuda_contig("group_cu", decode["group_cu"], torch.int32)
            _cuda_contig("group_prefix_len", decode["group_prefix_len"], torch.int32)
            st.group_cu = decode["group_cu"].data_ptr()
            st.group_prefix_len = decode["group_prefix_len"].data_ptr()
            st.n_groups = decode["group_cu"].numel() - 1
            st.max_group_size = int(decode["max_group_size"])
    g = geom_of(k_cache, hq if hq is not None else k_cache.shape[2])
    lib = load_library()
    with torch.cuda.device(k_cache.device):
        need = int(lib.paged_mixed_step_workspace_size(st.decode_batch, ctypes.byref(g)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=k_cache.device)
    fn = lib.paged_mixed_step_one_launch if one_launch else lib.paged_mixed_step
    with torch.cuda.device(k_cache.device):
        rc = fn(ctypes.byref(st), _ptr(k_cache), _ptr(v_cache), _ptr(workspace),
                workspace.numel(), ctypes.byref(g), _stream(k_cache))
    _check("paged_mixed_step_one_launch" if one_launch else "paged_mixed_step", rc)
    return pout, dout
