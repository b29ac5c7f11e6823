"""Helpers for the GPU parity tests: move a synthetic step to the device, run
the library's kernels through the binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_70_gb300 as pkv


def to_dev(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy; bf16 comes back as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def widen(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class DevStep:
    """Device copies of a workloads.Step."""

    def __init__(self, step):
        self.s = step
        self.table = to_dev(step.table)
        self.k_cache = to_dev(step.k_cache)
        self.v_cache = to_dev(step.v_cache)
        self.new_k = to_dev(step.new_k)
        self.new_v = to_dev(step.new_v)
        self.token_seq = to_dev(step.token_seq)
        self.token_pos = to_dev(step.token_pos)
        if step.n_decode:
            self.q_decode = to_dev(step.q_decode)
            self.cache_seqlens = to_dev(step.cache_seqlens)
            self.decode_table = self.table[: step.n_decode].contiguous()
        if step.n_prefill:
            self.q_prefill = to_dev(step.q_prefill)
            self.cu_q = to_dev(step.cu_q)
            self.cu_k = to_dev(step.cu_k)
            self.prefill_table = self.table[step.n_decode: step.n_decode + step.n_prefill].contiguous()

    def write(self) -> torch.Tensor:
        s = self.s
        slots = pkv.paged_build_slot_mapping(self.table, self.token_seq, self.token_pos,
                                             s.block_size)
        pkv.paged_kv_write(self.new_k, self.new_v, slots, self.k_cache, self.v_cache)
        return slots

    def decode(self, **kw) -> torch.Tensor:
        return pkv.paged_decode(self.q_decode, self.k_cache, self.v_cache, self.decode_table,
                                self.cache_seqlens, self.s.scale, **kw)

    def prefill(self, **kw) -> torch.Tensor:
        s = self.s
        return pkv.paged_varlen_prefill(self.q_prefill, self.k_cache, self.v_cache, self.cu_q,
                                        self.cu_k, s.max_seqlen_q, s.max_seqlen_k,
                                        self.prefill_table, causal=s.causal, scale=s.scale, **kw)


def oracle_write(step):
    """Oracle caches after the step's write (copies of the step's pools)."""
    import oracle
    kc, vc = step.k_cache.copy(), step.v_cache.copy()
    slots = oracle.build_slot_mapping(step.table, step.token_seq, step.token_pos, step.block_size)
    oracle.kv_write(step.new_k, step.new_v, slots, kc, vc)
    return slots, kc, vc


def tolerance(dtype: str):
    """(max-abs, mean-abs) bounds of the parity tests: fp32 inputs 1e-4 max-abs;
    bf16 inputs (fp32 accumulation, bf16 output) 2e-2 max-abs and 2e-3 mean-abs."""
    return (1e-4, 1e-4) if dtype == "f32" else (2e-2, 2e-3)


def assert_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    mx_tol, mean_tol = tolerance(dtype)
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= mx_tol and mean <= mean_tol, f"{what}: max-abs {mx:.3g}, mean-abs {mean:.3g}"
    return mx, mean
