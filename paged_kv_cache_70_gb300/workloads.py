"""Seeded synthetic inputs for the paged KV-cache hot path.

This module only draws inputs: lengths, block placement and N(0,1) values.  It
holds none of the method's arithmetic (no addressing, no slot ids, no softmax),
so both the CUDA path and the CPU oracle can consume what it produces without
sharing any of the computation.  It needs numpy and torch (CPU, for the
fp32 -> bf16 cast of the drawn values) and never touches the GPU.

Shapes follow the workloads of the pages: Qwen3-0.6B-style attention (16 query
heads, 8 KV heads, head_dim 128, bf16) over a paged pool, block sizes 16-256,
contexts up to 40K tokens ("从零开始写Qwen3（六）PagedAttention", section
"KVCache大小计算"), the decode example of "Sayfalı dikkat" (cache_seqlens
[30, 32, 70], block size 32, at most 4 blocks per sequence), and chunked
prefill over a prefix cache ("fast-attn 库的使用").

Recipe (all configs): ``numpy.random.Generator(PCG64(seed))`` with
seed = 1000 + config id; lengths uniform on the stated integer ranges;
physical blocks handed out in the order of a seeded permutation of the pool
(pool = blocks needed + 10% free unless stated); table padding -1; values
standard normal, rounded to the cache dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "bf16")


def _to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    import torch
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


_CHUNK = 1 << 22  # elements per independently seeded chunk


def _normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) values rounded to ``dtype``.  Large arrays are filled in fixed
    chunks, each from its own generator seeded by (a draw of ``rng``, chunk
    index), on a thread pool; the values do not depend on the thread count."""
    n = int(np.prod(shape))
    base = int(rng.integers(0, 2**63 - 1))
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)
    chunks = [(i, min(i + _CHUNK, n)) for i in range(0, n, _CHUNK)]

    def fill(k):
        lo, hi = chunks[k]
        g = np.random.default_rng([base, k])
        out[lo:hi] = _to_dtype(g.standard_normal(hi - lo, dtype=np.float32), dtype)

    if len(chunks) <= 1:
        for k in range(len(chunks)):
            fill(k)
    else:
        from concurrent.futures import ThreadPoolExecutor
        import os
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(len(chunks))))
    return out.reshape(shape)


@dataclass
class Step:
    """One step of the hot path over a paged pool.

    ``table`` has one row per sequence (decode sequences first, then prefill
    requests), padded with -1 to ``max_blocks`` columns.  The step first writes
    ``new_k``/``new_v`` row n at logical position ``token_pos[n]`` of sequence
    ``token_seq[n]`` (``token_seq[n] == -1`` marks a padding row that must not be
    written), then runs decode over the first ``n_decode`` sequences and varlen
    prefill over the next ``n_prefill`` ones.
    """
    name: str
    dtype: str
    hq: int
    hkv: int
    d: int
    block_size: int
    num_blocks: int
    scale: float
    table: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    new_k: np.ndarray
    new_v: np.ndarray
    token_seq: np.ndarray
    token_pos: np.ndarray
    n_decode: int = 0
    q_decode: np.ndarray | None = None
    cache_seqlens: np.ndarray | None = None
    n_prefill: int = 0
    q_prefill: np.ndarray | None = None
    cu_q: np.ndarray | None = None
    cu_k: np.ndarray | None = None
    causal: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.table.shape[1])

    @property
    def kv_dim(self) -> int:
        return self.hkv * self.d

    @property
    def elt(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def decode_table(self) -> np.ndarray:
        return self.table[: self.n_decode]

    @property
    def prefill_table(self) -> np.ndarray:
        return self.table[self.n_decode: self.n_decode + self.n_prefill]

    @property
    def max_seqlen_q(self) -> int:
        return int(np.max(np.diff(self.cu_q))) if self.n_prefill else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(np.max(np.diff(self.cu_k))) if self.n_prefill else 0


class _Pool:
    """Hands out physical block ids in the order of a seeded permutation."""

    def __init__(self, rng: np.random.Generator, num_blocks: int):
        self.order = rng.permutation(num_blocks).astype(np.int32)
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        if self.next + n > len(self.order):
            raise ValueError("pool exhausted")
        out = self.order[self.next: self.next + n]
        self.next += n
        return out


def _blocks_for(tokens: int, block_size: int) -> int:
    return -(-tokens // block_size)


def _table(rows: list[np.ndarray], width: int) -> np.ndarray:
    t = np.full((len(rows), max(width, 1)), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        t[i, : len(r)] = r
    return t


def make_step(*, name: str, dtype: str, hq: int, hkv: int, d: int, block_size: int,
              decode_lens=(), prefill_q=(), prefill_cached=(), seed: int = 0,
              pool_extra: float = 0.10, max_blocks: int | None = None,
              shared_prefix: tuple[int, int] | None = None, pad_fraction: float = 0.0,
              causal: bool = True, scale: float | None = None,
              num_blocks: int | None = None) -> Step:
    """General step generator.

    decode_lens[b]      cached tokens of decode sequence b before the step; the
                        step appends one token at that position and decodes over
                        decode_lens[b] + 1 keys.
    prefill_q[r]        new query tokens of prefill request r, appended after
                        prefill_cached[r] already-cached tokens.
    shared_prefix       (groups, prefix_tokens): decode sequences are split into
                        ``groups`` equal groups whose tables share the physical
                        blocks of a ``prefix_tokens``-long prefix (a multiple of
                        the block size); decode_lens then counts prefix+suffix.
    pad_fraction        fraction of padding rows (token_seq = -1) interleaved at
                        seeded positions among the new-token rows.
    """
    assert dtype in DTYPES
    rng = np.random.default_rng(seed)
    decode_lens = [int(x) for x in decode_lens]
    prefill_q = [int(x) for x in prefill_q]
    prefill_cached = [int(x) for x in prefill_cached] or [0] * len(prefill_q)
    nd, npf = len(decode_lens), len(prefill_q)
    B = block_size

    # blocks each sequence needs once the step's new tokens are in
    need_dec = [_blocks_for(L + 1, B) for L in decode_lens]
    need_pre = [_blocks_for(c + q, B) for q, c in zip(prefill_q, prefill_cached)]
    if shared_prefix is not None:
        groups, ptoks = shared_prefix
        assert ptoks % B == 0 and nd % groups == 0
        pblocks = ptoks // B
        unique_dec = [n - pblocks for n in need_dec]
        total = groups * pblocks + sum(unique_dec) + sum(need_pre)
    else:
        total = sum(need_dec) + sum(need_pre)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(total * (1.0 + pool_extra)))
    pool = _Pool(rng, num_blocks)

    rows: list[np.ndarray] = []
    if shared_prefix is not None:
        per_group = nd // groups
        prefixes = [pool.take(pblocks) for _ in range(groups)]
        for b in range(nd):
            g = b // per_group
            rows.append(np.concatenate([prefixes[g], pool.take(unique_dec[b])]))
    else:
        for n in need_dec:
            rows.append(pool.take(n))
    for n in need_pre:
        rows.append(pool.take(n))
    width = max([len(r) for r in rows] + [0])
    if max_blocks is not None:
        assert max_blocks >= width
        width = max_blocks
    table = _table(rows, width)

    kv_shape = (num_blocks, B, hkv, d)
    k_cache = _normal(rng, kv_shape, dtype)
    v_cache = _normal(rng, kv_shape, dtype)

    # new tokens: one per decode sequence, then every new prefill token
    seqs = [b for b in range(nd)]
    poss = [decode_lens[b] for b in range(nd)]
    for r in range(npf):
        for i in range(prefill_q[r]):
            seqs.append(nd + r)
            poss.append(prefill_cached[r] + i)
    seqs = np.asarray(seqs, dtype=np.int32)
    poss = np.asarray(poss, dtype=np.int32)
    if pad_fraction > 0 and len(seqs):
        n_pad = int(round(pad_fraction * len(seqs)))
        total_rows = len(seqs) + n_pad
        pad_at = np.sort(rng.choice(total_rows, size=n_pad, replace=False))
        is_pad = np.zeros(total_rows, dtype=bool)
        is_pad[pad_at] = True
        s2 = np.full(total_rows, -1, dtype=np.int32)
        p2 = np.full(total_rows, -1, dtype=np.int32)
        s2[~is_pad] = seqs
        p2[~is_pad] = poss
        seqs, poss = s2, p2
    n_new = len(seqs)
    new_k = _normal(rng, (n_new, hkv, d), dtype)
    new_v = _normal(rng, (n_new, hkv, d), dtype)

    step = Step(name=name, dtype=dtype, hq=hq, hkv=hkv, d=d, block_size=B,
                num_blocks=num_blocks, scale=scale if scale is not None else 1.0 / math.sqrt(d),
                table=table, k_cache=k_cache, v_cache=v_cache, new_k=new_k, new_v=new_v,
                token_seq=seqs, token_pos=poss, causal=causal)
    if nd:
        step.n_decode = nd
        step.q_decode = _normal(rng, (nd, hq, d), dtype)
        step.cache_seqlens = np.asarray([L + 1 for L in decode_lens], dtype=np.int32)
    if npf:
        step.n_prefill = npf
        cu_q = np.zeros(npf + 1, dtype=np.int32)
        cu_k = np.zeros(npf + 1, dtype=np.int32)
        cu_q[1:] = np.cumsum(prefill_q)
        cu_k[1:] = np.cumsum([q + c for q, c in zip(prefill_q, prefill_cached)])
        step.cu_q, step.cu_k = cu_q, cu_k
        step.q_prefill = _normal(rng, (int(cu_q[-1]), hq, d), dtype)
    return step


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny fp32 decode: lens [30,32,70], B=32, pool 8, Hq=2, Hkv=1, d=64",
    2: "Qwen3-0.6B decode: batch 64, L~U[128,4096], B=16, GQA 16/8, d=128, bf16",
    3: "long-context decode: batch 8, L~U[16384,40960], B=256, GQA 16/8, d=128, bf16",
    4: "causal varlen prefill: 16 req, q~U[1,2048], cached~U[0,2048], B=256, GQA 16/8, d=128, bf16",
    5: "continuous-batching step: 256 decode (8x32 shared 2048-token prefixes, suffix U[0,512]) "
       "+ 4x512 prefill, B=16, 5% padded slots, GQA 16/8, d=128, bf16",
}


def config(cfg: int, seed: int | None = None) -> Step:
    """The seeded synthetic step of workload ``cfg`` (1..5)."""
    seed = 1000 + cfg if seed is None else seed
    rng = np.random.default_rng(seed + 7_000_000)  # lengths; values use ``seed``
    if cfg == 1:
        return make_step(name="cfg1", dtype="f32", hq=2, hkv=1, d=64, block_size=32,
                         decode_lens=[30, 32, 70], seed=seed, num_blocks=8, max_blocks=4)
    if cfg == 2:
        lens = rng.integers(128, 4096, size=64, endpoint=True)
        return make_step(name="cfg2", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                         decode_lens=lens, seed=seed)
    if cfg == 3:
        lens = rng.integers(16384, 40960, size=8, endpoint=True)
        return make_step(name="cfg3", dtype="bf16", hq=16, hkv=8, d=128, block_size=256,
                         decode_lens=lens, seed=seed)
    if cfg == 4:
        q = rng.integers(1, 2048, size=16, endpoint=True)
        c = rng.integers(0, 2048, size=16, endpoint=True)
        return make_step(name="cfg4", dtype="bf16", hq=16, hkv=8, d=128, block_size=256,
                         prefill_q=q, prefill_cached=c, seed=seed)
    if cfg == 5:
        suffix = rng.integers(0, 512, size=256, endpoint=True)
        return make_step(name="cfg5", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                         decode_lens=2048 + suffix, prefill_q=[512] * 4, prefill_cached=[0] * 4,
                         shared_prefix=(8, 2048), pad_fraction=0.05, seed=seed)
    raise ValueError(f"unknown config {cfg}")
