"""GPU parity of the shared-prefix decode: groups of sequences whose first
keys sit in the same physical blocks read those blocks once per group (the
prefix attention on the tensor cores, merged with each sequence's own keys by
the boxed rule); the result must be plain paged attention over all keys."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep, assert_close, oracle_write, to_dev, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


def _bf(x):
    return W._to_dtype(np.asarray(x, np.float32), "bf16")


def test_mixed_step_decode_half():
    """The continuous-batching workload's 256 decode sequences (8 groups of 32
    sharing a 2048-token prefix, suffixes U[0,512]) after the step's write."""
    step = W.config(5)
    dev = DevStep(step)
    dev.write()
    nd = step.n_decode
    group_cu = np.arange(0, nd + 1, nd // 8, dtype=np.int32)
    plen = np.full(8, 2048, np.int32)
    out = pkv.paged_decode_shared_prefix(dev.q_decode, dev.k_cache, dev.v_cache,
                                         dev.decode_table, dev.cache_seqlens, to_dev(group_cu),
                                         to_dev(plen), nd // 8, step.scale)
    plain = dev.decode()
    torch.cuda.synchronize()
    _, kc, vc = oracle_write(step)
    want = oracle.decode(step.q_decode, kc, vc, step.decode_table, step.cache_seqlens,
                         step.scale)
    assert_close(widen(out), want, "bf16", "shared-prefix decode")
    assert_close(widen(out), widen(plain), "bf16", "shared vs plain decode")
    assert pkv.paged_error_flags() == 0


def build_groups(rng, sizes, prefixes, suffix_max, B, hq=16, hkv=8, d=128):
    """Tables where the members of group g share the first prefixes[g] keys'
    blocks; each member adds U[0, suffix_max] keys of its own."""
    rows, lens = [], []
    nxt = 0
    for gsize, p in zip(sizes, prefixes):
        shared = list(range(nxt, nxt + p // B))
        nxt += p // B
        for _ in range(gsize):
            L = p + int(rng.integers(0, suffix_max + 1))
            own = -(-L // B) - len(shared)
            rows.append(shared + list(range(nxt, nxt + own)))
            nxt += own
            lens.append(L)
    nb = nxt + 3
    perm = rng.permutation(nb).astype(np.int32)
    width = max(len(r) for r in rows)
    table = np.full((len(rows), width), -1, np.int32)
    for i, r in enumerate(rows):
        table[i, : len(r)] = perm[np.array(r, dtype=np.int64)] if r else []
    kc = _bf(rng.standard_normal((nb, B, hkv, d)))
    vc = _bf(rng.standard_normal((nb, B, hkv, d)))
    q = _bf(rng.standard_normal((len(rows), hq, d)))
    group_cu = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return q, kc, vc, table, np.array(lens, np.int32), group_cu, np.array(prefixes, np.int32)


@pytest.mark.parametrize("sizes,prefixes,suffix_max,B", [
    ([1, 5, 40, 130], [0, 64, 320, 1024], 300, 16),   # group of one, > 128 members
    ([3, 3], [256, 512], 0, 256),                      # some members have no own keys
    ([7], [128], 700, 64),
    ([2, 2, 2], [0, 0, 0], 200, 32),                   # no sharing at all
    ([32] * 8, [4096] * 8, 0, 16),                     # prefix only: the split has no tile
])
def test_groups(sizes, prefixes, suffix_max, B):
    rng = np.random.default_rng(sum(sizes) + B)
    q, kc, vc, table, lens, gcu, plen = build_groups(rng, sizes, prefixes, suffix_max, B)
    scale = 1 / math.sqrt(128)
    out = pkv.paged_decode_shared_prefix(to_dev(q), to_dev(kc), to_dev(vc), to_dev(table),
                                         to_dev(lens), to_dev(gcu), to_dev(plen), max(sizes),
                                         scale)
    torch.cuda.synchronize()
    want = oracle.decode(q, kc, vc, table, lens, scale)
    assert_close(widen(out), want, "bf16", f"groups {sizes}")
    assert pkv.paged_error_flags() == 0


def test_prefix_not_a_whole_block_is_flagged():
    rng = np.random.default_rng(1)
    q, kc, vc, table, lens, gcu, plen = build_groups(rng, [4], [64], 50, 16)
    plen[0] = 40
    pkv.paged_decode_shared_prefix(to_dev(q), to_dev(kc), to_dev(vc), to_dev(table),
                                   to_dev(lens), to_dev(gcu), to_dev(plen), 4)
    torch.cuda.synchronize()
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_LENGTH


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 8), (8, 2), (64, 8), (32, 2)])
def test_group_sizes(hq, hkv):
    """GQA group 1 (the prefix pass takes one head per work item), 4, 8 and 16
    (two and four decode warps per KV head), and a KV-head count below the
    decode kernel's warp count."""
    rng = np.random.default_rng(hq * 7 + hkv)
    q, kc, vc, table, lens, gcu, plen = build_groups(rng, [6, 9], [256, 512], 200, 32,
                                                     hq=hq, hkv=hkv)
    scale = 1 / math.sqrt(128)
    out = pkv.paged_decode_shared_prefix(to_dev(q), to_dev(kc), to_dev(vc), to_dev(table),
                                         to_dev(lens), to_dev(gcu), to_dev(plen), 9, scale)
    torch.cuda.synchronize()
    want = oracle.decode(q, kc, vc, table, lens, scale)
    assert_close(widen(out), want, "bf16", f"{hq}/{hkv}")
    assert pkv.paged_error_flags() == 0


def test_head_dim_64():
    """head_dim 64: the prefix pass on the head_dim-64 tensor-core kernel."""
    rng = np.random.default_rng(64)
    q, kc, vc, table, lens, gcu, plen = build_groups(rng, [5, 40], [128, 512], 300, 16, d=64)
    scale = 1 / math.sqrt(64)
    out = pkv.paged_decode_shared_prefix(to_dev(q), to_dev(kc), to_dev(vc), to_dev(table),
                                         to_dev(lens), to_dev(gcu), to_dev(plen), 40, scale)
    torch.cuda.synchronize()
    want = oracle.decode(q, kc, vc, table, lens, scale)
    assert_close(widen(out), want, "bf16", "head_dim 64")
    assert pkv.paged_error_flags() == 0
