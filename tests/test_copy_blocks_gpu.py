"""GPU parity of paged_copy_blocks (bit-exact against the oracle's block
copy) and of a whole copy-on-write step: the native block manager forks a
sequence, the fork's next token lands in a shared partial block, the block is
copied on the GPU, the token's K/V written and both sequences decoded."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from oracle.block_manager import BlockManager as Oracle, copy_blocks
from gpu_helpers import assert_close, to_dev, to_host, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


def pools(rng, nb, B, hkv, d, dtype):
    if dtype == "bf16":
        mk = lambda: rng.integers(0, 1 << 16, size=(nb, B, hkv, d), dtype=np.uint16)
    else:
        mk = lambda: rng.standard_normal((nb, B, hkv, d)).astype(np.float32)
    return mk(), mk()


@pytest.mark.parametrize("nb,B,hkv,d,dtype,npairs", [
    (64, 16, 8, 128, "bf16", 20),     # 32 KiB blocks
    (40, 256, 8, 128, "bf16", 7),     # 512 KiB blocks, several CTAs per block
    (50, 1, 1, 64, "f32", 25),
    (30, 3, 1, 5, "bf16", 9),         # 30-byte blocks: byte-wise path
    (20, 32, 2, 64, "f32", 0),        # nothing to copy
])
def test_copy_blocks_bit_exact(nb, B, hkv, d, dtype, npairs):
    rng = np.random.default_rng(nb * 7 + B)
    kc, vc = pools(rng, nb, B, hkv, d, dtype)
    perm = rng.permutation(nb)
    src, dst = perm[:npairs].astype(np.int32), perm[npairs: 2 * npairs].astype(np.int32)
    dk, dv = to_dev(kc), to_dev(vc)
    if npairs:
        pkv.paged_copy_blocks(dk, dv, to_dev(src), to_dev(dst))
    else:
        e = torch.empty(0, dtype=torch.int32, device="cuda")
        pkv.paged_copy_blocks(dk, dv, e, e)
    torch.cuda.synchronize()
    copy_blocks(kc, vc, src, dst)
    assert np.array_equal(to_host(dk).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(to_host(dv).view(np.uint8), vc.view(np.uint8))
    assert pkv.paged_error_flags() == 0


def test_copy_blocks_bad_id_is_skipped_and_flagged():
    rng = np.random.default_rng(3)
    kc, vc = pools(rng, 10, 16, 8, 128, "bf16")
    src, dst = np.array([1, 2, 11], np.int32), np.array([3, -1, 4], np.int32)
    dk, dv = to_dev(kc), to_dev(vc)
    pkv.paged_copy_blocks(dk, dv, to_dev(src), to_dev(dst))
    torch.cuda.synchronize()
    copy_blocks(kc, vc, src[:1], dst[:1])  # only the valid pair happens
    assert np.array_equal(to_host(dk), kc) and np.array_equal(to_host(dv), vc)
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_BLOCK


def test_copy_on_write_step():
    """fork + append: the child's new token goes into a copy of the shared
    partial block; afterwards each sequence decodes over its own keys."""
    rng = np.random.default_rng(11)
    B, hkv, hq, d, nb = 16, 2, 4, 128, 32
    nat, ora = pkv.BlockManager(nb, B), Oracle(nb, B)
    prompt = list(rng.integers(0, 50, size=40))       # 2 full blocks + 8 tokens
    a, _ = nat.allocate(prompt)
    oa, _ = ora.allocate(prompt)
    b, ob = nat.fork(a), ora.fork(oa)
    bf = lambda *shape: oracle.f32_to_bf16(
        rng.standard_normal(shape).astype(np.float32)).reshape(shape)
    kc, vc = bf(nb, B, hkv, d), bf(nb, B, hkv, d)
    dk, dv = to_dev(kc), to_dev(vc)
    # the child appends a token: shared partial block -> copy first
    cow = nat.append(b, 7)
    assert cow == ora.append(ob, 7) and cow[0] >= 0
    pkv.paged_copy_blocks(dk, dv, to_dev(np.array([cow[0]], np.int32)),
                          to_dev(np.array([cow[1]], np.int32)))
    copy_blocks(kc, vc, [cow[0]], [cow[1]])
    # the parent appends too (its block is now its own: no copy)
    assert nat.append(a, 9) == (-1, -1) == ora.append(oa, 9)
    tables = np.full((2, 4), -1, np.int32)
    for r, s in enumerate((a, b)):
        t = nat.table(s)
        tables[r, : len(t)] = t
    # each sequence's new token (position 40) goes to its own block
    new_k, new_v = bf(2, hkv, d), bf(2, hkv, d)
    slots = pkv.paged_build_slot_mapping(to_dev(tables), to_dev(np.array([0, 1], np.int32)),
                                         to_dev(np.array([40, 40], np.int32)), B)
    pkv.paged_kv_write(to_dev(new_k), to_dev(new_v), slots, dk, dv)
    oslots = oracle.build_slot_mapping(tables, np.array([0, 1], np.int32),
                                       np.array([40, 40], np.int32), B)
    assert np.array_equal(to_host(slots), oslots) and oslots[0] != oslots[1]
    oracle.kv_write(new_k, new_v, oslots, kc, vc)
    assert np.array_equal(to_host(dk), kc) and np.array_equal(to_host(dv), vc)
    q = bf(1, hq, d).repeat(2, 0)
    lens = np.array([41, 41], np.int32)
    out = pkv.paged_decode(to_dev(q), dk, dv, to_dev(tables), to_dev(lens), 1 / math.sqrt(d))
    torch.cuda.synchronize()
    want = oracle.decode(q, kc, vc, tables, lens, 1 / math.sqrt(d))
    assert_close(widen(out), want, "bf16", "copy-on-write decode")
    # same query, same first 40 keys: only the 41st key (each its own) differs
    assert not np.array_equal(widen(out)[0], widen(out)[1])
    assert pkv.paged_error_flags() == 0
