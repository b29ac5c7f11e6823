"""GPU parity of decode with the in-place append (the new token's K/V is
written into the cache and attended to in the same call) against the oracle:
write the new rows, then plain paged attention over L+1 keys."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep, assert_close, oracle_write, to_dev, to_host, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_config_step_with_append(cfg):
    """The workload's decode step in one call: cache_seqlens before the step,
    the step's new rows as k_new / v_new."""
    step = W.config(cfg)
    assert np.all(step.token_seq == np.arange(step.n_decode))  # one new row per sequence
    dev = DevStep(step)
    before = to_dev(step.cache_seqlens - 1)
    out = pkv.paged_decode_append(dev.q_decode, dev.new_k, dev.new_v, dev.k_cache, dev.v_cache,
                                  dev.decode_table, before, step.scale)
    torch.cuda.synchronize()
    _, kc, vc = oracle_write(step)
    assert np.array_equal(to_host(dev.k_cache), kc) and np.array_equal(to_host(dev.v_cache), vc)
    want = oracle.decode(step.q_decode, kc, vc, step.decode_table, step.cache_seqlens, step.scale)
    assert_close(widen(out), want, step.dtype, f"cfg{cfg} append")
    # the same as the separate write + decode
    dev2 = DevStep(step)
    dev2.write()
    assert_close(widen(out), widen(dev2.decode()), step.dtype, f"cfg{cfg} append vs write+decode")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_cache_returns_v_new(dtype):
    """L = 0: the only key is the new one, so out = v_new (softmax of one key)."""
    rng = np.random.default_rng(4)
    hq, hkv, d, B, nb = 4, 2, 64, 16, 6
    conv = (lambda x: W._to_dtype(x.astype(np.float32), "bf16")) if dtype == "bf16" else \
        (lambda x: x.astype(np.float32))
    q = conv(rng.standard_normal((3, hq, d)))
    kn, vn = conv(rng.standard_normal((3, hkv, d))), conv(rng.standard_normal((3, hkv, d)))
    kc = conv(rng.standard_normal((nb, B, hkv, d)))
    vc = conv(rng.standard_normal((nb, B, hkv, d)))
    table = np.array([[4, -1], [1, -1], [0, 2]], np.int32)
    lens = np.array([0, 0, 0], np.int32)
    dk, dv = to_dev(kc), to_dev(vc)
    out = pkv.paged_decode_append(to_dev(q), to_dev(kn), to_dev(vn), dk, dv, to_dev(table),
                                  to_dev(lens))
    torch.cuda.synchronize()
    got = to_host(out)
    for b in range(3):
        for h in range(hq):
            assert np.array_equal(got[b, h], vn[b, h // 2])
    for b, blk in enumerate([4, 1, 0]):
        kc[blk, 0], vc[blk, 0] = kn[b], vn[b]
    assert np.array_equal(to_host(dk), kc) and np.array_equal(to_host(dv), vc)


def test_position_past_the_table_is_flagged_and_not_written():
    rng = np.random.default_rng(5)
    step = W.config(1)
    dev = DevStep(step)
    before = step.cache_seqlens - 1
    before[2] = step.table.shape[1] * step.block_size  # one past the row's capacity
    kc0 = to_host(dev.k_cache).copy()
    pkv.paged_decode_append(dev.q_decode, dev.new_k, dev.new_v, dev.k_cache, dev.v_cache,
                            dev.decode_table, to_dev(before.astype(np.int32)), step.scale)
    torch.cuda.synchronize()
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_LENGTH
    kc = to_host(dev.k_cache)
    # sequences 0 and 1 were written, sequence 2 was not
    slots = oracle.build_slot_mapping(step.table, np.array([0, 1], np.int32),
                                      before[:2].astype(np.int32), step.block_size)
    kc0.reshape(-1, *kc0.shape[2:])[slots] = step.new_k[:2]
    assert np.array_equal(kc, kc0)


@pytest.mark.parametrize("dtype,hq,hkv,d,B", [("f32", 8, 2, 64, 1), ("bf16", 32, 8, 128, 48),
                                              ("f32", 16, 16, 128, 16), ("bf16", 64, 8, 128, 16),
                                              ("bf16", 32, 2, 64, 256)])
def test_append_shapes(dtype, hq, hkv, d, B):
    """Other dtypes, head sizes, GQA groups and block sizes (B = 1, B not a
    power of two, Hkv above the decode kernel's warp count; bf16 groups of 8
    and 16, whose whole pages go through the tensor-core pass)."""
    lens = [0, 1, B, 3 * B + 1, 700]
    step = W.make_step(name="app", dtype=dtype, hq=hq, hkv=hkv, d=d, block_size=B,
                       decode_lens=lens, seed=sum(lens) + hq + d)
    dev = DevStep(step)
    out = pkv.paged_decode_append(dev.q_decode, dev.new_k, dev.new_v, dev.k_cache, dev.v_cache,
                                  dev.decode_table, to_dev(np.array(lens, np.int32)), step.scale)
    torch.cuda.synchronize()
    _, kc, vc = oracle_write(step)
    assert np.array_equal(to_host(dev.k_cache), kc) and np.array_equal(to_host(dev.v_cache), vc)
    want = oracle.decode(step.q_decode, kc, vc, step.decode_table, step.cache_seqlens, step.scale)
    assert_close(widen(out), want, dtype, f"{dtype} {hq}/{hkv} d{d} B{B}")
    assert pkv.paged_error_flags() == 0
