"""GPU parity of the slot_mapping build and the cache write: bit-exact against
the oracle (addressing and byte work are exact)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep, oracle_write, to_dev, to_host

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


def test_token9_and_decode_example_slots():
    """题目5 (B=4, table [3,1,5]) and the Sayfalı dikkat decode example."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_token9.json")))
    table = to_dev(np.array([g["block_table"]], np.int32))
    pos = np.arange(g["num_tokens"], dtype=np.int32)
    slots = pkv.paged_build_slot_mapping(table, to_dev(np.zeros_like(pos)), to_dev(pos),
                                         g["block_size"])
    want = oracle.build_slot_mapping(np.array([g["block_table"]], np.int32), np.zeros_like(pos),
                                     pos, g["block_size"])
    assert np.array_equal(to_host(slots), want)
    assert to_host(slots)[9] == 5 * 4 + 1
    d = json.load(open(os.path.join(GOLDEN, "decode_example.json")))
    t = np.array(d["block_table"], np.int32)
    seq = np.array([0, 1, 2, -1], np.int32)
    pos = np.array(d["cache_seqlens"] + [0], np.int32)
    s = to_host(pkv.paged_build_slot_mapping(to_dev(t), to_dev(seq), to_dev(pos), 32))
    assert list(s) == [94, 32, 198, -1]
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("cfg", [1, 4, 5])
def test_config_write_bit_exact(cfg):
    """Write every new token of the workload (config 5 has 5% -1 padding rows)."""
    step = W.config(cfg)
    dev = DevStep(step)
    slots = dev.write()
    torch.cuda.synchronize()
    want_slots, kc, vc = oracle_write(step)
    assert np.array_equal(to_host(slots), want_slots)
    assert np.array_equal(to_host(dev.k_cache), kc)
    assert np.array_equal(to_host(dev.v_cache), vc)
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("src,dst,hkv,d", [("f32", "f32", 1, 64), ("bf16", "bf16", 8, 128),
                                           ("f32", "bf16", 2, 64), ("bf16", "f32", 3, 24),
                                           ("f32", "f32", 3, 5)])
def test_write_dtypes_and_skip(src, dst, hkv, d):
    """Negative slots write nothing (canary intact); fp32 -> bf16 rounds to
    nearest even; ragged row widths take the element-wise path."""
    rng = np.random.default_rng(7)
    nb, B, n = 9, 4, 20
    slots = rng.permutation(nb * B)[:n].astype(np.int32)
    slots[::3] = -1
    def mk(shape, dt):
        x = rng.standard_normal(shape).astype(np.float32)
        return W._to_dtype(x, dt)
    k, v = mk((n, hkv, d), src), mk((n, hkv, d), src)
    canary = mk((nb, B, hkv, d), dst)
    kc, vc = canary.copy(), canary.copy()
    oracle.kv_write(k, v, slots, kc, vc)
    dk, dv = to_dev(canary.copy()), to_dev(canary.copy())
    pkv.paged_kv_write(to_dev(k), to_dev(v), to_dev(slots), dk, dv)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(dk), kc)
    assert np.array_equal(to_host(dv), vc)


def test_out_of_range_slot_is_skipped_and_flagged():
    nb, B, hkv, d = 4, 4, 2, 64
    k = torch.randn(3, hkv, d, device="cuda")
    kc = torch.zeros(nb, B, hkv, d, device="cuda")
    vc = torch.zeros(nb, B, hkv, d, device="cuda")
    slots = torch.tensor([1, nb * B, -1], dtype=torch.int32, device="cuda")
    pkv.paged_kv_write(k, k, slots, kc, vc)
    torch.cuda.synchronize()
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_SLOT
    assert torch.equal(kc.view(-1, hkv, d)[1], k[0])
    assert int((kc != 0).any(dim=(2, 3)).sum()) == 1


def test_slot_builder_flags_bad_entries():
    table = to_dev(np.array([[3, -1], [0, 1]], np.int32))
    seq = to_dev(np.array([0, 0, 1, 2, 1], np.int32))
    pos = to_dev(np.array([1, 5, 7, 0, 9], np.int32))
    s = to_host(pkv.paged_build_slot_mapping(table, seq, pos, 4))
    assert list(s) == [13, -1, 7, -1, -1]
    f = pkv.paged_error_flags()
    assert f & pkv.PKV_FLAG_BAD_BLOCK and f & pkv.PKV_FLAG_BAD_SEQ and f & pkv.PKV_FLAG_BAD_LENGTH


@pytest.mark.parametrize("cfg", [1, 4, 5])
def test_write_positions_matches_oracle(cfg):
    """paged_kv_write_positions (slot build and write in one launch): the same
    caches and slot mapping as the oracle's two steps, padding rows skipped."""
    step = W.config(cfg)
    dev = DevStep(step)
    out = torch.full((step.token_seq.size,), 12345, dtype=torch.int32, device="cuda")
    pkv.paged_kv_write_positions(dev.new_k, dev.new_v, dev.table, dev.token_seq, dev.token_pos,
                                 dev.k_cache, dev.v_cache, slot_mapping_out=out)
    torch.cuda.synchronize()
    want_slots, kc, vc = oracle_write(step)
    assert np.array_equal(to_host(out), want_slots)
    assert np.array_equal(to_host(dev.k_cache), kc)
    assert np.array_equal(to_host(dev.v_cache), vc)
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("src,dst,hkv,d", [("f32", "bf16", 2, 64), ("bf16", "f32", 3, 24),
                                           ("bf16", "bf16", 8, 128)])
def test_write_positions_dtypes_and_bad_entries(src, dst, hkv, d):
    """Every write path of the fused call; bad sequence ids, positions and
    table entries write nothing and set their flags; no slot output."""
    rng = np.random.default_rng(11)
    nb, B = 6, 4
    table = np.array([[3, 0, -1], [5, 1, 2]], np.int32)
    seq = np.array([0, 1, 1, -1, 0, 2, 1, 0], np.int32)
    pos = np.array([1, 4, 11, 0, 9, 0, 12, 5], np.int32)
    n = seq.size

    def mk(shape, dt):
        return W._to_dtype(rng.standard_normal(shape).astype(np.float32), dt)
    k, v = mk((n, hkv, d), src), mk((n, hkv, d), src)
    canary = mk((nb, B, hkv, d), dst)
    # rows 0-2 and 7 are valid (the oracle's addressing); row 3 is padding;
    # row 4 meets a -1 table entry, row 5 a sequence id past the table, row 6
    # a position past its row: slot -1, nothing written
    valid = np.array([0, 1, 2, 7])
    slots = np.full(n, -1, np.int32)
    slots[valid] = oracle.build_slot_mapping(table, seq[valid], pos[valid], B)
    assert list(slots) == [13, 4, 11, -1, -1, -1, -1, 1]
    kc, vc = canary.copy(), canary.copy()
    oracle.kv_write(k, v, slots, kc, vc)
    dk, dv = to_dev(canary.copy()), to_dev(canary.copy())
    pkv.paged_kv_write_positions(to_dev(k), to_dev(v), to_dev(table), to_dev(seq), to_dev(pos),
                                 dk, dv)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(dk), kc)
    assert np.array_equal(to_host(dv), vc)
    f = pkv.paged_error_flags()
    assert f & pkv.PKV_FLAG_BAD_BLOCK and f & pkv.PKV_FLAG_BAD_SEQ and f & pkv.PKV_FLAG_BAD_LENGTH
