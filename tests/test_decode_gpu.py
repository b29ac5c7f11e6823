"""GPU parity of paged decode (block-table reads + online-softmax merge +
split-KV combine) against the fp64 oracle, through the C ABI."""
import ctypes
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import DevStep, assert_close, oracle_write, to_dev, to_host, widen

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


def _oracle_decode(step, kc, vc):
    return oracle.decode(step.q_decode, kc, vc, step.decode_table, step.cache_seqlens, step.scale)


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_config_step(cfg):
    """The workload's step: write the new tokens, then decode over L+1 keys."""
    step = W.config(cfg)
    dev = DevStep(step)
    dev.write()
    out = dev.decode()
    torch.cuda.synchronize()
    _, kc, vc = oracle_write(step)
    assert np.array_equal(to_host(dev.k_cache), kc)
    want = _oracle_decode(step, kc, vc)
    assert_close(widen(out), want, step.dtype, f"cfg{cfg}")
    assert pkv.paged_error_flags() == 0


def test_decode_example_state():
    """Sayfalı dikkat decode example as printed: cache_seqlens [30,32,70],
    B=32, table [[2,-1,-1,-1],[0,1,-1,-1],[3,5,6,-1]] (fp32, Hq=2, Hkv=1, d=64)."""
    g = json.load(open(os.path.join(GOLDEN, "decode_example.json")))
    rng = np.random.default_rng(1001)
    kc = rng.standard_normal((8, 32, 1, 64)).astype(np.float32)
    vc = rng.standard_normal((8, 32, 1, 64)).astype(np.float32)
    q = rng.standard_normal((3, 2, 64)).astype(np.float32)
    table = np.array(g["block_table"], np.int32)
    lens = np.array(g["cache_seqlens"], np.int32)
    out = pkv.paged_decode(to_dev(q), to_dev(kc), to_dev(vc), to_dev(table), to_dev(lens), 0.125)
    want = oracle.decode(q, kc, vc, table, lens, 0.125)
    assert_close(widen(out), want, "f32", "p4 example")


CASES = [
    # (dtype, hq, hkv, d, B, lens)
    ("bf16", 16, 8, 128, 16, [0, 1, 15, 16, 17, 33, 1000]),
    ("bf16", 16, 8, 128, 256, [255, 256, 257, 0, 5000]),
    ("f32", 16, 8, 128, 32, [1, 31, 64, 100]),
    ("bf16", 8, 8, 128, 64, [3, 130, 700]),        # G = 1
    ("bf16", 32, 8, 128, 16, [77, 500, 1]),         # G = 4
    ("f32", 16, 4, 64, 16, [5, 700, 33]),           # G = 4, fp32, d = 64
    ("bf16", 4, 1, 128, 32, [1, 63, 2000]),         # G = 4, Hkv = 1 (8 warps share the head)
    ("bf16", 32, 8, 128, 256, [20000, 3]),          # G = 4, long context
    ("f32", 4, 1, 64, 32, [30, 32, 70, 0]),         # Hkv = 1 (warps share a head)
    ("bf16", 4, 2, 64, 48, [47, 48, 49, 200]),      # B not a power of two
    ("bf16", 8, 4, 64, 1, [1, 2, 9]),               # B = 1
    ("f32", 32, 16, 128, 16, [40, 300]),            # Hkv > 8: heads split across CTAs
    ("bf16", 2, 2, 128, 3, [0, 0, 0]),              # all empty
    ("bf16", 16, 8, 128, 16, [4096] * 3 + [0] * 500 + [17] * 200),  # many sequences
    ("bf16", 64, 8, 128, 16, [900, 1, 33, 4000]),   # G = 8: pages on the tensor cores
    ("f32", 32, 4, 64, 32, [5, 64, 700]),           # G = 8, fp32: two split warps per KV head
    ("bf16", 8, 1, 128, 64, [129, 2000]),           # G = 8, Hkv = 1
    ("bf16", 128, 8, 128, 256, [3000, 20000]),      # G = 16, long context
    ("f32", 32, 2, 128, 16, [1, 300, 17]),          # G = 16, fp32: four split warps per KV head
    ("bf16", 32, 1, 64, 16, [50, 1000]),            # G = 32
    ("bf16", 64, 8, 128, 48, [47, 48, 49, 3000]),   # G = 8, B = 48: the CUDA-core split alone
    ("bf16", 64, 8, 64, 128, [127, 128, 129, 0, 5000]),  # G = 8 on the tensor cores, d = 64
    ("bf16", 16, 1, 128, 8, [1, 7, 8, 9, 1000] * 40),    # G = 16, 200 sequences of pages of 8
]


@pytest.mark.parametrize("dtype,hq,hkv,d,B,lens", CASES)
def test_decode_shapes(dtype, hq, hkv, d, B, lens):
    step = W.make_step(name="edge", dtype=dtype, hq=hq, hkv=hkv, d=d, block_size=B,
                       decode_lens=[max(L - 1, 0) for L in lens], seed=sum(lens) + hq + B)
    step.cache_seqlens = np.asarray(lens, np.int32)  # attend over exactly these lengths
    dev = DevStep(step)
    out = dev.decode()
    torch.cuda.synchronize()
    want = _oracle_decode(step, step.k_cache, step.v_cache)
    assert_close(widen(out), want, dtype, str(lens[:6]))
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("hq,hkv,B", [(32, 8, 16), (64, 8, 256), (16, 8, 16), (32, 4, 48)])
def test_nonfinite_pool_past_the_keys_is_ignored(hq, hkv, B):
    """Every pool row past a sequence's keys holds NaN, in the last page and
    in every unused block: nothing of it may reach the output.  Groups of 4 and
    8 with B = 16 or 256 take the tensor-core route (masked scores, zeroed V
    rows of the partial last page); 16/8 heads and B = 48 take the split."""
    lens = [1, 15, 17, 130, 1000, 4000]
    step = W.make_step(name="nan", dtype="bf16", hq=hq, hkv=hkv, d=128, block_size=B,
                       decode_lens=[L - 1 for L in lens], seed=77 + hq + B)
    step.cache_seqlens = np.asarray(lens, np.int32)
    kc, vc = step.k_cache.copy(), step.v_cache.copy()
    keep = np.zeros(kc.shape[:2], dtype=bool)  # [blocks, B]: rows that hold a key
    for b, L in enumerate(lens):
        for p in range(L):
            keep[step.decode_table[b, p // B], p % B] = True
    kc[~keep] = 0x7fc0  # bf16 NaN
    vc[~keep] = 0x7fc0
    step.k_cache, step.v_cache = kc, vc
    out = widen(DevStep(step).decode())
    torch.cuda.synchronize()
    assert np.all(np.isfinite(out))
    want = _oracle_decode(step, kc, vc)
    assert_close(out, want, "bf16", f"nan pool {hq}/{hkv} B{B}")
    assert pkv.paged_error_flags() == 0


def test_single_key_returns_v0():
    step = W.make_step(name="one", dtype="f32", hq=4, hkv=2, d=128, block_size=16,
                       decode_lens=[0, 0], seed=3)
    step.cache_seqlens = np.array([1, 1], np.int32)
    out = DevStep(step).decode()
    for b in range(2):
        v0 = step.v_cache[step.table[b, 0], 0]  # [Hkv, d]
        for h in range(4):
            assert np.allclose(widen(out)[b, h], v0[h // 2], atol=1e-6, rtol=0)


def test_physical_permutation_bitwise():
    """Moving physical blocks (data + table) leaves the GPU output bit-identical:
    the reduction order depends only on logical positions."""
    step = W.config(2)
    dev = DevStep(step)
    a = to_host(dev.decode())
    nb = step.num_blocks
    perm = np.random.default_rng(9).permutation(nb)
    inv = np.argsort(perm)
    dev.k_cache = dev.k_cache[torch.from_numpy(inv).cuda()].contiguous()
    dev.v_cache = dev.v_cache[torch.from_numpy(inv).cuda()].contiguous()
    t = step.decode_table
    dev.decode_table = to_dev(np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32))
    b = to_host(dev.decode())
    assert np.array_equal(a, b)


def test_repeatable_and_out_buffer():
    step = W.config(3)
    dev = DevStep(step)
    a = to_host(dev.decode())
    out = torch.full_like(dev.q_decode, float("nan"))
    ws = torch.empty(pkv.paged_decode_workspace_size(step.n_decode, step.hq, dev.k_cache),
                     dtype=torch.uint8, device="cuda")
    dev.decode(out=out, workspace=ws)
    assert np.array_equal(a, to_host(out))


def test_bad_block_id_is_flagged_not_read():
    step = W.make_step(name="bad", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                       decode_lens=[40, 40], seed=5)
    step.table[1, 1] = step.num_blocks + 1000  # out of range inside the valid length
    dev = DevStep(step)
    out = dev.decode()
    torch.cuda.synchronize()
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_BLOCK
    want = oracle.decode(step.q_decode[:1], step.k_cache, step.v_cache, step.decode_table[:1],
                         step.cache_seqlens[:1], step.scale)
    assert_close(widen(out)[:1], want, "bf16", "untouched sequence")


def test_length_beyond_table_is_clamped_and_flagged():
    step = W.make_step(name="long", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                       decode_lens=[20], seed=6, max_blocks=2)
    step.cache_seqlens = np.array([10_000], np.int32)
    DevStep(step).decode()
    torch.cuda.synchronize()
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_LENGTH


def test_workspace_and_support_errors():
    step = W.make_step(name="ws", dtype="bf16", hq=16, hkv=8, d=128, block_size=16,
                       decode_lens=[10], seed=8)
    dev = DevStep(step)
    with pytest.raises(pkv.PagedKVError) as e:
        dev.decode(workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == -3
    q = torch.zeros(1, 16, 96, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode(q, kc, kc, dev.decode_table, dev.cache_seqlens)
    assert e.value.status == -2
    # a GQA group of 12 (not 1, 2, 4, 8, 16 or 32)
    q = torch.zeros(1, 96, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_decode(q, kc, kc, dev.decode_table, dev.cache_seqlens)
    assert e.value.status == -2


def test_split_points_vary_with_the_batch():
    """One 20000-key sequence decoded with the other sequences of the batch
    empty (its keys spread over every CTA) and non-empty (its keys cut into
    other shares and merged from other partial states): within tolerance of
    the oracle each time, and of each other."""
    others = [40000] * 3 + [5, 17, 3000] * 6
    lens = [20000] + others
    step = W.make_step(name="split", dtype="bf16", hq=16, hkv=8, d=128, block_size=64,
                       decode_lens=[L - 1 for L in lens], seed=77)
    want = oracle.decode(step.q_decode[:1], step.k_cache, step.v_cache, step.decode_table[:1],
                         np.array([20000], np.int32), step.scale)
    dev = DevStep(step)
    outs = []
    for variant in (np.zeros(len(others)), np.array(others), np.array(others[::-1]) // 3):
        dev.cache_seqlens = to_dev(np.concatenate([[20000], variant]).astype(np.int32))
        out = widen(dev.decode())
        torch.cuda.synchronize()
        assert_close(out[:1], want, "bf16", "sequence 0")
        outs.append(out[0])
    assert_close(outs[1], outs[0].astype(np.float64), "bf16", "split vs alone")
    assert_close(outs[2], outs[0].astype(np.float64), "bf16", "split vs alone")


@pytest.mark.gpu
def test_one_workspace_across_calls_with_different_tile_starts():
    """Calls that reuse one workspace but cut their keys differently (other
    tile starts, pieces and partial-state slots) each match the oracle: a
    call reads only its own tile starts and partial states, never what the
    call before left in the workspace."""
    full = [3000, 17, 40000, 5, 12000, 800, 25000, 64]
    step = W.make_step(name="reuse", dtype="bf16", hq=16, hkv=8, d=128, block_size=64,
                       decode_lens=[L - 1 for L in full], seed=91)
    dev = DevStep(step)
    g = pkv.geom_of(dev.k_cache, step.hq)
    need = int(pkv._binding.load_library().paged_decode_workspace_size(len(full), ctypes.byref(g)))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    pkv.paged_error_flags()  # clear
    variants = [full, [L // 3 + 1 for L in full], [0 if i % 2 else L for i, L in enumerate(full)],
                full[:1] + [1] * (len(full) - 1), full]
    for lens in variants:
        lens = np.array(lens, np.int32)
        dev.cache_seqlens = to_dev(lens)
        out = widen(dev.decode(workspace=ws))
        torch.cuda.synchronize()
        want = oracle.decode(step.q_decode, step.k_cache, step.v_cache, step.decode_table, lens,
                             step.scale)
        assert_close(out, want, "bf16", f"lengths {lens.tolist()}")
    assert pkv.paged_error_flags() == 0
