"""GPU parity of the causal varlen prefill (tcgen05/TMEM, paged K/V through
the block table) against the fp64 oracle, through the C ABI."""
import math

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


def _bf(x):
    return W._to_dtype(np.asarray(x, np.float32), "bf16")


def make_case(qlens, klens, B, hq=16, hkv=8, d=128, seed=0, extra_blocks=3):
    """Pool + table holding each request's keys (any q/k lengths, k may be < q)."""
    rng = np.random.default_rng(seed)
    need = [-(-k // B) for k in klens]
    nb = sum(need) + extra_blocks
    order = rng.permutation(nb).astype(np.int32)
    width = max(need + [1])
    table = np.full((len(qlens), width), -1, np.int32)
    nxt = 0
    for r, n in enumerate(need):
        table[r, :n] = order[nxt: nxt + n]
        nxt += n
    kc = _bf(rng.standard_normal((nb, B, hkv, d)))
    vc = _bf(rng.standard_normal((nb, B, hkv, d)))
    cq = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(klens)]).astype(np.int32)
    q = _bf(rng.standard_normal((int(cq[-1]), hq, d)))
    return dict(q=q, kc=kc, vc=vc, table=table, cq=cq, ck=ck, B=B, scale=1 / math.sqrt(d))


def run_gpu(c, causal=True):
    return pkv.paged_varlen_prefill(
        to_dev(c["q"]), to_dev(c["kc"]), to_dev(c["vc"]), to_dev(c["cq"]), to_dev(c["ck"]),
        int(np.diff(c["cq"]).max()), int(np.diff(c["ck"]).max()), to_dev(c["table"]),
        causal=causal, scale=c["scale"])


def run_oracle(c, causal=True, rows=None):
    return oracle.prefill(c["q"], c["kc"], c["vc"], c["cq"], c["ck"], c["scale"], causal=causal,
                          block_table=c["table"], block_size=c["B"], row_subset=rows)


def test_varlen_example_lengths():
    """Sayfalı dikkat varlen example lengths: q [10,3,1], k [0,1,7]; rows that
    see no key (all of r0, rows 0-1 of r1) are 0."""
    c = make_case([10, 3, 1], [0, 1, 7], B=16, seed=1)
    out = run_gpu(c)
    torch.cuda.synchronize()
    got = widen(out)
    assert np.all(got[:12] == 0)
    assert_close(got, run_oracle(c), "bf16", "varlen example")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("B", [8, 16, 32, 64, 128, 256, 512])
def test_block_sizes(B):
    qlens = [1, 127, 128, 129, 300]
    cached = [0, 5, 256, 1000 % B + 3, 77]
    c = make_case(qlens, [q + k for q, k in zip(qlens, cached)], B=B, seed=B)
    out = run_gpu(c)
    torch.cuda.synchronize()
    assert_close(widen(out), run_oracle(c), "bf16", f"B={B}")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (16, 4), (32, 4), (4, 1)])
def test_gqa_groups(hq, hkv):
    c = make_case([200, 64], [260, 64], B=64, hq=hq, hkv=hkv, seed=hq * 10 + hkv)
    assert_close(widen(run_gpu(c)), run_oracle(c), "bf16", f"{hq}/{hkv}")


@pytest.mark.parametrize("hq,hkv,B", [(16, 8, 16), (8, 8, 256), (32, 8, 64)])
@pytest.mark.parametrize("causal", [True, False])
def test_head_dim_64(hq, hkv, B, causal):
    """head_dim 64: one 64-dim swizzled region per tile row, PV with N = 64;
    with paired heads (16/8, 32/8) and paired query tiles (8/8)."""
    qlens = [1, 127, 128, 129, 300, 700]
    klens = [1, 300, 128, 500, 300, 900]
    c = make_case(qlens, klens, B=B, hq=hq, hkv=hkv, d=64, seed=hq + B + int(causal))
    out = run_gpu(c, causal)
    torch.cuda.synchronize()
    assert_close(widen(out), run_oracle(c, causal), "bf16", f"d64 {hq}/{hkv} B={B} {causal}")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (12, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_query_tile_pairs(hq, hkv, causal):
    """An odd GQA group (1, 3): a CTA takes two consecutive query tiles of one
    head instead of two heads.  Query lengths give odd and even tile counts,
    ragged last tiles and a single tile; cached keys shift the causal
    diagonal, and a request with fewer keys than queries leaves rows that see
    no key."""
    qlens = [1, 127, 128, 129, 255, 256, 300, 513]
    klens = [40, 127, 300, 129, 600, 256, 1000, 300]
    c = make_case(qlens, klens, B=64, hq=hq, hkv=hkv, seed=hq + hkv + int(causal))
    out = run_gpu(c, causal)
    torch.cuda.synchronize()
    assert_close(widen(out), run_oracle(c, causal), "bf16", f"{hq}/{hkv} causal={causal}")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("causal", [True, False])
def test_causal_flag(causal):
    c = make_case([131, 7, 256], [131, 300, 600], B=32, seed=5)
    assert_close(widen(run_gpu(c, causal)), run_oracle(c, causal), "bf16", str(causal))


def test_single_query_equals_decode():
    """q_len = 1 prefill (causal or not) equals paged decode over the same keys."""
    lens = [1, 200, 513, 4096]
    c = make_case([1] * 4, lens, B=16, seed=9)
    dec = pkv.paged_decode(to_dev(c["q"]), to_dev(c["kc"]), to_dev(c["vc"]), to_dev(c["table"]),
                           to_dev(np.array(lens, np.int32)), c["scale"])
    for causal in (True, False):
        pre = run_gpu(c, causal)
        torch.cuda.synchronize()
        err = np.abs(widen(pre) - widen(dec))
        assert err.max() <= 2e-2 and err.mean() <= 2e-3


@pytest.mark.parametrize("cfg", [5, 4])
def test_config_prefill(cfg):
    """Workload step: write the new tokens, then prefill, compared with the
    oracle on every query row and head (workload 4: 17,928 rows, a few seconds
    of the multi-threaded oracle)."""
    step = W.config(cfg)
    dev = DevStep(step)
    dev.write()
    out = dev.prefill()
    torch.cuda.synchronize()
    _, kc, vc = oracle_write(step)
    want = oracle.prefill(step.q_prefill, kc, vc, step.cu_q, step.cu_k, step.scale, causal=True,
                          block_table=step.prefill_table, block_size=step.block_size)
    assert_close(widen(out), want, "bf16", f"cfg{cfg}")
    assert pkv.paged_error_flags() == 0


def test_physical_permutation_bitwise():
    c = make_case([300, 90], [700, 90], B=16, seed=3)
    a = to_host(run_gpu(c))
    nb = c["kc"].shape[0]
    perm = np.random.default_rng(4).permutation(nb)
    inv = np.argsort(perm)
    c2 = dict(c, kc=c["kc"][inv], vc=c["vc"][inv],
              table=np.where(c["table"] >= 0, perm[np.maximum(c["table"], 0)], -1).astype(np.int32))
    b = to_host(run_gpu(c2))
    assert np.array_equal(a, b)


def test_nonfinite_pool_padding_is_ignored():
    """Pool slots past a request's keys hold NaN: they must not leak into the
    output (p = 0 for those keys)."""
    c = make_case([50, 3], [70, 3], B=64, seed=11)
    kc, vc = c["kc"].copy(), c["vc"].copy()
    for r, k in enumerate([70, 3]):
        blk = c["table"][r, (k - 1) // 64]
        kc[blk, k % 64:] = 0x7fc0  # bf16 NaN
        vc[blk, k % 64:] = 0x7fc0
    c2 = dict(c, kc=kc, vc=vc)
    out = widen(run_gpu(c2))
    assert np.all(np.isfinite(out))
    assert_close(out, run_oracle(c), "bf16", "nan padding")


@pytest.mark.parametrize("B,entry", [(64, 2), (16, 3), (16, 4), (16, 2), (16, 9), (32, 5)])
def test_bad_block_id_is_flagged(B, entry):
    """A table entry outside the pool is flagged and its page skipped.  With
    several pages per 128-key tile (B < 128) the pages of a tile are shared by
    three producer warps (page p of a tile by warp p mod 3); the cases put the
    bad page in each of them.  Nothing waits past its time limit."""
    c = make_case([40], [300], B=B, seed=12)
    c["table"][0, entry] = 10_000
    run_gpu(c)
    torch.cuda.synchronize()
    flags = pkv.paged_error_flags()
    assert flags & pkv.PKV_FLAG_BAD_BLOCK
    assert not flags & pkv.PKV_FLAG_TIMEOUT


def test_unsupported_combinations():
    c = make_case([4], [4], B=16, d=96, seed=1)
    with pytest.raises(pkv.PagedKVError) as e:
        run_gpu(c)
    assert e.value.status == -2
    c = make_case([4], [4], B=24, seed=1)
    with pytest.raises(pkv.PagedKVError) as e:
        run_gpu(c)
    assert e.value.status == -2


@pytest.mark.parametrize("step", [0.15, 0.6])
def test_growing_scores(step):
    """Keys whose scores rise tile by tile: each 128-key tile of row 0 lies
    ~`step` * 16 (log2 units) above the previous one, so the softmax's row
    sum outgrows 2^8 without the reference moving (step 0.15) and the
    reference itself moves and O is rescaled mid-row (both steps)."""
    rng = np.random.default_rng(21)
    d, B, qlen, klen = 128, 64, 130, 900
    q = rng.standard_normal((qlen, 2, d))
    u = q[qlen - 1, 0] / np.linalg.norm(q[qlen - 1, 0])
    gain = step * (np.arange(klen) // 128) + 0.05 * rng.standard_normal(klen)
    k = 0.3 * rng.standard_normal((klen, 1, d)) + (gain[:, None] * u[None, :] * 12.0)[:, None, :]
    v = rng.standard_normal((klen, 1, d))
    nb = -(-klen // B) + 2
    order = rng.permutation(nb).astype(np.int32)
    table = order[: -(-klen // B)][None, :].copy()
    kc = np.zeros((nb, B, 1, d))
    vc = np.zeros((nb, B, 1, d))
    for j in range(klen):
        kc[table[0, j // B], j % B] = k[j]
        vc[table[0, j // B], j % B] = v[j]
    c = dict(q=_bf(q), kc=_bf(kc), vc=_bf(vc), table=table,
             cq=np.array([0, qlen], np.int32), ck=np.array([0, klen], np.int32), B=B,
             scale=1 / math.sqrt(d))
    for causal in (True, False):
        got = widen(run_gpu(c, causal))
        assert np.all(np.isfinite(got))
        assert_close(got, run_oracle(c, causal), "bf16", f"step {step} causal {causal}")
    assert pkv.paged_error_flags() == 0


def packed_case(qlens, klens, hq=16, hkv=8, d=128, seed=0, tail=0):
    """Packed K/V [sum(klens) + tail, Hkv, d]; request r's keys are rows
    cu_k[r] .. cu_k[r+1]-1 (tail rows after the last request hold NaN)."""
    rng = np.random.default_rng(seed)
    cq = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(klens)]).astype(np.int32)
    k = _bf(rng.standard_normal((int(ck[-1]) + tail, hkv, d)))
    v = _bf(rng.standard_normal((int(ck[-1]) + tail, hkv, d)))
    k[int(ck[-1]):] = 0x7fc0
    v[int(ck[-1]):] = 0x7fc0
    q = _bf(rng.standard_normal((int(cq[-1]), hq, d)))
    return dict(q=q, k=k, v=v, cq=cq, ck=ck, scale=1 / math.sqrt(d))


def run_packed(c, causal=True):
    return pkv.paged_varlen_prefill(
        to_dev(c["q"]), to_dev(c["k"]), to_dev(c["v"]), to_dev(c["cq"]), to_dev(c["ck"]),
        int(np.diff(c["cq"]).max()), int(np.diff(c["ck"]).max()), None, causal=causal,
        scale=c["scale"])


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qlens,klens,tail", [
    ([10, 3, 1], [0, 1, 7], 0),                       # the varlen example's lengths
    ([1, 127, 128, 129, 300], [1, 200, 128, 400, 1000], 0),
    ([64, 700], [64, 1500], 37),                      # NaN rows after the last request
    ([200, 64], [260, 64], 0),
])
def test_contiguous_varlen(qlens, klens, tail, causal):
    """block_table = NULL: plain varlen attention over packed K/V."""
    c = packed_case(qlens, klens, seed=sum(qlens) + tail, tail=tail)
    got = widen(run_packed(c, causal))
    want = oracle.prefill(c["q"], c["k"], c["v"], c["cq"], c["ck"], c["scale"], causal=causal)
    assert np.all(np.isfinite(got))
    assert_close(got, want, "bf16", f"packed {qlens}/{klens}")
    assert pkv.paged_error_flags() == 0


def test_contiguous_equals_paged_bitwise():
    """The same keys read packed or through a block table give identical bits."""
    qlens, klens, B = [100, 256, 33], [300, 900, 33], 64
    c = packed_case(qlens, klens, seed=5)
    rng = np.random.default_rng(6)
    need = [-(-k // B) for k in klens]
    nb = sum(need) + 2
    order = rng.permutation(nb).astype(np.int32)
    table = np.full((len(klens), max(need)), -1, np.int32)
    kc = np.zeros((nb, B) + c["k"].shape[1:], np.uint16)
    vc = np.zeros_like(kc)
    nxt = 0
    for r, kl in enumerate(klens):
        table[r, : need[r]] = order[nxt: nxt + need[r]]
        nxt += need[r]
        for j in range(kl):
            kc[table[r, j // B], j % B] = c["k"][c["ck"][r] + j]
            vc[table[r, j // B], j % B] = c["v"][c["ck"][r] + j]
    paged = pkv.paged_varlen_prefill(
        to_dev(c["q"]), to_dev(kc), to_dev(vc), to_dev(c["cq"]), to_dev(c["ck"]), max(qlens),
        max(klens), to_dev(table), causal=True, scale=c["scale"])
    assert np.array_equal(to_host(paged), to_host(run_packed(c)))


def test_contiguous_keys_past_the_arrays_are_flagged():
    c = packed_case([8], [40], seed=2)
    c["ck"] = np.array([0, 60], np.int32)  # claims more keys than the arrays hold
    run_packed(c)
    torch.cuda.synchronize()
    assert pkv.paged_error_flags() & pkv.PKV_FLAG_BAD_LENGTH
