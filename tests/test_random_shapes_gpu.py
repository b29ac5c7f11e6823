"""Seeded sweep over random shapes against the oracle: prefill (head_dim 64 and
128, GQA groups 1-4, block sizes 8-256, causal or not, paged or packed K/V,
requests with fewer keys than queries), decode (fp32 and bf16, groups 1, 2
and 4, block sizes 1-256) and shared-prefix decode (random groups and prefix
lengths).  Deterministic: each case's shapes come from a fixed seed."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import assert_close, to_dev, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


def _bf(x):
    return W._to_dtype(np.asarray(x, np.float32), "bf16")


@pytest.mark.parametrize("seed", range(12))
def test_random_prefill(seed):
    rng = np.random.default_rng(500 + seed)
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    hq = hkv * int(rng.choice([1, 2, 3, 4]))
    B = int(rng.choice([8, 16, 32, 64, 128, 256]))
    nreq = int(rng.integers(1, 6))
    qlens = [int(rng.integers(1, 600)) for _ in range(nreq)]
    klens = [max(0, q + int(rng.integers(-50, 700))) for q in qlens]
    causal = bool(rng.random() < 0.7)
    packed = seed % 4 == 3
    cq = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(klens)]).astype(np.int32)
    q = _bf(rng.standard_normal((int(cq[-1]), hq, d)))
    scale = 1 / math.sqrt(d)
    if packed:
        kp = _bf(rng.standard_normal((max(1, int(ck[-1])), hkv, d)))
        vp = _bf(rng.standard_normal((max(1, int(ck[-1])), hkv, d)))
        out = pkv.paged_varlen_prefill(to_dev(q), to_dev(kp), to_dev(vp), to_dev(cq), to_dev(ck),
                                       max(qlens), max(klens), None, causal=causal, scale=scale)
        torch.cuda.synchronize()
        want = oracle.prefill(q, kp, vp, cq, ck, scale, causal=causal)
    else:
        need = [-(-k // B) for k in klens]
        nb = sum(need) + 2
        order = rng.permutation(nb).astype(np.int32)
        table = np.full((nreq, max(need + [1])), -1, np.int32)
        nxt = 0
        for r, m in enumerate(need):
            table[r, :m] = order[nxt:nxt + m]
            nxt += m
        kc = _bf(rng.standard_normal((nb, B, hkv, d)))
        vc = _bf(rng.standard_normal((nb, B, hkv, d)))
        out = pkv.paged_varlen_prefill(to_dev(q), to_dev(kc), to_dev(vc), to_dev(cq), to_dev(ck),
                                       max(qlens), max(klens), to_dev(table), causal=causal,
                                       scale=scale)
        torch.cuda.synchronize()
        want = oracle.prefill(q, kc, vc, cq, ck, scale, causal=causal, block_table=table,
                              block_size=B)
    assert_close(widen(out), want, "bf16",
                 f"d{d} {hq}/{hkv} B{B} q{qlens} k{klens} causal={causal} packed={packed}")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("seed", range(12))
def test_random_decode(seed):
    rng = np.random.default_rng(700 + seed)
    dtype = str(rng.choice(["bf16", "f32"]))
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4, 8, 16]))
    hq = hkv * int(rng.choice([1, 2, 4, 8]))
    B = int(rng.choice([1, 3, 16, 32, 48, 256]))
    lens = [int(rng.integers(0, 3000)) for _ in range(int(rng.integers(1, 40)))]
    step = W.make_step(name="rnd", dtype=dtype, hq=hq, hkv=hkv, d=d, block_size=B,
                       decode_lens=[max(L - 1, 0) for L in lens], seed=900 + seed)
    step.cache_seqlens = np.asarray(lens, np.int32)
    out = pkv.paged_decode(to_dev(step.q_decode), to_dev(step.k_cache), to_dev(step.v_cache),
                           to_dev(step.decode_table), to_dev(step.cache_seqlens), step.scale)
    torch.cuda.synchronize()
    want = oracle.decode(step.q_decode, step.k_cache, step.v_cache, step.decode_table,
                         step.cache_seqlens, step.scale)
    assert_close(widen(out), want, dtype, f"{dtype} d{d} {hq}/{hkv} B{B} n{len(lens)}")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_shared_prefix(seed):
    rng = np.random.default_rng(1100 + seed)
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    hq = hkv * int(rng.choice([1, 2, 4, 8]))
    B = int(rng.choice([8, 16, 32, 64, 128, 256]))
    ngr = int(rng.integers(1, 5))
    sizes = [int(rng.integers(1, 40)) for _ in range(ngr)]
    prefixes = [int(rng.integers(0, 6)) * B for _ in range(ngr)]
    rows, lens, nxt = [], [], 0
    for gs, pl in zip(sizes, prefixes):
        shared = list(range(nxt, nxt + pl // B))
        nxt += pl // B
        for _ in range(gs):
            L = pl + int(rng.integers(0, 400))
            own = -(-L // B) - len(shared)
            rows.append(shared + list(range(nxt, nxt + own)))
            nxt += own
            lens.append(L)
    nb = nxt + 2
    perm = rng.permutation(nb).astype(np.int32)
    table = np.full((len(rows), max(len(r) for r in rows) + 1), -1, np.int32)
    for i, r in enumerate(rows):
        if r:
            table[i, : len(r)] = perm[np.array(r, dtype=np.int64)]
    kc = _bf(rng.standard_normal((nb, B, hkv, d)))
    vc = _bf(rng.standard_normal((nb, B, hkv, d)))
    q = _bf(rng.standard_normal((len(rows), hq, d)))
    gcu = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    lens = np.array(lens, np.int32)
    scale = 1 / math.sqrt(d)
    out = pkv.paged_decode_shared_prefix(to_dev(q), to_dev(kc), to_dev(vc), to_dev(table),
                                         to_dev(lens), to_dev(gcu),
                                         to_dev(np.array(prefixes, np.int32)), max(sizes), scale)
    torch.cuda.synchronize()
    want = oracle.decode(q, kc, vc, table, lens, scale)
    assert_close(widen(out), want, "bf16", f"d{d} {hq}/{hkv} B{B} {sizes} {prefixes}")
    assert pkv.paged_error_flags() == 0
