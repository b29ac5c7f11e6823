"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each ``pin_*`` takes a loaded oracle library (``oracle.load()`` or a variant
compiled with a planted mistake) and raises AssertionError when the oracle
disagrees with the pinned fact.  ``tests/test_oracle_pins.py`` runs them on the
real oracle; ``tests/test_oracle_mutations.py`` checks that every planted
mistake is caught by at least one of them.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _sdpa(q, k, v, scale, mask=None):
    """torch fp64 scaled-dot-product attention; q [Hq, Lq, d], k/v [Hkv, Lk, d]."""
    q = torch.as_tensor(q, dtype=torch.float64)[None]
    k = torch.as_tensor(k, dtype=torch.float64)[None]
    v = torch.as_tensor(v, dtype=torch.float64)[None]
    out = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=scale, enable_gqa=q.shape[1] != k.shape[1])
    return out[0].numpy()


# ---------------------------------------------------------------------------
# worked examples printed on the pages
# ---------------------------------------------------------------------------

def pin_online_trace(lib):
    """题目2: x=[2,1,4,3] -> [m,l] = [2,1],[2,1.3679],[4,1.1851],[4,1.5529]."""
    g = golden("online_softmax_trace.json")
    m, l = oracle.online_softmax_trace(np.array(g["x"], dtype=np.float64), lib=lib)
    printed = np.array(g["printed_states_after_each_element"], dtype=np.float64)
    assert np.allclose(m, printed[:, 0], atol=0, rtol=0), (m, printed)
    assert np.allclose(l, printed[:, 1], atol=2e-4, rtol=0), (l, printed)
    # closed forms of the same states
    e = math.exp
    exact = [1.0, 1.0 + e(-1), (1.0 + e(-1)) * e(-2) + 1.0, (1.0 + e(-1)) * e(-2) + 1.0 + e(-1)]
    assert np.allclose(l, exact, atol=1e-13, rtol=0)
    assert abs(l[-1] - (e(-2) + e(-3) + e(-1) + 1.0)) < 1e-13


def pin_flash_example(lib):
    """题目3: N=4, d=2, Br=Bc=2 FlashAttention walk-through."""
    g = golden("flash_worked_example.json")
    Q, K, V = (np.array(g[x], dtype=np.float64) for x in "QKV")
    scale = 1.0 / math.sqrt(2.0)
    O, mh, lh, ch = oracle.flash_tiles(Q, K, V, g["Br"], g["Bc"], scale, lib=lib)
    pr = g["printed"]
    assert np.allclose(ch[0, 0], pr["Q1_correction_at_K1"], atol=0)
    assert np.allclose(mh[0, 0], pr["Q1_m_after_K1"], atol=5e-4)
    assert np.allclose(lh[0, 0], pr["Q1_l_after_K1"], atol=5e-4)
    assert np.allclose(ch[0, 1], pr["Q1_correction_at_K2"], atol=1e-15)
    # closed form of the final outputs, a = e^(-1/sqrt 2)
    a = math.exp(-1.0 / math.sqrt(2.0))
    expect = np.array([[1 / (1 + a), 0.5],
                       [0.5, 0.5],
                       [1 / (1 + a), 2 * a / (1 + a) ** 2],
                       [0.5, 0.5]])
    assert np.allclose(O, expect, atol=1e-13, rtol=0), (O, expect)
    assert np.allclose(lh[0, 1], [2 + 2 * a, 2 + 2 * a], atol=1e-13)
    assert np.allclose(lh[1, 1], [(1 + a) ** 2, 4.0], atol=1e-13)
    # the tiled walk equals the one-shot definition (decode on a dense layout)
    for r in range(4):
        out, _, _ = oracle.online_attention(Q[r], K, V, scale, [4], lib=lib)
        assert np.allclose(out, expect[r], atol=1e-13)


def pin_token9(lib):
    """题目5: B=4, table [3,1,5]; token 9 -> logical 2, physical 5, offset 1."""
    g = golden("block_table_token9.json")
    B, table = g["block_size"], np.array(g["block_table"], dtype=np.int32)
    slots = [oracle.slot_id(table, B, p, lib=lib) for p in range(g["num_tokens"])]
    t = g["token"]
    assert slots[t] // B == g["physical_block"] and slots[t] % B == g["offset_in_block"]
    assert t // B == g["logical_block"]
    # physical layout: which tokens each physical block holds (12-slot view)
    full = [oracle.slot_id(table, B, p, lib=lib) for p in range(len(table) * B)]
    layout = {}
    for p, s in enumerate(full):
        layout.setdefault(str(s // B), []).append(p)
    assert layout == g["physical_layout"], layout
    stored_last = [p for p, s in enumerate(slots) if s // B == g["physical_block"]]
    assert stored_last == g["last_block_tokens_stored"]
    assert (len(stored_last) == B) == g["last_block_full"]
    # element offset = phys*B*kvDim + slot*kvDim (kvDim = 8 here)
    assert oracle.element_offset(table, B, 8, t, lib=lib) == (5 * B + 1) * 8


def pin_decode_example(lib):
    """Sayfalı dikkat decode example: cache_seqlens [30,32,70], B=32."""
    g = golden("decode_example.json")
    table = np.array(g["block_table"], dtype=np.int32)
    B, lens = g["block_size"], g["cache_seqlens"]
    seq = np.arange(3, dtype=np.int32)
    slots = oracle.build_slot_mapping(table, seq, np.array(lens, dtype=np.int32), B, lib=lib)
    assert list(slots) == [2 * 32 + 30, 1 * 32 + 0, 6 * 32 + 6], slots
    for b, L in enumerate(lens):
        prev = oracle.slot_id(table[b], B, L - 1, lib=lib) // B
        new = slots[b] // B
        assert (prev == new) == g["new_token_fits_in_last_cached_block"][b]
        assert new in g["blocks_listed_per_sequence"][b]
        assert len({oracle.slot_id(table[b], B, p, lib=lib) // B for p in range(L)}) == \
            g["blocks_needed_for_cached_tokens"][b]
    # padding rows map to -1
    s2 = oracle.build_slot_mapping(table, np.array([0, -1, 2], np.int32),
                                   np.array([30, 5, 70], np.int32), B, lib=lib)
    assert list(s2) == [94, -1, 198]


def pin_cu_seqlens(lib):
    """Sayfalı dikkat varlen example: cu_seq_lens_q [0,10,13,14], _k [0,0,1,8]."""
    g = golden("cu_seqlens_example.json")
    cq, ck = np.array(g["cu_seq_lens_q"]), np.array(g["cu_seq_lens_k"])
    assert list(np.diff(cq)) == g["q_lens"] and list(np.diff(ck)) == g["k_lens"]
    assert np.diff(cq).max() == g["max_length_q"] and np.diff(ck).max() == g["max_length_k"]
    assert list(oracle.request_index(cq, lib=lib)) == g["q_request_index"]
    assert list(oracle.request_index(ck, lib=lib)) == g["k_request_index"]


def pin_prefill_example(lib):
    """Prefill on the varlen example's lengths under bottom-right causal
    alignment: r0 (10 queries, 0 keys) and r1 rows 0-1 see nothing (output 0);
    r1 row 2 sees exactly key 0 (output = that V row); r2's single query sees
    all 7 keys.  Checked for the packed (no table) and the paged layouts."""
    g = golden("cu_seqlens_example.json")
    cq = np.array(g["cu_seq_lens_q"], np.int32)
    ck = np.array(g["cu_seq_lens_k"], np.int32)
    rng = np.random.default_rng(5)
    hq, hkv, d = 4, 2, 8
    q = rng.standard_normal((14, hq, d)).astype(np.float32)
    k = rng.standard_normal((8, hkv, d)).astype(np.float32)
    v = rng.standard_normal((8, hkv, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    out = oracle.prefill(q, k, v, cq, ck, scale, causal=True, lib=lib)
    assert np.all(out[0:12] == 0.0)
    for h in range(hq):
        assert np.array_equal(out[12, h], v[0, h // 2].astype(np.float64))
    ref = _sdpa(q[13][:, None, :], k[1:8].transpose(1, 0, 2), v[1:8].transpose(1, 0, 2), scale)
    assert np.allclose(out[13], ref[:, 0, :], atol=1e-12)
    # paged layout: B=2, requests' keys scattered over a pool of 8 blocks
    B = 2
    perm = np.array([6, 1, 4, 0, 7, 3, 2, 5], np.int32)
    table = np.full((3, 4), -1, np.int32)
    table[1, :1] = perm[:1]
    table[2, :4] = perm[1:5]
    kc = rng.standard_normal((8, B, hkv, d)).astype(np.float32)
    vc = rng.standard_normal((8, B, hkv, d)).astype(np.float32)
    for r, (lo, hi) in enumerate(zip(ck[:-1], ck[1:])):
        for j in range(hi - lo):
            blk, off = table[r, j // B], j % B
            kc[blk, off], vc[blk, off] = k[lo + j], v[lo + j]
    out2 = oracle.prefill(q, kc, vc, cq, ck, scale, causal=True, block_table=table,
                          block_size=B, lib=lib)
    assert np.array_equal(out2, out)


# ---------------------------------------------------------------------------
# library routines and closed forms
# ---------------------------------------------------------------------------

def pin_bf16_rounding(lib):
    """fp32 -> bf16 round-to-nearest-even equals torch's cast, incl. ties."""
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(2000).astype(np.float32),
        (rng.standard_normal(500) * 1e-39).astype(np.float32),  # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38, 1.0, 1.00390625, 1.01171875,
                  1.0078125 + 2.0 ** -8, 65504.0], dtype=np.float32),
    ])
    # exact ties: bf16 value + half an ulp, for both even and odd mantissas
    base = np.arange(0x3f80, 0x3f90, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties])
    got = oracle.f32_to_bf16(vals, lib=lib)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), np.nonzero(got != want)


def pin_kv_write(lib):
    """Write: rows land at slot*kvDim, negative slots write nothing, fp32->bf16
    casts round to nearest even, equal dtypes copy bits."""
    rng = np.random.default_rng(3)
    nb, B, hkv, d = 6, 4, 2, 8
    kv_dim = hkv * d
    slots = np.array([5, -1, 0, 23, -1, 12], np.int32)
    k = rng.standard_normal((6, hkv, d)).astype(np.float32)
    v = rng.standard_normal((6, hkv, d)).astype(np.float32)
    canary = np.float32(-12345.5)
    kc = np.full((nb, B, hkv, d), canary, np.float32)
    vc = np.full((nb, B, hkv, d), canary, np.float32)
    oracle.kv_write(k, v, slots, kc, vc, lib=lib)
    kf, vf = kc.reshape(-1, kv_dim), vc.reshape(-1, kv_dim)
    written = {int(s): n for n, s in enumerate(slots) if s >= 0}
    for s in range(nb * B):
        if s in written:
            assert np.array_equal(kf[s], k[written[s]].ravel())
            assert np.array_equal(vf[s], v[written[s]].ravel())
        else:
            assert np.all(kf[s] == canary) and np.all(vf[s] == canary)
    # fp32 source into a bf16 cache
    kb = np.zeros((nb, B, hkv, d), np.uint16)
    vb = np.zeros((nb, B, hkv, d), np.uint16)
    oracle.kv_write(k, v, slots, kb, vb, lib=lib)
    want = torch.from_numpy(k).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(kb.reshape(-1, kv_dim)[23], want[3].ravel())
    assert np.all(kb.reshape(-1, kv_dim)[1] == 0)


def _paged_from_sequences(rng, seqs_k, seqs_v, B, num_blocks):
    """Scatter contiguous per-sequence K/V [L, Hkv, d] into a shuffled pool."""
    hkv, d = seqs_k[0].shape[1:]
    kc = rng.standard_normal((num_blocks, B, hkv, d)).astype(np.float32)
    vc = rng.standard_normal((num_blocks, B, hkv, d)).astype(np.float32)
    order = rng.permutation(num_blocks).astype(np.int32)
    width = max(1, max(-(-len(s) // B) for s in seqs_k))
    table = np.full((len(seqs_k), width), -1, np.int32)
    nxt = 0
    for b, (ks, vs) in enumerate(zip(seqs_k, seqs_v)):
        nblk = -(-len(ks) // B)
        table[b, :nblk] = order[nxt: nxt + nblk]
        nxt += nblk
        for j in range(len(ks)):
            kc[table[b, j // B], j % B] = ks[j]
            vc[table[b, j // B], j % B] = vs[j]
    return kc, vc, table


def pin_decode_vs_sdpa(lib):
    """Paged decode equals torch fp64 SDPA (GQA) on the contiguous sequences."""
    rng = np.random.default_rng(21)
    hq, hkv, d, B = 6, 2, 16, 4
    lens = [1, 5, 13, 8, 0]
    ks = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in lens]
    vs = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in lens]
    kc, vc, table = _paged_from_sequences(rng, ks, vs, B, 12)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float32)
    scale = 0.37
    out = oracle.decode(q, kc, vc, table, np.array(lens, np.int32), scale, lib=lib)
    for b, L in enumerate(lens):
        if L == 0:
            assert np.all(out[b] == 0)
            continue
        ref = _sdpa(q[b][:, None, :], ks[b].transpose(1, 0, 2), vs[b].transpose(1, 0, 2), scale)
        assert np.allclose(out[b], ref[:, 0, :], atol=1e-12), b


def pin_prefill_vs_sdpa(lib):
    """Paged causal prefill over a cached prefix equals torch fp64 SDPA with
    the lower-right causal bias (rows that see no key: output 0)."""
    from torch.nn.attention.bias import causal_lower_right
    rng = np.random.default_rng(22)
    hq, hkv, d, B = 4, 2, 16, 4
    qlens, cached = [5, 1, 7, 3], [3, 0, 9, 0]
    klens = [a + b for a, b in zip(qlens, cached)]
    ks = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in klens]
    vs = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in klens]
    kc, vc, table = _paged_from_sequences(rng, ks, vs, B, 16)
    cq = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(klens)]).astype(np.int32)
    q = rng.standard_normal((cq[-1], hq, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    for causal in (True, False):
        out = oracle.prefill(q, kc, vc, cq, ck, scale, causal=causal, block_table=table,
                             block_size=B, lib=lib)
        packed_k = np.concatenate(ks)
        packed_v = np.concatenate(vs)
        out_packed = oracle.prefill(q, packed_k, packed_v, cq, ck, scale, causal=causal, lib=lib)
        assert np.array_equal(out, out_packed)
        for r in range(len(qlens)):
            qq = q[cq[r]:cq[r + 1]].transpose(1, 0, 2)
            mask = causal_lower_right(qlens[r], klens[r]) if causal else None
            ref = _sdpa(qq, ks[r].transpose(1, 0, 2), vs[r].transpose(1, 0, 2), scale, mask)
            assert np.allclose(out[cq[r]:cq[r + 1]], ref.transpose(1, 0, 2), atol=1e-12), r


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

def _compositions(n):
    for cuts in itertools.product([0, 1], repeat=n - 1):
        lens, cur = [], 1
        for c in cuts:
            if c:
                lens.append(cur)
                cur = 1
            else:
                cur += 1
        lens.append(cur)
        yield lens


def pin_online_equals_one_shot(lib):
    """Block-wise merge over every chunking of n <= 12 keys equals the one-shot
    softmax (same keys, dense layout) within 1e-12."""
    rng = np.random.default_rng(31)
    for n in (1, 2, 3, 5, 8, 12):
        d = 4
        q = rng.standard_normal(d)
        K = rng.standard_normal((n, d)) * 2.0
        V = rng.standard_normal((n, d))
        scale = 0.7
        kc = K.astype(np.float32)[None, :, None, :]
        vc = V.astype(np.float32)[None, :, None, :]
        ref = oracle.decode(q.astype(np.float32)[None, None, :], kc, vc,
                            np.zeros((1, 1), np.int32), np.array([n], np.int32), scale,
                            lib=lib)[0, 0]
        Kf = kc[0, :, 0, :].astype(np.float64)
        Vf = vc[0, :, 0, :].astype(np.float64)
        qf = q.astype(np.float32).astype(np.float64)
        for lens in _compositions(n):
            out, m, l = oracle.online_attention(qf, Kf, Vf, scale, lens, lib=lib)
            assert np.allclose(out, ref, atol=1e-12, rtol=0), (n, lens)
            s = scale * Kf @ qf
            assert abs(m - s.max()) < 1e-12 and abs(l - np.exp(s - s.max()).sum()) < 1e-12


def pin_permutation_invariance(lib):
    """Moving physical blocks (data and table together) leaves decode and
    prefill outputs unchanged (bit for bit: the gather order is logical)."""
    rng = np.random.default_rng(41)
    hq, hkv, d, B, nb = 4, 2, 8, 4, 10
    kc = rng.standard_normal((nb, B, hkv, d)).astype(np.float32)
    vc = rng.standard_normal((nb, B, hkv, d)).astype(np.float32)
    table = np.array([[3, 7, 1, -1], [0, 9, 4, 2]], np.int32)
    lens = np.array([11, 16], np.int32)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    out = oracle.decode(q, kc, vc, table, lens, 0.5, lib=lib)
    perm = rng.permutation(nb)
    inv = np.argsort(perm)
    kc2, vc2 = kc[inv], vc[inv]  # new block p holds old block inv[p]; old b -> perm[b]
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    out2 = oracle.decode(q, kc2, vc2, table2, lens, 0.5, lib=lib)
    assert np.array_equal(out, out2)
    cq = np.array([0, 3, 5], np.int32)
    ck = np.array([0, 11, 27], np.int32)
    qp = rng.standard_normal((5, hq, d)).astype(np.float32)
    a = oracle.prefill(qp, kc, vc, cq, ck, 0.5, block_table=table, block_size=B, lib=lib)
    b = oracle.prefill(qp, kc2, vc2, cq, ck, 0.5, block_table=table2, block_size=B, lib=lib)
    assert np.array_equal(a, b)


def pin_special_cases(lib):
    """L=1 returns v0 exactly; identical keys give the mean of V; zero length
    gives 0; non-causal (and causal) prefill with one query equals decode."""
    rng = np.random.default_rng(51)
    hq, hkv, d, B = 2, 1, 8, 4
    kc = rng.standard_normal((3, B, hkv, d)).astype(np.float32)
    vc = rng.standard_normal((3, B, hkv, d)).astype(np.float32)
    table = np.array([[2, 0, 1]], np.int32)
    q = rng.standard_normal((1, hq, d)).astype(np.float32)
    out = oracle.decode(q, kc, vc, table, np.array([1], np.int32), 0.3, lib=lib)
    assert np.array_equal(out[0, 0], vc[2, 0, 0].astype(np.float64))
    out0 = oracle.decode(q, kc, vc, table, np.array([0], np.int32), 0.3, lib=lib)
    assert np.all(out0 == 0)
    kc_same = kc.copy()
    kc_same[:] = kc[0, 0]
    out = oracle.decode(q, kc_same, vc, table, np.array([10], np.int32), 0.3, lib=lib)
    rows = [vc[table[0, j // B], j % B, 0].astype(np.float64) for j in range(10)]
    assert np.allclose(out[0, 1], np.mean(rows, axis=0), atol=1e-13)
    dec = oracle.decode(q, kc, vc, table, np.array([9], np.int32), 0.3, lib=lib)
    for causal in (False, True):
        pre = oracle.prefill(q, kc, vc, np.array([0, 1], np.int32), np.array([0, 9], np.int32),
                             0.3, causal=causal, block_table=table, block_size=B, lib=lib)
        assert np.array_equal(pre, dec)


def _bf16_to_f64(u16: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns with torch (a library routine, not the oracle's)."""
    return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def pin_bf16_inputs(lib):
    """bf16 q/K/V are widened exactly: decode and prefill on bf16 inputs equal
    torch fp64 SDPA on torch's own widening; a bf16 -> fp32 cache write is the
    exact widening."""
    rng = np.random.default_rng(61)
    hq, hkv, d, B = 4, 2, 16, 8
    lens = [9, 17, 3]
    def bf(x):
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
    ks = [bf(rng.standard_normal((L, hkv, d))) for L in lens]
    vs = [bf(rng.standard_normal((L, hkv, d))) for L in lens]
    nb = 8
    kc = bf(rng.standard_normal((nb, B, hkv, d)))
    vc = bf(rng.standard_normal((nb, B, hkv, d)))
    table = np.array([[5, 2, -1], [0, 7, 3], [6, -1, -1]], np.int32)
    for b, L in enumerate(lens):
        for j in range(L):
            kc[table[b, j // B], j % B] = ks[b][j]
            vc[table[b, j // B], j % B] = vs[b][j]
    q = bf(rng.standard_normal((3, hq, d)))
    out = oracle.decode(q, kc, vc, table, np.array(lens, np.int32), 0.25, lib=lib)
    for b, L in enumerate(lens):
        ref = _sdpa(_bf16_to_f64(q[b])[:, None, :], _bf16_to_f64(ks[b]).transpose(1, 0, 2),
                    _bf16_to_f64(vs[b]).transpose(1, 0, 2), 0.25)
        assert np.allclose(out[b], ref[:, 0, :], atol=1e-12), b
    cq = np.array([0, 2, 3, 6], np.int32)
    ck = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    qp = bf(rng.standard_normal((6, hq, d)))
    outp = oracle.prefill(qp, kc, vc, cq, ck, 0.25, causal=False, block_table=table,
                          block_size=B, lib=lib)
    for r in range(3):
        qq = _bf16_to_f64(qp[cq[r]:cq[r + 1]]).transpose(1, 0, 2)
        ref = _sdpa(qq, _bf16_to_f64(ks[r]).transpose(1, 0, 2),
                    _bf16_to_f64(vs[r]).transpose(1, 0, 2), 0.25)
        assert np.allclose(outp[cq[r]:cq[r + 1]], ref.transpose(1, 0, 2), atol=1e-12), r
    kf = np.zeros((nb, B, hkv, d), np.float32)
    vf = np.zeros((nb, B, hkv, d), np.float32)
    oracle.kv_write(ks[0], vs[0], np.arange(9, dtype=np.int32), kf, vf, lib=lib)
    assert np.array_equal(kf.reshape(-1, hkv, d)[:9].astype(np.float64), _bf16_to_f64(ks[0]))


ALL_PINS = [
    pin_online_trace, pin_flash_example, pin_token9, pin_decode_example, pin_cu_seqlens,
    pin_prefill_example, pin_bf16_rounding, pin_kv_write, pin_decode_vs_sdpa,
    pin_prefill_vs_sdpa, pin_online_equals_one_shot, pin_permutation_invariance,
    pin_special_cases, pin_bf16_inputs,
]
