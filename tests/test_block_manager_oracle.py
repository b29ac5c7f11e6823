"""The block-manager oracle against what the pages fix: the worked prefix-cache
trace (refcounts, shared blocks, released block, final table) and the
reference-counting / copy-on-write rules, plus invariants over random
operation sequences and a brute-force cross-check of prefix sharing."""
import json
import os
import random

import numpy as np
import pytest

from oracle.block_manager import BlockManager, NoSpace, copy_blocks

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "prefix_cache_refcount_trace.json")


def test_prefix_cache_trace():
    """题目6: prefix ABCD -> blocks 0,1 (refs 1,1); request 1 shares 0,1 and
    takes 2; request 2 shares 0,1 and takes 3; freeing request 1 releases only
    block 2; request 2's table is [0,1,3]."""
    g = json.load(open(GOLDEN))
    bm = BlockManager(8, g["block_size"])
    ids = {}
    for st in g["steps"]:
        if st["op"] == "allocate":
            sid, cached = bm.allocate([g["tokens"][c] for c in st["tokens"]])
            ids[st["name"]] = sid
            assert bm.table(sid) == st["table"]
            assert cached == g["block_size"] * len(st.get("shared", []))
        elif st["op"] == "free":
            before = set(bm.free_stack())
            bm.free_seq(ids[st["name"]])
            assert sorted(set(bm.free_stack()) - before) == st["released"]
        else:
            assert bm.table(ids[st["name"]]) == st["table"]
            continue
        for b, r in st["refs"].items():
            assert bm.ref[int(b)] == r, (st, b)


def test_release_of_shared_block_only_drops_a_reference():
    """§11.3: freeing a block that is still shared withdraws one reference and
    leaves the other holder's data in place."""
    bm = BlockManager(6, 4)
    a, _ = bm.allocate(range(10))           # blocks 0,1,2 (2 partial)
    b = bm.fork(a)
    assert [bm.ref[x] for x in bm.table(a)] == [2, 2, 2]
    bm.free_seq(a)
    assert bm.table(b) == [0, 1, 2] and [bm.ref[x] for x in bm.table(b)] == [1, 1, 1]
    assert bm.num_free() == 3
    bm.free_seq(b)
    assert bm.num_free() == 6 and bm.free_stack()[-1] == 0  # released in reverse: 0 on top


def test_copy_on_write():
    """§11.3: a write into a shared block first copies it into a new block,
    which the writer then owns; the other holder keeps the old block."""
    bm = BlockManager(6, 4)
    a, _ = bm.allocate(range(6))            # [0,1], block 1 holds 2 of 4 tokens
    b = bm.fork(a)
    assert bm.append(b, 99) == (1, 2)       # shared partial block 1 -> copy into 2
    assert bm.table(a) == [0, 1] and bm.table(b) == [0, 2]
    assert bm.ref[0] == 2 and bm.ref[1] == 1 and bm.ref[2] == 1
    assert bm.append(a, 7) == (-1, -1)      # block 1 is now a's alone: in place
    assert bm.append(b, 98) == (-1, -1)     # fills block 2 (4 tokens)
    assert bm.append(b, 97) == (-1, -1) and bm.table(b) == [0, 2, 3]  # new block, no copy
    k = np.arange(6 * 4 * 3).reshape(6, 4, 3)
    v = -k
    copy_blocks(k, v, [1], [2])
    assert np.array_equal(k[2], k[1]) and np.array_equal(v[2], v[1])


def test_full_block_filled_by_append_is_shared_later():
    bm = BlockManager(8, 2)
    a, _ = bm.allocate([5])
    bm.append(a, 6)                          # block 0 = (5,6) now full -> cached
    b, cached = bm.allocate([5, 6, 7])
    assert cached == 2 and bm.table(b)[0] == bm.table(a)[0] and bm.ref[bm.table(a)[0]] == 2


def test_no_space_changes_nothing():
    bm = BlockManager(3, 2)
    a, _ = bm.allocate([1, 2, 3, 4])
    snap = (list(bm.ref), bm.free_stack(), dict(bm.cache))
    with pytest.raises(NoSpace):
        bm.allocate([9, 9, 9, 9, 9])
    assert (list(bm.ref), bm.free_stack(), dict(bm.cache)) == snap
    b, cached = bm.allocate([1, 2, 3, 4, 5])  # 2 shared + 1 new fits
    assert cached == 4 and bm.num_free() == 0
    c = bm.fork(b)
    snap = (list(bm.ref), bm.free_stack(), bm.table(b), bm.table(c))
    with pytest.raises(NoSpace):
        bm.append(c, 6)                      # the shared partial block needs a copy
    assert (list(bm.ref), bm.free_stack(), bm.table(b), bm.table(c)) == snap


def check_invariants(bm: BlockManager):
    held = [0] * bm.num_blocks
    for s in bm.seqs.values():
        B = bm.block_size
        assert len(s["table"]) == -(-len(s["tokens"]) // B)
        for b in s["table"]:
            held[b] += 1
    assert held == bm.ref                                   # ref = holders
    free = bm.free_stack()
    assert len(set(free)) == len(free)
    assert set(free) == {b for b in range(bm.num_blocks) if bm.ref[b] == 0}
    for key, b in bm.cache.items():
        assert bm.ref[b] > 0 and bm.key_of[b] == key
        parent, toks = key
        # some live sequence holds `b` right after `parent` with these tokens
        ok = False
        for s in bm.seqs.values():
            t = s["table"]
            for i, x in enumerate(t):
                if x == b and (t[i - 1] if i else -1) == parent and \
                        tuple(s["tokens"][i * bm.block_size:(i + 1) * bm.block_size]) == toks:
                    ok = True
        assert ok


def shared_prefix_blocks(bm, t1, t2):
    """Brute force: full leading blocks two token lists have in common."""
    B, n = bm.block_size, 0
    while (n + 1) * B <= min(len(t1), len(t2)) and t1[:(n + 1) * B] == t2[:(n + 1) * B]:
        n += 1
    return n


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_keep_invariants(seed):
    rng = random.Random(seed)
    bm = BlockManager(40, rng.choice([1, 2, 3, 4]))
    prompts = [[rng.randrange(3) for _ in range(rng.randrange(1, 14))] for _ in range(6)]
    for _ in range(300):
        op = rng.random()
        live = list(bm.seqs)
        try:
            if op < 0.3 or not live:
                p = list(rng.choice(prompts))
                sid, cached = bm.allocate(p)
                # prefix sharing found exactly the common full blocks with live sequences
                # whose blocks are still cached along the chain
                assert cached % bm.block_size == 0
            elif op < 0.45:
                bm.fork(rng.choice(live))
            elif op < 0.8:
                bm.append(rng.choice(live), rng.randrange(3))
            else:
                bm.free_seq(rng.choice(live))
        except NoSpace:
            pass
        check_invariants(bm)


def test_sharing_matches_brute_force():
    """Two sequences allocated back to back share exactly their common full
    leading blocks (nothing else is live)."""
    rng = random.Random(7)
    for _ in range(200):
        B = rng.choice([1, 2, 3, 4])
        bm = BlockManager(64, B)
        t1 = [rng.randrange(2) for _ in range(rng.randrange(1, 12))]
        t2 = [rng.randrange(2) for _ in range(rng.randrange(1, 12))]
        a, _ = bm.allocate(t1)
        b, cached = bm.allocate(t2)
        n = shared_prefix_blocks(bm, t1, t2)
        assert cached == n * B
        assert bm.table(a)[:n] == bm.table(b)[:n]
        assert not set(bm.table(a)[n:]) & set(bm.table(b)[n:])
