"""The library's native block manager (paged_bm_*) against the oracle:
identical block tables, reference counts, free stacks, cached-token counts,
copy-on-write pairs and out-of-space behaviour over random operation
sequences, and the worked prefix-cache trace.  Host code: no GPU needed."""
import json
import os
import random

import pytest

import paged_kv_cache_70_gb300 as pkv
from oracle.block_manager import BlockManager as Oracle, NoSpace

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "prefix_cache_refcount_trace.json")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_70_gb300 import build
    build.build()


def same_state(nat, ora, seqs):
    assert nat.free_stack() == ora.free_stack()
    assert [nat.ref_count(b) for b in range(ora.num_blocks)] == ora.ref
    for n_id, o_id in seqs.items():
        assert nat.table(n_id) == ora.table(o_id)
        assert nat.seq_len(n_id) == ora.seq_len(o_id)


def test_trace_through_native_manager():
    g = json.load(open(GOLDEN))
    bm = pkv.BlockManager(8, g["block_size"])
    ids = {}
    for st in g["steps"]:
        if st["op"] == "allocate":
            ids[st["name"]], _ = bm.allocate([g["tokens"][c] for c in st["tokens"]])
            assert bm.table(ids[st["name"]]) == st["table"]
        elif st["op"] == "free":
            bm.free(ids[st["name"]])
        else:
            assert bm.table(ids[st["name"]]) == st["table"]
            continue
        for b, r in st["refs"].items():
            assert bm.ref_count(int(b)) == r


@pytest.mark.parametrize("seed", range(8))
def test_random_operations_match_oracle(seed):
    rng = random.Random(100 + seed)
    nblocks, B = rng.choice([(24, 1), (40, 2), (40, 3), (64, 4), (16, 8)])
    nat, ora = pkv.BlockManager(nblocks, B), Oracle(nblocks, B)
    prompts = [[rng.randrange(3) for _ in range(rng.randrange(0, 3 * B + 3))] for _ in range(6)]
    seqs = {}  # native id -> oracle id
    for _ in range(400):
        op = rng.random()
        live = list(seqs)
        if op < 0.3 or not live:
            p = rng.choice(prompts)
            try:
                o = ora.allocate(p)
            except NoSpace:
                with pytest.raises(pkv.PagedKVError) as e:
                    nat.allocate(p)
                assert e.value.status == pkv.PKV_ERR_NO_SPACE
            else:
                n = nat.allocate(p)
                assert n[1] == o[1]
                seqs[n[0]] = o[0]
        elif op < 0.45:
            s = rng.choice(live)
            seqs[nat.fork(s)] = ora.fork(seqs[s])
        elif op < 0.8:
            s, tok = rng.choice(live), rng.randrange(3)
            try:
                o = ora.append(seqs[s], tok)
            except NoSpace:
                with pytest.raises(pkv.PagedKVError) as e:
                    nat.append(s, tok)
                assert e.value.status == pkv.PKV_ERR_NO_SPACE
            else:
                assert nat.append(s, tok) == o
        else:
            s = rng.choice(live)
            nat.free(s)
            ora.free_seq(seqs.pop(s))
        same_state(nat, ora, seqs)
    nat.close()


def test_invalid_arguments():
    bm = pkv.BlockManager(4, 2)
    for bad in (lambda: bm.table(7), lambda: bm.free(7), lambda: bm.fork(7),
                lambda: bm.append(7, 1), lambda: bm.ref_count(4), lambda: bm.ref_count(-1)):
        with pytest.raises(pkv.PagedKVError) as e:
            bad()
        assert e.value.status == -1
    with pytest.raises(pkv.PagedKVError):
        pkv.BlockManager(4, 0)
    empty, cached = bm.allocate([])
    assert bm.table(empty) == [] and cached == 0 and bm.num_free() == 4
