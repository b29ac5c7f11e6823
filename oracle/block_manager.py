"""Oracle of the paged KV cache's block manager: reference counts, the free
stack, prefix sharing of full blocks and copy-on-write.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this module.  It imports
nothing from the product and shares no code with the library's block manager.

Sources:
  [P1] "11. Paged attention 与 online softmax" (dilfish.github.io), §11.3
       block sharing and copy-on-write: sequences with a common prefix point
       their block tables at the same physical blocks, which are then
       read-only; a sequence about to write a new token into a shared block
       first takes a new block, copies the old contents into it and writes
       there.  refs[p] counts the block tables / prefix-cache entries that
       point at block p: allocation sets it to 1, sharing increments it,
       release decrements it, and only at 0 does the block return to the free
       stack -- releasing a block that is still shared only withdraws one
       reference.
  [P2] "结合nanovllm的FlashAttention和PagedAttention主要原理概述"
       (meredith2328.github.io), 题目6 prefix cache with reference counts: a
       block's content hash is chained from the previous block's hash
       (compute_hash(token_ids, prefix_hash)); a hit increments the found
       block's ref_count, a miss allocates a new block; a finished request is
       released by walking its block table in reverse; a block whose count
       reaches 0 leaves the hash map and goes back to the free list.

Readings where the pages leave a step open (also listed in the design notes):
  - The free blocks form a stack ([P1] "空闲栈"): allocation pops the top and a
    released block is pushed on top.  Initially the top is block 0, then 1,
    2, ... ([P2]'s trace allocates 0, 1, 2, 3 in that order).
  - Only FULL blocks are entered into the prefix cache and shared by lookup;
    a partial last block is private unless a fork shares it.
  - The chained hash is taken exactly: the cache key of block i of a token
    sequence is (physical block of block i-1, or -1 for i = 0; the B token ids
    of block i).  The physical block of the previous block identifies the
    whole prefix, so this key is what a collision-free compute_hash computes;
    a lookup therefore hits only while every earlier block of the sequence hit.
  - A full block filled by appended tokens enters the cache when it fills
    (unless its key is already present).
  - fork(seq) gives a new sequence the same blocks and tokens (every block's
    count +1); appending into a shared partial last block is the
    copy-on-write case of [P1].
"""
from __future__ import annotations


class NoSpace(Exception):
    """Not enough free blocks; the manager's state is unchanged."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        assert num_blocks >= 0 and block_size >= 1
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.ref = [0] * num_blocks
        # stack: the LAST element is the top
        self.free = list(range(num_blocks - 1, -1, -1))
        self.cache = {}      # (parent block, tuple of B token ids) -> block
        self.key_of = {}     # block -> its cache key
        self.seqs = {}       # seq id -> {"table": [...], "tokens": [...]}
        self.next_seq = 0

    # -- [P1] §11.3 counts and the free stack ---------------------------------
    def _take(self) -> int:
        b = self.free.pop()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        assert self.ref[b] > 0
        self.ref[b] -= 1
        if self.ref[b] == 0:
            key = self.key_of.pop(b, None)
            if key is not None:
                del self.cache[key]
            self.free.append(b)

    # -- [P2] 题目6 allocation with prefix lookup -----------------------------
    def allocate(self, tokens) -> tuple[int, int]:
        """New sequence holding `tokens`; returns (seq id, cached tokens)."""
        B = self.block_size
        tokens = [int(t) for t in tokens]
        nblk = -(-len(tokens) // B)
        # count the misses first so that a shortage changes nothing
        parent, misses = -1, 0
        for i in range(nblk):
            blk = tuple(tokens[i * B:(i + 1) * B])
            hit = self.cache.get((parent, blk)) if len(blk) == B else None
            if hit is None:
                misses = nblk - i
                break
            parent = hit
        if misses > len(self.free):
            raise NoSpace()
        table, cached, parent = [], 0, -1
        for i in range(nblk):
            blk = tuple(tokens[i * B:(i + 1) * B])
            key = (parent, blk) if len(blk) == B else None
            b = self.cache.get(key) if key is not None else None
            if b is not None:
                self.ref[b] += 1            # shared: one more reference
                cached += B
            else:
                b = self._take()            # new block, count 1
                if key is not None:
                    self.cache[key] = b
                    self.key_of[b] = key
            table.append(b)
            parent = b
        sid = self.next_seq
        self.next_seq += 1
        self.seqs[sid] = {"table": table, "tokens": tokens}
        return sid, cached

    def fork(self, sid: int) -> int:
        s = self.seqs[sid]
        for b in s["table"]:
            self.ref[b] += 1
        cid = self.next_seq
        self.next_seq += 1
        self.seqs[cid] = {"table": list(s["table"]), "tokens": list(s["tokens"])}
        return cid

    def append(self, sid: int, token: int) -> tuple[int, int]:
        """One more token for `sid`.  Returns (src, dst) of the block copy the
        write needs first ([P1] copy-on-write), or (-1, -1)."""
        B = self.block_size
        s = self.seqs[sid]
        L = len(s["tokens"])
        cow = (-1, -1)
        if L % B == 0:
            if not self.free:
                raise NoSpace()
            s["table"].append(self._take())
        else:
            last = s["table"][-1]
            if self.ref[last] > 1:
                if not self.free:
                    raise NoSpace()
                nb = self._take()
                self._release(last)
                s["table"][-1] = nb
                cow = (last, nb)
        s["tokens"].append(int(token))
        if (L + 1) % B == 0:
            parent = s["table"][-2] if len(s["table"]) >= 2 else -1
            key = (parent, tuple(s["tokens"][-B:]))
            b = s["table"][-1]
            if key not in self.cache and b not in self.key_of:
                self.cache[key] = b
                self.key_of[b] = key
        return cow

    def free_seq(self, sid: int) -> None:
        """Release a finished sequence, walking its table in reverse ([P2])."""
        s = self.seqs.pop(sid)
        for b in reversed(s["table"]):
            self._release(b)

    # -- queries -----------------------------------------------------------
    def table(self, sid: int) -> list[int]:
        return list(self.seqs[sid]["table"])

    def seq_len(self, sid: int) -> int:
        return len(self.seqs[sid]["tokens"])

    def num_free(self) -> int:
        return len(self.free)

    def free_stack(self) -> list[int]:
        """Free blocks, bottom of the stack first."""
        return list(self.free)


def copy_blocks(k_cache, v_cache, src, dst) -> None:
    """The copy a copy-on-write needs ([P1] §11.3): block dst of each pool
    becomes a copy of block src (numpy arrays [num_blocks, ...], in place)."""
    for s, d in zip(src, dst):
        k_cache[d] = k_cache[s]
        v_cache[d] = v_cache[s]
