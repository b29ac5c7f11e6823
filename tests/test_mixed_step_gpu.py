"""GPU parity of paged_mixed_step on the continuous-batching workload: the
prefill requests' new rows written (padding rows skipped), their causal
prefill, and the decode sequences' in-place append + decode (through the
shared-prefix path or not), against the oracle's write followed by plain
paged attention; the pools bit-exact afterwards."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_70_gb300 as pkv
from paged_kv_cache_70_gb300 import workloads as W
from gpu_helpers import assert_close, oracle_write, to_dev, to_host, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_flags():
    pkv.paged_error_flags(clear=True)
    yield


def split_step(step):
    """The step's new rows split into the decode tokens (one per sequence, in
    sequence order) and the rest (prefill tokens and padding rows)."""
    nd = step.n_decode
    is_dec = (step.token_seq >= 0) & (step.token_seq < nd)
    dec_rows = np.where(is_dec)[0]
    dec_rows = dec_rows[np.argsort(step.token_seq[dec_rows])]
    assert np.array_equal(step.token_seq[dec_rows], np.arange(nd))
    pf_rows = np.where(~is_dec)[0]
    slots = oracle.build_slot_mapping(step.table, step.token_seq, step.token_pos, step.block_size)
    return dec_rows, pf_rows, slots


def test_head_dim_64_without_groups():
    """A step with head_dim 64 (prefill part on the head_dim-64 tensor-core
    kernel, decode with append), no shared prefixes."""
    step = W.make_step(name="mix64", dtype="bf16", hq=16, hkv=8, d=64, block_size=16,
                       decode_lens=[5, 300, 1000, 16], prefill_q=[200, 1, 129],
                       prefill_cached=[0, 64, 300], seed=64)
    dec_rows, pf_rows, slots = split_step(step)
    kc, vc = to_dev(step.k_cache), to_dev(step.v_cache)
    decode = dict(q=to_dev(step.q_decode), k_new=to_dev(step.new_k[dec_rows]),
                  v_new=to_dev(step.new_v[dec_rows]), table=to_dev(step.decode_table.copy()),
                  seqlens=to_dev(step.cache_seqlens - 1))
    prefill = dict(k_new=to_dev(step.new_k[pf_rows]), v_new=to_dev(step.new_v[pf_rows]),
                   slots=to_dev(slots[pf_rows]), q=to_dev(step.q_prefill), cu_q=to_dev(step.cu_q),
                   cu_k=to_dev(step.cu_k), max_q=step.max_seqlen_q, max_k=step.max_seqlen_k,
                   table=to_dev(step.prefill_table.copy()))
    pout, dout = pkv.paged_mixed_step(kc, vc, step.scale, prefill=prefill, decode=decode)
    torch.cuda.synchronize()
    _, okc, ovc = oracle_write(step)
    assert np.array_equal(to_host(kc), okc) and np.array_equal(to_host(vc), ovc)
    want_d = oracle.decode(step.q_decode, okc, ovc, step.decode_table, step.cache_seqlens,
                           step.scale)
    assert_close(widen(dout), want_d, "bf16", "d64 mixed decode")
    want_p = oracle.prefill(step.q_prefill, okc, ovc, step.cu_q, step.cu_k, step.scale,
                            causal=True, block_table=step.prefill_table,
                            block_size=step.block_size)
    assert_close(widen(pout), want_p, "bf16", "d64 mixed prefill")
    assert pkv.paged_error_flags() == 0


@pytest.mark.parametrize("grouped,one_launch", [(True, False), (False, False), (True, True),
                                                (False, True)])
def test_continuous_batching_step(grouped, one_launch):
    """The whole step against the oracle, chained and in one launch (without
    groups the one-launch entry hands the step to the chained form)."""
    step = W.config(5)
    dec_rows, pf_rows, slots = split_step(step)
    kc, vc = to_dev(step.k_cache), to_dev(step.v_cache)
    nd = step.n_decode
    decode = dict(q=to_dev(step.q_decode), k_new=to_dev(step.new_k[dec_rows]),
                  v_new=to_dev(step.new_v[dec_rows]), table=to_dev(step.decode_table.copy()),
                  seqlens=to_dev(step.cache_seqlens - 1))
    if grouped:
        decode.update(group_cu=to_dev(np.arange(0, nd + 1, nd // 8, dtype=np.int32)),
                      group_prefix_len=to_dev(np.full(8, 2048, np.int32)), max_group_size=nd // 8)
    prefill = dict(k_new=to_dev(step.new_k[pf_rows]), v_new=to_dev(step.new_v[pf_rows]),
                   slots=to_dev(slots[pf_rows]), q=to_dev(step.q_prefill), cu_q=to_dev(step.cu_q),
                   cu_k=to_dev(step.cu_k), max_q=step.max_seqlen_q, max_k=step.max_seqlen_k,
                   table=to_dev(step.prefill_table.copy()))
    pout, dout = pkv.paged_mixed_step(kc, vc, step.scale, prefill=prefill, decode=decode,
                                      one_launch=one_launch)
    torch.cuda.synchronize()
    _, okc, ovc = oracle_write(step)
    assert np.array_equal(to_host(kc), okc) and np.array_equal(to_host(vc), ovc)
    want_d = oracle.decode(step.q_decode, okc, ovc, step.decode_table, step.cache_seqlens,
                           step.scale)
    assert_close(widen(dout), want_d, "bf16", "mixed step decode")
    want_p = oracle.prefill(step.q_prefill, okc, ovc, step.cu_q, step.cu_k, step.scale,
                            causal=True, block_table=step.prefill_table,
                            block_size=step.block_size)
    assert_close(widen(pout), want_p, "bf16", "mixed step prefill")
    assert pkv.paged_error_flags() == 0


def test_parts_alone():
    """Decode only and prefill only."""
    step = W.config(5)
    dec_rows, pf_rows, slots = split_step(step)
    kc, vc = to_dev(step.k_cache), to_dev(step.v_cache)
    _, dout = pkv.paged_mixed_step(kc, vc, step.scale, decode=dict(
        q=to_dev(step.q_decode), k_new=to_dev(step.new_k[dec_rows]),
        v_new=to_dev(step.new_v[dec_rows]), table=to_dev(step.decode_table.copy()),
        seqlens=to_dev(step.cache_seqlens - 1)))
    pout, _ = pkv.paged_mixed_step(kc, vc, step.scale, prefill=dict(
        k_new=to_dev(step.new_k[pf_rows]), v_new=to_dev(step.new_v[pf_rows]),
        slots=to_dev(slots[pf_rows]), q=to_dev(step.q_prefill), cu_q=to_dev(step.cu_q),
        cu_k=to_dev(step.cu_k), max_q=step.max_seqlen_q, max_k=step.max_seqlen_k,
        table=to_dev(step.prefill_table.copy())))
    torch.cuda.synchronize()
    _, okc, ovc = oracle_write(step)
    assert np.array_equal(to_host(kc), okc)
    want_d = oracle.decode(step.q_decode, okc, ovc, step.decode_table, step.cache_seqlens,
                           step.scale)
    assert_close(widen(dout), want_d, "bf16", "decode part")
    want_p = oracle.prefill(step.q_prefill, okc, ovc, step.cu_q, step.cu_k, step.scale,
                            causal=True, block_table=step.prefill_table,
                            block_size=step.block_size)
    assert_close(widen(pout), want_p, "bf16", "prefill part")


def test_one_launch_equals_chained():
    """The one-launch step runs the same CTA functions on the same partition of
    the work as the chained launches: its outputs and caches are bit-identical."""
    step = W.config(5)
    dec_rows, pf_rows, slots = split_step(step)
    nd = step.n_decode
    outs = []
    for one in (False, True):
        kc, vc = to_dev(step.k_cache), to_dev(step.v_cache)
        decode = dict(q=to_dev(step.q_decode), k_new=to_dev(step.new_k[dec_rows]),
                      v_new=to_dev(step.new_v[dec_rows]), table=to_dev(step.decode_table.copy()),
                      seqlens=to_dev(step.cache_seqlens - 1),
                      group_cu=to_dev(np.arange(0, nd + 1, nd // 8, dtype=np.int32)),
                      group_prefix_len=to_dev(np.full(8, 2048, np.int32)), max_group_size=nd // 8)
        prefill = dict(k_new=to_dev(step.new_k[pf_rows]), v_new=to_dev(step.new_v[pf_rows]),
                       slots=to_dev(slots[pf_rows]), q=to_dev(step.q_prefill),
                       cu_q=to_dev(step.cu_q), cu_k=to_dev(step.cu_k), max_q=step.max_seqlen_q,
                       max_k=step.max_seqlen_k, table=to_dev(step.prefill_table.copy()))
        pout, dout = pkv.paged_mixed_step(kc, vc, step.scale, prefill=prefill, decode=decode,
                                          one_launch=one)
        torch.cuda.synchronize()
        outs.append([to_host(t) for t in (pout, dout, kc, vc)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    assert pkv.paged_error_flags() == 0
