"""The CPU oracle against the pages' worked examples, closed forms, library
routines and invariants (no GPU)."""
import pytest

import oracle
from oracle_pins import ALL_PINS, golden


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_pool_sizing():
    """§11.1 example (B=16, T=100, L=28, kvDim=1024, fp32) and the Qwen3-0.6B
    per-token figure of "KVCache大小计算"."""
    g = golden("pool_sizing.json")
    e = g["p1_example"]
    assert oracle.blocks_per_layer(e["T"], e["B"]) == e["blocks_per_layer"]
    assert oracle.pool_blocks(e["T"], e["B"], e["L"]) == e["total_blocks"]
    assert oracle.pool_bytes(1, e["B"], e["kvDim"], e["elt_bytes"]) == e["bytes_per_block"]
    total = oracle.pool_bytes(e["total_blocks"], e["B"], e["kvDim"], e["elt_bytes"])
    assert total / 2**20 == e["total_mib_printed"]
    assert oracle.tokens_in_last_block(e["T"], e["B"]) == e["last_block_slots_used"]
    qn = g["qwen3_0p6b"]
    per_tok = oracle.kv_bytes_per_token(qn["layers"], qn["kv_heads"] * qn["head_dim"],
                                        qn["elt_bytes"])
    assert per_tok == qn["kib_per_token"] * 1024
    assert per_tok * qn["tokens"] == qn["mib_total"] * 2**20


def test_threads_reported(lib):
    assert oracle.num_threads(lib) >= 1
