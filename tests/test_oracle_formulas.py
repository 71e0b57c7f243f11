"""Pins of the oracle's byte accounting against the numbers printed on the pages.

Fixture: tests/golden/kv_cache_arithmetic.json (each case carries its page
and section).
"""
import json
import math
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_arithmetic.json")
CASES = json.load(open(GOLDEN))["cases"]


def _value(case):
    q, a = case["quantity"], case["inputs"]
    if q == "kv_bytes_per_token":
        return oracle.kv_bytes_per_token(**a)
    if q == "kv_bytes":
        return oracle.kv_bytes(**a)
    if q == "decode_kv_read_seconds":
        return oracle.decode_kv_read_seconds(**a)
    if q == "decode_kv_read_seconds_100k":
        b = oracle.kv_bytes(a["n_layers"], a["n_kv_heads"], a["head_dim"], a["dtype_bytes"],
                            a["seq_len"], 1)
        return oracle.decode_kv_read_seconds(b, a["hbm_bytes_per_s"])
    if q == "tokens_that_fit":
        return oracle.tokens_that_fit(**a)
    if q == "requests_at_2048":
        return [math.floor(t / a["avg_context"]) for t in a["tokens"]]
    if q == "naive_utilisation":
        return oracle.naive_utilisation(**a)
    if q == "max_last_block_waste":
        bs = a["block_size"]
        return max(oracle.last_block_waste_tokens(n, bs) for n in range(1, 10 * bs))
    if q == "grouped_reduction":
        full = oracle.kv_bytes_per_token(a["n_layers"], a["mha_heads"], 128, 2)
        grouped = oracle.kv_bytes_per_token_grouped(a["n_layers"], a["layers_per_group"],
                                                    a["mha_heads"], 128, 2)
        grouped_gqa = oracle.kv_bytes_per_token_grouped(a["n_layers"], a["layers_per_group"],
                                                        a["gqa_kv_heads"], 128, 2)
        return {"layer_factor": full / grouped, "total_factor": full / grouped_gqa}
    raise KeyError(q)


@pytest.mark.parametrize("case", CASES, ids=[c["id"] for c in CASES])
def test_printed_value(case):
    got = _value(case)
    want = case["value"]
    if case.get("comparison") == "greater":
        assert got > want
    elif isinstance(want, dict):
        assert got == pytest.approx(want, rel=case["rel_tol"], abs=0)
    elif isinstance(want, list):
        assert got == want
    else:
        assert got == pytest.approx(want, rel=case["rel_tol"], abs=0)


def test_blocks_and_waste_bounds():
    # only the last block is partly filled: ceil(n / bs) blocks, waste < bs
    for bs in (16, 32):
        for n in range(0, 200):
            nb = oracle.blocks_for_tokens(n, bs)
            assert (nb - 1) * bs < n <= nb * bs or (n == 0 and nb == 0)
            assert 0 <= oracle.last_block_waste_tokens(n, bs) < bs


def test_workload_step_bytes():
    # per-layer KV bytes read by one decode step of the benchmark workloads
    assert oracle.kv_bytes(1, 8, 128, 2, 4096, 64) == 1 << 30            # Llama-3.1-8B layer
    assert oracle.kv_bytes(1, 8, 128, 2, 32768, 4) == 1 << 29            # 70B-shaped, batch 4
    assert oracle.kv_bytes(1, 8, 128, 2, 131072, 1) == 1 << 29           # 70B-shaped, batch 1
    assert oracle.kv_bytes(1, 8, 128, 1, 8192, 128) == 1 << 31           # FP8, one layer call
