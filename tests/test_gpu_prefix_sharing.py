"""The prefix cache driving block sharing on the GPU: requests with a
common system prompt reuse the cached physical blocks (their block tables
alias them), append only the tokens after the cached prefix, and decode;
the result must equal attention over each request's dense, private K/V.

"KV-Cache Engineering: Paged Attention, Prefix Cache, Disaggregation
(2026)", prefix caching answer: matching blocks are reused through the block
table and only the first non-matching block triggers prefill.  The K/V of a
token here is a seeded function of (token id, position), standing in for a
model whose cache for a given prefix is deterministic."""
import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv
from workloads import bf16_bits_to_f32, normal_bf16_bits
from tests._gpu import DEV, assert_close, bf16_dev_to_f64, to_dev, to_dev_bf16
from tests._paged import sdpa_reference

pytestmark = pytest.mark.gpu


def _kv_rows(tokens, start, Hkv, D, role):
    rows = [normal_bf16_bits(1_000_003 * role + 7919 * int(t) + p, (1, Hkv, D))
            for p, t in enumerate(tokens, start=start)]
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, Hkv, D), np.uint16)


def test_prefix_cache_shared_blocks_decode():
    bs, Hkv, Hq, D, NB = 16, 8, 32, 128, 64
    rng = np.random.Generator(np.random.PCG64(3))
    system = rng.integers(0, 32000, size=5 * bs + 3).tolist()      # 5 full blocks + 3 tokens
    requests = [system + rng.integers(0, 32000, size=n).tolist() for n in (9, 30, 1, 45)]
    requests.append(rng.integers(0, 32000, size=40).tolist())         # no shared prefix
    k = torch.zeros((1, NB, Hkv, bs, D), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros_like(k)
    cache = pkv.PrefixCache(bs)
    free = list(range(NB - 1, -1, -1))
    MB = max(-(-len(r) // bs) for r in requests)
    tables = np.full((len(requests), MB), -1, np.int32)
    computed = 0
    for i, toks in enumerate(requests):
        reused = cache.match(toks)
        blocks = reused + [free.pop() for _ in range(-(-len(toks) // bs) - len(reused))]
        tables[i, :len(blocks)] = blocks
        start = len(reused) * bs                    # prefill starts at the first miss
        slots = np.array([blocks[p // bs] * bs + p % bs for p in range(start, len(toks))], np.int64)
        kn = _kv_rows(toks[start:], start, Hkv, D, 1)
        vn = _kv_rows(toks[start:], start, Hkv, D, 2)
        pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), k, v)
        computed += len(toks) - start
        cache.insert(toks, blocks)
    # the four sharers reused the 5 system-prompt blocks
    assert computed == sum(len(r) for r in requests) - 3 * 5 * bs
    entries, lookups, hits = cache.stats()
    assert hits == 3 * 5
    q = normal_bf16_bits(11, (len(requests), Hq, D))
    ctx = np.array([len(r) for r in requests], np.int32)
    out = pkv.paged_decode(to_dev_bf16(q), k, v, to_dev(tables), to_dev(ctx))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    kd = [bf16_bits_to_f32(_kv_rows(r, 0, Hkv, D, 1)).astype(np.float64) for r in requests]
    vd = [bf16_bits_to_f32(_kv_rows(r, 0, Hkv, D, 2)).astype(np.float64) for r in requests]
    want = sdpa_reference(q, kd, vd, D ** -0.5)
    assert_close(bf16_dev_to_f64(out), want, "prefix-cache sharing")
