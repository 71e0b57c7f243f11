"""The fused step (append on the planner's extra CTAs, then decode) against
the two separate calls: the same cache bytes and the same output bits, for
bf16, E4M3 and INT8 caches, single- and multi-token queries, and a batch of
no sequences; and against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import normal_bf16_bits, random_case
from tests._gpu import DeviceCase, assert_close, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _new_tokens(c, T, seed):
    # the last T positions of every sequence get new K/V
    pos = c.context_lens.astype(np.int64)[:, None] - T + np.arange(T)[None, :]
    blk = c.block_tables[np.arange(c.B)[:, None], pos // c.bs].astype(np.int64)
    slots = (blk * c.bs + pos % c.bs).reshape(-1)
    kn = normal_bf16_bits(seed, (len(slots), c.Hkv, c.D))
    vn = normal_bf16_bits(seed + 1, (len(slots), c.Hkv, c.D))
    return kn, vn, slots


def _bytes(t):
    return t.view(torch.uint8).cpu().numpy() if t.dtype != torch.bfloat16 else \
        t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int8a"])
@pytest.mark.parametrize("T", [1, 4])
def test_fused_equals_separate(dtype, T):
    lens = [T + 5, 200, 517, 64]
    c = random_case(140 + T, len(lens), 32, 8, 128, 16, lens, kv_dtype=dtype)
    kn, vn, slots = _new_tokens(c, T, 141)
    q = normal_bf16_bits(142, (c.B, T, 32, 128) if T > 1 else (c.B, 32, 128))
    a, b = DeviceCase(c), DeviceCase(c)
    fused = pkv.append_and_decode(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), to_dev_bf16(q), a.k, a.v,
                                  a.bt, a.cl, [0], 0, c.scale, k_scale=a.ks, v_scale=a.vs)
    pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), b.k, b.v, b.ks, b.vs)
    if T > 1:
        sep = pkv.paged_decode_multi(to_dev_bf16(q), b.k, b.v, b.bt, b.cl, [0], 0, c.scale, k_scale=b.ks,
                                     v_scale=b.vs)
    else:
        sep = pkv.paged_decode(to_dev_bf16(q), b.k, b.v, b.bt, b.cl, [0], 0, c.scale, k_scale=b.ks, v_scale=b.vs)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert np.array_equal(_bytes(a.k), _bytes(b.k)) and np.array_equal(_bytes(a.v), _bytes(b.v))
    assert torch.equal(fused, sep)
    # and the oracle, on its own append of the same tokens
    ko, vo = a.k_host.copy(), a.v_host.copy()
    assert oracle.kv_append(kn, vn, slots, ko, vo, c.k_scale, c.v_scale) == 0
    qm = q if T > 1 else q[:, None]
    want = oracle.paged_decode_multi(qm, ko, vo, c.block_tables, c.context_lens, c.kv_group_ptr, 0, c.scale,
                                     k_scale=c.k_scale, v_scale=c.v_scale)
    got = bf16_dev_to_f64(fused if T > 1 else fused[:, None])
    assert_close(got, want, f"fused {dtype} T={T}")


def test_fused_with_empty_batch_only_appends():
    c = random_case(150, 2, 8, 2, 64, 16, [20, 33])
    kn, vn, slots = _new_tokens(c, 1, 151)
    dc = DeviceCase(c)
    q = torch.empty((0, 8, 64), dtype=torch.bfloat16, device=dc.k.device)
    bt = dc.bt[:0]
    cl = dc.cl[:0]
    pkv.append_and_decode(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), q, dc.k, dc.v, bt, cl)
    torch.cuda.synchronize()
    ko, vo = dc.k_host.copy(), dc.v_host.copy()
    assert oracle.kv_append(kn, vn, slots, ko, vo) == 0
    assert np.array_equal(_bytes(dc.k), ko) and np.array_equal(_bytes(dc.v), vo)
