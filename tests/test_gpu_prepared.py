"""Prepared calls: a decode, multi-token decode or append-and-decode whose
arguments were checked and marshalled once, then called step after step with
new contents in its bound buffers, gives the same output bits and cache bytes
as the plain calls on an identical cache."""
import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv
from workloads import normal_bf16_bits, random_case
from tests._gpu import DeviceCase, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("T,append", [(1, False), (1, True), (40, False), (40, True)])
def test_prepared_matches_plain_calls(T, append):
    c = random_case(1501 + T + append, 5, 32, 8, 128, 16, [T + 30, 700, 1500, 77, T + 3])
    dp, de = DeviceCase(c), DeviceCase(c)
    pos = c.context_lens.astype(np.int64)[:, None] - T + np.arange(T)[None, :]
    blk = c.block_tables[np.arange(c.B)[:, None], pos // c.bs].astype(np.int64)
    slots = to_dev((blk * c.bs + pos % c.bs).reshape(-1))
    gp = c.kv_group_ptr.tolist()
    qshape = (c.B, c.Hq, c.D) if T == 1 else (c.B, T, c.Hq, c.D)

    def inputs(seed):
        return (to_dev_bf16(normal_bf16_bits(seed, (c.B * T, c.Hkv, c.D))),
                to_dev_bf16(normal_bf16_bits(seed + 1, (c.B * T, c.Hkv, c.D))),
                to_dev_bf16(normal_bf16_bits(seed + 2, qshape)))

    kn, vn, q = inputs(1600)
    call = pkv.PreparedDecode(q, dp.k, dp.v, dp.bt, dp.cl, gp, 0, c.scale,
                              k_new=kn if append else None, v_new=vn if append else None,
                              slot_mapping=slots if append else None)
    assert call.out.shape == q.shape
    for i in range(3):
        k2, v2, q2 = inputs(1700 + 10 * i)
        kn.copy_(k2)
        vn.copy_(v2)
        q.copy_(q2)
        got = call()
        if append:
            ref = pkv.append_and_decode(k2, v2, slots, q2, de.k, de.v, de.bt, de.cl, gp, 0, c.scale)
        elif T == 1:
            ref = pkv.paged_decode(q2, de.k, de.v, de.bt, de.cl, gp, 0, c.scale)
        else:
            ref = pkv.paged_decode_multi(q2, de.k, de.v, de.bt, de.cl, gp, 0, c.scale)
        torch.cuda.synchronize()
        assert got is call.out
        assert np.array_equal(_bits(got), _bits(ref)), f"step {i}: output differs from the plain call"
        assert np.array_equal(_bits(dp.k), _bits(de.k)) and np.array_equal(_bits(dp.v), _bits(de.v))
    assert pkv.read_device_error() == 0


def test_prepared_on_a_bound_stream():
    c = random_case(1801, 3, 32, 8, 128, 16, [100, 2000, 33])
    dc = DeviceCase(c)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    call = pkv.PreparedDecode(dc.q[0], dc.k, dc.v, dc.bt, dc.cl, stream=s)
    call()
    s.synchronize()
    ref = pkv.paged_decode(dc.q[0], dc.k, dc.v, dc.bt, dc.cl)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(call.out), _bits(ref))
