"""GPU block copy against the oracle's copy: bit-exact, between device pools,
to and from pinned host memory, with E4M3 scales and INT8 (scale, zero)
pairs; plus copy-on-write of a
shared prefix block followed by an append and a decode."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import normal_bf16_bits, random_case
from tests._gpu import DEV, DeviceCase, assert_close, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _pools(seed, nb, shape, dtype):
    rng = np.random.Generator(np.random.PCG64(seed))
    if dtype == "bf16":
        return (rng.integers(0, 1 << 16, size=(nb,) + shape, dtype=np.uint16),
                rng.integers(0, 1 << 16, size=(nb,) + shape, dtype=np.uint16))
    dt = np.uint8 if dtype == "fp8" else np.int8
    lo, hi = (0, 256) if dtype == "fp8" else (-128, 128)
    return (rng.integers(lo, hi, size=(nb,) + shape, dtype=dt),
            rng.integers(lo, hi, size=(nb,) + shape, dtype=dt))


def _tensor(a, where):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    if where == "device":
        return t.to(DEV)
    return t.clone().pin_memory()


def _host(t):
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@pytest.mark.parametrize("dtype,shape", [("bf16", (8, 16, 128)), ("bf16", (2, 32, 64)), ("fp8", (8, 32, 128)),
                                         ("int8", (4, 16, 128))])
@pytest.mark.parametrize("src_where,dst_where", [("device", "device"), ("device", "host"), ("host", "device")])
def test_copy_bit_exact(dtype, shape, src_where, dst_where):
    src_nb, dst_nb, n = 40, 25, 17
    sk, sv = _pools(1, src_nb, shape, dtype)
    dk, dv = _pools(2, dst_nb, shape, dtype)
    rng = np.random.Generator(np.random.PCG64(3))
    pairs = np.stack([rng.choice(src_nb, n, replace=False), rng.choice(dst_nb, n, replace=False)],
                     axis=1).astype(np.int32)
    scales = {}
    if dtype != "bf16":
        per_page = (shape[0],) if dtype == "fp8" else (shape[0], 2)
        for name, nb in (("sks", src_nb), ("svs", src_nb), ("dks", dst_nb), ("dvs", dst_nb)):
            scales[name] = rng.uniform(0.01, 1.0, size=(nb,) + per_page).astype(np.float32)
    t_sk, t_sv = _tensor(sk, src_where), _tensor(sv, src_where)
    t_dk, t_dv = _tensor(dk, dst_where), _tensor(dv, dst_where)
    ts = {k: (v := _tensor(a, "device" if k[0] == "s" and src_where == "device" or
                           k[0] == "d" and dst_where == "device" else "host")) for k, a in scales.items()}
    pkv.copy_blocks(t_sk, t_sv, t_dk, t_dv, to_dev(pairs), ts.get("sks"), ts.get("svs"),
                    ts.get("dks"), ts.get("dvs"))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    args = [scales.get("sks"), scales.get("svs"), scales.get("dks"), scales.get("dvs")]
    assert oracle.copy_blocks(sk, sv, dk, dv, pairs, *args) == 0
    assert np.array_equal(_host(t_dk), dk) and np.array_equal(_host(t_dv), dv)
    if dtype != "bf16":
        assert np.array_equal(_host(ts["dks"]), scales["dks"])
        assert np.array_equal(_host(ts["dvs"]), scales["dvs"])


def test_swap_out_and_back_in():
    # a sequence's blocks go to a host pool and come back into other blocks
    shape = (8, 16, 128)
    sk, sv = _pools(4, 64, shape, "bf16")
    k, v = _tensor(sk, "device"), _tensor(sv, "device")
    hk = torch.zeros((10,) + shape, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    seq = np.array([5, 61, 17, 33, 2, 40], np.int32)
    out_pairs = np.stack([seq, np.arange(len(seq))], axis=1).astype(np.int32)
    pkv.copy_blocks(k, v, hk, hv, to_dev(out_pairs))
    new_home = np.array([8, 9, 10, 11, 12, 13], np.int32)
    in_pairs = np.stack([np.arange(len(seq)), new_home], axis=1).astype(np.int32)
    pkv.copy_blocks(hk, hv, k, v, to_dev(in_pairs))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    got_k, got_v = _host(k), _host(v)
    assert np.array_equal(got_k[new_home], sk[seq]) and np.array_equal(got_v[new_home], sv[seq])


def test_out_of_range_pairs_flagged_and_skipped():
    shape = (2, 16, 64)
    sk, sv = _pools(5, 8, shape, "bf16")
    dk, dv = _pools(6, 8, shape, "bf16")
    pairs = np.array([[1, 2], [8, 3], [4, -1], [6, 7]], np.int32)
    t_dk, t_dv = _tensor(dk, "device"), _tensor(dv, "device")
    pkv.copy_blocks(_tensor(sk, "device"), _tensor(sv, "device"), t_dk, t_dv, to_dev(pairs))
    assert pkv.read_device_error() & pkv.DEVERR_BLOCK_ID
    assert oracle.copy_blocks(sk, sv, dk, dv, pairs[[0, 3]]) == 0
    assert np.array_equal(_host(t_dk), dk) and np.array_equal(_host(t_dv), dv)


def test_validate_mode_rejects_repeated_destination(monkeypatch):
    shape = (2, 16, 64)
    sk, sv = _pools(7, 8, shape, "bf16")
    t = [_tensor(a, "device") for a in (sk, sv, sk, sv)]
    monkeypatch.setenv("PKV_VALIDATE", "1")
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks(*t, to_dev(np.array([[1, 2], [3, 2]], np.int32)))


def test_copy_on_write_then_append_and_decode():
    # sequences 0 and 1 share their first block; before sequence 1 writes
    # into it, the block is copied to a spare block and its table updated
    c = random_case(41, 2, 16, 4, 128, 16, [10, 12], spare_blocks=4)
    c.block_tables[1, 0] = c.block_tables[0, 0]   # aliased prefix block
    c.context_lens = np.array([10, 11], np.int32)  # sequence 1 is about to write token 11
    spare = int(next(i for i in range(c.NB) if i not in set(c.block_tables[:, 0].tolist())))
    dc = DeviceCase(c)
    shared = int(c.block_tables[0, 0])
    pkv.copy_blocks(dc.k[0], dc.v[0], dc.k[0], dc.v[0], to_dev(np.array([[shared, spare]], np.int32)))
    c.block_tables[1, 0] = spare
    c.context_lens = np.array([10, 12], np.int32)
    dc.bt = to_dev(c.block_tables)
    dc.cl = to_dev(c.context_lens)
    kn = normal_bf16_bits(42, (1, c.Hkv, c.D))
    vn = normal_bf16_bits(43, (1, c.Hkv, c.D))
    slot = np.array([spare * c.bs + 11], np.int64)
    pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slot), dc.k, dc.v)
    got = bf16_dev_to_f64(dc.decode())
    # the oracle applies the same three steps to its own copy of the cache
    ko, vo = dc.k_host.copy(), dc.v_host.copy()
    assert oracle.copy_blocks(ko[0], vo[0], ko[0], vo[0], np.array([[shared, spare]], np.int32)) == 0
    assert oracle.kv_append(kn, vn, slot, ko, vo) == 0
    want = oracle.paged_decode(c.q[0], ko, vo, c.block_tables, c.context_lens, c.kv_group_ptr, 0, c.scale)
    assert_close(got, want, "copy-on-write")
    # the shared block itself is unchanged for sequence 0
    assert np.array_equal(_host(dc.k[0, shared]), dc.k_host[0, shared])
