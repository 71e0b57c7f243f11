"""GPU kv_append: bit-exact against the oracle's scatter (bf16) and against the
oracle's E4M3 encoder (FP8), with every byte outside the written slots
unchanged."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import bf16_bits_to_f32, normal_bf16_bits
from tests._gpu import DEV, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _caches(shape, dtype, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    if dtype == "bf16":
        k = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
        v = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    elif dtype == "int8":
        k = rng.integers(-128, 128, size=shape, dtype=np.int8)
        v = rng.integers(-128, 128, size=shape, dtype=np.int8)
    else:
        k = rng.integers(0, 256, size=shape, dtype=np.uint8)
        v = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return k, v


def _dev_cache(a):
    return to_dev_bf16(a) if a.dtype == np.uint16 else to_dev(a)


@pytest.mark.parametrize("scale,zero", [(1.0, 0.0), (0.031, 0.0), (0.02, -17.0), (1e-3, 5.0), (250.0, 127.0)])
def test_int8_quantisation_every_bf16_pattern(scale, zero):
    # all 65536 bf16 bit patterns (NaN included) through the INT8 append,
    # against the oracle's encoder
    Hkv, D, bs = 1, 128, 32
    N = (1 << 16) // D
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(N, Hkv, D)
    NB = N // bs
    shape = (1, NB, Hkv, bs, D)
    kd = torch.zeros(shape, dtype=torch.int8, device=DEV)
    vd = torch.zeros(shape, dtype=torch.int8, device=DEV)
    prm = np.zeros((1, NB, Hkv, 2), dtype=np.float32)
    prm[..., 0] = scale
    prm[..., 1] = zero
    slots = np.arange(N, dtype=np.int64)
    pkv.kv_append(to_dev_bf16(bits), to_dev_bf16(bits), to_dev(slots), kd, vd, to_dev(prm), to_dev(prm))
    torch.cuda.synchronize()
    ko = np.zeros(shape, np.int8)
    vo = np.zeros(shape, np.int8)
    assert oracle.kv_append(bits, bits, slots, ko, vo, prm, prm) == 0
    assert np.array_equal(kd.cpu().numpy(), ko)
    assert np.array_equal(vd.cpu().numpy(), vo)


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("D,bs", [(64, 16), (128, 16), (128, 32)])
@pytest.mark.parametrize("slot", [0, 1])
def test_append_bit_exact(dtype, D, bs, slot):
    if dtype != "bf16" and D != 128:
        pytest.skip("one-byte caches need head_dim 128")
    S, NB, Hkv, N = 2, 37, 4, 64
    shape = (S, NB, Hkv, bs, D)
    k, v = _caches(shape, dtype, 1 + D + bs)       # random canary bytes everywhere
    rng = np.random.Generator(np.random.PCG64(7 + D))
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    slots[5] = -1
    slots[17] = -1
    kn = normal_bf16_bits(100 + D, (N, Hkv, D))
    vn = normal_bf16_bits(200 + D, (N, Hkv, D))
    ks = vs = None
    if dtype == "fp8":
        ks = rng.uniform(0.002, 0.03, size=(S, NB, Hkv)).astype(np.float32)
        vs = rng.uniform(0.002, 0.03, size=(S, NB, Hkv)).astype(np.float32)
    elif dtype == "int8":
        # half the pages symmetric (zero 0), half with a zero point
        z = np.where(rng.random((S, NB, Hkv)) < 0.5, 0, rng.integers(-30, 31, size=(S, NB, Hkv)))
        ks = np.stack([rng.uniform(0.01, 0.05, size=(S, NB, Hkv)), z], axis=-1).astype(np.float32)
        vs = np.stack([rng.uniform(0.01, 0.05, size=(S, NB, Hkv)), z[..., ::-1]], axis=-1).astype(np.float32)
    kd, vd = _dev_cache(k), _dev_cache(v)
    pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), kd, vd,
                  None if ks is None else to_dev(ks), None if vs is None else to_dev(vs), slot=slot)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert oracle.kv_append(kn, vn, slots, k, v, ks, vs, slot=slot) == 0
    assert np.array_equal(_host(kd), k)
    assert np.array_equal(_host(vd), v)


@pytest.mark.parametrize("scale", [1.0, 1 / 448, 0.0091, 3.7, 1e-3, 250.0])
def test_e4m3_quantisation_every_bf16_pattern(scale):
    # all 65536 bf16 bit patterns (NaN included) through the FP8 append,
    # against the oracle's encoder; NaN inputs only need to stay NaN
    Hkv, D, bs = 1, 128, 32
    N = (1 << 16) // D
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(N, Hkv, D)
    NB = N // bs
    shape = (1, NB, Hkv, bs, D)
    kd = torch.zeros(shape, dtype=torch.uint8, device=DEV)
    vd = torch.zeros(shape, dtype=torch.uint8, device=DEV)
    sc = np.full((1, NB, Hkv), scale, dtype=np.float32)
    slots = np.arange(N, dtype=np.int64)
    pkv.kv_append(to_dev_bf16(bits), to_dev_bf16(bits), to_dev(slots), kd, vd, to_dev(sc), to_dev(sc))
    torch.cuda.synchronize()
    got = kd.cpu().numpy().reshape(N, D)
    want = oracle.e4m3_quantize(bits.reshape(N, D), np.float32(scale))
    x = bf16_bits_to_f32(bits.reshape(N, D))
    nan_in = np.isnan(x)
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert np.all((got[nan_in] & 0x7F) == 0x7F)
    assert np.array_equal(vd.cpu().numpy(), kd.cpu().numpy())


def test_append_out_of_range_slot_flagged_and_skipped():
    S, NB, Hkv, bs, D = 1, 4, 2, 16, 64
    k, v = _caches((S, NB, Hkv, bs, D), "bf16", 3)
    kd, vd = _dev_cache(k), _dev_cache(v)
    slots = np.array([3, NB * bs, -7, 10], dtype=np.int64)
    kn = normal_bf16_bits(1, (4, Hkv, D))
    pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(kn), to_dev(slots), kd, vd)
    assert pkv.read_device_error() & pkv.DEVERR_SLOT
    ok = slots.copy()
    ok[1:3] = -1
    assert oracle.kv_append(kn, kn, ok, k, v) == 0
    assert np.array_equal(_host(kd), k)


def test_append_validate_mode_rejects_duplicates(monkeypatch):
    S, NB, Hkv, bs, D = 1, 4, 2, 16, 64
    kd = torch.zeros((S, NB, Hkv, bs, D), dtype=torch.bfloat16, device=DEV)
    vd = torch.zeros_like(kd)
    kn = to_dev_bf16(normal_bf16_bits(2, (3, Hkv, D)))
    monkeypatch.setenv("PKV_VALIDATE", "1")
    with pytest.raises(pkv.PkvError):
        pkv.kv_append(kn, kn, to_dev(np.array([5, 9, 5], np.int64)), kd, vd)


def test_append_then_decode_reads_new_token():
    # a decode step: append token n-1 of each sequence, then attend over n tokens
    from workloads import random_case
    from tests._gpu import DeviceCase, assert_close, bf16_dev_to_f64
    c = random_case(31, 3, 16, 4, 128, 16, [33, 64, 100])
    dc = DeviceCase(c)
    N = c.B
    pos = c.context_lens - 1
    slots = np.array([c.block_tables[b, pos[b] // c.bs] * c.bs + pos[b] % c.bs for b in range(N)],
                     dtype=np.int64)
    kn = normal_bf16_bits(32, (N, c.Hkv, c.D))
    vn = normal_bf16_bits(33, (N, c.Hkv, c.D))
    pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), dc.k, dc.v)
    got = bf16_dev_to_f64(dc.decode())
    assert oracle.kv_append(kn, vn, slots, dc.k_host, dc.v_host) == 0
    assert_close(got, dc.oracle(), "append + decode")
