"""GPU parity of paged_decode against the CPU oracle on small seeded cases
that still span several pages, partitions and a ragged tail.

Tolerance (bf16 output, fp32 accumulation): |gpu - oracle| <= 1e-2 + 1e-2 |oracle|.
"""
import itertools

import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv
from workloads import random_case, tiny_case, normal_bf16_bits, bf16_bits_from_f32
from tests._gpu import (DeviceCase, assert_close, bf16_dev_to_bits, bf16_dev_to_f64, to_dev,
                        to_dev_bf16)

pytestmark = pytest.mark.gpu

MATHS = {"mma": pkv.MATH_MMA, "ffma": pkv.MATH_FFMA}


def _run(case, math="mma", ppu=0, warps=0, stages=0, layer=0):
    dc = DeviceCase(case)
    out = dc.decode(layer=layer, opts=pkv.decode_opts(ppu, MATHS[math], warps, stages))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    return bf16_dev_to_f64(out), dc.oracle(layer=layer), dc, out


@pytest.mark.parametrize("math", ["mma", "ffma"])
def test_tiny_workload(math):
    got, want, _, _ = _run(tiny_case(), math)
    assert_close(got, want, f"tiny/{math}")


SWEEP = [  # (D, bs, Hq, Hkv, dtype)
    (64, 16, 8, 2, "bf16"), (64, 32, 4, 4, "bf16"), (128, 16, 32, 8, "bf16"),
    (128, 32, 64, 8, "bf16"), (128, 16, 8, 1, "bf16"), (128, 32, 16, 2, "bf16"),
    (128, 32, 32, 8, "fp8"), (128, 16, 8, 2, "fp8"), (128, 32, 8, 8, "fp8"),
    (128, 32, 32, 8, "int8"), (128, 16, 8, 2, "int8a"), (128, 32, 16, 1, "int8a"),
]
LENS = [1, 15, 16, 17, 100, 257, 0, 513, 1031]


@pytest.mark.parametrize("D,bs,Hq,Hkv,dtype", SWEEP)
@pytest.mark.parametrize("math", ["mma", "ffma"])
@pytest.mark.parametrize("ppu", [0, 2, 64])
def test_random_sweep(D, bs, Hq, Hkv, dtype, math, ppu):
    G = Hq // Hkv
    if math == "ffma" and G not in (1, 2, 4, 8):
        pytest.skip("ffma supports G in {1, 2, 4, 8}")
    seed = D * 1000 + bs * 10 + Hq + 7 * Hkv + {"bf16": 0, "fp8": 50000, "int8": 60000, "int8a": 70000}[dtype]
    c = random_case(seed, len(LENS), Hq, Hkv, D, bs, LENS, kv_dtype=dtype, poison=True)
    got, want, _, _ = _run(c, math, ppu)
    assert_close(got, want, f"D{D} bs{bs} G{G} {dtype} {math} ppu{ppu}")


@pytest.mark.parametrize("math", ["mma", "ffma"])
def test_large_logits(math):
    c = random_case(77, 3, 16, 2, 128, 16, [300, 45, 1000], value_scale=6.0)
    got, want, _, _ = _run(c, math, ppu=4)
    assert_close(got, want, "large logits")


@pytest.mark.parametrize("math", ["mma", "ffma"])
@pytest.mark.parametrize("G", [1, 8, 16])
def test_head_groupings(math, G):
    if math == "ffma" and G == 16:
        pytest.skip("ffma supports G <= 8")
    Hkv = 2
    c = random_case(90 + G, 4, G * Hkv, Hkv, 128, 16, [33, 200, 64, 1])
    got, want, _, _ = _run(c, math, ppu=3)
    assert_close(got, want, f"G{G}")


@pytest.mark.parametrize("math", ["mma", "ffma"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int8a"])
def test_single_token_is_v_exactly(math, dtype):
    # one token: softmax weight 1, the output is bf16(V_0) bit for bit
    c = random_case(5, 3, 8, 2, 128, 32, [1, 1, 1], kv_dtype=dtype)
    got, want, dc, out = _run(c, math)
    if dtype == "bf16":
        bits = bf16_dev_to_bits(out)
        want_bits = bf16_bits_from_f32(want.astype(np.float32))
        assert np.array_equal(bits, want_bits)
    else:
        # one-byte caches: the dequantised value is rounded to fp32 first
        assert_close(got, want, "single token fp8")


@pytest.mark.parametrize("math", ["mma", "ffma"])
def test_physical_permutation_bitwise_identical(math):
    # the same logical sequences stored in two different block permutations
    lens = [70, 300, 16, 129]
    a = random_case(11, 4, 32, 8, 128, 16, lens)
    b = random_case(11, 4, 32, 8, 128, 16, lens)
    perm = np.random.Generator(np.random.PCG64(3)).permutation(a.NB)
    inv = np.argsort(perm)
    b.k_src = a.k_src[:, inv].copy()
    b.v_src = a.v_src[:, inv].copy()
    b.block_tables = np.where(a.block_tables >= 0, perm[np.maximum(a.block_tables, 0)], -1).astype(np.int32)
    for ppu in (0, 3):
        _, _, _, oa = _run(a, math, ppu)
        _, _, _, ob = _run(b, math, ppu)
        assert torch.equal(oa, ob)


@pytest.mark.parametrize("math", ["mma", "ffma"])
def test_aliased_prefix_bitwise_identical(math):
    # sequences 1 and 2 point at sequence 0's first 4 blocks instead of
    # private copies holding the same tokens
    lens = [100, 90, 80]
    c = random_case(12, 3, 16, 4, 128, 16, lens)
    for b in (1, 2):
        for j in range(4):
            dst = c.block_tables[b, j]
            src = c.block_tables[0, j]
            c.k_src[:, dst] = c.k_src[:, src]
            c.v_src[:, dst] = c.v_src[:, src]
    private = DeviceCase(c)
    o_priv = private.decode(opts=pkv.decode_opts(2, MATHS[math]))
    c2 = random_case(12, 3, 16, 4, 128, 16, lens)
    c2.k_src, c2.v_src = c.k_src.copy(), c.v_src.copy()
    for b in (1, 2):
        c2.block_tables[b, :4] = c.block_tables[0, :4]
    shared = DeviceCase(c2)
    o_shared = shared.decode(opts=pkv.decode_opts(2, MATHS[math]))
    torch.cuda.synchronize()
    assert torch.equal(o_priv, o_shared)


@pytest.mark.parametrize("math", ["mma", "ffma"])
def test_split_matches_single_pass(math):
    c = random_case(13, 3, 32, 8, 128, 16, [1000, 513, 64])
    single, want, _, _ = _run(c, math, ppu=64)
    split, _, _, _ = _run(c, math, ppu=3)
    assert_close(single, want, "single pass")
    assert_close(split, want, "split")
    assert_close(split, single, "split vs single")


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int8"])
def test_shared_with_pointer(dtype):
    # two cache slots; layers 0..3 read slots [1, 0, 1, 1]
    c = random_case(14, 3, 16, 4, 128, 32, [40, 200, 77], kv_dtype=dtype, S=2,
                    kv_group_ptr=[1, 0, 1, 1])
    dc = DeviceCase(c)
    for layer in range(4):
        got = bf16_dev_to_f64(dc.decode(layer=layer))
        assert_close(got, dc.oracle(layer=layer), f"layer {layer}")


@pytest.mark.parametrize("warps,stages", [(1, 2), (2, 3), (4, 4), (8, 2), (3, 5)])
def test_launch_shapes(warps, stages):
    c = random_case(15, 5, 32, 8, 128, 16, [1, 700, 33, 256, 95])
    got, want, _, _ = _run(c, "mma", ppu=5, warps=warps, stages=stages)
    assert_close(got, want, f"warps{warps} stages{stages}")


def test_poisoned_tails_do_not_leak():
    # NaN everywhere a sequence does not read, out-of-range ids in unused
    # table entries: output stays finite and equal to the oracle's
    c = random_case(16, 4, 8, 2, 128, 32, [5, 33, 64, 95], poison=True)
    for math in ("mma", "ffma"):
        got, want, _, _ = _run(c, math)
        assert_close(got, want, f"poison {math}")


def test_zero_length_sequences_give_zeros():
    c = random_case(17, 3, 8, 2, 64, 16, [0, 20, 0])
    dc = DeviceCase(c)
    out = torch.full_like(dc.q[0], float("nan"))
    dc.decode(out=out)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[2] == 0) and np.all(np.isfinite(o[1]))


def test_out_of_range_block_id_flagged_and_skipped():
    c = random_case(18, 2, 8, 2, 64, 16, [40, 40])
    c.block_tables[1, 1] = c.NB + 5          # a block the sequence does read
    dc = DeviceCase(c)
    dc.decode()
    assert pkv.read_device_error() & pkv.DEVERR_BLOCK_ID
    assert pkv.read_device_error() == 0      # reading clears it


def test_context_len_over_capacity_flagged():
    c = random_case(19, 2, 8, 2, 64, 16, [40, 20])
    dc = DeviceCase(c)
    dc.cl = to_dev(np.array([40, 10 ** 6], np.int32))
    out = dc.decode()
    torch.cuda.synchronize()
    assert pkv.read_device_error() & pkv.DEVERR_CONTEXT_LEN
    assert torch.all(out[1] == 0)


def test_validate_mode_rejects_bad_tables(monkeypatch):
    c = random_case(20, 2, 8, 2, 64, 16, [40, 40])
    c.block_tables[0, 2] = -3
    dc = DeviceCase(c)
    monkeypatch.setenv("PKV_VALIDATE", "1")
    with pytest.raises(pkv.PkvError) as ei:
        dc.decode()
    assert ei.value.status == 1


def test_host_argument_errors():
    c = random_case(21, 2, 8, 2, 64, 16, [40, 40])
    dc = DeviceCase(c)
    with pytest.raises(pkv.PkvError) as ei:       # layer outside kv_group_ptr
        pkv.paged_decode(dc.q[0], dc.k, dc.v, dc.bt, dc.cl, [0], 1)
    assert ei.value.status == 1
    with pytest.raises(pkv.PkvError) as ei:       # shared-with pointer outside the slots
        pkv.paged_decode(dc.q[0], dc.k, dc.v, dc.bt, dc.cl, [3], 0)
    assert ei.value.status == 1
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:       # workspace too small
        pkv.paged_decode(dc.q[0], dc.k, dc.v, dc.bt, dc.cl, [0], 0,
                         workspace=ws, opts=pkv.decode_opts(partition_blocks=1))
    assert ei.value.status == 6
    with pytest.raises(pkv.PkvError) as ei:       # out aliases q
        pkv.paged_decode(dc.q[0], dc.k, dc.v, dc.bt, dc.cl, [0], 0, out=dc.q[0])
    assert ei.value.status == 1


@pytest.mark.parametrize("math", ["mma", "ffma"])
def test_fp8_scales_spanning_orders_of_magnitude(math):
    # per-page E4M3 scales spread over three decades within one sequence
    # (V pages scaled by 1e-3 .. 1, K pages by 0.1 .. 3); values stay O(1),
    # the range the tolerance is written for.  The oracle dequantises the
    # same bytes.
    from workloads import bf16_bits_to_f32, bf16_bits_from_f32, fp8_tile_scales
    c = random_case(23, 3, 16, 4, 128, 32, [600, 333, 64], kv_dtype="fp8")
    rng = np.random.Generator(np.random.PCG64(24))
    fv = (10.0 ** rng.uniform(-3, 0, size=(1, c.NB, 1, 1, 1))).astype(np.float32)
    fk = rng.uniform(0.1, 3.0, size=(1, c.NB, 1, 1, 1)).astype(np.float32)
    c.k_src = bf16_bits_from_f32(bf16_bits_to_f32(c.k_src) * fk)
    c.v_src = bf16_bits_from_f32(bf16_bits_to_f32(c.v_src) * fv)
    c.k_scale = fp8_tile_scales(c.k_src)
    c.v_scale = fp8_tile_scales(c.v_src)
    for ppu in (0, 3):
        got, want, _, _ = _run(c, math, ppu)
        assert_close(got, want, f"fp8 wide scales {math} ppu{ppu}")
