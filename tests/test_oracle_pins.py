"""Pins of the CPU oracle against things other than itself.

* torch's float64 scaled_dot_product_attention on the dense logical sequence
  (a library routine; the paged cache here is built by scattering the dense
  sequence into random physical blocks, the opposite direction of the
  oracle's gather) -- "PagedAttention" on the bandwidth-wall page: the block
  table maps logical to physical blocks and the kernel finds K/V through it;
* torch's float8_e4m3fn conversion (library) and the OCP E4M3 field values
  for the codec -- "Quantized KV Cache / FP8 KV cache";
* closed forms (one token, equal keys, one dominant key) and invariants
  (physical block permutation, shared prefix blocks, poisoned unused rows,
  GQA vs repeated MHA heads, the cross-layer shared-with pointer).

Every pin is a function of the oracle library so that ``test_planted_mistakes``
can run the same pins against copies of the oracle with a mistake planted in
them and check that at least one pin fails for each.
"""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from workloads import bf16_bits_from_f32, bf16_bits_to_f32, normal_bf16_bits
from tests._paged import (dense_bf16_seqs, paged_from_dense, sdpa_causal_tail_reference,
                          sdpa_reference, torch_e4m3_to_f64, torch_f32_to_e4m3)

TOL = 1e-12


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# attention pins
# ---------------------------------------------------------------------------
def pin_sdpa_bf16(lib=None):
    configs = [  # (Hq, Hkv, D, bs, lens)
        (8, 2, 64, 16, [37, 100]),
        (4, 4, 64, 16, [1, 16, 17, 0]),
        (8, 1, 128, 32, [33, 64, 5]),
        (16, 2, 128, 16, [48, 250]),
        (8, 8, 128, 32, [31, 32, 95]),
    ]
    for i, (Hq, Hkv, D, bs, lens) in enumerate(configs):
        ks, vs = dense_bf16_seqs(100 + i, lens, Hkv, D)
        kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=200 + i)
        q = normal_bf16_bits(300 + i, (len(lens), Hq, D))
        scale = float(np.float32(1 / np.sqrt(D)))
        got = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, scale, lib=lib)
        want = sdpa_reference(q, [_f64(k) for k in ks], [_f64(v) for v in vs], scale)
        np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL, err_msg=f"config {i}")


def pin_large_logits(lib=None):
    # logits of order +-1e3: the softmax must subtract the running maximum
    lens, Hq, Hkv, D, bs = [40, 7], 4, 2, 64, 16
    rng = np.random.Generator(np.random.PCG64(5))
    ks = [bf16_bits_from_f32(rng.standard_normal((n, Hkv, D), dtype=np.float32) * 20) for n in lens]
    vs = [bf16_bits_from_f32(rng.standard_normal((n, Hkv, D), dtype=np.float32)) for n in lens]
    q = bf16_bits_from_f32(rng.standard_normal((2, Hq, D), dtype=np.float32) * 20)
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=6)
    got = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, lib=lib)
    want = sdpa_reference(q, [_f64(k) for k in ks], [_f64(v) for v in vs], 0.125)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


def pin_closed_forms(lib=None):
    Hq, Hkv, D, bs = 4, 2, 64, 16
    # one token: the output is that token's V, exactly
    ks, vs = dense_bf16_seqs(7, [1], Hkv, D)
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=8)
    q = normal_bf16_bits(9, (1, Hq, D))
    got = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, lib=lib)
    for h in range(Hq):
        assert np.array_equal(got[0, h], _f64(vs[0][0, h // (Hq // Hkv)]))
    # all keys equal: the output is the mean of V
    n = 45
    k_one = normal_bf16_bits(10, (1, Hkv, D))
    ks = [np.repeat(k_one, n, axis=0)]
    vs = [normal_bf16_bits(11, (n, Hkv, D))]
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=12)
    got = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, lib=lib)
    mean = _f64(vs[0]).mean(axis=0)
    for h in range(Hq):
        np.testing.assert_allclose(got[0, h], mean[h // (Hq // Hkv)], rtol=TOL, atol=TOL)
    # one dominant key: the output is that token's V
    n, j = 50, 29
    kd = np.zeros((n, Hkv, D), dtype=np.float32)
    kd[j, :, 0] = 64.0
    qd = np.zeros((1, Hq, D), dtype=np.float32)
    qd[0, :, 0] = 8.0
    ks = [bf16_bits_from_f32(kd)]
    vs = [normal_bf16_bits(13, (n, Hkv, D))]
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=14)
    got = oracle.paged_decode(bf16_bits_from_f32(qd), kc, vc, bt, ctx, [0], 0, 0.125, lib=lib)
    for h in range(Hq):
        np.testing.assert_allclose(got[0, h], _f64(vs[0][j, h // (Hq // Hkv)]), rtol=0, atol=1e-12)


def pin_permutation_invariance(lib=None):
    Hq, Hkv, D, bs, lens = 8, 2, 64, 16, [70, 33, 16]
    ks, vs = dense_bf16_seqs(20, lens, Hkv, D)
    q = normal_bf16_bits(21, (3, Hq, D))
    outs = []
    for seed in (1, 2, 3):
        kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=seed, spare=4)
        outs.append(oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, lib=lib))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_shared_prefix(lib=None):
    # three sequences whose first two blocks hold the same tokens: aliasing
    # those blocks in the tables must give the same result as private copies
    Hq, Hkv, D, bs = 4, 1, 64, 16
    prefix_k = normal_bf16_bits(30, (32, Hkv, D))
    prefix_v = normal_bf16_bits(31, (32, Hkv, D))
    tails = [10, 0, 21]
    ks = [np.concatenate([prefix_k, normal_bf16_bits(32 + i, (t, Hkv, D))]) for i, t in enumerate(tails)]
    vs = [np.concatenate([prefix_v, normal_bf16_bits(40 + i, (t, Hkv, D))]) for i, t in enumerate(tails)]
    q = normal_bf16_bits(33, (3, Hq, D))
    kc, vc, bt, ctx, pl = paged_from_dense(ks, vs, bs, seed=34)
    private = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, lib=lib)
    bt2 = bt.copy()
    for b in (1, 2):
        bt2[b, :2] = bt[0, :2]          # alias sequence 0's prefix blocks
        for p in pl[b][:2]:             # and poison the private copies
            kc[0, p] = 0x7FC0
            vc[0, p] = 0x7FC0
    aliased = oracle.paged_decode(q, kc, vc, bt2, ctx, [0], 0, 0.125, lib=lib)
    assert np.array_equal(private, aliased)


def pin_poisoned_unused(lib=None):
    Hq, Hkv, D, bs, lens = 8, 2, 64, 16, [37, 100, 16]
    ks, vs = dense_bf16_seqs(50, lens, Hkv, D)
    q = normal_bf16_bits(51, (3, Hq, D))
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=52, spare=3, MB=9)
    clean = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, lib=lib)
    kp = np.where(kc == 0, np.uint16(0x7FC0), kc)   # unused rows were zero-filled
    vp = np.where(vc == 0, np.uint16(0x7FC0), vc)
    btp = np.where(bt < 0, np.int32(10 ** 6), bt)
    dirty = oracle.paged_decode(q, kp, vp, btp, ctx, [0], 0, 0.125, lib=lib)
    assert np.all(np.isfinite(dirty))
    assert np.array_equal(clean, dirty)


def pin_gqa_equals_repeated_mha(lib=None):
    Hq, Hkv, D, bs, lens = 8, 2, 128, 32, [40, 77]
    G = Hq // Hkv
    ks, vs = dense_bf16_seqs(60, lens, Hkv, D)
    q = normal_bf16_bits(61, (2, Hq, D))
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=62)
    gqa = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.0883883, lib=lib)
    kr = np.ascontiguousarray(np.repeat(kc, G, axis=2))
    vr = np.ascontiguousarray(np.repeat(vc, G, axis=2))
    mha = oracle.paged_decode(q, kr, vr, bt, ctx, [0], 0, 0.0883883, lib=lib)
    assert np.array_equal(gqa, mha)


def pin_shared_with_pointer(lib=None):
    # two cache slots with different contents; layer l reads slot ptr[l]
    Hq, Hkv, D, bs, lens = 4, 2, 64, 16, [20, 50]
    ptr = [1, 0, 1]
    ks0, vs0 = dense_bf16_seqs(70, lens, Hkv, D)
    ks1, vs1 = dense_bf16_seqs(71, lens, Hkv, D)
    kc, vc, bt, ctx, _ = paged_from_dense(ks0, vs0, bs, seed=72, slots=2, slot=0)
    kc1, vc1, _, _, _ = paged_from_dense(ks1, vs1, bs, seed=72, slots=2, slot=1)
    kc[1], vc[1] = kc1[1], vc1[1]
    q = normal_bf16_bits(73, (2, Hq, D))
    for layer, slot in enumerate(ptr):
        got = oracle.paged_decode(q, kc, vc, bt, ctx, ptr, layer, 0.125, lib=lib)
        ks, vs = (ks0, vs0) if slot == 0 else (ks1, vs1)
        want = sdpa_reference(q, [_f64(k) for k in ks], [_f64(v) for v in vs], 0.125)
        np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL)


def pin_sdpa_fp8(lib=None):
    # E4M3 pages with one scale per (block, KV head): the reference decodes
    # the same codes with torch and multiplies by the page's scale
    Hq, Hkv, D, bs, lens = 8, 2, 128, 32, [70, 31]
    rng = np.random.Generator(np.random.PCG64(80))
    codes = [rng.integers(0, 256, size=(n, Hkv, D), dtype=np.uint8) for n in lens]
    vcodes = [rng.integers(0, 256, size=(n, Hkv, D), dtype=np.uint8) for n in lens]
    for c in codes + vcodes:                        # no NaN codes in real data
        c[(c & 0x7F) == 0x7F] = 0x3F
    kc, vc, bt, ctx, pl = paged_from_dense(codes, vcodes, bs, seed=81)
    NB = kc.shape[1]
    ks = rng.uniform(0.01, 2.0, size=(1, NB, Hkv)).astype(np.float32)
    vsc = rng.uniform(0.01, 2.0, size=(1, NB, Hkv)).astype(np.float32)
    q = normal_bf16_bits(82, (2, Hq, D))
    got = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.0883883, k_scale=ks, v_scale=vsc, lib=lib)
    kd, vd = [], []
    for b, n in enumerate(lens):
        tok_blk = np.array([pl[b][t // bs] for t in range(n)])
        kd.append(torch_e4m3_to_f64(codes[b]) * ks[0, tok_blk][:, :, None].astype(np.float64))
        vd.append(torch_e4m3_to_f64(vcodes[b]) * vsc[0, tok_blk][:, :, None].astype(np.float64))
    want = sdpa_reference(q, kd, vd, 0.0883883)
    np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL)


def pin_bad_inputs_rejected(lib=None):
    Hq, Hkv, D, bs, lens = 4, 2, 64, 16, [20]
    ks, vs = dense_bf16_seqs(90, lens, Hkv, D)
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=91)
    q = normal_bf16_bits(92, (1, Hq, D))
    bad = bt.copy()
    bad[0, 1] = kc.shape[1]
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kc, vc, bad, ctx, [0], 0, 0.125, lib=lib)
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kc, vc, bt, np.array([bt.shape[1] * bs + 1], np.int32), [0], 0, 0.125, lib=lib)


# ---------------------------------------------------------------------------
# codec pins
# ---------------------------------------------------------------------------
def pin_e4m3_decode_all_codes(lib=None):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes, lib=lib)
    want = torch_e4m3_to_f64(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    # OCP E4M3 anchors: max 448 = S.1111.110, min normal 2^-6, min subnormal 2^-9, 1.0
    anchors = {0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x38: 1.0, 0x00: 0.0}
    for c, v in anchors.items():
        assert got[c] == v
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def pin_e4m3_encode_matches_library(lib=None):
    # every bf16 pattern whose magnitude is below 464 (where a non-saturating
    # RNE conversion and the saturating one agree), as float32
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = bf16_bits_to_f32(bits)
    keep = np.isfinite(x) & (np.abs(x) < 464)
    x = x[keep]
    got = oracle.e4m3_quantize(bf16_bits_from_f32(x), np.float32(1.0), lib=lib)
    want = torch_f32_to_e4m3(x)
    assert np.array_equal(got, want)
    # saturation of finite values above the range, and NaN stays NaN
    for v in (464.0, 480.0, 1e4, 3e38, float("inf")):
        assert oracle.e4m3_encode(v, lib=lib) == 0x7E
        assert oracle.e4m3_encode(-v, lib=lib) == 0xFE
    assert oracle.e4m3_encode(float("nan"), lib=lib) & 0x7F == 0x7F
    # round trip of every finite code
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        v = oracle.e4m3_decode(np.array([c], np.uint8), lib=lib)[0]
        assert oracle.e4m3_encode(v, lib=lib) == c


def pin_e4m3_scaled_quantize(lib=None):
    rng = np.random.Generator(np.random.PCG64(95))
    x = normal_bf16_bits(96, (4096,))
    for s in (np.float32(1.0), np.float32(0.0091), np.float32(3.7), np.float32(1 / 448)):
        got = oracle.e4m3_quantize(x, s, lib=lib)
        q = (bf16_bits_to_f32(x) / s).astype(np.float32)
        q = np.clip(q, -448, 448)
        assert np.array_equal(got, torch_f32_to_e4m3(q))
    del rng


# ---------------------------------------------------------------------------
# append pins
# ---------------------------------------------------------------------------
def pin_append_scatter(lib=None):
    S, NB, Hkv, bs, D = 2, 9, 2, 16, 64
    rng = np.random.Generator(np.random.PCG64(97))
    kc = rng.integers(0, 1 << 16, size=(S, NB, Hkv, bs, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(S, NB, Hkv, bs, D), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    N = 20
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    slots[3] = -1
    kn = normal_bf16_bits(98, (N, Hkv, D))
    vn = normal_bf16_bits(99, (N, Hkv, D))
    assert oracle.kv_append(kn, vn, slots, kc, vc, slot=1, lib=lib) == 0
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        for h in range(Hkv):
            assert np.array_equal(kc[1, blk, h, off], kn[i, h])
            assert np.array_equal(vc[1, blk, h, off], vn[i, h])
            k0[1, blk, h, off] = kn[i, h]
            v0[1, blk, h, off] = vn[i, h]
    assert np.array_equal(kc, k0) and np.array_equal(vc, v0)   # nothing else moved
    bad = slots.copy()
    bad[0] = NB * bs
    kc2 = kc.copy()
    assert oracle.kv_append(kn, vn, bad, kc2, vc, slot=1, lib=lib) == oracle.ORACLE_BAD_SLOT
    assert np.array_equal(kc2, kc)


def pin_append_fp8(lib=None):
    S, NB, Hkv, bs, D = 1, 6, 2, 32, 128
    rng = np.random.Generator(np.random.PCG64(100))
    kc = np.zeros((S, NB, Hkv, bs, D), np.uint8)
    vc = np.zeros((S, NB, Hkv, bs, D), np.uint8)
    ks = rng.uniform(0.005, 0.05, size=(S, NB, Hkv)).astype(np.float32)
    vs = rng.uniform(0.005, 0.05, size=(S, NB, Hkv)).astype(np.float32)
    N = 12
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    kn = normal_bf16_bits(101, (N, Hkv, D))
    vn = normal_bf16_bits(102, (N, Hkv, D))
    assert oracle.kv_append(kn, vn, slots, kc, vc, ks, vs, lib=lib) == 0
    for i, s in enumerate(slots):
        blk, off = divmod(int(s), bs)
        for h in range(Hkv):
            qk = np.clip(bf16_bits_to_f32(kn[i, h]) / ks[0, blk, h], -448, 448).astype(np.float32)
            qv = np.clip(bf16_bits_to_f32(vn[i, h]) / vs[0, blk, h], -448, 448).astype(np.float32)
            assert np.array_equal(kc[0, blk, h, off], torch_f32_to_e4m3(qk))
            assert np.array_equal(vc[0, blk, h, off], torch_f32_to_e4m3(qv))


def pin_copy_blocks(lib=None):
    # every destination block equals its source block; nothing else moves;
    # copying back restores the source pool
    rng = np.random.Generator(np.random.PCG64(120))
    shape_a, shape_b = (11, 2, 16, 64), (7, 2, 16, 64)
    ak = rng.integers(0, 1 << 16, size=shape_a, dtype=np.uint16)
    av = rng.integers(0, 1 << 16, size=shape_a, dtype=np.uint16)
    bk = rng.integers(0, 1 << 16, size=shape_b, dtype=np.uint16)
    bv = rng.integers(0, 1 << 16, size=shape_b, dtype=np.uint16)
    pairs = np.array([[3, 0], [9, 5], [0, 2], [10, 6]], np.int32)
    bk0, bv0 = bk.copy(), bv.copy()
    assert oracle.copy_blocks(ak, av, bk, bv, pairs, lib=lib) == 0
    for s_, d_ in pairs:
        assert np.array_equal(bk[d_], ak[s_]) and np.array_equal(bv[d_], av[s_])
    untouched = [i for i in range(shape_b[0]) if i not in set(pairs[:, 1])]
    assert np.array_equal(bk[untouched], bk0[untouched]) and np.array_equal(bv[untouched], bv0[untouched])
    ak2, av2 = ak.copy(), av.copy()
    ak2[pairs[:, 0]] = 0
    av2[pairs[:, 0]] = 0
    assert oracle.copy_blocks(bk, bv, ak2, av2, pairs[:, ::-1].copy(), lib=lib) == 0
    assert np.array_equal(ak2, ak) and np.array_equal(av2, av)
    assert oracle.copy_blocks(ak, av, bk, bv, np.array([[11, 0]], np.int32), lib=lib) == oracle.ORACLE_BAD_BLOCK


def pin_int8_codec(lib=None):
    # reference: numpy's IEEE float32 division and round-half-even rint,
    # plus the clamp and the NaN rule; closed forms for ties and range ends
    rng = np.random.Generator(np.random.PCG64(130))
    xs = np.concatenate([rng.standard_normal(400).astype(np.float32) * 3,
                         np.array([0.0, -0.0, 1e30, -1e30], np.float32)])
    for scale, zero in ((0.031, 0.0), (0.5, 0.0), (0.02, -17.0), (0.2, 100.0), (1.0, -128.0)):
        sc, z = np.float32(scale), np.float32(zero)
        lo = -127.0 if zero == 0 else -128.0
        want = np.clip(np.rint(xs / sc) + z, lo, 127).astype(np.int64)
        got = np.array([oracle.int8_encode(x, scale, zero, lib=lib) for x in xs])
        assert np.array_equal(got, want), (scale, zero)
        assert oracle.int8_encode(float("nan"), scale, zero, lib=lib) == int(zero)
    # ties go to the even integer; exact multiples are exact; decode is (q - z) s
    assert [oracle.int8_encode(v, 1.0, lib=lib) for v in (0.5, 1.5, 2.5, -2.5, 7.0)] == [0, 2, 2, -2, 7]
    assert oracle.int8_encode(-500.0, 1.0, 0.0, lib=lib) == -127
    assert oracle.int8_encode(-500.0, 1.0, 5.0, lib=lib) == -128
    for q in (-128, -1, 0, 1, 127):
        assert oracle.int8_decode(q, 0.25, 3.0, lib=lib) == (q - 3) * 0.25


def pin_sdpa_int8(lib=None):
    # INT8 pages with (scale, zero) per (block, KV head): the reference is
    # SDPA over (code - zero) * scale computed here in float64
    Hq, Hkv, D, bs, lens = 8, 2, 128, 16, [70, 31]
    rng = np.random.Generator(np.random.PCG64(131))
    codes = [rng.integers(-128, 128, size=(n, Hkv, D), dtype=np.int8) for n in lens]
    vcodes = [rng.integers(-128, 128, size=(n, Hkv, D), dtype=np.int8) for n in lens]
    kc, vc, bt, ctx, pl = paged_from_dense(codes, vcodes, bs, seed=132)
    NB = kc.shape[1]
    kp = np.stack([rng.uniform(0.001, 0.05, size=(1, NB, Hkv)),
                   rng.integers(-20, 21, size=(1, NB, Hkv))], axis=-1).astype(np.float32)
    vp = np.stack([rng.uniform(0.001, 0.05, size=(1, NB, Hkv)),
                   rng.integers(-20, 21, size=(1, NB, Hkv))], axis=-1).astype(np.float32)
    q = normal_bf16_bits(133, (2, Hq, D))
    got = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.0883883, k_scale=kp, v_scale=vp, lib=lib)
    kd, vd = [], []
    for b, n in enumerate(lens):
        blk = np.array([pl[b][t // bs] for t in range(n)])
        ks, kz = kp[0, blk, :, 0][:, :, None].astype(np.float64), kp[0, blk, :, 1][:, :, None].astype(np.float64)
        vs, vz = vp[0, blk, :, 0][:, :, None].astype(np.float64), vp[0, blk, :, 1][:, :, None].astype(np.float64)
        kd.append((codes[b].astype(np.float64) - kz) * ks)
        vd.append((vcodes[b].astype(np.float64) - vz) * vs)
    want = sdpa_reference(q, kd, vd, 0.0883883)
    np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL)


def pin_multi_token_causal(lib=None):
    # T new query tokens per sequence against torch's causal SDPA on the dense
    # sequence (bottom-right aligned: the new tokens are the last T positions)
    configs = [  # (T, Hq, Hkv, D, bs, lens)
        (2, 8, 2, 64, 16, [37, 100, 2]),
        (4, 4, 4, 64, 16, [1, 16, 17, 3]),   # lengths below T: leading rows are zero
        (3, 8, 1, 128, 32, [33, 64, 5]),
        (5, 16, 4, 128, 16, [48, 250]),
        (1, 8, 2, 64, 16, [20, 9]),
    ]
    for i, (T, Hq, Hkv, D, bs, lens) in enumerate(configs):
        ks, vs = dense_bf16_seqs(400 + i, lens, Hkv, D)
        kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=500 + i)
        q = normal_bf16_bits(600 + i, (len(lens), T, Hq, D))
        scale = float(np.float32(1 / np.sqrt(D)))
        got = oracle.paged_decode_multi(q, kc, vc, bt, ctx, [0], 0, scale, lib=lib)
        want = sdpa_causal_tail_reference(q, [_f64(k) for k in ks], [_f64(v) for v in vs], scale)
        np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL, err_msg=f"config {i}")
        if T == 1:  # the single-token entry point is the T = 1 case
            one = oracle.paged_decode(q[:, 0], kc, vc, bt, ctx, [0], 0, scale, lib=lib)
            np.testing.assert_array_equal(one, got[:, 0])


PINS = [pin_sdpa_bf16, pin_large_logits, pin_closed_forms, pin_permutation_invariance,
        pin_shared_prefix, pin_poisoned_unused, pin_gqa_equals_repeated_mha,
        pin_shared_with_pointer, pin_sdpa_fp8, pin_bad_inputs_rejected,
        pin_e4m3_decode_all_codes, pin_e4m3_encode_matches_library, pin_e4m3_scaled_quantize,
        pin_append_scatter, pin_append_fp8, pin_copy_blocks, pin_int8_codec, pin_sdpa_int8,
        pin_multi_token_causal]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
MUTANTS = [
    ("gather_wrong_block", "block_tables[(int64_t)b * MB + j / bs];\n        int64_t page",
     "block_tables[(int64_t)b * MB + (j / bs) / 2];\n        int64_t page"),
    ("gqa_strided_heads", "int32_t g = h / G;", "int32_t g = h % Hkv;"),
    ("scale_dropped", "s[j] = (double)scale * dot;", "s[j] = dot;"),
    ("no_max_subtraction", "s[j] = exp(s[j] - smax);", "s[j] = exp(s[j]);"),
    ("no_normalisation", "double p = s[j] / z;", "double p = s[j];"),
    ("rows_reversed", "page, bs, D, j % bs, d)", "page, bs, D, bs - 1 - j % bs, d)"),
    ("last_dim_dropped", "for (int32_t d = 0; d < D; ++d)\n          dot +=",
     "for (int32_t d = 0; d < D - 1; ++d)\n          dot +="),
    ("v_from_k_cache", "cache_value(v_cache, fp8, v_scale", "cache_value(k_cache, fp8, k_scale"),
    ("slot_ignored", "int64_t page = ((int64_t)slot * NB + blk) * Hkv + g;",
     "int64_t page = ((int64_t)0 * NB + blk) * Hkv + g;"),
    ("fp8_scale_dropped", "* (double)scales[page];", "* 1.0;"),
    ("e4m3_wrong_bias", "mag = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);",
     "mag = ldexp(1.0 + (double)mantissa / 8.0, exponent - 6);"),
    ("e4m3_ties_up", "else code = (lo % 2 == 0) ? lo : lo + 1;", "else code = lo + 1;"),
    ("copy_wrong_source", "memcpy(dst_k + d * block_bytes, src_k + s * block_bytes",
     "memcpy(dst_k + d * block_bytes, src_k + d * block_bytes"),
    ("int8_rounds_down", "double q = nearbyint((double)t) + (double)zero;",
     "double q = floor((double)t) + (double)zero;"),
    ("int8_zero_sign", "return ((double)q - (double)zero) * (double)scale;",
     "return ((double)q + (double)zero) * (double)scale;"),
    ("int8_symmetric_clamp", "double lo = (zero == 0.0f) ? -127.0 : -128.0;", "double lo = -128.0;"),
    ("causal_off_by_one", "int32_t m = context_lens[b] - T + t + 1;",
     "int32_t m = context_lens[b] - T + t;"),
    ("causal_ignored", "int32_t m = context_lens[b] - T + t + 1;", "int32_t m = context_lens[b];"),
    ("query_token_order", "int32_t t = r / Hq, h = r % Hq;", "int32_t t = (T - 1) - r / Hq, h = r % Hq;"),
    ("append_wrong_offset", "int64_t blk = s / bs, off = s % bs;", "int64_t blk = s / bs, off = (s + 1) % bs;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistakes(name, old, new, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mutated = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(c), "-lm"], check=True)
    lib = oracle.load_library(str(so))
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"


def test_sampled_pairs_with_repeats_match_full_run():
    # a (b, h) listed more than once must give the same row as a full run
    Hq, Hkv, D, bs, lens = 8, 2, 64, 16, [300, 41, 77]
    ks, vs = dense_bf16_seqs(110, lens, Hkv, D)
    kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=111)
    q = normal_bf16_bits(112, (3, Hq, D))
    full = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125)
    pairs = np.array([[0, 1]] * 16 + [[2, 7], [0, 1], [1, 0]] * 8, dtype=np.int32)
    part = oracle.paged_decode(q, kc, vc, bt, ctx, [0], 0, 0.125, pairs=pairs)
    for b, h in pairs:
        assert np.array_equal(part[b, h], full[b, h])
