"""Pins of the oracle's matrix-product form (``oracle.paged_decode_multi_gemm``).

It states the same definition as the element-by-element C oracle with the
logits and the weighted value sums of a (sequence, KV head) taken as float64
matrix products, so that the full-size parity tests finish in seconds.  It is
pinned to things other than itself:

* torch's float64 causal scaled_dot_product_attention on the dense logical
  sequence, with the paged cache built by scattering that sequence into
  random physical blocks (the opposite direction of the oracle's gather);
* the SDPA reference over E4M3 codes decoded by torch and over INT8
  (code - zero) * scale, page parameters per (block, KV head);
* the C oracle on random paged cases (aliased blocks, ragged and short
  lengths, every cache kind), to float64 rounding.

``test_planted_mistakes_gemm`` plants plausible mistakes in a copy of the
function and checks that the pins catch each one.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from workloads import normal_bf16_bits, random_case
from tests._paged import (dense_bf16_seqs, paged_from_dense, sdpa_causal_tail_reference,
                          torch_e4m3_to_f64)
from workloads import bf16_bits_to_f32

TOL = 1e-12


def _f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def pin_gemm_sdpa_bf16(fn):
    configs = [  # (T, Hq, Hkv, D, bs, lens)
        (1, 8, 2, 64, 16, [37, 100, 1]),
        (2, 8, 2, 64, 16, [37, 100, 2]),
        (4, 4, 4, 64, 16, [1, 16, 17, 3]),   # lengths below T: leading rows are zero
        (3, 8, 1, 128, 32, [33, 64, 5]),
        (5, 16, 4, 128, 16, [48, 250]),
        (9, 32, 8, 128, 16, [70, 9, 0]),
    ]
    for i, (T, Hq, Hkv, D, bs, lens) in enumerate(configs):
        ks, vs = dense_bf16_seqs(700 + i, lens, Hkv, D)
        kc, vc, bt, ctx, _ = paged_from_dense(ks, vs, bs, seed=710 + i)
        q = normal_bf16_bits(720 + i, (len(lens), T, Hq, D))
        scale = float(np.float32(1 / np.sqrt(D)))
        got = fn(q, kc, vc, bt, ctx, [0], 0, scale)
        want = sdpa_causal_tail_reference(q, [_f64(k) for k in ks], [_f64(v) for v in vs], scale)
        np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL, err_msg=f"config {i}")


def pin_gemm_sdpa_one_byte(fn):
    T, Hq, Hkv, D, bs, lens = 3, 8, 2, 128, 32, [70, 31, 2]
    rng = np.random.Generator(np.random.PCG64(730))
    # E4M3 codes (no NaN codes), scale per (block, KV head)
    codes = [rng.integers(0, 256, size=(n, Hkv, D), dtype=np.uint8) for n in lens]
    vcodes = [rng.integers(0, 256, size=(n, Hkv, D), dtype=np.uint8) for n in lens]
    for c in codes + vcodes:
        c[(c & 0x7F) == 0x7F] = 0x3F
    kc, vc, bt, ctx, pl = paged_from_dense(codes, vcodes, bs, seed=731)
    NB = kc.shape[1]
    ks = rng.uniform(0.01, 2.0, size=(1, NB, Hkv)).astype(np.float32)
    vsc = rng.uniform(0.01, 2.0, size=(1, NB, Hkv)).astype(np.float32)
    q = normal_bf16_bits(732, (len(lens), T, Hq, D))
    got = fn(q, kc, vc, bt, ctx, [0], 0, 0.0883883, k_scale=ks, v_scale=vsc)
    kd, vd = [], []
    for b, n in enumerate(lens):
        blk = np.array([pl[b][t // bs] for t in range(n)])
        kd.append(torch_e4m3_to_f64(codes[b]) * ks[0, blk][:, :, None].astype(np.float64))
        vd.append(torch_e4m3_to_f64(vcodes[b]) * vsc[0, blk][:, :, None].astype(np.float64))
    want = sdpa_causal_tail_reference(q, kd, vd, 0.0883883)
    np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL, err_msg="e4m3")
    # INT8 (code - zero) * scale
    codes = [rng.integers(-128, 128, size=(n, Hkv, D), dtype=np.int8) for n in lens]
    vcodes = [rng.integers(-128, 128, size=(n, Hkv, D), dtype=np.int8) for n in lens]
    kc, vc, bt, ctx, pl = paged_from_dense(codes, vcodes, bs, seed=733)
    NB = kc.shape[1]
    kp = np.stack([rng.uniform(0.001, 0.05, size=(1, NB, Hkv)),
                   rng.integers(-20, 21, size=(1, NB, Hkv))], axis=-1).astype(np.float32)
    vp = np.stack([rng.uniform(0.001, 0.05, size=(1, NB, Hkv)),
                   rng.integers(-20, 21, size=(1, NB, Hkv))], axis=-1).astype(np.float32)
    got = fn(q, kc, vc, bt, ctx, [0], 0, 0.0883883, k_scale=kp, v_scale=vp)
    kd, vd = [], []
    for b, n in enumerate(lens):
        blk = np.array([pl[b][t // bs] for t in range(n)])
        kd.append((codes[b].astype(np.float64) - kp[0, blk, :, 1][:, :, None]) * kp[0, blk, :, 0][:, :, None])
        vd.append((vcodes[b].astype(np.float64) - vp[0, blk, :, 1][:, :, None]) * vp[0, blk, :, 0][:, :, None])
    want = sdpa_causal_tail_reference(q, kd, vd, 0.0883883)
    np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL, err_msg="int8")


def pin_gemm_matches_c_oracle(fn):
    # random paged cases (random block permutation, spare blocks, two cache
    # slots read through the shared-with pointer) against the C oracle
    cases = [
        (random_case(740, 3, 8, 2, 64, 16, [1, 40, 333]), 4),
        (random_case(741, 2, 16, 16, 128, 32, [64, 2]), 3),
        (random_case(742, 3, 32, 8, 128, 16, [300, 17, 5], kv_dtype="fp8"), 6),
        (random_case(743, 2, 32, 8, 128, 32, [96, 130], kv_dtype="int8a"), 2),
        (random_case(744, 2, 8, 2, 128, 16, [50, 77], S=2, kv_group_ptr=[1, 0]), 1),
    ]
    for c, T in cases:
        if c.kv_dtype == "fp8":
            k = oracle.quantize_cache(c.k_src, c.k_scale)
            v = oracle.quantize_cache(c.v_src, c.v_scale)
        elif c.kv_dtype.startswith("int8"):
            k = oracle.int8_quantize_cache(c.k_src, c.k_scale)
            v = oracle.int8_quantize_cache(c.v_src, c.v_scale)
        else:
            k, v = c.k_src, c.v_src
        q = normal_bf16_bits(c.B + 745, (c.B, T, c.Hq, c.D))
        want = oracle.paged_decode_multi(q, k, v, c.block_tables, c.context_lens, c.kv_group_ptr, 0, c.scale,
                                         k_scale=c.k_scale, v_scale=c.v_scale)
        got = fn(q, k, v, c.block_tables, c.context_lens, c.kv_group_ptr, 0, c.scale,
                 k_scale=c.k_scale, v_scale=c.v_scale)
        np.testing.assert_allclose(got, want, rtol=TOL, atol=TOL, err_msg=c.name)


def pin_gemm_rejects_bad_tables(fn):
    c = random_case(750, 2, 8, 2, 64, 16, [20, 40])
    bt = c.block_tables.copy()
    bt[1, 1] = c.NB + 3
    with pytest.raises(ValueError):
        fn(normal_bf16_bits(751, (2, 1, 8, 64)), c.k_src, c.v_src, bt, c.context_lens, [0], 0, c.scale)
    with pytest.raises(ValueError):
        fn(normal_bf16_bits(751, (2, 1, 8, 64)), c.k_src, c.v_src, c.block_tables,
           np.array([20, 10_000], np.int32), [0], 0, c.scale)


GEMM_PINS = [pin_gemm_sdpa_bf16, pin_gemm_sdpa_one_byte, pin_gemm_matches_c_oracle, pin_gemm_rejects_bad_tables]


@pytest.mark.parametrize("pin", GEMM_PINS, ids=[p.__name__ for p in GEMM_PINS])
def test_gemm_pin(pin):
    pin(oracle.paged_decode_multi_gemm)


GEMM_MUTANTS = [
    ("causal_off_by_one", "keys = n - T + pos_t + 1", "keys = n - T + pos_t"),
    ("causal_ignored", "keys = n - T + pos_t + 1", "keys = n + 0 * pos_t"),
    ("gqa_strided_heads", "Q = qf[b, :, g * G:(g + 1) * G, :]", "Q = qf[b, :, g::Hkv, :]"),
    ("scale_dropped", "S = sc * (Q @ K[g].T)", "S = (Q @ K[g].T)"),
    ("no_normalisation", "O = (E / np.where(z > 0, z, 1.0)) @ V[g]", "O = E @ V[g]"),
    ("v_from_k", "O = (E / np.where(z > 0, z, 1.0)) @ V[g]", "O = (E / np.where(z > 0, z, 1.0)) @ K[g]"),
    ("rows_reversed", ".reshape(Hkv, -1, D)[:, :n]\n        V", ".reshape(Hkv, -1, D)[:, :n][:, ::-1]\n        V"),
    ("block_order_ignored", "blocks = bt[b, :(n + bs - 1) // bs]", "blocks = np.sort(bt[b, :(n + bs - 1) // bs])"),
    ("slot_ignored", "slot = int(np.asarray(kv_group_ptr)[layer])", "slot = 0"),
    ("zero_point_sign", "pr[:, :, None, None, 1])", "-pr[:, :, None, None, 1])"),
    ("e4m3_scale_dropped", "return table[pages] * sc[:, :, None, None]", "return table[pages]"),
    ("token_order", "out[b, :, g * G:(g + 1) * G, :] = O.reshape(T, G, D)",
     "out[b, :, g * G:(g + 1) * G, :] = O.reshape(T, G, D)[::-1]"),
]


def _mutated(old, new):
    src = textwrap.dedent(inspect.getsource(oracle.paged_decode_multi_gemm)) + "\n" + \
        textwrap.dedent(inspect.getsource(oracle._cache_values))
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["paged_decode_multi_gemm"]


@pytest.mark.parametrize("name,old,new", GEMM_MUTANTS, ids=[m[0] for m in GEMM_MUTANTS])
def test_planted_mistakes_gemm(name, old, new):
    fn = _mutated(old, new)
    failed = []
    for pin in GEMM_PINS:
        try:
            pin(fn)
        except (AssertionError, ValueError, IndexError, pytest.fail.Exception):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
