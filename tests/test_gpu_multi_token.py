"""GPU multi-token query decode (T new tokens per sequence, causal among
them) against the oracle: sweeps over head grouping x T (one and several row
tiles), block sizes, cache dtypes, split-K partition sizes, contexts shorter
than T; the T = 1 case against the single-token call; each query token
against a single-token decode of the truncated context (bitwise); and the
speculative-decoding flow (append T tokens, then verify them)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import normal_bf16_bits, random_case
from tests._gpu import ATOL, DEV, DeviceCase, assert_close, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _q(seed, B, T, Hq, D):
    return normal_bf16_bits(seed, (B, T, Hq, D))


def _run(dc, qbits, ppu=0, layer=0):
    c = dc.c
    opts = pkv.decode_opts(partition_blocks=ppu)
    out = pkv.paged_decode_multi(to_dev_bf16(qbits), dc.k, dc.v, dc.bt, dc.cl, c.kv_group_ptr.tolist(),
                                 layer, c.scale, k_scale=dc.ks, v_scale=dc.vs, opts=opts)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    return out


def _oracle(dc, qbits, layer=0):
    c = dc.c
    return oracle.paged_decode_multi(qbits, dc.k_host, dc.v_host, c.block_tables, c.context_lens,
                                     c.kv_group_ptr, layer, c.scale, k_scale=c.k_scale, v_scale=c.v_scale)


SWEEP = [  # (D, bs, Hq, Hkv, T, dtype, lens)
    (128, 16, 32, 8, 2, "bf16", [1, 2, 3, 17, 300, 33]),     # G 4: 8 rows, one tile
    (128, 16, 32, 8, 4, "bf16", [4, 5, 16, 100, 1000]),       # 16 rows, one tile
    (128, 16, 32, 8, 8, "bf16", [3, 8, 9, 64, 700]),          # two tiles; a context below T
    (128, 32, 32, 8, 5, "bf16", [5, 31, 32, 33, 513]),        # ragged last tile
    (64, 16, 8, 8, 16, "bf16", [16, 17, 40, 200]),            # MHA: 16 tokens in one tile
    (64, 32, 8, 8, 20, "bf16", [19, 20, 21, 333]),            # two tiles of 16 and 4 tokens
    (128, 16, 16, 1, 3, "bf16", [3, 50, 129]),                # MQA G 16: one token per tile
    (128, 32, 64, 8, 2, "bf16", [2, 77, 260]),                # G 8
    (128, 32, 32, 8, 4, "fp8", [4, 70, 300]),
    (128, 16, 32, 8, 8, "fp8", [8, 20, 129]),
    (128, 32, 32, 8, 4, "int8a", [4, 70, 300]),
    (128, 16, 16, 4, 6, "int8", [6, 33, 250]),
]


@pytest.mark.parametrize("D,bs,Hq,Hkv,T,dtype,lens", SWEEP)
@pytest.mark.parametrize("ppu", [0, 1, 3])
def test_multi_token_sweep(D, bs, Hq, Hkv, T, dtype, lens, ppu):
    seed = D + 3 * bs + 7 * Hq + 11 * Hkv + 13 * T + len(lens)
    c = random_case(seed, len(lens), Hq, Hkv, D, bs, lens, kv_dtype=dtype)
    dc = DeviceCase(c)
    q = _q(seed + 1, c.B, T, Hq, D)
    got = bf16_dev_to_f64(_run(dc, q, ppu))
    want = _oracle(dc, q)
    assert_close(got, want, f"T={T} {dtype} ppu={ppu}")


def test_one_token_is_the_single_token_call():
    c = random_case(71, 4, 32, 8, 128, 16, [1, 40, 300, 0])
    dc = DeviceCase(c)
    q = _q(72, c.B, 1, 32, 128)
    multi = _run(dc, q)
    single = pkv.paged_decode(to_dev_bf16(q[:, 0]), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(multi[:, 0], single)


@pytest.mark.parametrize("Hq,Hkv,T", [(32, 8, 4), (32, 8, 8), (8, 8, 5)])
def test_each_token_equals_truncated_single_token_decode(Hq, Hkv, T):
    # query token t over context n is a single-token decode over n - T + t + 1
    # tokens: same tiles per row, same masking, same partitions -> same bits
    lens = [T + 3, 100, 257]
    c = random_case(80 + T, len(lens), Hq, Hkv, 128, 16, lens)
    dc = DeviceCase(c)
    q = _q(81 + T, c.B, T, Hq, 128)
    opts = pkv.decode_opts(partition_blocks=4, math=pkv.MATH_MMA)  # the same mma.sync kernels
    multi = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=opts)
    for t in range(T):
        cl = to_dev((c.context_lens - T + t + 1).astype(np.int32))
        single = pkv.paged_decode(to_dev_bf16(np.ascontiguousarray(q[:, t])), dc.k, dc.v, dc.bt, cl, [0], 0,
                                  c.scale, opts=opts)
        torch.cuda.synchronize()
        assert torch.equal(multi[:, t], single), f"token {t}"


def test_contexts_shorter_than_t_give_zero_rows():
    T = 6
    c = random_case(90, 4, 8, 2, 64, 16, [0, 2, 5, 6])
    dc = DeviceCase(c)
    q = _q(91, c.B, T, 8, 64)
    got = bf16_dev_to_f64(_run(dc, q))
    want = _oracle(dc, q)
    assert_close(got, want, "short contexts")
    assert np.all(got[0] == 0) and np.all(got[1, :4] == 0) and np.all(got[2, :1] == 0)


def test_poisoned_tails_do_not_leak():
    c = random_case(95, 3, 32, 8, 128, 16, [7, 33, 100], poison=True)
    dc = DeviceCase(c)
    q = _q(96, c.B, 4, 32, 128)
    got = bf16_dev_to_f64(_run(dc, q, ppu=2))
    assert_close(got, _oracle(dc, q), "poisoned")


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int8a"])
def test_speculative_verify_flow(dtype):
    # a step that appends T draft tokens per sequence, then scores them
    T, Hq, Hkv, D, bs = 4, 32, 8, 128, 16
    before = np.array([60, 15, 200], np.int32)
    c = random_case(100, 3, Hq, Hkv, D, bs, (before + T).tolist(), kv_dtype=dtype, spare_blocks=2)
    dc = DeviceCase(c)
    # the draft tokens' K/V: the rows at positions before[b] .. before[b] + T - 1
    slots = np.array([c.block_tables[b, p // bs] * bs + p % bs
                      for b in range(c.B) for p in range(before[b], before[b] + T)], np.int64)
    kn = normal_bf16_bits(101, (len(slots), Hkv, D))
    vn = normal_bf16_bits(102, (len(slots), Hkv, D))
    pkv.kv_append(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), dc.k, dc.v, dc.ks, dc.vs)
    q = _q(103, c.B, T, Hq, D)
    got = bf16_dev_to_f64(_run(dc, q))
    ko, vo = dc.k_host.copy(), dc.v_host.copy()
    assert oracle.kv_append(kn, vn, slots, ko, vo, c.k_scale, c.v_scale) == 0
    assert np.array_equal(dc.k.cpu().numpy().view(ko.dtype) if dtype != "bf16" else
                          dc.k.view(torch.int16).cpu().numpy().view(np.uint16), ko)
    want = oracle.paged_decode_multi(q, ko, vo, c.block_tables, c.context_lens, c.kv_group_ptr, 0,
                                     c.scale, k_scale=c.k_scale, v_scale=c.v_scale)
    assert_close(got, want, f"verify {dtype}")


def test_ffma_rejects_multi_token():
    c = random_case(110, 2, 8, 2, 64, 16, [10, 20])
    dc = DeviceCase(c)
    q = to_dev_bf16(_q(111, 2, 2, 8, 64))
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode_multi(q, dc.k, dc.v, dc.bt, dc.cl, opts=pkv.decode_opts(math=pkv.MATH_FFMA))


@pytest.mark.parametrize("stages", [2, 3, 6])
@pytest.mark.parametrize("T,Hq,Hkv", [(8, 32, 8), (16, 32, 8), (3, 16, 1)])
def test_multi_tile_ring_depths(stages, T, Hq, Hkv):
    # several row tiles per KV head, each its own stream over the pages, at
    # every ring depth, over many units and partitions
    lens = [T + 1, 300, 611, 64]
    c = random_case(120 + T + stages, len(lens), Hq, Hkv, 128, 16, lens, poison=True)
    dc = DeviceCase(c)
    q = _q(121 + T, c.B, T, Hq, 128)
    opts = pkv.decode_opts(stages=stages, partition_blocks=5, math=pkv.MATH_MMA)
    plan = pkv.decode_plan(dc.k, c.B, Hq, c.MB, opts, T)
    assert plan["row_tiles"] > 1 and plan["stages"] == stages
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=opts)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert_close(bf16_dev_to_f64(out), _oracle(dc, q), f"T={T} stages={stages}")


# ---------------------------------------------------------------------------
# tcgen05 tiles (128 query rows, TMEM accumulators)
# ---------------------------------------------------------------------------
TC_SWEEP = [  # (bs, Hq, Hkv, T, lens)
    (16, 32, 8, 8, [1, 9, 40, 300, 1000]),      # G 4: 32 rows of 128; a context below T
    (32, 32, 8, 5, [5, 31, 32, 33, 513]),       # bs 32: one page per step
    (16, 16, 1, 3, [3, 50, 129]),               # G 16
    (16, 8, 8, 20, [19, 20, 21, 333]),          # MHA, 20 rows
    (16, 32, 8, 33, [40, 100, 260]),            # two tiles (32 + 1 tokens)
    (16, 64, 8, 128, [130, 300]),               # G 8: eight tiles, a prefill chunk
    (32, 16, 2, 17, [17, 64, 65, 700]),
    # two or more tiles per KV head: CTAs that hold a pair of tiles
    (16, 32, 8, 64, [64, 65, 300, 1000]),        # one full pair
    (32, 32, 8, 96, [96, 200, 701]),             # three tiles: the second pair half empty
    (16, 8, 1, 40, [41, 500, 77]),               # G 8: 16 tokens a tile, three tiles
    (16, 24, 8, 50, [50, 51, 260]),              # G 3: 42 tokens (126 rows) a tile
    (32, 32, 8, 256, [256, 300, 1100]),          # a 256-token prefill chunk, eight tiles
]


def _tc_opts(ppu=0):
    return pkv.decode_opts(partition_blocks=ppu, math=pkv.MATH_TC)


@pytest.mark.parametrize("bs,Hq,Hkv,T,lens", TC_SWEEP)
@pytest.mark.parametrize("ppu", [0, 1, 3, 7])
def test_tc_sweep(bs, Hq, Hkv, T, lens, ppu):
    seed = 900 + 3 * bs + 7 * Hq + 11 * Hkv + 13 * T
    c = random_case(seed, len(lens), Hq, Hkv, 128, bs, lens, poison=True)
    dc = DeviceCase(c)
    q = _q(seed + 1, c.B, T, Hq, 128)
    plan = pkv.decode_plan(dc.k, c.B, Hq, c.MB, _tc_opts(ppu), T)
    assert plan["math"] == pkv.MATH_TC
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=_tc_opts(ppu))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert_close(bf16_dev_to_f64(out), _oracle(dc, q), f"tc T={T} G={Hq // Hkv} bs={bs} ppu={ppu}")


@pytest.mark.parametrize("value_scale", [1.0, 4.0])
def test_tc_large_logits_and_auto_choice(value_scale):
    # logits of order +-100 make the lazy running maximum rescale O often
    c = random_case(950, 3, 32, 8, 128, 16, [64, 500, 1200], value_scale=value_scale)
    dc = DeviceCase(c)
    q = _q(951, c.B, 16, 32, 128)
    assert pkv.decode_plan(dc.k, c.B, 32, c.MB, None, 16)["math"] == pkv.MATH_TC   # auto picks tcgen05
    tc = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale)
    mma = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale,
                                 opts=pkv.decode_opts(math=pkv.MATH_MMA))
    torch.cuda.synchronize()
    want = _oracle(dc, q)
    # N(0,1) values (the workloads' distribution) are held to the unit bound
    # 1e-2 + 1e-2 |oracle|.  With K and V scaled by 4 the bound takes an
    # absolute term derived from the arithmetic: both back-ends round the
    # attention weights P to bf16 (unit roundoff 2^-8) before P . V, so the
    # numerator's error is up to 2^-8 sum_k w_k |V_k| <= 2^-8 max|V|, which
    # outputs near 0 by cancellation cannot absorb in their relative term.
    # A float64 emulation of the tcgen05 kernel's steps (64-token steps, lazy
    # running maximum, bf16 P, fp32 sums) reproduces the elements that exceed
    # the unit bound at that scale, with the same maximum error.
    atol = ATOL
    if value_scale != 1.0:
        v = bf16_dev_to_f64(dc.v)
        atol = ATOL + 2.0 ** -8 * float(np.abs(v).max())
    assert_close(bf16_dev_to_f64(tc), want, "tc", atol=atol)
    assert_close(bf16_dev_to_f64(mma), want, "mma", atol=atol)


def test_tc_speculative_verify_flow():
    T, Hq, Hkv, D, bs = 8, 32, 8, 128, 16
    before = np.array([60, 15, 200, 1000], np.int32)
    c = random_case(960, 4, Hq, Hkv, D, bs, (before + T).tolist(), spare_blocks=2)
    dc = DeviceCase(c)
    slots = np.array([c.block_tables[b, p // bs] * bs + p % bs
                      for b in range(c.B) for p in range(before[b], before[b] + T)], np.int64)
    kn = normal_bf16_bits(961, (len(slots), Hkv, D))
    vn = normal_bf16_bits(962, (len(slots), Hkv, D))
    q = _q(963, c.B, T, Hq, D)
    got = pkv.append_and_decode(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), to_dev_bf16(q), dc.k, dc.v,
                                dc.bt, dc.cl, [0], 0, c.scale)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    ko, vo = dc.k_host.copy(), dc.v_host.copy()
    assert oracle.kv_append(kn, vn, slots, ko, vo) == 0
    want = oracle.paged_decode_multi(q, ko, vo, c.block_tables, c.context_lens, c.kv_group_ptr, 0, c.scale)
    assert_close(bf16_dev_to_f64(got), want, "tc verify")


def test_tc_unsupported_shapes_rejected():
    c64 = random_case(970, 2, 32, 8, 64, 16, [40, 50])   # head_dim 64
    d64 = DeviceCase(c64)
    q = to_dev_bf16(_q(971, 2, 8, 32, 64))
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode_multi(q, d64.k, d64.v, d64.bt, d64.cl, opts=_tc_opts())
    c = random_case(972, 2, 32, 8, 128, 16, [40, 50])
    dc = DeviceCase(c)
    with pytest.raises(pkv.PkvError):   # T = 1
        pkv.paged_decode_multi(to_dev_bf16(_q(973, 2, 1, 32, 128)), dc.k, dc.v, dc.bt, dc.cl, opts=_tc_opts())


def test_tc_bad_block_id_flagged_and_skipped():
    # an out-of-range id inside a sequence: flagged, its page contributes nothing
    T, Hq, Hkv = 16, 32, 8
    c = random_case(980, 2, Hq, Hkv, 128, 16, [100, 200])
    dc = DeviceCase(c)
    bt = c.block_tables.copy()
    bt[1, 3] = c.NB + 5
    dc.bt = to_dev(bt)
    q = _q(981, c.B, T, Hq, 128)
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=_tc_opts())
    torch.cuda.synchronize()
    assert pkv.read_device_error() & pkv.DEVERR_BLOCK_ID
    got = bf16_dev_to_f64(out)
    # sequence 0 is untouched; sequence 1 equals attention without tokens 48..63
    want0 = _oracle(dc, q)[0]
    assert_close(got[0], want0, "tc sequence 0")
    assert np.all(np.isfinite(got[1]))


@pytest.mark.parametrize("T,ppu", [(8, 0), (8, 1), (32, 0), (32, 1), (64, 0), (64, 1)])
def test_tc_first_token_is_v0_exactly(T, ppu):
    # context_lens == T: the first query token attends to position 0 alone,
    # so its softmax weight is 1 and its output is bf16(V_0) bit for bit, in
    # the rotated (T x G = 32) and the full-tile (128 rows) instance, with and
    # without split-K partitions (a partition with no key of the row has
    # weight 0 in the merge)
    c = random_case(990 + T + ppu, 3, 32, 8, 128, 16, [T, T, T])
    dc = DeviceCase(c)
    q = _q(991 + T, c.B, T, 32, 128)
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=_tc_opts(ppu))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    got = out[:, 0].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)   # [B][Hq][D]
    G = c.Hq // c.Hkv
    for b in range(c.B):
        blk = int(c.block_tables[b, 0])
        for h in range(c.Hq):
            assert np.array_equal(got[b, h], dc.v_host[0, blk, h // G, 0]), (b, h)


@pytest.mark.parametrize("T", [8, 32, 64])
def test_tc_physical_permutation_bitwise_identical(T):
    # the same logical sequences stored in two different block permutations
    # give the same output bits: the order of every sum depends only on
    # logical positions (and the partition length)
    lens = [70, 300, 40, 129]
    a = random_case(13 + T, 4, 32, 8, 128, 16, lens)
    b = random_case(13 + T, 4, 32, 8, 128, 16, lens)
    perm = np.random.Generator(np.random.PCG64(4)).permutation(a.NB)
    inv = np.argsort(perm)
    b.k_src = a.k_src[:, inv].copy()
    b.v_src = a.v_src[:, inv].copy()
    b.block_tables = np.where(a.block_tables >= 0, perm[np.maximum(a.block_tables, 0)], -1).astype(np.int32)
    da, db = DeviceCase(a), DeviceCase(b)
    q = to_dev_bf16(_q(14 + T, a.B, T, 32, 128))
    for ppu in (0, 3):
        oa = pkv.paged_decode_multi(q, da.k, da.v, da.bt, da.cl, [0], 0, a.scale, opts=_tc_opts(ppu))
        ob = pkv.paged_decode_multi(q, db.k, db.v, db.bt, db.cl, [0], 0, b.scale, opts=_tc_opts(ppu))
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"T={T} ppu={ppu}"


@pytest.mark.parametrize("T", [8, 32, 64])
def test_tc_aliased_prefix_bitwise_identical(T):
    # sequences 1 and 2 point at sequence 0's first 4 blocks instead of
    # private copies holding the same tokens
    lens = [100, 90, 80]
    c = random_case(15 + T, 3, 32, 8, 128, 16, lens)
    for s in (1, 2):
        for j in range(4):
            dst, src = c.block_tables[s, j], c.block_tables[0, j]
            c.k_src[:, dst] = c.k_src[:, src]
            c.v_src[:, dst] = c.v_src[:, src]
    private = DeviceCase(c)
    c2 = random_case(15 + T, 3, 32, 8, 128, 16, lens)
    c2.k_src, c2.v_src = c.k_src.copy(), c.v_src.copy()
    for s in (1, 2):
        c2.block_tables[s, :4] = c.block_tables[0, :4]
    shared = DeviceCase(c2)
    q = to_dev_bf16(_q(16 + T, c.B, T, 32, 128))
    op = pkv.paged_decode_multi(q, private.k, private.v, private.bt, private.cl, [0], 0, c.scale, opts=_tc_opts(2))
    osh = pkv.paged_decode_multi(q, shared.k, shared.v, shared.bt, shared.cl, [0], 0, c2.scale, opts=_tc_opts(2))
    torch.cuda.synchronize()
    assert torch.equal(op, osh)


@pytest.mark.parametrize("T,ppu", [(512, 0), (512, 5), (200, 3)])
def test_tc_prefill_chunks(T, ppu):
    # chunked prefill over a paged cache ("Continuous Batching"): windows of
    # up to 512 new tokens per sequence, with and without split-K partitions,
    # every element against the oracle
    Hq, Hkv = 32, 8
    lens = [T, T + 37, 1500]
    c = random_case(1100 + T + ppu, len(lens), Hq, Hkv, 128, 16, lens, poison=True)
    dc = DeviceCase(c)
    q = _q(1101 + T, c.B, T, Hq, 128)
    plan = pkv.decode_plan(dc.k, c.B, Hq, c.MB, _tc_opts(ppu), T)
    assert plan["math"] == pkv.MATH_TC and plan["row_tiles"] == (T * 4 + 127) // 128
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=_tc_opts(ppu))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    want = oracle.paged_decode_multi_gemm(q, dc.k_host, dc.v_host, c.block_tables, c.context_lens,
                                          c.kv_group_ptr, 0, c.scale)
    assert_close(bf16_dev_to_f64(out), want, f"prefill T={T} ppu={ppu}")


@pytest.mark.parametrize("B,lens_hi", [(24, 4096), (40, 2600), (9, 700)])
def test_tc_pair_half_length_partitions(B, lens_hi):
    # the tile-pair kernel's last-round balancing: with automatic partitions
    # and a last round of units at most half full, the last sequences take
    # partitions of half the length and the merge covers their rows only;
    # ragged lengths (some shorter than one partition), every element
    # against the oracle
    Hq, Hkv, T = 32, 8, 64
    rng = np.random.Generator(np.random.PCG64(1200 + B))
    lens = [int(x) for x in rng.integers(T, lens_hi + 1, size=B)]
    lens[-1] = lens_hi
    c = random_case(1201 + B, B, Hq, Hkv, 128, 16, lens, poison=True)
    dc = DeviceCase(c)
    q = _q(1202 + B, c.B, T, Hq, 128)
    plan = pkv.decode_plan(dc.k, c.B, Hq, c.MB, _tc_opts(0), T)
    assert plan["math"] == pkv.MATH_TC and plan["row_tiles"] == 2
    full = (c.MB + plan["partition_blocks"] - 1) // plan["partition_blocks"]
    units = B * full * Hkv   # pair units at the longest context
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    halved = 0 < units % sms <= sms // 2
    assert (plan["max_partitions"] > full) == halved, (units, sms, plan)
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=_tc_opts(0))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    want = oracle.paged_decode_multi_gemm(q, dc.k_host, dc.v_host, c.block_tables, c.context_lens,
                                          c.kv_group_ptr, 0, c.scale)
    assert_close(bf16_dev_to_f64(out), want, f"half-length partitions B={B}")


def test_tc_pair_matches_one_tile_kernel():
    # the pair kernel and the one-tile kernel (PKV_TC_PAIR=0 in a child
    # process) compute the same products; their outputs agree to rounding
    import os
    import subprocess
    import sys
    env = dict(os.environ, PKV_TC_PAIR="0")
    code = (
        "import sys, numpy as np, torch\n"
        "sys.path.insert(0, %r)\n"
        "import paged_kv_cache_274_gb300 as pkv\n"
        "from workloads import random_case, normal_bf16_bits\n"
        "from tests._gpu import DeviceCase, to_dev_bf16\n"
        "c = random_case(1200, 3, 32, 8, 128, 16, [64, 300, 900])\n"
        "dc = DeviceCase(c)\n"
        "q = normal_bf16_bits(1201, (3, 64, 32, 128))\n"
        "o = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale,"
        " opts=pkv.decode_opts(math=pkv.MATH_TC))\n"
        "np.save(sys.argv[1], o.float().cpu().numpy())\n"
    ) % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),)
    import tempfile
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "one_tile.npy")
        subprocess.run([sys.executable, "-c", code, path], env=env, check=True, timeout=600)
        one_tile = np.load(path).astype(np.float64)
    c = random_case(1200, 3, 32, 8, 128, 16, [64, 300, 900])
    dc = DeviceCase(c)
    q = _q(1201, 3, 64, 32, 128)
    pair = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale, opts=_tc_opts())
    torch.cuda.synchronize()
    assert_close(bf16_dev_to_f64(pair), one_tile, "pair vs one-tile kernel")


# ---------------------------------------------------------------------------
# one-byte caches (E4M3, INT8) on the tcgen05 tiles: products on exact code
# values (E4M3 K pages as they are, against a two-part E4M3 query; INT8 K
# and all V pages widened to f16 in shared memory), the page scales applied
# to the scores and to P
# ---------------------------------------------------------------------------
TC_1B_SWEEP = [  # (dtype, bs, Hq, Hkv, T, lens)
    ("fp8", 16, 32, 8, 8, [1, 9, 40, 300, 1000]),      # 32 rows of 128, a context below T
    ("fp8", 32, 32, 8, 33, [40, 100, 260]),            # two tiles
    ("fp8", 16, 16, 1, 20, [20, 50, 129]),             # G 16
    ("int8", 16, 16, 1, 3, [3, 50, 129]),
    ("int8a", 32, 32, 8, 32, [32, 64, 700]),           # one full tile
    ("int8a", 16, 8, 8, 20, [19, 20, 21, 333]),        # MHA
]


@pytest.mark.parametrize("dtype,bs,Hq,Hkv,T,lens", TC_1B_SWEEP)
@pytest.mark.parametrize("ppu", [0, 3])
def test_tc_one_byte_sweep(dtype, bs, Hq, Hkv, T, lens, ppu):
    seed = 1300 + 3 * bs + 7 * Hq + 11 * Hkv + 13 * T + len(dtype)
    c = random_case(seed, len(lens), Hq, Hkv, 128, bs, lens, kv_dtype=dtype, poison=True)
    dc = DeviceCase(c)
    q = _q(seed + 1, c.B, T, Hq, 128)
    plan = pkv.decode_plan(dc.k, c.B, Hq, c.MB, _tc_opts(ppu), T)
    assert plan["math"] == pkv.MATH_TC
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale,
                                 k_scale=dc.ks, v_scale=dc.vs, opts=_tc_opts(ppu))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert_close(bf16_dev_to_f64(out), _oracle(dc, q), f"tc {dtype} T={T} G={Hq // Hkv} bs={bs} ppu={ppu}")


@pytest.mark.parametrize("dtype", ["fp8", "int8a"])
@pytest.mark.parametrize("ppu", [0, 3])
def test_tc_one_byte_wide_scales(dtype, ppu):
    # per-page scales spread over three decades within one sequence (V pages
    # scaled by 1e-3 .. 1, K pages by 0.1 .. 3), values O(1): P carries
    # v_scale / v_max of its page in f16, which keeps 11 bits down to a
    # ratio of 2^-14 of a weight; the oracle dequantises the same bytes
    from workloads import bf16_bits_to_f32, bf16_bits_from_f32, fp8_tile_scales, int8_tile_params
    c = random_case(1480 + ppu, 3, 16, 4, 128, 32, [600, 333, 64], kv_dtype=dtype)
    rng = np.random.Generator(np.random.PCG64(1481))
    fv = (10.0 ** rng.uniform(-3, 0, size=(1, c.NB, 1, 1, 1))).astype(np.float32)
    fk = rng.uniform(0.1, 3.0, size=(1, c.NB, 1, 1, 1)).astype(np.float32)
    c.k_src = bf16_bits_from_f32(bf16_bits_to_f32(c.k_src) * fk)
    c.v_src = bf16_bits_from_f32(bf16_bits_to_f32(c.v_src) * fv)
    if dtype == "fp8":
        c.k_scale, c.v_scale = fp8_tile_scales(c.k_src), fp8_tile_scales(c.v_src)
    else:
        c.k_scale, c.v_scale = int8_tile_params(c.k_src, False), int8_tile_params(c.v_src, False)
    dc = DeviceCase(c)
    T = 32
    q = _q(1482 + ppu, c.B, T, 16, 128)
    plan = pkv.decode_plan(dc.k, c.B, 16, c.MB, _tc_opts(ppu), T)
    assert plan["math"] == pkv.MATH_TC
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale,
                                 k_scale=dc.ks, v_scale=dc.vs, opts=_tc_opts(ppu))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert_close(bf16_dev_to_f64(out), _oracle(dc, q), f"tc {dtype} wide scales ppu={ppu}")


@pytest.mark.parametrize("dtype", ["fp8", "int8a"])
def test_tc_one_byte_query_dynamic_range(dtype):
    # query rows whose elements span 16 binades (|q| = |N(0,1)| x 2^U(-14, 2)),
    # rows of zeros, and rows with one element 2^10 above the rest: the E4M3
    # path splits each scaled row into two E4M3 parts that are exact down to
    # 2^-10 of the row's largest element and within 2^-17 of it below; the
    # INT8 path holds the row in f16 scaled to [2^14, 2^15)
    c = random_case(1470, 3, 32, 8, 128, 16, [500, 129, 64], kv_dtype=dtype)
    dc = DeviceCase(c)
    T = 32
    rng = np.random.Generator(np.random.PCG64(1471))
    q = rng.standard_normal((c.B, T, 32, 128)) * 2.0 ** rng.uniform(-14, 2, size=(c.B, T, 32, 128))
    q[0, 3] = 0.0                                      # every head of one token: zeros
    q[1, :, 5] = 1e-3 * rng.standard_normal((T, 128))  # one head: small but not tiny
    q[1, :, 5, 7] = 1.0                                 # ... with one element 2^10 above
    from workloads import bf16_bits_from_f32
    q = bf16_bits_from_f32(q.astype(np.float32))
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale,
                                 k_scale=dc.ks, v_scale=dc.vs, opts=_tc_opts(0))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert_close(bf16_dev_to_f64(out), _oracle(dc, q), f"tc {dtype} query dynamic range")


def _widened_bits(dc, blk, kvh, row):
    """bf16 bits of bf16(fp32(code value) x fp32 scale) ((code - zero) for
    INT8) of V row `row` of page (blk, kvh): the dequantised row, rounded
    once.  A query row whose only key is that row (weight 1, one page in its
    unit) gets exactly these bits: the kernel multiplies the exact f16 code
    value by the page scale once, in fp32."""
    c = dc.c
    codes = dc.v_host[0, blk, kvh, row]
    if c.kv_dtype == "fp8":
        val = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32)
        val = val * torch.tensor(float(c.v_scale[0, blk, kvh]), dtype=torch.float32)
    else:
        s_, z_ = c.v_scale[0, blk, kvh]
        val = (torch.from_numpy(codes.astype(np.float32)) - torch.tensor(float(z_))) * torch.tensor(float(s_))
    return val.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["fp8", "int8a"])
@pytest.mark.parametrize("T,ppu", [(8, 0), (32, 1)])
def test_tc_one_byte_first_token_is_widened_v0_exactly(dtype, T, ppu):
    # context_lens == T: the first query token attends to position 0 alone
    # (weight 1), so its output is the widened V_0 row bit for bit
    c = random_case(1400 + T + ppu, 3, 32, 8, 128, 16, [T, T, T], kv_dtype=dtype)
    dc = DeviceCase(c)
    q = _q(1401 + T, c.B, T, 32, 128)
    out = pkv.paged_decode_multi(to_dev_bf16(q), dc.k, dc.v, dc.bt, dc.cl, [0], 0, c.scale,
                                 k_scale=dc.ks, v_scale=dc.vs, opts=_tc_opts(ppu))
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    got = out[:, 0].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    G = c.Hq // c.Hkv
    for b in range(c.B):
        blk = int(c.block_tables[b, 0])
        for h in range(c.Hq):
            assert np.array_equal(got[b, h], _widened_bits(dc, blk, h // G, 0)), (b, h)


def test_tc_one_byte_physical_permutation_bitwise_identical():
    lens = [70, 300, 40, 129]
    a = random_case(1450, 4, 32, 8, 128, 16, lens, kv_dtype="fp8")
    b = random_case(1450, 4, 32, 8, 128, 16, lens, kv_dtype="fp8")
    perm = np.random.Generator(np.random.PCG64(5)).permutation(a.NB)
    inv = np.argsort(perm)
    b.k_src, b.v_src = a.k_src[:, inv].copy(), a.v_src[:, inv].copy()
    b.k_scale, b.v_scale = a.k_scale[:, inv].copy(), a.v_scale[:, inv].copy()
    b.block_tables = np.where(a.block_tables >= 0, perm[np.maximum(a.block_tables, 0)], -1).astype(np.int32)
    da, db = DeviceCase(a), DeviceCase(b)
    q = to_dev_bf16(_q(1451, a.B, 8, 32, 128))
    for ppu in (0, 3):
        oa = pkv.paged_decode_multi(q, da.k, da.v, da.bt, da.cl, [0], 0, a.scale, k_scale=da.ks, v_scale=da.vs,
                                    opts=_tc_opts(ppu))
        ob = pkv.paged_decode_multi(q, db.k, db.v, db.bt, db.cl, [0], 0, b.scale, k_scale=db.ks, v_scale=db.vs,
                                    opts=_tc_opts(ppu))
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"ppu={ppu}"
