"""CPU-side checks of the C ABI: the library builds, loads, exports every
function the header declares, and the host-only entry points validate their
arguments (no GPU needed: these paths return before touching CUDA)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv
from paged_kv_cache_274_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def declared_functions():
    src = "".join(open(os.path.join(ROOT, "include", f)).read()
                  for f in sorted(os.listdir(os.path.join(ROOT, "include"))) if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pkv_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_api():
    names = declared_functions()
    for n in ("pkv_kv_append", "pkv_paged_decode", "pkv_decode_workspace_bytes",
              "pkv_read_device_error", "pkv_status_string", "pkv_paged_decode_multi",
              "pkv_copy_blocks", "pkv_prefix_cache_match", "pkv_read_probe"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"


def test_abi_version_and_status_strings(lib):
    assert lib.pkv_abi_version() == 2
    assert lib.pkv_status_string(0) == b"ok"
    assert b"aligned" in lib.pkv_status_string(3)


def _desc(**kw):
    d = dict(num_slots=1, num_blocks=100, block_size=16, num_kv_heads=8, head_dim=128, dtype=0)
    d.update(kw)
    return pkv.CacheDesc(**d)


def test_workspace_bytes_host_only(lib):
    d = _desc()
    n1 = lib.pkv_decode_workspace_bytes(ctypes.byref(d), 64, 32, 256, None)
    assert n1 > 0
    # one partition per sequence: no split-K partials
    opts = pkv.decode_opts(partition_blocks=64)
    small = lib.pkv_decode_workspace_bytes(ctypes.byref(d), 4, 32, 64, ctypes.byref(opts))
    assert 0 < small < 4096
    # more partitions need more partial storage
    o8 = pkv.decode_opts(partition_blocks=8)
    o32 = pkv.decode_opts(partition_blocks=32)
    assert (lib.pkv_decode_workspace_bytes(ctypes.byref(d), 64, 32, 256, ctypes.byref(o8)) >
            lib.pkv_decode_workspace_bytes(ctypes.byref(d), 64, 32, 256, ctypes.byref(o32)))


@pytest.mark.parametrize("bad", [
    dict(block_size=8), dict(head_dim=96), dict(dtype=1, head_dim=64), dict(num_kv_heads=0),
    dict(dtype=7), dict(num_blocks=0)])
def test_bad_cache_descriptors_rejected(lib, bad):
    d = _desc(**bad)
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d), 4, 32, 16, None) == 0
    st = lib.pkv_kv_append(ctypes.byref(d), 0, None, None, None, 4, None, None, None, None, None)
    assert st in (1, 2)


def test_bad_head_grouping_rejected(lib):
    d = _desc()
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d), 4, 12, 16, None) == 0   # 12 % 8 != 0
    ffma = pkv.decode_opts(math=pkv.MATH_FFMA)
    d1 = _desc(num_kv_heads=1)
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d1), 4, 16, 16, ctypes.byref(ffma)) == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d1), 4, 16, 16, None) > 0   # mma: G = 16 ok
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d1), 4, 32, 16, None) == 0  # G = 32


def test_append_argument_checks(lib):
    d = _desc()
    # slot outside the cache slots
    assert lib.pkv_kv_append(ctypes.byref(d), 1, None, None, None, 1, None, None, None, None, None) == 1
    # zero tokens is a no-op
    assert lib.pkv_kv_append(ctypes.byref(d), 0, None, None, None, 0, None, None, None, None, None) == 0
    # null pointers
    assert lib.pkv_kv_append(ctypes.byref(d), 0, None, None, None, 3, None, None, None, None, None) == 1
    # misaligned pointers (never dereferenced: the check comes first)
    p = ctypes.c_void_p(0x1008)
    assert lib.pkv_kv_append(ctypes.byref(d), 0, p, p, ctypes.c_void_p(0x2000), 3, p, p, None,
                             None, None) == 3
    # E4M3 cache without scales
    d8 = _desc(dtype=1)
    a = ctypes.c_void_p(0x1000)
    assert lib.pkv_kv_append(ctypes.byref(d8), 0, a, a, a, 3, a, a, None, None, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    # monkeypatch puts the loaded library and its path back afterwards
    monkeypatch.setattr(pkv, "_lib", None)
    monkeypatch.setattr(pkv, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(pkv.PkvError):
        pkv.load()


def test_binding_rejects_host_tensors():
    # every call checks its tensors before anything is launched
    kc = torch.zeros((1, 4, 2, 16, 64), dtype=torch.bfloat16)
    q = torch.zeros((2, 8, 64), dtype=torch.bfloat16)
    bt = torch.zeros((2, 4), dtype=torch.int32)
    cl = torch.ones(2, dtype=torch.int32)
    for call in (pkv.paged_decode, pkv.PreparedDecode):
        with pytest.raises(pkv.PkvError) as ei:
            call(q, kc, kc, bt, cl)
        assert ei.value.status == 1 and "CUDA tensor" in str(ei.value)


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_274_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "pkv_oracle" not in text, f


def _plan(lib, d, B, T, Hq, MB, opts=None):
    plan = pkv.DecodePlan()
    st = lib.pkv_decode_multi_describe(ctypes.byref(d), B, T, Hq, MB,
                                       ctypes.byref(opts) if opts is not None else None,
                                       ctypes.byref(plan))
    return st, plan


@pytest.mark.parametrize("Hq,Hkv,T,tokens_per_tile,tiles", [
    (32, 8, 1, 1, 1), (32, 8, 4, 4, 1), (32, 8, 8, 4, 2), (32, 8, 5, 4, 2),
    (16, 1, 3, 1, 3), (8, 8, 16, 16, 1), (8, 8, 17, 16, 2), (24, 8, 6, 5, 2)])
def test_multi_token_row_tiles(lib, Hq, Hkv, T, tokens_per_tile, tiles):
    # mma.sync: (query token, head) rows form tiles of at most 16 rows, whole tokens each
    d = _desc(num_kv_heads=Hkv)
    st, plan = _plan(lib, d, 8, T, Hq, 64, pkv.decode_opts(math=pkv.MATH_MMA))
    assert st == 0
    assert (plan.query_tokens_per_tile, plan.row_tiles) == (tokens_per_tile, tiles)
    assert (Hq // Hkv) * plan.query_tokens_per_tile <= 16


@pytest.mark.parametrize("Hq,Hkv,T,math,tokens_per_tile,tiles", [
    (32, 8, 4, 2, 4, 1),        # 16 rows: auto keeps mma.sync
    (32, 8, 8, 3, 8, 1),        # 32 rows: auto picks tcgen05 (one 128-row tile)
    (32, 8, 16, 3, 16, 1),      # 64 rows: auto picks tcgen05 (128-row tiles)
    (32, 8, 33, 3, 32, 2),
    (16, 1, 9, 3, 8, 2),        # G 16: 8 tokens per 128-row tile
    (8, 8, 128, 3, 128, 1),     # MHA: 128 tokens in one tile
    (64, 8, 2, 2, 2, 1)])       # G 8, 16 rows
def test_auto_back_end_and_tiles(lib, Hq, Hkv, T, math, tokens_per_tile, tiles):
    d = _desc(num_kv_heads=Hkv)
    st, plan = _plan(lib, d, 8, T, Hq, 64)
    assert st == 0 and plan.math == math
    assert (plan.query_tokens_per_tile, plan.row_tiles) == (tokens_per_tile, tiles)


def test_tc_argument_checks(lib):
    tc = pkv.decode_opts(math=pkv.MATH_TC)
    assert _plan(lib, _desc(), 8, 1, 32, 64, tc)[0] == 2                  # T = 1
    st, plan = _plan(lib, _desc(dtype=1), 8, 4, 32, 64, tc)                # E4M3 cache: widened
    assert st == 0 and plan.math == pkv.MATH_TC and plan.warps_per_cta == 8  # + the converter warp
    assert _plan(lib, _desc(head_dim=64), 8, 4, 32, 64, tc)[0] == 2       # head_dim 64
    assert _plan(lib, _desc(), 8, 4, 32, 64, tc)[0] == 0


@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_tc_one_tile_fits_two_ctas_per_sm(lib, dtype):
    # the one-tile tcgen05 kernel runs two CTAs per SM (each overlaps the
    # other's waits; 256 TMEM columns each): its shared memory, plus the
    # 1 KiB the SM keeps per CTA, must fit twice into the SM's 228 KiB.  The
    # one-byte instances add the unit slots' page parameters (2 x 4 KiB).
    st, plan = _plan(lib, _desc(dtype=dtype), 8, 32, 32, 64, pkv.decode_opts(math=pkv.MATH_TC))
    assert st == 0 and plan.math == pkv.MATH_TC and plan.row_tiles == 1
    assert plan.warps_per_cta == (7 if dtype == 0 else 8)
    assert 2 * (plan.smem_bytes_per_cta + 1024) <= 228 * 1024


def test_multi_token_arguments(lib):
    d = _desc()
    assert _plan(lib, d, 8, 0, 32, 64)[0] == 1                       # T = 0
    assert _plan(lib, d, 8, pkv.MAX_QUERY_TOKENS + 1, 32, 64)[0] == 1
    assert _plan(lib, d, 8, 2, 32, 64, pkv.decode_opts(math=pkv.MATH_FFMA))[0] == 2  # mma only
    assert _plan(lib, d, 8, 1, 32, 64, pkv.decode_opts(math=pkv.MATH_FFMA))[0] == 0
    # T = 1 is the single-token call
    one = pkv.DecodePlan()
    assert lib.pkv_decode_describe(ctypes.byref(d), 8, 32, 64, None, ctypes.byref(one)) == 0
    st, multi = _plan(lib, d, 8, 1, 32, 64)
    assert st == 0 and bytes(one) == bytes(multi)
    # partial storage grows with the query rows
    o = pkv.decode_opts(partition_blocks=8)
    w1 = lib.pkv_decode_multi_workspace_bytes(ctypes.byref(d), 8, 1, 32, 64, ctypes.byref(o))
    w4 = lib.pkv_decode_multi_workspace_bytes(ctypes.byref(d), 8, 4, 32, 64, ctypes.byref(o))
    assert w4 > 3 * w1 > 0


@pytest.mark.parametrize("B,MB,ppu", [
    (64, 256, 256),   # 64 sequences x 8 KV heads of 4096 tokens: 512 whole-sequence units (2 rounds of 304)
    (4, 256, 64),     # 4 sequences: 64-block units, 128 of them, one round
    (64, 40, 40)])    # short contexts: one partition per sequence
def test_tc_partition_length(lib, B, MB, ppu):
    # the tcgen05 kernel's partition length: the size of {64, 128, 256}
    # blocks with the least modelled time (rounds of 2 x 152 units x (64-token
    # steps + 6.5)), capped at the table width; explicit sizes 1..256
    st, plan = _plan(lib, _desc(num_blocks=20000), B, 32, 32, MB)
    assert st == 0 and plan.math == pkv.MATH_TC
    assert plan.partition_blocks == ppu
    assert plan.max_partitions == (MB + ppu - 1) // ppu
    st, p128 = _plan(lib, _desc(num_blocks=20000), B, 32, 32, MB, pkv.decode_opts(partition_blocks=128))
    assert st == 0 and p128.partition_blocks == min(128, MB)
    assert _plan(lib, _desc(num_blocks=20000), B, 32, 32, MB, pkv.decode_opts(partition_blocks=257))[0] == 1


def test_read_probe_argument_errors(lib):
    # host checks come before any CUDA call
    a = ctypes.c_void_p(0x1000)
    assert lib.pkv_read_probe(None, 16, a, None) == 1
    assert lib.pkv_read_probe(a, 16, None, None) == 1
    assert lib.pkv_read_probe(a, 24, a, None) == 1          # not a multiple of 16
    assert lib.pkv_read_probe(ctypes.c_void_p(0x1008), 16, a, None) == 3   # data not 16-byte aligned
    assert lib.pkv_read_probe(a, 16, ctypes.c_void_p(0x1004), None) == 3   # sum not 8-byte aligned


@pytest.mark.parametrize("T,ppu,pmax", [(8, 256, 1), (32, 256, 1), (64, 256, 2), (128, 256, 1)])
def test_tc_partition_length_counts_split_k(lib, T, ppu, pmax):
    # the verify steps of the Llama-8B layer (64 sequences of 256 blocks):
    # at T = 64 (two row tiles per KV head) 128-block units would take fewer
    # modelled rounds (7 x 38.5 = 269.5 against 4 x 70.5 = 282), but each
    # writes 128 rows x 130 fp32 of split-K partials that the merge reads back
    # (2048 x 133 KB at 4 MB per step: +68), so whole sequences win.  Then the
    # tile-pair kernel's last round (512 pair units on 152 SMs: 56) is under
    # half full, so the last ceil(56 / 8) = 7 sequences take half-length
    # partitions (and a merge launch over their rows); at T = 128 it is 112
    # of 152, and nothing changes
    st, plan = _plan(lib, _desc(num_blocks=20000), 64, T, 32, 256)
    assert st == 0 and plan.math == pkv.MATH_TC
    assert plan.partition_blocks == ppu and plan.max_partitions == pmax
    assert plan.kernels_per_call == (3 if pmax > 1 else 2)


def test_kernel_digest_ignores_comments_only(tmp_path):
    # profiles name the sources they were taken on by this digest: a comment
    # edit keeps it, a code edit changes it
    import shutil
    d = tmp_path / "csrc"
    shutil.copytree(os.path.join(ROOT, "paged_kv_cache_274_gb300", "csrc"), d)
    base = _build.kernel_digest(str(d))
    assert base == _build.kernel_digest()
    f = d / "read_probe.cu"
    src = f.read_text()
    f.write_text(src.replace("// Read-only HBM probe", "// A read-only HBM probe", 1) + "\n/* a note */\n")
    assert _build.kernel_digest(str(d)) == base
    f.write_text(src.replace("kProbeUnroll = 4", "kProbeUnroll = 2", 1))
    assert _build.kernel_digest(str(d)) != base


def test_plans_are_consistent_over_random_shapes(lib):
    # host planning only: for seeded random shapes every accepted plan covers
    # the table with its partitions, tiles whole query tokens, fits shared
    # memory, launches a merge exactly when a sequence can span more
    # partitions than the decode merges itself, and sizes a workspace the
    # library accepts
    rng = np.random.Generator(np.random.PCG64(2024))
    checked = 0
    for _ in range(400):
        D = int(rng.choice([64, 128]))
        bs = int(rng.choice([16, 32]))
        dtype = int(rng.choice([0, 1, 2])) if D == 128 else 0
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        T = int(rng.choice([1, 2, 4, 8, 16, 33, 64, 128]))
        B = int(rng.integers(1, 300))
        MB = int(rng.integers(1, 1200))
        math = int(rng.choice([0, 1, 2, 3]))
        ppu = int(rng.choice([0, 0, 1, 5, 64]))
        d = _desc(num_blocks=50000, block_size=bs, num_kv_heads=Hkv, head_dim=D, dtype=dtype)
        opts = pkv.decode_opts(partition_blocks=ppu, math=math)
        st, plan = _plan(lib, d, B, T, G * Hkv, MB, opts)
        if st != 0:
            assert st in (1, 2)   # refused shapes: invalid argument or unsupported
            continue
        checked += 1
        assert plan.math in (pkv.MATH_FFMA, pkv.MATH_MMA, pkv.MATH_TC)
        assert plan.partition_blocks >= 1 and plan.partition_blocks * plan.max_partitions >= MB
        # the tile-pair kernel (tcgen05, two or more row tiles, bf16) may give
        # the last sequences partitions of half the length
        pair = plan.math == pkv.MATH_TC and plan.row_tiles >= 2 and dtype == 0
        if pair and (plan.max_partitions - 1) * plan.partition_blocks >= MB:
            assert (plan.max_partitions - 1) * ((plan.partition_blocks + 1) // 2) < MB
        else:
            assert (plan.max_partitions - 1) * plan.partition_blocks < MB
        tt, nt = plan.query_tokens_per_tile, plan.row_tiles
        assert 1 <= tt <= T and nt == (T + tt - 1) // tt
        rows = 128 if plan.math == pkv.MATH_TC else 16
        assert tt * G <= rows or tt == 1
        assert plan.smem_bytes_per_cta <= 227 * 1024
        fused = plan.math != pkv.MATH_TC and plan.max_partitions <= 4
        assert plan.kernels_per_call == (3 if plan.max_partitions > 1 and not fused else 2)
        n = lib.pkv_decode_multi_workspace_bytes(ctypes.byref(d), B, T, G * Hkv, MB, ctypes.byref(opts))
        assert n == plan.workspace_bytes and n > 0
    assert checked > 150


def test_two_part_e4m3_query_split():
    # the E4M3 tcgen05 path holds a query row, scaled to a largest |q'| in
    # [2^7, 2^8), as qh = e4m3(q') plus ql = e4m3(q' - qh), both rounded to
    # nearest: for every bf16 value below 2^8 the sum is q' exactly from 2^-2
    # up (the residual's 4 significant bits are no finer than E4M3's 2^-9),
    # and within 2^-10 of it below
    import torch
    bits = np.arange(0x0001, 0x4380, dtype=np.uint16)  # 0x4380: 256.0 as bf16
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32)
    x = torch.cat([x, -x])
    qh = x.to(torch.float8_e4m3fn).to(torch.float32)
    ql = (x - qh).to(torch.float8_e4m3fn).to(torch.float32)  # x - qh is exact in fp32
    err = (qh + ql - x).abs()
    big = x.abs() >= 0.25
    assert bool((err[big] == 0).all())
    assert float(err[~big].max()) <= 2.0 ** -10
