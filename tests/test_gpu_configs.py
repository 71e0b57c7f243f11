"""The five workloads and the verify steps at full size, in the launch
configuration the benchmark times (default options), compared with the
oracle on every output element (|gpu - oracle| <= 1e-2 + 1e-2 |oracle|);
plus the invariants that hold at any size (aliased prefix == private copies,
bitwise).  Single-token calls use the element-by-element C oracle; the
multi-token verify steps use its matrix-product form, which states the same
definition and is pinned to it and to torch's SDPA on the CPU."""
import gc

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import (fp8_shared_case, llama8b_layer_case, long_context_case, mixed_prefix_case,
                       normal_bf16_bits, tiny_case)
from workloads.gen import unalias_prefix
from tests._gpu import DeviceCase, assert_close, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _check_full(dc, out, layer, what, want=None):
    """Every (sequence, head, column) of `out` against the oracle; returns
    the oracle's output so that another back-end can be checked against it."""
    if want is None:
        want = dc.oracle(layer=layer)
    assert_close(bf16_dev_to_f64(out), want, what)
    return want


def test_tiny_full():
    c = tiny_case()
    dc = DeviceCase(c)
    out = dc.decode()
    assert_close(bf16_dev_to_f64(out), dc.oracle(), "tiny")


def test_llama8b_layer_step():
    # step = append each sequence's newest token, then decode at context 4096
    c = llama8b_layer_case()
    dc = DeviceCase(c)
    pkv.kv_append(to_dev_bf16(c.k_new), to_dev_bf16(c.v_new), to_dev(c.slot_mapping), dc.k, dc.v)
    out = dc.decode()
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert oracle.kv_append(c.k_new, c.v_new, c.slot_mapping, dc.k_host, dc.v_host) == 0
    # the appended rows are bit-exact
    for b in range(0, c.B, 7):
        s = int(c.slot_mapping[b])
        blk, off = divmod(s, c.bs)
        row = dc.k[0, blk, :, off].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(row, c.k_new[b])
    want = _check_full(dc, out, 0, "llama8b layer")
    out_ffma = dc.decode(opts=pkv.decode_opts(math=pkv.MATH_FFMA))
    _check_full(dc, out_ffma, 0, "llama8b layer (ffma)", want)


@pytest.mark.parametrize("T", [4, 8, 32, 64, 128, 256])
def test_spec_verify_full(T):
    # the verify step the benchmark times: T draft tokens per sequence appended
    # at the end of its context (4096 after the append), then one T-token
    # decode with default options (mma.sync tiles for 16 rows per KV head,
    # the tcgen05 kernel with long units above), every output element
    # against the oracle
    c = llama8b_layer_case()
    dc = DeviceCase(c)
    pos = c.context_lens.astype(np.int64)[:, None] - T + np.arange(T)[None, :]
    blk = c.block_tables[np.arange(c.B)[:, None], pos // c.bs].astype(np.int64)
    slots = (blk * c.bs + pos % c.bs).reshape(-1)
    kn = normal_bf16_bits(301 + T, (c.B * T, c.Hkv, c.D))
    vn = normal_bf16_bits(302 + T, (c.B * T, c.Hkv, c.D))
    q = normal_bf16_bits(303 + T, (c.B, T, c.Hq, c.D))
    plan = pkv.decode_plan(dc.k, c.B, c.Hq, c.MB, None, T)
    assert plan["math"] == (pkv.MATH_MMA if T * c.G <= 16 else pkv.MATH_TC)
    out = pkv.append_and_decode(to_dev_bf16(kn), to_dev_bf16(vn), to_dev(slots), to_dev_bf16(q), dc.k, dc.v,
                                dc.bt, dc.cl, c.kv_group_ptr.tolist(), 0, c.scale)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    assert oracle.kv_append(kn, vn, slots, dc.k_host, dc.v_host) == 0
    want = oracle.paged_decode_multi_gemm(q, dc.k_host, dc.v_host, c.block_tables, c.context_lens,
                                          c.kv_group_ptr, 0, c.scale)
    assert_close(bf16_dev_to_f64(out), want, f"verify T={T} ({plan['partition_blocks']}-block partitions)")


def test_mixed_prefix_batch():
    c = mixed_prefix_case()
    dc = DeviceCase(c)
    out = dc.decode()
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    _check_full(dc, out, 0, "mixed prefix")
    # aliasing the prefix blocks or giving every sharer private copies: same bits
    cp = unalias_prefix(c)
    del dc
    gc.collect()
    dp = DeviceCase(cp)
    out_p = dp.decode()
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), out_p.cpu())


@pytest.mark.parametrize("variant", ["b4_32k", "b1_128k"])
def test_long_context(variant):
    c = long_context_case(variant)
    dc = DeviceCase(c)
    out = dc.decode()
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    _check_full(dc, out, 0, f"long {variant}")


def test_fp8_shared_four_layers():
    c = fp8_shared_case()
    dc = DeviceCase(c)
    assert c.kv_group_ptr.tolist() == [0, 0, 0, 0]
    for layer in range(c.L):
        out = dc.decode(layer=layer)
        torch.cuda.synchronize()
        assert pkv.read_device_error() == 0
        _check_full(dc, out, layer, f"fp8 layer {layer}")


def test_int8_shared_two_layers():
    # the same workload with an asymmetric INT8 cache
    c = fp8_shared_case(kv_dtype="int8a", L=2)
    dc = DeviceCase(c)
    for layer in range(c.L):
        out = dc.decode(layer=layer)
        torch.cuda.synchronize()
        assert pkv.read_device_error() == 0
        _check_full(dc, out, layer, f"int8 layer {layer}")
