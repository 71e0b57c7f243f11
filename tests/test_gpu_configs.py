"""The five workloads at full size, in the launch configuration the benchmark
times (default options), compared with the oracle on sampled (sequence,
head) outputs that it computes one by one; plus the invariants that hold at
any size (aliased prefix == private copies, bitwise)."""
import gc

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import (fp8_shared_case, llama8b_layer_case, long_context_case, mixed_prefix_case,
                       tiny_case)
from workloads.gen import unalias_prefix
from tests._gpu import DeviceCase, assert_close, bf16_dev_to_f64, sample_pairs, to_dev, to_dev_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def _free():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _check_sampled(dc, out, layer, n, seed, what):
    pairs = sample_pairs(dc.c, n, seed)
    want = dc.oracle(layer=layer, pairs=pairs)
    got = bf16_dev_to_f64(out)
    b, h = pairs[:, 0], pairs[:, 1]
    assert_close(got[b, h], want[b, h], what)


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
    _check_sampled(dc, out, 0, 48, 2, "llama8b layer")
    out_ffma = dc.decode(opts=pkv.decode_opts(math=pkv.MATH_FFMA))
    _check_sampled(dc, out_ffma, 0, 16, 3, "llama8b layer (ffma)")


def test_mixed_prefix_batch():
    c = mixed_prefix_case()
    dc = DeviceCase(c)
    out = dc.decode()
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    # sample shared and private, short and long sequences
    shared = np.flatnonzero(c.notes["shared"])
    private = np.flatnonzero(~c.notes["shared"])
    order = np.argsort(c.context_lens)
    seqs = sorted(set([int(shared[0]), int(shared[-1]), int(private[0]), int(private[-1]),
                       int(order[0]), int(order[-1]), int(order[len(order) // 2])]))
    pairs = np.array([(b, h) for b in seqs for h in (0, 13, 31)], dtype=np.int32)
    want = dc.oracle(pairs=pairs)
    got = bf16_dev_to_f64(out)
    assert_close(got[pairs[:, 0], pairs[:, 1]], want[pairs[:, 0], pairs[:, 1]], "mixed prefix")
    _check_sampled(dc, out, 0, 32, 4, "mixed prefix (random sample)")
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
    _check_sampled(dc, out, 0, 16, 5, f"long {variant}")


def test_fp8_shared_four_layers():
    c = fp8_shared_case()
    dc = DeviceCase(c)
    assert c.kv_group_ptr.tolist() == [0, 0, 0, 0]
    for layer in range(c.L):
        out = dc.decode(layer=layer)
        torch.cuda.synchronize()
        assert pkv.read_device_error() == 0
        _check_sampled(dc, out, layer, 12, 10 + layer, f"fp8 layer {layer}")


def test_int8_shared_two_layers():
    # the same workload with an asymmetric INT8 cache
    c = fp8_shared_case(kv_dtype="int8a", L=2)
    dc = DeviceCase(c)
    for layer in range(c.L):
        out = dc.decode(layer=layer)
        torch.cuda.synchronize()
        assert pkv.read_device_error() == 0
        _check_sampled(dc, out, layer, 12, 20 + layer, f"int8 layer {layer}")
