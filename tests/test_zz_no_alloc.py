"""The decode entry point that needs no workspace from its caller.

Some callers cannot allocate device memory when they decode (a runtime that
owns every allocation, a plugin that is handed only its buffers), so the
library offers pkv_paged_decode_static_workspace, whose scratch is a static
device array inside the library.  These tests call it through the C ABI
(ctypes binding) and check it against pkv_paged_decode with a caller
workspace, on two calls in a row with different inputs so that what the
first call leaves in the shared array cannot leak into the second.
This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv
from workloads import random_case
from tests._gpu import DeviceCase, assert_close, bf16_dev_to_f64

pytestmark = pytest.mark.gpu


def _static_decode(dc, opts):
    c = dc.c
    out = torch.full_like(dc.q[0], float("nan"))
    pkv.paged_decode_static_workspace(dc.q[0], dc.k, dc.v, dc.bt, dc.cl, c.kv_group_ptr.tolist(), 0,
                                      c.scale, out=out, k_scale=dc.ks, v_scale=dc.vs, opts=opts)
    torch.cuda.synchronize()
    assert pkv.read_device_error() == 0
    return out


@pytest.mark.parametrize("math", [pkv.MATH_MMA, pkv.MATH_FFMA])
def test_two_calls_match_workspace_entry_point(math):
    # first call: split-K partials in the array; second call: different
    # shapes and lengths (fewer partitions, one sequence inactive)
    cases = [
        (random_case(301, 4, 32, 8, 128, 16, [700, 33, 1000, 257]), pkv.decode_opts(3, math)),
        (random_case(302, 3, 16, 4, 128, 32, [64, 0, 95], kv_dtype="fp8"), pkv.decode_opts(2, math)),
    ]
    for c, opts in cases:
        dc = DeviceCase(c)
        ref = dc.decode(opts=opts)
        got = _static_decode(dc, opts)
        assert_close(bf16_dev_to_f64(got), bf16_dev_to_f64(ref), c.name)
        assert_close(bf16_dev_to_f64(got), dc.oracle(), c.name + " vs oracle")


def test_oversized_request_is_rejected():
    # 4096 sequences x 64 heads x 4096 one-block partitions: far beyond the array
    desc = pkv.CacheDesc(1, 1 << 16, 16, 8, 128, pkv.KV_BF16)
    opts = pkv.decode_opts(partition_blocks=1)
    gp = (ctypes.c_int32 * 1)(0)
    lib = pkv.load()
    need = lib.pkv_decode_workspace_bytes(ctypes.byref(desc), 4096, 64, 4096, ctypes.byref(opts))
    assert need > pkv.STATIC_WORKSPACE_MAX_BYTES
    st = lib.pkv_paged_decode_static_workspace(
        ctypes.byref(desc), None, 4096, 64, None, None, None, None, None, 4096, None, gp, 1, 0,
        0.088, None, ctypes.byref(opts), None)
    assert st == 6
    assert b"built-in workspace" in lib.pkv_last_error_message()
