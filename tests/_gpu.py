"""Helpers for the GPU parity tests: move a DecodeCase to the device, run the
library through its binding, run the oracle on the same inputs, compare."""
import numpy as np
import torch

import oracle
import paged_kv_cache_274_gb300 as pkv
from workloads import DecodeCase

DEV = torch.device("cuda:0")
ATOL = 1e-2   # |gpu - oracle| <= ATOL + RTOL * |oracle|  (bf16 out, fp32 accumulate)
RTOL = 1e-2


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(DEV)


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceCase:
    """Host cache arrays (as the oracle sees them) and their device copies."""

    def __init__(self, c: DecodeCase):
        self.c = c
        if c.kv_dtype in ("int8", "int8a"):
            self.k_host = oracle.int8_quantize_cache(c.k_src, c.k_scale)
            self.v_host = oracle.int8_quantize_cache(c.v_src, c.v_scale)
            self.k = to_dev(self.k_host)
            self.v = to_dev(self.v_host)
            self.ks = to_dev(c.k_scale)
            self.vs = to_dev(c.v_scale)
        elif c.kv_dtype == "fp8":
            self.k_host = oracle.quantize_cache(c.k_src, c.k_scale)
            self.v_host = oracle.quantize_cache(c.v_src, c.v_scale)
            self.k = to_dev(self.k_host)
            self.v = to_dev(self.v_host)
            self.ks = to_dev(c.k_scale)
            self.vs = to_dev(c.v_scale)
        else:
            self.k_host, self.v_host = c.k_src, c.v_src
            self.k = to_dev_bf16(c.k_src)
            self.v = to_dev_bf16(c.v_src)
            self.ks = self.vs = None
        self.bt = to_dev(c.block_tables.astype(np.int32))
        self.cl = to_dev(c.context_lens.astype(np.int32))
        self.q = [to_dev_bf16(c.q[l]) for l in range(c.L)]

    def decode(self, layer=0, opts=None, out=None, workspace=None):
        c = self.c
        return pkv.paged_decode(self.q[layer], self.k, self.v, self.bt, self.cl,
                                c.kv_group_ptr.tolist(), layer, c.scale, out=out,
                                workspace=workspace, k_scale=self.ks, v_scale=self.vs, opts=opts)

    def oracle(self, layer=0, pairs=None):
        c = self.c
        return oracle.paged_decode(c.q[layer], self.k_host, self.v_host, c.block_tables,
                                   c.context_lens, c.kv_group_ptr, layer, c.scale,
                                   k_scale=c.k_scale, v_scale=c.v_scale, pairs=pairs)


def assert_close(got: np.ndarray, want: np.ndarray, what: str = "", atol: float = ATOL):
    assert got.shape == want.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    err = np.abs(got - want)
    bound = atol + RTOL * np.abs(want)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; max err "
                             f"{err.max():.3e}; first {idx.tolist()}")


def sample_pairs(c: DecodeCase, n: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    b = rng.integers(0, c.B, size=n)
    h = rng.integers(0, c.Hq, size=n)
    # always include the first and last (sequence, head)
    b[0], h[0] = 0, 0
    b[-1], h[-1] = c.B - 1, c.Hq - 1
    return np.stack([b, h], axis=1).astype(np.int32)
