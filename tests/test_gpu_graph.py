"""The library's calls inside CUDA graphs: one decode step (the append on the
planner's extra CTAs, then the decode and its merge) captured once and
replayed with new inputs copied into its buffers gives the same output bits
and cache bytes as eager calls on an identical cache, for single-token
(mma.sync) and multi-token (tcgen05) queries."""
import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv
from workloads import normal_bf16_bits, random_case
from tests._gpu import DeviceCase, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("T", [1, 40])
def test_graph_replay_matches_eager(T):
    c = random_case(1201 + T, 6, 32, 8, 128, 16, [T + 30, 300, 1000, 77, 2000, T + 5])
    dg, de = DeviceCase(c), DeviceCase(c)  # one cache for the graph, an identical one for eager calls
    pos = c.context_lens.astype(np.int64)[:, None] - T + np.arange(T)[None, :]
    blk = c.block_tables[np.arange(c.B)[:, None], pos // c.bs].astype(np.int64)
    slots = to_dev((blk * c.bs + pos % c.bs).reshape(-1))
    gp = c.kv_group_ptr.tolist()

    def inputs(seed):
        return (to_dev_bf16(normal_bf16_bits(seed, (c.B * T, c.Hkv, c.D))),
                to_dev_bf16(normal_bf16_bits(seed + 1, (c.B * T, c.Hkv, c.D))),
                to_dev_bf16(normal_bf16_bits(seed + 2, (c.B, T, c.Hq, c.D))))

    kn, vn, q = inputs(1300)  # the captured step's buffers
    out = torch.empty_like(q)
    ws = pkv.new_decode_workspace(dg.k, c.B, c.Hq, c.MB, None, T)
    step = lambda d, k_, v_, q_, o_=None, w_=None: pkv.append_and_decode(  # noqa: E731
        k_, v_, slots, q_, d.k, d.v, d.bt, d.cl, gp, 0, c.scale, out=o_, workspace=w_)
    # one call outside the graph on each cache (library set-up), then capture
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(dg, kn, vn, q, out, ws)
    torch.cuda.current_stream().wait_stream(side)
    step(de, kn, vn, q)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(dg, kn, vn, q, out, ws)
    for i in range(3):
        k2, v2, q2 = inputs(1400 + 10 * i)
        kn.copy_(k2)
        vn.copy_(v2)
        q.copy_(q2)
        graph.replay()
        ref = step(de, k2, v2, q2)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(out), _bits(ref)), f"step {i}: output differs from the eager call"
        assert np.array_equal(_bits(dg.k), _bits(de.k)) and np.array_equal(_bits(dg.v), _bits(de.v))
    assert pkv.read_device_error() == 0
