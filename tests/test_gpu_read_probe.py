"""The read-only HBM probe reads every byte once: its sum of 32-bit words
equals the host's, for sizes from one 16-byte chunk to beyond L2, ragged
against the grid's stride and unroll."""
import numpy as np
import pytest
import torch

import paged_kv_cache_274_gb300 as pkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, (1 << 20) + 48, (200 << 20) + 16 * 12345])
def test_read_probe_sums_every_word(nbytes):
    rng = np.random.Generator(np.random.PCG64(nbytes))
    host = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    want = int(host.astype(np.uint64).sum(dtype=np.uint64))
    data = torch.from_numpy(host.view(np.int32)).cuda()
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    pkv.read_probe(data, out)
    pkv.read_probe(data, out)   # adds to the running sum
    torch.cuda.synchronize()
    got = int(out.cpu().numpy().view(np.uint64)[0])
    assert got == (2 * want) % 2**64


def test_read_probe_empty_launches_nothing():
    out = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    pkv.read_probe(torch.empty(0, dtype=torch.uint8, device="cuda"), out)
    torch.cuda.synchronize()
    assert int(out.item()) == 7
