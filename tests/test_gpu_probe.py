"""GPU check of the read-bandwidth probe (pn_read_ranges): it must read every
16-byte word of every range exactly once, which the XOR of the words read
shows (computed on the host with numpy)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_pn_gb300 import build, pn as pn_mod
    build.build()
    return pn_mod


def test_read_ranges_xor(pn):
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(11)
    sizes = [16, 4096, 37_879_808, 0, 16 * 12345, 2_228_224]
    host = [rng.integers(0, 2 ** 32, size=n // 4, dtype=np.uint32) for n in sizes]
    tensors = [torch.from_numpy(h.view(np.int32)).to(dev) if h.size else torch.empty(0, dtype=torch.int32, device=dev)
               for h in host]
    sink = torch.zeros(len(tensors), dtype=torch.int32, device=dev)
    pn.read_ranges(tensors, sink)
    got = sink.cpu().numpy().view(np.uint32)
    want = np.array([np.bitwise_xor.reduce(h) if h.size else 0 for h in host], dtype=np.uint32)
    assert np.array_equal(got, want)
