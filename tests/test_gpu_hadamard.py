"""GPU parity of the runtime Hadamard rotation (pn_hadamard) with the CPU oracle.

The rotation's arithmetic is fixed (fp32 butterflies in ascending stages, one
fp32 scale, fp16 round-to-nearest-even), so the device output is compared bit
for bit.  Inputs are seeded fp16 activations of the workloads' widths plus
magnitudes that reach the edges of fp16 (subnormal inputs, outputs that
overflow to infinity).  A rotated GEMV is checked end to end: the GPU rotation
followed by the GPU GEMV against the oracle's rotation and GEMV.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import PN3T, PN4T, assert_gemv_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_pn_gb300 import build, pn as pn_mod
    build.build()
    pn_mod.lib()
    return pn_mod


def activations(rng, M, K):
    x = rng.standard_normal((M, K))
    scale = rng.choice([1.0, 1.0, 1.0, 300.0, 1e-5], size=(M, K))       # large and subnormal values
    x = (x * scale).astype(np.float16)
    x[rng.random((M, K)) < 0.02] = 0.0
    return x


@pytest.mark.parametrize("M,K,block", [(1, 5120, 1024), (8, 6144, 2048), (3, 17408, 1024), (2, 8192, 4096),
                                       (1, 96, 2), (5, 96, 32), (7, 4096, 512), (4, 640, 128)])
def test_hadamard_bit_exact(pn, oracle, M, K, block):
    dev = torch.device("cuda", 0)
    x = activations(np.random.default_rng(K + block + M), M, K)
    got = pn.hadamard(torch.from_numpy(x).to(dev), block).cpu().numpy()
    want = oracle.hadamard(x, block)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_hadamard_overflow_and_in_place(pn, oracle):
    dev = torch.device("cuda", 0)
    x = np.full((2, 16), 65504.0, dtype=np.float16)          # sums overflow fp16 after scaling
    x[1, ::2] = -65504.0
    xd = torch.from_numpy(x).to(dev)
    pn.hadamard(xd, 4, out=xd)                                # in place
    want = oracle.hadamard(x, 4)
    got = xd.cpu().numpy()
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    assert np.isinf(got).any()


@pytest.mark.parametrize("pn_type,K,block", [(PN3T, 5120, 1024), (PN4T, 6144, 2048)])
def test_rotated_gemv(pn, oracle, pn_type, K, block):
    # rotation then GEMV on the device against the oracle's rotation and GEMV
    from bit_weight_only_pn_gb300 import synth
    dev = torch.device("cuda", 0)
    N, M = 333, 2
    w = synth.weights(0x4AD, N, K)
    x = synth.activations(0x4AE, M, K)
    W = oracle.pack(pn_type, w)
    xr = oracle.hadamard(x, block)
    y_ref, abs_sum = oracle.gemv(pn_type, W, K, xr)
    xd = pn.hadamard(torch.from_numpy(x).to(dev), block)
    assert np.array_equal(xd.cpu().numpy().view(np.uint16), xr.view(np.uint16))
    y = pn.gemv(pn_type, torch.from_numpy(W).to(dev), K, xd, workspace=pn.Workspace(N, dev)).cpu().numpy()
    assert_gemv_close(y, y_ref, abs_sum)
