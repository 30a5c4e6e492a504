"""GPU parity of the device GPTQ-style quantiser (pn_gptq) with the CPU oracle.

Both sides run the same fp64 / fp32 IEEE operations in the same order (each
sum in index order, nothing fused), so the PN bytes must be identical: the
scales, and every code, including the ones the error feedback moved.  Shapes
cover both formats, row counts that do not fill the last group of rows, and
correlated calibration inputs (the case where the feedback matters); a
diagonal Hessian reduces GPTQ to the round-to-nearest packer, and a singular
one is refused.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import PN3T, PN4T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_pn_gb300 import build, pn as pn_mod
    build.build()
    pn_mod.lib()
    return pn_mod


def case(seed, N, K, n):
    rng = np.random.default_rng(seed)
    w = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    A = rng.standard_normal((K, K)) * (0.3 / np.sqrt(K / 64)) + np.eye(K)
    X = (rng.standard_normal((n, K)) @ A).astype(np.float32)
    return w, X


@pytest.mark.parametrize("pn_type,N,K,n", [(PN3T, 13, 160, 300), (PN3T, 33, 320, 500), (PN3T, 8, 640, 700),
                                           (PN4T, 17, 256, 400), (PN4T, 64, 512, 600), (PN4T, 3, 64, 80)])
def test_gptq_bytes_equal_oracle(pn, oracle, pn_type, N, K, n):
    w, X = case(N * 1000 + K + n, N, K, n)
    dev = torch.device("cuda", 0)
    got = pn.gptq(pn_type, torch.from_numpy(w).to(dev), torch.from_numpy(X).to(dev), 0.01).cpu().numpy()
    want = oracle.gptq(pn_type, w, X, 0.01)
    assert np.array_equal(got, want)
    # and the feedback did something: not all equal to round-to-nearest
    assert not np.array_equal(got, oracle.pack(pn_type, w))


def test_gptq_diagonal_hessian_is_rtn(pn):
    rng = np.random.default_rng(7)
    dev = torch.device("cuda", 0)
    for pn_type, K in ((PN3T, 160), (PN4T, 128)):
        w = (0.02 * rng.standard_normal((11, K))).astype(np.float32)
        X = np.diag(rng.uniform(0.5, 2.0, K)).astype(np.float32)
        got = pn.gptq(pn_type, torch.from_numpy(w).to(dev), torch.from_numpy(X).to(dev), 0.01)
        assert torch.equal(got, pn.pack(pn_type, torch.from_numpy(w).to(dev)))


def test_gptq_refusals(pn):
    dev = torch.device("cuda", 0)
    w = torch.zeros((4, 160), dtype=torch.float32, device=dev)
    with pytest.raises(pn.PnError) as err:                     # H = 0: not positive definite
        pn.gptq(PN3T, w, torch.zeros((10, 160), dtype=torch.float32, device=dev), 0.01)
    assert err.value.status == 1
    W = pn.gptq(PN3T, w[:0], torch.ones((10, 160), dtype=torch.float32, device=dev), 0.01)
    assert W.shape == (0, 2 * 34)
    torch.cuda.synchronize()
