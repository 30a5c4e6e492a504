"""GPU parity on the zero code: blocks whose weights are almost all n = z.

Format page, "Zero is a code, and the scale has a sign": a mid-tread code set
has an exact zero, and most weights of a block may sit on it.  The GEMV bound
|y - y_ref| <= 1e-5 * sum_k |w_k x_k| + 1e-6 counts only the non-zero
weights, so a kernel must not let zero-code weights carry rounding error: a
computation of sum n*x - z*sum x cancels, and its error grows with
sum |x| over the whole block.  These inputs (one full-range step per block,
at most two other non-zero steps, tiny x there and x up to 1e3 on every zero
code; scales from 2^-14 to about 8 and a few fp16 subnormals) make that error
far larger than the bound.  Every output is compared with the oracle, for
every kernel and every token count class, at the pages' widths.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import GEOMETRY, PN3T, PN4T, assert_gemv_close, zero_code_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_pn_gb300 import build, pn as pn_mod
    build.build()
    pn_mod.lib()
    return pn_mod


@pytest.fixture(scope="module")
def dev(pn):
    return torch.device("cuda", 0)


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


@pytest.mark.parametrize("algo", ["tc", "cuda_core", "cuda_core_staged"])
@pytest.mark.parametrize("pn_type,K", [(PN3T, 5120), (PN4T, 5120), (PN4T, 17408)])
def test_zero_code_blocks(pn, dev, oracle, pn_type, K, algo):
    a = {"tc": pn.ALGO_TENSOR_CORE, "cuda_core": pn.ALGO_CUDA_CORE,
         "cuda_core_staged": pn.ALGO_CUDA_CORE_STAGED}[algo]
    bpb = GEOMETRY[pn_type][0]
    N = 1000
    rng = np.random.default_rng(0x2E40 + K + pn_type)
    w, x16 = zero_code_case(rng, pn_type, N, K // bpb, 16)
    W = oracle.pack(pn_type, w)
    Wd = to_dev(W, dev)
    ws = pn.Workspace(N, dev)
    for M in (1, 2, 3, 8, 16):
        if algo == "cuda_core_staged" and M > 8:
            continue
        x = x16[:M]
        y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
        y = pn.gemv(pn_type, Wd, K, to_dev(x, dev), workspace=ws, algo=a).cpu().numpy()
        assert ws.status() == 0
        assert_gemv_close(y, y_ref, abs_sum)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_zero_code_layer(pn, dev, oracle, M):
    # the fused layer call over mixed types, every output compared
    shapes = [(PN3T, 5120, 700), (PN4T, 17408, 300), (PN4T, 5120, 129), (PN3T, 5120, 61)]
    entries, refs = [], []
    rng = np.random.default_rng(0x2E41 + M)
    for t, K, N in shapes:
        w, x = zero_code_case(rng, t, N, K // GEOMETRY[t][0], M)
        W = oracle.pack(t, w)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        entries.append((t, to_dev(W, dev), K, to_dev(x, dev), y))
        refs.append(oracle.gemv(t, W, K, x))
    ws = pn.Workspace(sum(s[2] for s in shapes), dev)
    pn.gemv_layer(entries, M, workspace=ws)
    assert ws.status() == 0
    for (t, Wd, K, xd, y), (y_ref, abs_sum) in zip(entries, refs):
        assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)
