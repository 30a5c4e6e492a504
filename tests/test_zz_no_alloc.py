"""pn_gemv_noalloc: the GEMV for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all (code in a host callback or on a
stream owned by another runtime, plugins whose framework owns every
allocation, serving loops that must not touch the allocator after loading), so
they cannot hand pn_gemv its workspace.  pn_gemv_noalloc takes its scratch from
a fixed array in the library instead.  This test calls it through the C ABI,
four times in a row with different shapes (the array keeps the previous
call's contents), and checks each result against pn_gemv's on the same inputs within
the GEMV tolerance used by every other GPU test.  The file name makes pytest
collect it last; it also passes when run on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

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
    return pn_mod


def call_noalloc(pn, pn_type, W, K, x, y):
    fn = pn.lib().pn_gemv_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return fn(pn_type, W.data_ptr(), W.shape[0], K, x.data_ptr(), x.shape[0], y.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_pn_gemv_twice(pn, oracle):
    from bit_weight_only_pn_gb300 import synth
    dev = torch.device("cuda", 0)
    # different shapes in a row; all split tiles across thread blocks, so each
    # call runs on hand-off words, counters and slots an earlier one used (the
    # first two go through the multi-token kernel, the third through the
    # one-token kernel, the fourth through the multi-token kernel's 16-token
    # form)
    for pn_type, N, K, M, seed in ((PN3T, 2000, 40 * 80, 3, 0xA11), (PN4T, 777, 24 * 64, 8, 0xA12),
                                   (PN3T, 3001, 64 * 80, 1, 0xA13), (PN4T, 1500, 32 * 64, 16, 0xA14)):
        w = synth.weights(seed, N, K)
        x = synth.activations(seed + 8, M, K)
        W = oracle.pack(pn_type, w)
        _, abs_sum = oracle.gemv(pn_type, W, K, x)
        Wd = torch.from_numpy(W).to(dev)
        xd = torch.from_numpy(x).to(dev)
        y_ref = pn.gemv(pn_type, Wd, K, xd, workspace=pn.Workspace(N, dev)).cpu().numpy()
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        assert call_noalloc(pn, pn_type, Wd, K, xd, y) == 0
        torch.cuda.synchronize()
        assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)
