"""pn_gemv_noalloc: the GEMV for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all (code in a host callback or on a
stream owned by another runtime, plugins whose framework owns every
allocation, serving loops that must not touch the allocator after loading), so
they cannot hand pn_gemv its workspace.  pn_gemv_noalloc takes its scratch from
a fixed array in the library instead.  These tests call it through the C ABI,
several times in a row with different shapes (the array keeps the previous
call's contents), and check every result against the CPU oracle within the
GEMV tolerance used by every other GPU test; after a call that gave up on a
device-side wait (leaving words of the array set), the next call must still be
right; and a call refused on its arguments must enqueue nothing.  The file
name makes pytest collect it last; it also passes when run on its own in a
fresh process.
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


def call_noalloc(pn, pn_type, W, K, x, y, M=None, stream=None):
    fn = pn.lib().pn_gemv_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    s = stream if stream is not None else torch.cuda.current_stream()
    return fn(pn_type, W.data_ptr(), W.shape[0], K, x.data_ptr(), x.shape[0] if M is None else M,
              y.data_ptr(), s.cuda_stream)


def case(oracle, pn_type, N, K, M, seed):
    from bit_weight_only_pn_gb300 import synth
    w = synth.weights(seed, N, K)
    x = synth.activations(seed + 8, M, K)
    W = oracle.pack(pn_type, w)
    y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
    dev = torch.device("cuda", 0)
    return torch.from_numpy(W).to(dev), torch.from_numpy(x).to(dev), y_ref, abs_sum


def test_noalloc_matches_oracle_on_calls_in_a_row(pn, oracle):
    dev = torch.device("cuda", 0)
    # different shapes in a row; all split tiles across thread blocks, so each
    # call runs on hand-off words, counters and slots an earlier one used (the
    # first two go through the multi-token kernel, the third through the
    # one-token kernel, the fourth through the multi-token kernel's 16-token
    # form, the last through the two-token form)
    for pn_type, N, K, M, seed in ((PN3T, 2000, 40 * 80, 3, 0xA11), (PN4T, 777, 24 * 64, 8, 0xA12),
                                   (PN3T, 3001, 64 * 80, 1, 0xA13), (PN4T, 1500, 32 * 64, 16, 0xA14),
                                   (PN4T, 2100, 272 * 64, 2, 0xA15)):
        Wd, xd, y_ref, abs_sum = case(oracle, pn_type, N, K, M, seed)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        assert call_noalloc(pn, pn_type, Wd, K, xd, y) == 0
        torch.cuda.synchronize()
        assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)


def test_noalloc_after_a_call_that_gave_up(pn, oracle):
    # A call whose device-side waits run out (testing aid: the first step's
    # bytes are announced but never copied) leaves hand-off words and the
    # status word of the shared array set; the next call must clear what it
    # needs and be right.  The waits are bounded, so nothing hangs.
    dev = torch.device("cuda", 0)
    for pn_type, N, K, M, seed in ((PN3T, 3001, 64 * 80, 1, 0xA21), (PN4T, 2000, 40 * 64, 8, 0xA22)):
        Wd, xd, y_ref, abs_sum = case(oracle, pn_type, N, K, M, seed)
        y = torch.zeros((M, N), dtype=torch.float32, device=dev)
        try:
            pn.set_wait_timeout_ns(2_000_000)
            pn.set_test_stall(True)
            assert call_noalloc(pn, pn_type, Wd, K, xd, y) == 0
            torch.cuda.synchronize()
        finally:
            pn.set_test_stall(False)
            pn.set_wait_timeout_ns(1_000_000_000)
        y.fill_(float("nan"))
        assert call_noalloc(pn, pn_type, Wd, K, xd, y) == 0
        torch.cuda.synchronize()
        assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)


def _cudart():
    for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("CUDA runtime library not found for the capture check")


def _captured_nodes(cudart, stream, fn):
    """Number of graph nodes that `fn` enqueues on `stream` (captured, never run)."""
    h = ctypes.c_void_p(stream.cuda_stream)
    assert cudart.cudaStreamBeginCapture(h, 2) == 0          # relaxed capture mode
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        assert cudart.cudaStreamEndCapture(h, ctypes.byref(graph)) == 0
    n = ctypes.c_size_t(0)
    assert cudart.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    cudart.cudaGraphDestroy(graph)
    return n.value


def test_noalloc_refused_call_enqueues_nothing(pn, oracle):
    dev = torch.device("cuda", 0)
    Wd, xd, y_ref, abs_sum = case(oracle, PN3T, 1000, 64 * 80, 1, 0xA31)
    y = torch.zeros((1, 1000), dtype=torch.float32, device=dev)
    assert call_noalloc(pn, PN3T, Wd, 64 * 80, xd, y) == 0          # set-up done before any capture
    torch.cuda.synchronize()
    cudart = _cudart()
    cudart.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
    cudart.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    cudart.cudaGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    cudart.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
    s = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    # control: the regular entry point's launch is seen as a node
    ws = pn.Workspace(1000, dev)
    torch.cuda.synchronize()
    assert _captured_nodes(cudart, s, lambda: pn.gemv(PN3T, Wd, 64 * 80, xd, y=y, workspace=ws, stream=s)) >= 1
    rcs = []
    bad = [dict(M=0), dict(M=17), dict(K=64 * 80 + 1), dict(type=7)]
    for b in bad:
        def go(b=b):
            rcs.append(call_noalloc(pn, b.get("type", PN3T), Wd, b.get("K", 64 * 80), xd, y, M=b.get("M"),
                                    stream=s))
        assert _captured_nodes(cudart, s, go) == 0
    assert all(rc == 1 for rc in rcs), rcs                      # PN_EINVAL, nothing enqueued
    # an output overlapping the weights is refused the same way
    rcs.clear()

    def go_alias():
        fn = pn.lib().pn_gemv_noalloc
        rcs.append(fn(PN3T, Wd.data_ptr(), 1000, 64 * 80, xd.data_ptr(), 1, Wd.data_ptr(), s.cuda_stream))
    assert _captured_nodes(cudart, s, go_alias) == 0
    assert rcs == [1]
    # and the array is still usable afterwards
    y.fill_(float("nan"))
    assert call_noalloc(pn, PN3T, Wd, 64 * 80, xd, y) == 0
    torch.cuda.synchronize()
    assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)
