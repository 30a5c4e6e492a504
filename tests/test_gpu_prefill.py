"""GPU parity of the prefill path (large M) with the CPU oracle.

pn_unpack_f16 rebuilds PN rows as fp16 (the exact decode rounded once, to
nearest even): compared bit for bit, on random blocks over the whole fp16
scale range and on hand-picked rounding cases.  pn_gemm_f16 (tcgen05 tensor
cores, fp32 accumulation over K in 16-wide steps) and pn_prefill (rebuild +
GEMM, chunk by chunk) are compared element by element with the oracle's fp64
GEMM of the same fp16 weights, within the bound the arithmetic gives:
(K/16 + 16) * 2^-24 * sum_k |w16 x| + 1e-6.  Shapes span several 128-row
and 256-token tiles with ragged tails in rows, tokens and K (K not a multiple
of the 64-wide staging step), M = 1, and prefill scratch of one and two row
tiles so that several chunks run; a full-size case is checked on sampled rows
and tokens.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import GEOMETRY, PN3T, PN4T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_pn_gb300 import build, pn as pn_mod
    build.build()
    pn_mod.lib()
    return pn_mod


DEV = torch.device("cuda", 0)


def assert_gemm_close(y, y_ref, abs_sum, K):
    y = np.asarray(y, dtype=np.float64)
    bound = (K / 16 + 16) * 2.0 ** -24 * abs_sum + 1e-6
    err = np.abs(y - y_ref)
    assert np.all(np.isfinite(y)), "non-finite output"
    bad = err > bound
    assert not bad.any(), f"{int(bad.sum())} outputs out of bound; worst excess {float((err - bound).max())}"


def random_pn(oracle, rng, pn_type, N, K):
    w = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    return oracle.pack(pn_type, w)


def activations(rng, M, K):
    return rng.standard_normal((M, K)).astype(np.float16)


@pytest.mark.parametrize("pn_type", [PN3T, PN4T])
def test_unpack_f16_bit_exact(pn, oracle, pn_type):
    rng = np.random.default_rng(71 + pn_type)
    bpb = GEOMETRY[pn_type][0]
    N, nb = 77, 13
    W = random_pn(oracle, rng, pn_type, N, nb * bpb)
    # scales over the whole fp16 range (incl. subnormal, overflowing products, -0)
    raw = W.reshape(N, nb, 34)
    dbits = rng.integers(0, 0x7C00, size=(N, nb)) | (rng.integers(0, 2, size=(N, nb)) << 15)
    raw[:, :, 0] = dbits & 0xFF
    raw[:, :, 1] = dbits >> 8
    raw[0, 0, :2] = [0x01, 0xBC]          # -(1 + 2^-10): ties to even in both directions
    raw[1, 0, :2] = [0xFF, 0x7B]          # 65504: products overflow to inf
    W = raw.reshape(N, nb * 34)
    got = pn.unpack_f16(pn_type, torch.from_numpy(W).to(DEV), nb * bpb).cpu().numpy()
    want = oracle.unpack_f16(pn_type, W, nb * bpb)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("N,K,M", [(128, 64, 256), (300, 640, 300), (129, 1280, 1), (257, 2048, 257),
                                   (64, 968, 513), (1000, 200, 40)])
def test_gemm_f16_matches_oracle(pn, oracle, N, K, M):
    rng = np.random.default_rng(N * 7 + K + M)
    w16 = (0.05 * rng.standard_normal((N, K))).astype(np.float16)
    x = activations(rng, M, K)
    y = pn.gemm_f16(torch.from_numpy(w16).to(DEV), torch.from_numpy(x).to(DEV)).cpu().numpy()
    y_ref, abs_sum = oracle.gemm_f16(w16, x)
    assert_gemm_close(y, y_ref, abs_sum, K)


def test_gemm_f16_output_stride_and_status(pn, oracle):
    # y rows longer than N (ldy > N): the columns past N stay untouched
    rng = np.random.default_rng(5)
    N, K, M = 200, 320, 70
    w16 = (0.05 * rng.standard_normal((N, K))).astype(np.float16)
    x = activations(rng, M, K)
    y = torch.full((M, N + 9), 7.0, dtype=torch.float32, device=DEV)
    ws = pn.Workspace(N, DEV)
    wd, xd = torch.from_numpy(w16).to(DEV), torch.from_numpy(x).to(DEV)   # kept alive past the launch
    rc = pn.lib().pn_gemm_f16(wd.data_ptr(), N, K, xd.data_ptr(), M, y.data_ptr(), N + 9, ws.ptr, ws.nbytes,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert ws.status() == 0
    out = y.cpu().numpy()
    assert np.all(out[:, N:] == 7.0)
    y_ref, abs_sum = oracle.gemm_f16(w16, x)
    assert_gemm_close(out[:, :N], y_ref, abs_sum, K)


@pytest.mark.parametrize("pn_type,N,K,M,scratch_rows", [(PN3T, 300, 640, 260, 128), (PN4T, 517, 1024, 33, 256),
                                                         (PN3T, 128, 5120, 1, 128), (PN4T, 700, 576, 300, 1024)])
def test_prefill_matches_oracle(pn, oracle, pn_type, N, K, M, scratch_rows):
    rng = np.random.default_rng(N + K + M)
    W = random_pn(oracle, rng, pn_type, N, K)
    x = activations(rng, M, K)
    scratch = torch.empty(scratch_rows * K, dtype=torch.float16, device=DEV)
    ws = pn.Workspace(N, DEV)
    y = pn.prefill(pn_type, torch.from_numpy(W).to(DEV), K, torch.from_numpy(x).to(DEV), scratch=scratch,
                   workspace=ws).cpu().numpy()
    assert ws.status() == 0
    y_ref, abs_sum = oracle.gemm_f16(oracle.unpack_f16(pn_type, W, K), x)
    assert_gemm_close(y, y_ref, abs_sum, K)


def test_prefill_full_size_sampled(pn, oracle):
    # pn3t 5120 -> 17408 (an FFN gate/up tensor) for a 1024-token prefill,
    # checked on sampled rows (both ends of every chunk edge) and tokens
    from bit_weight_only_pn_gb300 import synth
    N, K, M = 17408, 5120, 1024
    W = oracle.pack(PN3T, synth.weights(synth.weight_seed(1, 0), N, K))
    x = synth.activations(synth.x_seed(1, 0) + 77, M, K)
    scratch = torch.empty(4096 * K, dtype=torch.float16, device=DEV)
    y = pn.prefill(PN3T, torch.from_numpy(W).to(DEV), K, torch.from_numpy(x).to(DEV), scratch=scratch).cpu().numpy()
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 127, 128, 4095, 4096, 8191, 8192, N - 129, N - 1],
                                     rng.integers(0, N, size=60)]))
    toks = np.unique(np.concatenate([[0, 255, 256, M - 1], rng.integers(0, M, size=20)]))
    y_ref, abs_sum = oracle.gemm_f16(oracle.unpack_f16(PN3T, W[rows], K), x[toks])
    assert_gemm_close(y[np.ix_(toks, rows)], y_ref, abs_sum, K)


def test_gemm_wait_timeout_reports_status(pn, oracle):
    # Every CTA announces its first K slice's bytes but never copies them (a
    # barrier phase nothing completes): the MMA thread's wait must give up
    # after the time limit, the CTA must let its other copies land, free its
    # TMEM and return, the call must report PN_ETIMEOUT, and the next call
    # must be correct.
    rng = np.random.default_rng(9)
    N, K, M = 512, 1024, 300
    w16 = (0.05 * rng.standard_normal((N, K))).astype(np.float16)
    x = activations(rng, M, K)
    wd, xd = torch.from_numpy(w16).to(DEV), torch.from_numpy(x).to(DEV)
    ws = pn.Workspace(N, DEV)
    try:
        pn.set_wait_timeout_ns(2_000_000)
        pn.set_test_stall(True)
        pn.gemm_f16(wd, xd, workspace=ws)
        assert ws.status() == 5
    finally:
        pn.set_test_stall(False)
        pn.set_wait_timeout_ns(1_000_000_000)
    y = pn.gemm_f16(wd, xd, workspace=ws).cpu().numpy()
    assert ws.status() == 0
    y_ref, abs_sum = oracle.gemm_f16(w16, x)
    assert_gemm_close(y, y_ref, abs_sum, K)
