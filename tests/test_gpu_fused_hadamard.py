"""GPU parity of the GEMV with the Hadamard rotation fused into it.

pn_gemv_hadamard / pn_gemv_layer_hadamard rotate the activations inside the
GEMV launch (the runtime rotation of the tensorless docs, "How Qwen3.8-27B-PN3
uses it") instead of in a separate pn_hadamard launch.  Three checks:

* the rotated activations themselves, bit for bit: with identity weights
  (row j holds a single weight 1.0 at column j, which the signed-scale rule
  encodes exactly) every output y[m][j] is one rotated activation times 1.0
  plus zeros, so y equals the oracle's rotation exactly (as values: the sign
  of a zero may differ);
* y bit-identical to pn_hadamard followed by pn_gemv on the same device where
  both run the same kernel (same split, same summation order): single tensors
  and one-token layers;
* y within the GEMV tolerance of the oracle's rotation followed by the
  oracle's GEMV.

The inputs span several tiles, a ragged last tile and a thread-block split of
every row, and the refusals (M above 2, blocks out of range, activations that
do not fit shared memory) return their status without a launch.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import PN3T, PN4T, assert_gemv_close

pytestmark = pytest.mark.gpu

EINVAL, EUNSUPPORTED = 1, 3


@pytest.fixture(scope="module")
def pn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_pn_gb300 import build, pn as pn_mod
    build.build()
    pn_mod.lib()
    return pn_mod


def dev():
    return torch.device("cuda", 0)


def tensor_case(oracle, pn_type, N, K, M, seed):
    from bit_weight_only_pn_gb300 import synth
    W = oracle.pack(pn_type, synth.weights(seed, N, K))
    x = synth.activations(seed + 1, M, K)
    return W, x


@pytest.mark.parametrize("pn_type,K", [(PN3T, 5120), (PN4T, 6144)])
@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("block", [32, 256, 1024])
def test_identity_weights_read_back_the_rotation(pn, oracle, pn_type, K, M, block):
    # N = K identity rows: y[m][j] = rotated x[m][j] exactly
    w = np.eye(K, dtype=np.float32)
    W = oracle.pack(pn_type, w)
    x = np.random.default_rng(K + M + block).standard_normal((M, K)).astype(np.float16)
    want = oracle.hadamard(x, block).astype(np.float32)
    y = pn.gemv_hadamard(pn_type, torch.from_numpy(W).to(dev()), K, torch.from_numpy(x).to(dev()), block,
                         workspace=pn.Workspace(K, dev())).cpu().numpy()
    assert np.array_equal(y, want)


@pytest.mark.parametrize("pn_type,N,K,M", [(PN3T, 1000, 5120, 1), (PN3T, 1000, 5120, 2), (PN4T, 777, 17408, 1),
                                           (PN4T, 777, 17408, 2), (PN3T, 24, 40960, 1), (PN4T, 2100, 2048, 1),
                                           (PN4T, 2100, 2048, 2)])
@pytest.mark.parametrize("block", [64, 1024])
def test_fused_matches_two_launches_and_oracle(pn, oracle, pn_type, N, K, M, block):
    W, x = tensor_case(oracle, pn_type, N, K, M, 0xF00 + N + K + M)
    Wd, xd = torch.from_numpy(W).to(dev()), torch.from_numpy(x).to(dev())
    ws = pn.Workspace(N, dev())
    x_keep = xd.clone()
    y = pn.gemv_hadamard(pn_type, Wd, K, xd, block, workspace=ws)
    assert torch.equal(xd, x_keep)                                     # x is read, not modified
    y2 = pn.gemv(pn_type, Wd, K, pn.hadamard(xd, block), workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    y_ref, abs_sum = oracle.gemv(pn_type, W, K, oracle.hadamard(x, block))
    assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)


def layer_case(oracle, M, shapes, seed):
    from bit_weight_only_pn_gb300 import synth
    ents, host = [], []
    for i, (t, K, N) in enumerate(shapes):
        W = oracle.pack(t, synth.weights(seed + 2 * i, N, K))
        x = synth.activations(seed + 2 * i + 1, M, K)
        host.append((t, W, K, x))
        ents.append((t, torch.from_numpy(W).to(dev()), K, torch.from_numpy(x).to(dev()),
                     torch.full((M, N), float("nan"), dtype=torch.float32, device=dev())))
    return ents, host


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("block", [128, 1024])
def test_fused_layer(pn, oracle, M, block):
    # mixed formats and widths, as in one decoder layer (sizes reduced)
    shapes = [(PN3T, 5120, 1200), (PN4T, 5120, 200), (PN4T, 6144, 999), (PN4T, 17408, 640), (PN3T, 5120, 64)]
    ents, host = layer_case(oracle, M, shapes, 0xFA0 + M + block)
    ws = pn.Workspace(sum(e[1].shape[0] for e in ents), dev())
    pn.gemv_layer_hadamard(ents, M, block, workspace=ws)
    two = [(t, W, K, pn.hadamard(x, block), torch.empty_like(y)) for t, W, K, x, y in ents]
    pn.gemv_layer(two, M, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    for (t, W, K, x), e, f in zip(host, ents, two):
        y = e[4].cpu().numpy()
        y_ref, abs_sum = oracle.gemv(t, W, K, oracle.hadamard(x, block))
        assert_gemv_close(y, y_ref, abs_sum)
        if M == 1:
            # same kernel, split and order as the two-launch path (at M = 2
            # this layer's two-launch GEMV runs the batch kernel instead,
            # whose sums are ordered differently)
            assert np.array_equal(y.view(np.uint32), f[4].cpu().numpy().view(np.uint32))
        else:
            assert_gemv_close(f[4].cpu().numpy(), y_ref, abs_sum)


def test_fused_full_size_layer_sampled(pn, oracle):
    # the 27B-class decoder layer at full size, M = 1, block 1024: bit-identical
    # to the two-launch path everywhere, and the oracle on sampled rows
    from bit_weight_only_pn_gb300 import synth
    tensors = synth.CONFIGS[3]["tensors"]
    ents, rng = [], np.random.default_rng(0xFB)
    rows, host = [], []
    for e, (t, K, N) in enumerate(tensors):
        w = torch.from_numpy(synth.weights(synth.weight_seed(3, e), N, K)).to(dev())
        W = pn.pack(t, w)
        x = synth.activations(synth.x_seed(3, e), 1, K)
        ents.append((t, W, K, torch.from_numpy(x).to(dev()), torch.empty((1, N), dtype=torch.float32,
                                                                           device=dev())))
        r = np.unique(np.concatenate([rng.integers(0, N, 40), [0, N - 1]]))
        rows.append(r)
        host.append((W[torch.from_numpy(r).to(dev())].cpu().numpy(), x))
    ws = pn.Workspace(sum(N for _, _, N in tensors), dev())
    pn.gemv_layer_hadamard(ents, 1, 1024, workspace=ws)
    two = [(t, W, K, pn.hadamard(x, 1024), torch.empty_like(y)) for t, W, K, x, y in ents]
    pn.gemv_layer(two, 1, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    for (t, _, K, _, y), f, r, (Wr, x) in zip(ents, two, rows, host):
        yg = y.cpu().numpy()
        assert np.array_equal(yg.view(np.uint32), f[4].cpu().numpy().view(np.uint32))
        y_ref, abs_sum = oracle.gemv(t, Wr, K, oracle.hadamard(x, 1024))
        assert_gemv_close(yg[:, r], y_ref, abs_sum)


def test_fused_refusals(pn, oracle):
    W, x = tensor_case(oracle, PN3T, 64, 5120, 3, 0xFC0)
    Wd, xd = torch.from_numpy(W).to(dev()), torch.from_numpy(x).to(dev())
    ws = pn.Workspace(64, dev())
    y = torch.zeros((3, 64), dtype=torch.float32, device=dev())
    cases = [(xd, 1024, EUNSUPPORTED),            # three tokens
             (xd[:1], 16, EINVAL), (xd[:1], 2048, EINVAL), (xd[:1], 96, EINVAL),
             (xd[:1], 4096, EINVAL)]              # 4096 does not divide 5120
    for xs, block, want in cases:
        with pytest.raises(pn.PnError) as err:
            pn.gemv_hadamard(PN3T, Wd, 5120, xs, block, y=y[:xs.shape[0]], workspace=ws)
        assert err.value.status == want, (xs.shape, block)
    # rows of more than 64 chunks of 8 blocks
    W2, x2 = tensor_case(oracle, PN4T, 16, 65 * 512, 1, 0xFC1)
    with pytest.raises(pn.PnError) as err:
        pn.gemv_hadamard(PN4T, torch.from_numpy(W2).to(dev()), 65 * 512, torch.from_numpy(x2).to(dev()), 512,
                         workspace=ws)
    assert err.value.status == EUNSUPPORTED
    # two tokens of 40960 activations (160 KiB rotated) do not fit beside the ring
    W3, x3 = tensor_case(oracle, PN3T, 16, 40960, 2, 0xFC2)
    with pytest.raises(pn.PnError) as err:
        pn.gemv_hadamard(PN3T, torch.from_numpy(W3).to(dev()), 40960, torch.from_numpy(x3).to(dev()), 1024,
                         workspace=ws)
    assert err.value.status == EUNSUPPORTED
    torch.cuda.synchronize()
    assert ws.status() == 0


@pytest.mark.parametrize("rotated", [False, True])
def test_resident_wait_timeout_reports_status(pn, oracle, rotated):
    # A layer call (activations resident, rotated or copied) whose first weight
    # copy is announced but never made (testing aid): the waits give up after
    # the limit, the blocks let their other copies land, PN_ETIMEOUT is
    # reported, and the next call on the same workspace is right.
    shapes = [(PN3T, 5120, 640), (PN4T, 6144, 320)]
    ents, host = layer_case(oracle, 1, shapes, 0xFD0 + rotated)
    ws = pn.Workspace(sum(e[1].shape[0] for e in ents), dev())
    call = (lambda: pn.gemv_layer_hadamard(ents, 1, 1024, workspace=ws)) if rotated else \
        (lambda: pn.gemv_layer(ents, 1, workspace=ws))
    try:
        pn.set_wait_timeout_ns(2_000_000)
        pn.set_test_stall(True)
        call()
        assert ws.status() == 5
    finally:
        pn.set_test_stall(False)
        pn.set_wait_timeout_ns(1_000_000_000)
    for e in ents:
        e[4].fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    assert ws.status() == 0
    for (t, W, K, x), e in zip(host, ents):
        xr = oracle.hadamard(x, 1024) if rotated else x
        y_ref, abs_sum = oracle.gemv(t, W, K, xr)
        assert_gemv_close(e[4].cpu().numpy(), y_ref, abs_sum)


def test_fused_empty_rows(pn, oracle):
    # N = 0 is a no-op that returns PN_OK and writes nothing
    W, x = tensor_case(oracle, PN3T, 16, 5120, 1, 0xFE0)
    xd = torch.from_numpy(x).to(dev())
    Wd = torch.from_numpy(W).to(dev())[:0]
    y = torch.full((1, 1), 7.0, dtype=torch.float32, device=dev())
    pn.gemv_hadamard(PN3T, Wd, 5120, xd, 1024, y=y[:, :0], workspace=pn.Workspace(16, dev()))
    torch.cuda.synchronize()
    assert y.item() == 7.0


@pytest.mark.parametrize("M", [1, 2])
def test_layer_whose_activations_do_not_fit(pn, oracle, M):
    # three short 17408-wide tensors: a block's range spans all of them, whose
    # activations (M x 3 x 34 KB) do not fit beside the full ring, so the
    # one-token launch stages them per unit (M = 1) or the call goes to the
    # batch kernel (M = 2); the fused-rotation call still fits at M = 1
    shapes = [(PN4T, 17408, 40), (PN4T, 17408, 24), (PN4T, 17408, 33)]
    ents, host = layer_case(oracle, M, shapes, 0xFF0 + M)
    ws = pn.Workspace(200, dev())
    pn.gemv_layer(ents, M, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    for (t, W, K, x), e in zip(host, ents):
        y_ref, abs_sum = oracle.gemv(t, W, K, x)
        assert_gemv_close(e[4].cpu().numpy(), y_ref, abs_sum)
    if M == 1:
        for e in ents:
            e[4].fill_(float("nan"))
        pn.gemv_layer_hadamard(ents, M, 1024, workspace=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        for (t, W, K, x), e in zip(host, ents):
            y_ref, abs_sum = oracle.gemv(t, W, K, oracle.hadamard(x, 1024))
            assert_gemv_close(e[4].cpu().numpy(), y_ref, abs_sum)
