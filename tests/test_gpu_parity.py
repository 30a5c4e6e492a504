"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Decode and pack are compared byte for byte; GEMV outputs within
|y - y_ref| <= 1e-5 * sum_k |w_k x_k| + 1e-6 per element.  Inputs are the
seeded synthetic weights and activations of the workloads (N(0, 0.02) weights
quantised by the oracle's packer, fp16 N(0, 1) activations); every expected
value comes from the oracle.  Full-size workloads are checked on sampled rows
(rows are independent), computed by the oracle from the same packed bytes.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import GEOMETRY, PN3T, PN4T, assert_gemv_close

pytestmark = pytest.mark.gpu

TYPES = (PN3T, PN4T)


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


def to_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def synth_case(oracle, pn_type, N, K, M, seed):
    from bit_weight_only_pn_gb300 import synth
    w = synth.weights(seed, N, K)
    x = synth.activations(seed + 8, M, K)
    return oracle.pack(pn_type, w), x


# ----------------------------------------------------------------- decode ----

@pytest.mark.parametrize("pn_type", TYPES)
def test_unpack_bit_exact_random(pn, dev, oracle, pn_type):
    bpb = GEOMETRY[pn_type][0]
    for N, nb in ((257, 13), (64, 64), (3, 1)):
        W, _ = synth_case(oracle, pn_type, N, nb * bpb, 1, 0x51 + nb)
        got = pn.unpack(pn_type, to_dev(W, dev), nb * bpb).cpu().numpy()
        want = oracle.unpack(pn_type, W, nb * bpb)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("pn_type", TYPES)
def test_unpack_bit_exact_every_scale_and_bit(pn, dev, oracle, pn_type):
    # every finite fp16 scale (subnormals and -0 included) with random code
    # words, unused bits set at random
    bpb = GEOMETRY[pn_type][0]
    rng = np.random.default_rng(99)
    bits = np.arange(65536, dtype=np.uint16)
    bits = bits[np.isfinite(bits.view(np.float16))]
    W = rng.integers(0, 256, size=(bits.size, 34), dtype=np.uint8)
    W[:, 0:2] = bits.view(np.uint8).reshape(-1, 2)
    got = pn.unpack(pn_type, to_dev(W, dev), bpb).cpu().numpy()
    want = oracle.unpack(pn_type, W, bpb)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------------------- pack ----

@pytest.mark.parametrize("pn_type", TYPES)
def test_pack_byte_exact(pn, dev, oracle, pn_type):
    from bit_weight_only_pn_gb300 import synth
    bpb = GEOMETRY[pn_type][0]
    z = GEOMETRY[pn_type][3]
    rng = np.random.default_rng(5)
    w = synth.weights(0x77, 300, 16 * bpb)
    w[0:4] *= np.float32(1e-4)          # subnormal fp16 scales
    w[4:8] *= np.float32(1e-9)          # scales that underflow to the zero block
    w[8:12] = 0.0
    w[12:14] *= np.float32(1e9)         # scales that saturate at 65504
    w[14, :bpb] = 0.0
    w[14, 3], w[14, 9] = 0.25, -0.25    # tie of magnitudes, first index wins
    w[15] = np.round(w[15] / np.float32(2.0 ** -8)) * np.float32(2.0 ** -8)   # on a grid
    w[16, :] = -0.0
    w[17] = rng.integers(-z, z, size=w.shape[1]).astype(np.float32) * np.float32(0.5)  # rint ties
    want = oracle.pack(pn_type, w)
    got = pn.pack(pn_type, to_dev(w, dev)).cpu().numpy()
    assert np.array_equal(got, want)


# ------------------------------------------------------------------- GEMV ----

SHAPES = [(1000, 8), (16, 8), (17, 16), (129, 24), (300, 40)]   # (N, blocks per row)


@pytest.mark.parametrize("algo", ["tc", "cuda_core", "cuda_core_staged"])
@pytest.mark.parametrize("pn_type", TYPES)
def test_gemv_every_m(pn, dev, oracle, pn_type, algo):
    a = {"tc": pn.ALGO_TENSOR_CORE, "cuda_core": pn.ALGO_CUDA_CORE,
         "cuda_core_staged": pn.ALGO_CUDA_CORE_STAGED}[algo]
    bpb = GEOMETRY[pn_type][0]
    for N, nb in SHAPES:
        K = nb * bpb
        W, x16 = synth_case(oracle, pn_type, N, K, 16, 0x900 + N)
        Wd = to_dev(W, dev)
        ws = pn.Workspace(N, dev)
        for M in range(1, 9 if algo == "cuda_core_staged" else 17):
            x = x16[:M]
            y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
            y = pn.gemv(pn_type, Wd, K, to_dev(x, dev), workspace=ws, algo=a).cpu().numpy()
            assert ws.status() == 0
            assert_gemv_close(y, y_ref, abs_sum)


@pytest.mark.parametrize("pn_type", TYPES)
def test_gemv_deterministic(pn, dev, oracle, pn_type):
    bpb = GEOMETRY[pn_type][0]
    N, K = 2000, 40 * bpb
    W, x = synth_case(oracle, pn_type, N, K, 8, 0x31)
    Wd, xd = to_dev(W, dev), to_dev(x, dev)
    ws = pn.Workspace(N, dev)
    y1 = pn.gemv(pn_type, Wd, K, xd, workspace=ws).cpu().numpy()
    y2 = pn.gemv(pn_type, Wd, K, xd, workspace=ws).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
    assert_gemv_close(y1, y_ref, abs_sum)


@pytest.mark.parametrize("pn_type", TYPES)
def test_gemv_unaligned_and_ragged_k(pn, dev, oracle, pn_type):
    # K not a multiple of 8 blocks and W at a 2-byte offset: AUTO takes the
    # CUDA-core kernel; the tensor-core kernel refuses with PN_EALIGN.
    bpb = GEOMETRY[pn_type][0]
    for nb in (1, 3, 13):
        N, K = 77, nb * bpb
        W, x = synth_case(oracle, pn_type, N, K, 5, 0x40 + nb)
        y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
        ws = pn.Workspace(N, dev)
        y = pn.gemv(pn_type, to_dev(W, dev), K, to_dev(x, dev), workspace=ws).cpu().numpy()
        assert_gemv_close(y, y_ref, abs_sum)
        with pytest.raises(pn.PnError) as err:
            pn.gemv(pn_type, to_dev(W, dev), K, to_dev(x, dev), workspace=ws, algo=pn.ALGO_TENSOR_CORE)
        assert err.value.status == 2
    N, K = 200, 16 * bpb
    W, x = synth_case(oracle, pn_type, N, K, 3, 0x47)
    y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
    raw = torch.zeros(W.size + 16, dtype=torch.uint8, device=dev)
    raw[2:2 + W.size] = to_dev(W.reshape(-1), dev)
    Wodd = raw[2:2 + W.size].view(N, -1)
    y = pn.gemv(pn_type, Wodd, K, to_dev(x, dev), workspace=pn.Workspace(N, dev)).cpu().numpy()
    assert_gemv_close(y, y_ref, abs_sum)


def test_gemv_extreme_values(pn, dev, oracle):
    # largest fp16 activations and saturated scales stay finite and in tolerance
    from bit_weight_only_pn_gb300 import synth
    for pn_type in TYPES:
        bpb = GEOMETRY[pn_type][0]
        N, K = 64, 8 * bpb
        w = synth.weights(0x12, N, K) * np.float32(2000.0)
        W = oracle.pack(pn_type, w)
        x = np.full((16, K), 65504.0, dtype=np.float16)
        x[1::2] *= -1
        y_ref, abs_sum = oracle.gemv(pn_type, W, K, x)
        for a in (pn.ALGO_TENSOR_CORE, pn.ALGO_CUDA_CORE):
            y = pn.gemv(pn_type, to_dev(W, dev), K, to_dev(x, dev), workspace=pn.Workspace(N, dev), algo=a)
            assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)


def test_workspace_too_small(pn, dev, oracle):
    W, x = synth_case(oracle, PN3T, 1000, 640, 1, 3)
    ws = pn.Workspace(16, dev)
    ws.nbytes = 300
    with pytest.raises(pn.PnError) as err:
        pn.gemv(PN3T, to_dev(W, dev), 640, to_dev(x, dev), workspace=ws, algo=pn.ALGO_TENSOR_CORE)
    assert err.value.status == 1


def test_wait_timeout_reports_status(pn, dev, oracle):
    # Each thread block announces its first step's bytes but never copies them
    # (a barrier phase nothing completes): the waits must give up after the
    # time limit, the kernel must let its other copies land and return, report
    # PN_ETIMEOUT, and leave the context usable for the next call.
    N, K = 4096, 64 * 80
    W, x = synth_case(oracle, PN3T, N, K, 1, 0x99)
    Wd, xd = to_dev(W, dev), to_dev(x, dev)
    ws = pn.Workspace(N, dev)
    try:
        pn.set_wait_timeout_ns(2_000_000)
        pn.set_test_stall(True)
        pn.gemv(PN3T, Wd, K, xd, workspace=ws, algo=pn.ALGO_TENSOR_CORE)
        assert ws.status() == 5
    finally:
        pn.set_test_stall(False)
        pn.set_wait_timeout_ns(1_000_000_000)
    y = pn.gemv(PN3T, Wd, K, xd, workspace=ws, algo=pn.ALGO_TENSOR_CORE).cpu().numpy()
    assert ws.status() == 0
    y_ref, abs_sum = oracle.gemv(PN3T, W, K, x)
    assert_gemv_close(y, y_ref, abs_sum)


# ------------------------------------------------------- full-size, sampled --

def sample_rows(N, count, rng):
    edge = [0, 1, 15, 16, 127, 128, N // 2, N - 17, N - 16, N - 2, N - 1]
    rows = np.unique(np.concatenate([np.array([r for r in edge if 0 <= r < N]),
                                     rng.integers(0, N, size=count)]))
    return rows


@pytest.fixture(scope="module")
def big_inputs(oracle):
    """The single-tensor workloads at full size, packed by the oracle (cached)."""
    from bit_weight_only_pn_gb300 import synth
    cache = {}

    def get(cfg, tensor, pn_type, K, N, M):
        key = (cfg, tensor, M)
        if key not in cache:
            w = synth.weights(synth.weight_seed(cfg, tensor), N, K)
            W = oracle.pack(pn_type, w)
            del w
            x = synth.activations(synth.x_seed(cfg, tensor), M, K)
            cache[key] = (W, x)
        return cache[key]
    return get


@pytest.mark.parametrize("M", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("cfg", [0, 1, 2])
def test_gemv_full_size_sampled(pn, dev, oracle, big_inputs, cfg, M):
    from bit_weight_only_pn_gb300 import synth
    (pn_type, K, N), = synth.CONFIGS[cfg]["tensors"]
    W, x = big_inputs(cfg, 0, pn_type, K, N, 16)
    x = x[:M]
    ws = pn.Workspace(N, dev)
    y = pn.gemv(pn_type, to_dev(W, dev), K, to_dev(x, dev), workspace=ws).cpu().numpy()
    assert ws.status() == 0
    rows = sample_rows(N, 200, np.random.default_rng(cfg * 10 + M))
    y_ref, abs_sum = oracle.gemv(pn_type, W[rows], K, x)
    assert_gemv_close(y[:, rows], y_ref, abs_sum)


@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_layer_full_size_sampled(pn, dev, oracle, big_inputs, M):
    from bit_weight_only_pn_gb300 import synth
    cfg = {1: 3, 2: 3, 8: 4, 16: 5}[M]
    entries, host = [], []
    total_rows = 0
    for e, (pn_type, K, N) in enumerate(synth.LAYER_27B):
        W, x = big_inputs(3, e, pn_type, K, N, 16)
        x = x[:M]
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        entries.append((pn_type, to_dev(W, dev), K, to_dev(x, dev), y))
        host.append((pn_type, W, K, x))
        total_rows += N
    ws = pn.Workspace(total_rows, dev)
    pn.gemv_layer(entries, M, workspace=ws)
    assert ws.status() == 0
    for e, (pn_type, W, K, x) in enumerate(host):
        rows = sample_rows(W.shape[0], 60, np.random.default_rng(100 * cfg + e))
        y_ref, abs_sum = oracle.gemv(pn_type, W[rows], K, x)
        assert_gemv_close(entries[e][4].cpu().numpy()[:, rows], y_ref, abs_sum)


def test_layer_small_full_compare(pn, dev, oracle):
    # a scaled-down mixed layer compared on every output, both kernels
    shapes = [(PN3T, 640, 300), (PN4T, 512, 129), (PN3T, 1280, 1000), (PN4T, 1024, 16),
              (PN4T, 2048, 77)]
    for a in (pn.ALGO_AUTO, pn.ALGO_CUDA_CORE):
        for M in (1, 3, 8, 9, 16):
            entries, refs = [], []
            for i, (t, K, N) in enumerate(shapes):
                W, x = synth_case(oracle, t, N, K, M, 0x700 + i)
                y = torch.empty((M, N), dtype=torch.float32, device=dev)
                entries.append((t, to_dev(W, dev), K, to_dev(x, dev), y))
                refs.append(oracle.gemv(t, W, K, x))
            ws = pn.Workspace(sum(s[2] for s in shapes), dev)
            pn.gemv_layer(entries, M, workspace=ws, algo=a)
            assert ws.status() == 0
            for (t, Wd, K, xd, y), (y_ref, abs_sum) in zip(entries, refs):
                assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)


@pytest.mark.parametrize("pn_type", TYPES)
def test_gemv_long_rows_one_and_two_tokens(pn, dev, oracle, pn_type):
    # rows longer than the one-token kernel takes (more than 64 chunks of 8
    # blocks) go to the batch kernel at M = 1 and 2 as well; every output
    # against the oracle, single tensors and a mixed layer call
    bpb = GEOMETRY[pn_type][0]
    N, K = 300, 65 * 8 * bpb
    W, x = synth_case(oracle, pn_type, N, K, 2, 0x65)
    Wd = to_dev(W, dev)
    ws = pn.Workspace(N + 200, dev)
    for M in (1, 2):
        y_ref, abs_sum = oracle.gemv(pn_type, W, K, x[:M])
        y = pn.gemv(pn_type, Wd, K, to_dev(x[:M], dev), workspace=ws).cpu().numpy()
        assert ws.status() == 0
        assert_gemv_close(y, y_ref, abs_sum)
        W2, x2 = synth_case(oracle, PN3T, 200, 640, M, 0x66)
        entries = [(pn_type, Wd, K, to_dev(x[:M], dev), torch.empty((M, N), dtype=torch.float32, device=dev)),
                   (PN3T, to_dev(W2, dev), 640, to_dev(x2, dev), torch.empty((M, 200), dtype=torch.float32, device=dev))]
        pn.gemv_layer(entries, M, workspace=ws)
        assert ws.status() == 0
        assert_gemv_close(entries[0][4].cpu().numpy(), y_ref, abs_sum)
        y2_ref, a2 = oracle.gemv(PN3T, W2, 640, x2)
        assert_gemv_close(entries[1][4].cpu().numpy(), y2_ref, a2)


def test_cuda_core_staged_layer_and_limits(pn, dev, oracle):
    # the FMA-pipe kernel over a mixed layer at M = 8 (every output), and its
    # refusals: more than 8 tokens, rows longer than 64 chunks
    shapes = [(PN3T, 640, 300), (PN4T, 512, 129), (PN3T, 1280, 1000), (PN4T, 17408, 77)]
    M = 8
    entries, refs = [], []
    for i, (t, K, N) in enumerate(shapes):
        W, x = synth_case(oracle, t, N, K, M, 0x7A0 + i)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        entries.append((t, to_dev(W, dev), K, to_dev(x, dev), y))
        refs.append(oracle.gemv(t, W, K, x))
    ws = pn.Workspace(sum(s[2] for s in shapes), dev)
    pn.gemv_layer(entries, M, workspace=ws, algo=pn.ALGO_CUDA_CORE_STAGED)
    assert ws.status() == 0
    for (t, Wd, K, xd, y), (y_ref, abs_sum) in zip(entries, refs):
        assert_gemv_close(y.cpu().numpy(), y_ref, abs_sum)
    W, x = synth_case(oracle, PN3T, 64, 640, 9, 0x7B0)
    with pytest.raises(pn.PnError) as err:
        pn.gemv(PN3T, to_dev(W, dev), 640, to_dev(x, dev), workspace=ws, algo=pn.ALGO_CUDA_CORE_STAGED)
    assert err.value.status == 3
    W, x = synth_case(oracle, PN4T, 16, 65 * 512, 1, 0x7B1)
    with pytest.raises(pn.PnError) as err:
        pn.gemv(PN4T, to_dev(W, dev), 65 * 512, to_dev(x, dev), workspace=ws, algo=pn.ALGO_CUDA_CORE_STAGED)
    assert err.value.status == 3


def test_layer_host_buffers(pn, dev, oracle):
    # pn_gemv_layer_host: x from pinned host memory, y back to it, in one call;
    # device buffers partly contiguous (one copy) and partly apart, with an
    # empty entry in between
    from bit_weight_only_pn_gb300 import synth
    M = 2
    shapes = [(PN3T, 5120, 300), (PN4T, 6144, 0), (PN4T, 6144, 97), (PN3T, 640, 50)]
    host_x, host_ref, ents = [], [], []
    dx = torch.empty(sum(M * K for _, K, _ in shapes[:3]), dtype=torch.float16, device=dev)
    off = 0
    for i, (t, K, N) in enumerate(shapes):
        W = oracle.pack(t, synth.weights(0x7100 + i, max(N, 1), K))[:N]
        x = synth.activations(0x7200 + i, M, K)
        host_x.append(x.reshape(-1))
        if i < 3:
            xd = dx[off:off + M * K].view(M, K)
            off += M * K
        else:
            xd = torch.empty((M, K), dtype=torch.float16, device=dev)
        ents.append((t, torch.from_numpy(np.ascontiguousarray(W)).to(dev), K, xd,
                     torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)))
        host_ref.append((t, W, K, x, N))
    xh = torch.from_numpy(np.concatenate(host_x)).pin_memory()
    yh = torch.full((sum(M * N for _, _, N in shapes),), float("nan"), dtype=torch.float32).pin_memory()
    ws = pn.Workspace(500, dev)
    pn.gemv_layer_host(ents, M, xh, yh, ws)
    assert ws.status() == 0
    yo = 0
    for t, W, K, x, N in host_ref:
        if N:
            y_ref, abs_sum = oracle.gemv(t, W, K, x)
            assert_gemv_close(yh[yo:yo + M * N].numpy().reshape(M, N), y_ref, abs_sum)
        yo += M * N


def test_layer_call_reused(pn, dev, oracle):
    # pn.LayerCall marshals a layer's arguments once; device() and host()
    # reuse them across calls and steps
    from bit_weight_only_pn_gb300 import synth
    M = 1
    shapes = [(PN3T, 5120, 160), (PN4T, 6144, 77)]
    ents, refs, xs = [], [], []
    for i, (t, K, N) in enumerate(shapes):
        W = oracle.pack(t, synth.weights(0x7300 + i, N, K))
        x = synth.activations(0x7400 + i, M, K)
        ents.append((t, torch.from_numpy(W).to(dev), K, torch.from_numpy(x).to(dev),
                     torch.empty((M, N), dtype=torch.float32, device=dev)))
        refs.append(oracle.gemv(t, W, K, x))
        xs.append(x.reshape(-1))
    call = pn.LayerCall(ents, M, pn.Workspace(237, dev))
    xh = torch.from_numpy(np.concatenate(xs)).pin_memory()
    yh = torch.empty(sum(M * N for _, _, N in shapes), dtype=torch.float32).pin_memory()
    for _ in range(3):
        for e in ents:
            e[4].fill_(float("nan"))
        call.device()
        torch.cuda.synchronize()
        for e, (y_ref, abs_sum) in zip(ents, refs):
            assert_gemv_close(e[4].cpu().numpy(), y_ref, abs_sum)
        yh.fill_(float("nan"))
        call.host(xh, yh)
        yo = 0
        for (t, K, N), (y_ref, abs_sum) in zip(shapes, refs):
            assert_gemv_close(yh[yo:yo + M * N].numpy().reshape(M, N), y_ref, abs_sum)
            yo += M * N
    with pytest.raises(ValueError):
        call.host(xh[:-1], yh)
