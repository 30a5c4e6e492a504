"""Python binding of the PN CUDA library (include/pn.h): argument marshalling only.

PyTorch supplies device memory and the current CUDA stream; every step of the
computation runs in the library's kernels.  There is no CPU path: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PN3T = 124
PN4T = 125
ALGO_AUTO, ALGO_TENSOR_CORE, ALGO_CUDA_CORE, ALGO_CUDA_CORE_STAGED = 0, 1, 2, 3
MAX_M = 16
MAX_LAYER = 8
STATUS = {0: "PN_OK", 1: "PN_EINVAL", 2: "PN_EALIGN", 3: "PN_EUNSUPPORTED", 4: "PN_ECUDA",
          5: "PN_ETIMEOUT"}

LIBRARY = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpn_gb300.so")

_lock = threading.Lock()
_lib = None


class PnError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: str | None = None):
        detail = f" ({cuda_error})" if cuda_error else ""
        super().__init__(f"{what}: {STATUS.get(status, status)}{detail}")
        self.status = status
        self.cuda_error = cuda_error


class _Desc(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int), ("W", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise RuntimeError(f"PN CUDA library not built ({LIBRARY}); run "
                                   "`python -m bit_weight_only_pn_gb300.build`")
            L = ctypes.CDLL(LIBRARY)
            vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.pn_abi_version.restype = i32
            L.pn_status_string.restype = ctypes.c_char_p
            L.pn_status_string.argtypes = [i32]
            L.pn_last_cuda_error.restype = ctypes.c_char_p
            L.pn_last_cuda_error.argtypes = []
            L.pn_weights_per_block.restype = i32
            L.pn_weights_per_block.argtypes = [i32]
            L.pn_row_bytes.restype = sz
            L.pn_row_bytes.argtypes = [i32, i64]
            L.pn_pack.restype = i32
            L.pn_pack.argtypes = [i32, vp, i64, i64, vp, vp]
            L.pn_unpack.restype = i32
            L.pn_unpack.argtypes = [i32, vp, i64, i64, vp, vp]
            L.pn_workspace_bytes.restype = sz
            L.pn_workspace_bytes.argtypes = [i64]
            L.pn_workspace_init.restype = i32
            L.pn_workspace_init.argtypes = [vp, sz, vp]
            L.pn_workspace_status.restype = i32
            L.pn_workspace_status.argtypes = [vp, sz, vp]
            L.pn_gemv.restype = i32
            L.pn_gemv.argtypes = [i32, vp, i64, i64, vp, i32, vp, vp, sz, vp]
            L.pn_gemv_ex.restype = i32
            L.pn_gemv_ex.argtypes = [i32, vp, i64, i64, vp, i32, vp, vp, sz, i32, vp]
            L.pn_gemv_layer.restype = i32
            L.pn_gemv_layer.argtypes = [ctypes.POINTER(_Desc), i32, i32, vp, sz, vp]
            L.pn_gptq_scratch_bytes.restype = sz
            L.pn_gptq_scratch_bytes.argtypes = [i64, i64]
            L.pn_gptq.restype = i32
            L.pn_gptq.argtypes = [i32, vp, i64, i64, vp, i64, ctypes.c_double, vp, vp, sz, vp]
            L.pn_gemv_layer_host.restype = i32
            L.pn_gemv_layer_host.argtypes = [ctypes.POINTER(_Desc), i32, i32, vp, vp, vp, sz, vp]
            L.pn_gemv_hadamard.restype = i32
            L.pn_gemv_hadamard.argtypes = [i32, vp, i64, i64, vp, i32, i32, vp, vp, sz, vp]
            L.pn_gemv_layer_hadamard.restype = i32
            L.pn_gemv_layer_hadamard.argtypes = [ctypes.POINTER(_Desc), i32, i32, i32, vp, sz, vp]
            L.pn_gemv_layer_ex.restype = i32
            L.pn_gemv_layer_ex.argtypes = [ctypes.POINTER(_Desc), i32, i32, vp, sz, i32, vp]
            L.pn_unpack_f16.restype = i32
            L.pn_unpack_f16.argtypes = [i32, vp, i64, i64, vp, vp]
            L.pn_gemm_f16.restype = i32
            L.pn_gemm_f16.argtypes = [vp, i64, i64, vp, i64, vp, i64, vp, sz, vp]
            L.pn_prefill.restype = i32
            L.pn_prefill.argtypes = [i32, vp, i64, i64, vp, i64, vp, vp, sz, vp, sz, vp]
            L.pn_read_ranges.restype = i32
            L.pn_read_ranges.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(sz), i32, vp, vp]
            L.pn_hadamard.restype = i32
            L.pn_hadamard.argtypes = [vp, i32, i64, i32, vp, vp]
            L.pn_set_wait_timeout_ns.restype = None
            L.pn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
            L.pn_set_test_stall.restype = None
            L.pn_set_test_stall.argtypes = [ctypes.c_int]
            L.pn_tc_split.restype = i32
            L.pn_tc_split.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(i64), i32, i32,
                                      i32, ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(i32)]
            _lib = L
        return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        cuda = lib().pn_last_cuda_error().decode() if status == 4 else None
        raise PnError(status, what, cuda)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _require(t: torch.Tensor, dtype, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def weights_per_block(pn_type: int) -> int:
    return int(lib().pn_weights_per_block(pn_type))


def row_bytes(pn_type: int, K: int) -> int:
    return int(lib().pn_row_bytes(pn_type, K))


def pack(pn_type: int, w: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 weights [N][K] -> PN rows uint8 [N][row_bytes]."""
    _require(w, torch.float32, "w")
    N, K = w.shape
    rb = row_bytes(pn_type, K)
    if rb == 0:
        raise ValueError(f"K={K} is not a whole number of blocks")
    if out is None:
        out = torch.empty((N, rb), dtype=torch.uint8, device=w.device)
    _require(out, torch.uint8, "out")
    _check(lib().pn_pack(pn_type, _ptr(w), N, K, _ptr(out), _stream(stream)), "pn_pack")
    return out


def unpack(pn_type: int, W: torch.Tensor, K: int, out: torch.Tensor | None = None,
           stream=None) -> torch.Tensor:
    """PN rows uint8 [N][row_bytes] -> fp32 weights [N][K] (exact)."""
    _require(W, torch.uint8, "W")
    N = W.shape[0]
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=W.device)
    _require(out, torch.float32, "out")
    _check(lib().pn_unpack(pn_type, _ptr(W), N, K, _ptr(out), _stream(stream)), "pn_unpack")
    return out


class Workspace:
    """Zeroed device scratch for GEMV calls on one device (see pn_workspace_bytes)."""

    def __init__(self, total_rows: int, device=None, stream=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.device(self.device):
            self.nbytes = int(lib().pn_workspace_bytes(int(total_rows)))
            if self.nbytes == 0:
                raise PnError(4, "pn_workspace_bytes")
            self.buffer = torch.zeros(self.nbytes, dtype=torch.uint8, device=self.device)
        self.total_rows = int(total_rows)

    @property
    def ptr(self) -> int:
        return self.buffer.data_ptr()

    def status(self, stream=None) -> int:
        """Synchronise, read and clear the device status word (0 = ok)."""
        return int(lib().pn_workspace_status(self.ptr, self.nbytes, _stream(stream)))


def gemv(pn_type: int, W: torch.Tensor, K: int, x: torch.Tensor, y: torch.Tensor | None = None,
         workspace: Workspace | None = None, algo: int = ALGO_AUTO, stream=None) -> torch.Tensor:
    """y[M][N] = decode(W)[N][K] @ x[M][K]^T with fp32 accumulation (1 <= M <= 16)."""
    _require(W, torch.uint8, "W")
    _require(x, torch.float16, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    M = x.shape[0]
    N = W.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    _require(y, torch.float32, "y")
    ws_ptr, ws_bytes = (workspace.ptr, workspace.nbytes) if workspace is not None else (None, 0)
    _check(lib().pn_gemv_ex(pn_type, _ptr(W), N, K, _ptr(x), M, _ptr(y), ws_ptr, ws_bytes, algo,
                            _stream(stream)), "pn_gemv")
    return y


def gemv_layer(entries, M: int, workspace: Workspace | None = None, algo: int = ALGO_AUTO,
               stream=None):
    """Several independent GEMVs in one launch.

    ``entries`` is a sequence of (pn_type, W, K, x, y) with x fp16 [M][K] and y
    fp32 [M][N] preallocated.  Returns the list of y tensors.
    """
    entries = list(entries)
    arr = (_Desc * len(entries))()
    for i, (t, W, K, x, y) in enumerate(entries):
        _require(W, torch.uint8, "W")
        _require(x, torch.float16, "x")
        _require(y, torch.float32, "y")
        arr[i] = _Desc(t, _ptr(W), W.shape[0], K, _ptr(x), _ptr(y))
    ws_ptr, ws_bytes = (workspace.ptr, workspace.nbytes) if workspace is not None else (None, 0)
    _check(lib().pn_gemv_layer_ex(arr, len(entries), M, ws_ptr, ws_bytes, algo, _stream(stream)),
           "pn_gemv_layer")
    return [e[4] for e in entries]


def gemv_hadamard(pn_type: int, W: torch.Tensor, K: int, x: torch.Tensor, block: int,
                  y: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """y = decode(W) @ hadamard(x, block)^T in one launch (see pn_gemv_hadamard)."""
    _require(W, torch.uint8, "W")
    _require(x, torch.float16, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    M, N = x.shape[0], W.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    _require(y, torch.float32, "y")
    ws_ptr, ws_bytes = (workspace.ptr, workspace.nbytes) if workspace is not None else (None, 0)
    _check(lib().pn_gemv_hadamard(pn_type, _ptr(W), N, K, _ptr(x), M, block, _ptr(y), ws_ptr, ws_bytes,
                                  _stream(stream)), "pn_gemv_hadamard")
    return y


class LayerCall:
    """The marshalled arguments of one layer call (pn_gemv_layer /
    pn_gemv_layer_host) over fixed buffers, built once and reused: a serving
    loop that calls with the same tensors every step pays one ctypes call per
    step.  The entries' tensors are kept alive by this object."""

    def __init__(self, entries, M: int, workspace: Workspace):
        self.entries = list(entries)
        self.M = M
        self.workspace = workspace
        self._arr = (_Desc * len(self.entries))()
        for i, (t, W, K, x, y) in enumerate(self.entries):
            _require(W, torch.uint8, "W")
            _require(x, torch.float16, "x")
            _require(y, torch.float32, "y")
            self._arr[i] = _Desc(t, _ptr(W), W.shape[0], K, _ptr(x), _ptr(y))
        self._n = len(self.entries)
        self.x_elems = sum(M * K for _, _, K, _, _ in self.entries)
        self.y_elems = sum(M * W.shape[0] for _, W, _, _, _ in self.entries)

    def device(self, stream=None) -> None:
        """pn_gemv_layer on the entries' device buffers (enqueued on `stream`)."""
        _check(lib().pn_gemv_layer(self._arr, self._n, self.M, self.workspace.ptr, self.workspace.nbytes,
                                   _stream(stream)), "pn_gemv_layer")

    def host(self, x_host: torch.Tensor, y_host: torch.Tensor, stream=None) -> torch.Tensor:
        """pn_gemv_layer_host: x from host memory, y back to it; returns when
        y_host is written."""
        if x_host.is_cuda or y_host.is_cuda or x_host.dtype != torch.float16 or y_host.dtype != torch.float32:
            raise TypeError("x_host must be a CPU float16 tensor and y_host a CPU float32 tensor")
        if not (x_host.is_contiguous() and y_host.is_contiguous()):
            raise ValueError("host buffers must be contiguous")
        if x_host.numel() < self.x_elems or y_host.numel() < self.y_elems:
            raise ValueError("host buffers are too small")
        _check(lib().pn_gemv_layer_host(self._arr, self._n, self.M, x_host.data_ptr(), y_host.data_ptr(),
                                        self.workspace.ptr, self.workspace.nbytes, _stream(stream)),
               "pn_gemv_layer_host")
        return y_host


def gemv_layer_host(entries, M: int, x_host: torch.Tensor, y_host: torch.Tensor, workspace: Workspace,
                    stream=None) -> torch.Tensor:
    """pn_gemv_layer_host: x from host memory (every entry's x [M][K] in
    order, fp16), the GEMVs, y back to host memory (fp32), in one call that
    returns when y_host is written.  (LayerCall keeps the marshalled
    arguments for repeated calls.)"""
    return LayerCall(entries, M, workspace).host(x_host, y_host, stream)


def gemv_layer_hadamard(entries, M: int, block: int, workspace: Workspace | None = None, stream=None):
    """Several independent GEMVs on rotated activations in one launch (see pn_gemv_layer_hadamard)."""
    entries = list(entries)
    arr = (_Desc * len(entries))()
    for i, (t, W, K, x, y) in enumerate(entries):
        _require(W, torch.uint8, "W")
        _require(x, torch.float16, "x")
        _require(y, torch.float32, "y")
        arr[i] = _Desc(t, _ptr(W), W.shape[0], K, _ptr(x), _ptr(y))
    ws_ptr, ws_bytes = (workspace.ptr, workspace.nbytes) if workspace is not None else (None, 0)
    _check(lib().pn_gemv_layer_hadamard(arr, len(entries), M, block, ws_ptr, ws_bytes, _stream(stream)),
           "pn_gemv_layer_hadamard")
    return [e[4] for e in entries]


def gptq(pn_type: int, w: torch.Tensor, X: torch.Tensor, damp: float = 0.01, stream=None) -> torch.Tensor:
    """GPTQ-style quantisation (see pn_gptq): fp32 w [N][K] and calibration
    inputs X fp32 [n][K] -> PN rows [N][row_bytes].  Synchronous."""
    _require(w, torch.float32, "w")
    _require(X, torch.float32, "X")
    N, K = w.shape
    if X.dim() != 2 or X.shape[1] != K:
        raise ValueError("X must be [n][K]")
    rb = row_bytes(pn_type, K)
    if rb == 0:
        raise ValueError("K is not a whole number of blocks")
    W = torch.empty((N, rb), dtype=torch.uint8, device=w.device)
    nbytes = int(lib().pn_gptq_scratch_bytes(N, K))
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device=w.device)
    base = (scratch.data_ptr() + 255) // 256 * 256
    _check(lib().pn_gptq(pn_type, _ptr(w), N, K, _ptr(X), X.shape[0], float(damp), _ptr(W), base, nbytes,
                         _stream(stream)), "pn_gptq")
    return W


def hadamard(x: torch.Tensor, block: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Block Hadamard rotation of fp16 activations [M][K] (see pn_hadamard)."""
    _require(x, torch.float16, "x")
    if x.dim() == 1:
        x = x.view(1, -1)
    M, K = x.shape
    if out is None:
        out = torch.empty_like(x)
    _require(out, torch.float16, "out")
    _check(lib().pn_hadamard(_ptr(x), M, K, block, _ptr(out), _stream(stream)), "pn_hadamard")
    return out


def unpack_f16(pn_type: int, W: torch.Tensor, K: int, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """PN rows uint8 [N][row_bytes] -> fp16 weights [N][K] (exact decode, one rounding)."""
    _require(W, torch.uint8, "W")
    N = W.shape[0]
    if out is None:
        out = torch.empty((N, K), dtype=torch.float16, device=W.device)
    _require(out, torch.float16, "out")
    _check(lib().pn_unpack_f16(pn_type, _ptr(W), N, K, _ptr(out), _stream(stream)), "pn_unpack_f16")
    return out


def gemm_f16(w16: torch.Tensor, x: torch.Tensor, y: torch.Tensor | None = None,
             workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """y[M][N] = x[M][K] @ w16[N][K]^T, fp16 products, fp32 accumulation (tcgen05)."""
    _require(w16, torch.float16, "w16")
    _require(x, torch.float16, "x")
    N, K = w16.shape
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=w16.device)
    _require(y, torch.float32, "y")
    if workspace is None:
        workspace = Workspace(N, w16.device)
    _check(lib().pn_gemm_f16(_ptr(w16), N, K, _ptr(x), M, _ptr(y), y.shape[1], workspace.ptr,
                             workspace.nbytes, _stream(stream)), "pn_gemm_f16")
    return y


def prefill(pn_type: int, W: torch.Tensor, K: int, x: torch.Tensor, y: torch.Tensor | None = None,
            scratch: torch.Tensor | None = None, workspace: Workspace | None = None,
            stream=None) -> torch.Tensor:
    """y[M][N] for large M: PN rows rebuilt as fp16 chunk by chunk into
    ``scratch`` (default: room for every row), then the fp16 GEMM."""
    _require(W, torch.uint8, "W")
    _require(x, torch.float16, "x")
    N = W.shape[0]
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=W.device)
    _require(y, torch.float32, "y")
    if scratch is None:
        rows = max(128, (N + 127) // 128 * 128)
        scratch = torch.empty(rows * K, dtype=torch.float16, device=W.device)
    _require(scratch, torch.float16, "scratch")
    if workspace is None:
        workspace = Workspace(N, W.device)
    _check(lib().pn_prefill(pn_type, _ptr(W), N, K, _ptr(x), M, _ptr(y), _ptr(scratch),
                            scratch.numel() * 2, workspace.ptr, workspace.nbytes, _stream(stream)),
           "pn_prefill")
    return y


def read_ranges(tensors, sink: torch.Tensor, stream=None) -> torch.Tensor:
    """Diagnostic read-bandwidth probe (see pn_read_ranges): reads every
    tensor's bytes once and XORs its 32-bit words into sink[i] (int32 device
    tensor with one element per tensor)."""
    tensors = list(tensors)
    n = len(tensors)
    ptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in tensors])
    sizes = (ctypes.c_size_t * n)(*[t.numel() * t.element_size() for t in tensors])
    _require(sink, torch.int32, "sink")
    _check(lib().pn_read_ranges(ptrs, sizes, n, sink.data_ptr(), _stream(stream)), "pn_read_ranges")
    return sink


def set_wait_timeout_ns(ns: int) -> None:
    lib().pn_set_wait_timeout_ns(int(ns))


def set_test_stall(on: bool) -> None:
    lib().pn_set_test_stall(1 if on else 0)


def tc_split(shapes, M: int, num_sms: int) -> list[int]:
    """Testing aid (host only, see pn_tc_split): the unit ranges the
    tensor-core GEMV would give its thread blocks for tensors ``shapes`` =
    [(pn_type, N, K), ...] at M tokens on num_sms SMs; returns starts, with
    block c taking units [starts[c], starts[c + 1])."""
    shapes = list(shapes)
    n = len(shapes)
    types = (ctypes.c_int * n)(*[s[0] for s in shapes])
    Ns = (ctypes.c_int64 * n)(*[s[1] for s in shapes])
    Ks = (ctypes.c_int64 * n)(*[s[2] for s in shapes])
    starts = (ctypes.c_uint32 * (max(num_sms, 1) + 1))()
    grid = ctypes.c_int(0)
    _check(lib().pn_tc_split(types, Ns, Ks, n, M, num_sms, starts, ctypes.byref(grid)), "pn_tc_split")
    return list(starts[: grid.value + 1])
