"""The C-ABI library builds, loads and exports every symbol include/pn.h declares.

These run without a GPU: only calls that return before touching the device
(sizes, status strings, argument checks) are made.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pn.h")


@pytest.fixture(scope="module")
def lib():
    from bit_weight_only_pn_gb300 import build, pn
    build.build()
    return pn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pn_[a-z_0-9]+)\s*\(", text)
    return sorted(set(n for n in names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "pn_gemv" in names and "pn_gemv_layer" in names and "pn_pack" in names
    for name in names:
        assert hasattr(lib, name), f"{name} missing from the library"


def test_host_only_queries(lib):
    assert lib.pn_abi_version() == 1
    assert lib.pn_weights_per_block(124) == 80 and lib.pn_weights_per_block(125) == 64
    assert lib.pn_weights_per_block(3) == 0
    assert lib.pn_row_bytes(124, 5120) == 2176 and lib.pn_row_bytes(125, 17408) == 9248
    assert lib.pn_row_bytes(124, 6144) == 0 and lib.pn_row_bytes(125, 0) == 0
    assert lib.pn_row_bytes(125, -64) == 0
    for s in range(6):
        assert lib.pn_status_string(s)
    assert lib.pn_status_string(99) == b"unknown status"


PN_EINVAL, PN_EALIGN = 1, 2
FAKE = 0x10000      # a 64 KiB-aligned address that is never dereferenced: checks fail first


def test_argument_checks_return_before_any_launch(lib):
    g = lib.pn_gemv_ex
    # unknown type, K not a whole number of blocks, M out of range, negative N
    assert g(7, FAKE, 16, 5120, FAKE * 2, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    assert g(124, FAKE, 16, 5121, FAKE * 2, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    assert g(124, FAKE, 16, 5120, FAKE * 2, 0, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    assert g(124, FAKE, 16, 5120, FAKE * 2, 17, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    assert g(124, FAKE, -1, 5120, FAKE * 2, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    # null pointers, misaligned pointers
    assert g(124, None, 16, 5120, FAKE * 2, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    assert g(124, FAKE + 1, 16, 5120, FAKE * 2, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EALIGN
    assert g(124, FAKE, 16, 5120, FAKE * 2 + 1, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == PN_EALIGN
    assert g(124, FAKE, 16, 5120, FAKE * 2, 1, FAKE * 4 + 2, FAKE * 8, 1 << 20, 0, None) == PN_EALIGN
    # y overlapping W or x
    assert g(124, FAKE, 16, 5120, FAKE * 2, 1, FAKE + 64, FAKE * 8, 1 << 20, 0, None) == PN_EINVAL
    # N = 0 is a no-op
    assert g(124, FAKE, 0, 5120, FAKE * 2, 1, FAKE * 4, FAKE * 8, 1 << 20, 0, None) == 0
    # pack / unpack checks
    assert lib.pn_pack(124, FAKE, 4, 100, FAKE * 2, None) == PN_EINVAL
    assert lib.pn_pack(124, FAKE + 2, 4, 80, FAKE * 2, None) == PN_EALIGN
    assert lib.pn_unpack(125, FAKE * 2 + 1, 4, 64, FAKE, None) == PN_EALIGN
    assert lib.pn_unpack(125, FAKE, 4, 64, FAKE + 8, None) == PN_EINVAL   # overlap
    assert lib.pn_pack(125, FAKE, 0, 64, FAKE * 2, None) == 0
    # workspace helpers
    assert lib.pn_workspace_init(None, 1024, None) == PN_EINVAL
    assert lib.pn_workspace_init(FAKE + 16, 1024, None) == PN_EINVAL


def test_layer_checks(lib):
    from bit_weight_only_pn_gb300.pn import _Desc
    arr = (_Desc * 2)()
    arr[0] = _Desc(124, FAKE, 32, 5120, FAKE * 2, FAKE * 4)
    arr[1] = _Desc(125, FAKE * 8, 32, 6144, FAKE * 16, FAKE * 4 + 64)    # y overlaps entry 0's y
    assert lib.pn_gemv_layer(arr, 2, 1, FAKE * 32, 1 << 20, None) == PN_EINVAL
    assert lib.pn_gemv_layer(arr, 0, 1, FAKE * 32, 1 << 20, None) == PN_EINVAL
    assert lib.pn_gemv_layer(arr, 9, 1, FAKE * 32, 1 << 20, None) == PN_EINVAL
    assert lib.pn_gemv_layer(None, 1, 1, FAKE * 32, 1 << 20, None) == PN_EINVAL


def test_hadamard_checks(lib):
    h = lib.pn_hadamard
    h.restype = ctypes.c_int
    h.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    # block not a power of two, too small, too large, not dividing K; M out of range
    assert h(FAKE, 1, 96, 3, FAKE * 2, None) == PN_EINVAL
    assert h(FAKE, 1, 96, 1, FAKE * 2, None) == PN_EINVAL
    assert h(FAKE, 1, 8192, 8192, FAKE * 2, None) == PN_EINVAL
    assert h(FAKE, 1, 96, 64, FAKE * 2, None) == PN_EINVAL
    assert h(FAKE, 0, 96, 32, FAKE * 2, None) == PN_EINVAL
    # null, misaligned, partly overlapping buffers
    assert h(None, 1, 96, 32, FAKE * 2, None) == PN_EINVAL
    assert h(FAKE + 1, 1, 96, 32, FAKE * 2, None) == PN_EALIGN
    assert h(FAKE, 1, 96, 32, FAKE + 64, None) == PN_EINVAL


def test_fused_hadamard_checks(lib):
    # checks that come before any device query or launch
    g = lib.pn_gemv_hadamard
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    ws = FAKE * 8
    for block in (16, 96, 2048, 4096, 0, -32):                    # out of range, not 2^k, not dividing K
        assert g(124, FAKE, 16, 5120, FAKE * 2, 1, block, FAKE * 4, ws, 1 << 20, None) == PN_EINVAL
    assert g(124, FAKE, 16, 5120, FAKE * 2, 0, 1024, FAKE * 4, ws, 1 << 20, None) == PN_EINVAL     # M = 0
    assert g(124, FAKE, 16, 5121, FAKE * 2, 1, 1024, FAKE * 4, ws, 1 << 20, None) == PN_EINVAL     # K
    assert g(124, FAKE, 16, 5120, FAKE * 2 + 1, 1, 1024, FAKE * 4, ws, 1 << 20, None) == PN_EALIGN
    assert g(124, FAKE, 16, 5120, FAKE * 2, 1, 1024, FAKE + 64, ws, 1 << 20, None) == PN_EINVAL    # y on W
    from bit_weight_only_pn_gb300.pn import _Desc
    arr = (_Desc * 2)()
    arr[0] = _Desc(124, FAKE, 32, 5120, FAKE * 2, FAKE * 4)
    arr[1] = _Desc(125, FAKE * 8, 32, 6144, FAKE * 16, FAKE * 4 + 64)    # y overlaps entry 0's y
    L = lib.pn_gemv_layer_hadamard
    assert L(arr, 2, 1, 1024, FAKE * 32, 1 << 20, None) == PN_EINVAL
    arr[1] = _Desc(125, FAKE * 8, 32, 6144, FAKE * 16, FAKE * 64)
    assert L(arr, 2, 1, 4096, FAKE * 32, 1 << 20, None) == PN_EINVAL    # 4096 divides neither K
    assert L(arr, 0, 1, 1024, FAKE * 32, 1 << 20, None) == PN_EINVAL


def test_layer_host_checks(lib):
    from bit_weight_only_pn_gb300.pn import _Desc
    arr = (_Desc * 1)()
    arr[0] = _Desc(124, FAKE, 32, 5120, FAKE * 2, FAKE * 4)
    h = lib.pn_gemv_layer_host
    assert h(arr, 1, 1, None, FAKE * 8, FAKE * 32, 1 << 20, None) == PN_EINVAL          # no host x
    assert h(arr, 1, 1, FAKE * 8, None, FAKE * 32, 1 << 20, None) == PN_EINVAL          # no host y
    assert h(arr, 0, 1, FAKE * 8, FAKE * 16, FAKE * 32, 1 << 20, None) == PN_EINVAL     # count
    assert h(arr, 1, 17, FAKE * 8, FAKE * 16, FAKE * 32, 1 << 20, None) == PN_EINVAL    # M
    arr[0] = _Desc(124, FAKE, 32, 5120, FAKE * 2 + 1, FAKE * 4)
    assert h(arr, 1, 1, FAKE * 8, FAKE * 16, FAKE * 32, 1 << 20, None) == PN_EALIGN     # device x


def test_gptq_checks(lib):
    # checks that come before any device work
    g = lib.pn_gptq
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    sb = lib.pn_gptq_scratch_bytes
    sb.restype = ctypes.c_size_t
    sb.argtypes = [ctypes.c_int64, ctypes.c_int64]
    need = sb(8, 160)
    assert need >= (4 * 160 * 160 + 8 * 160) * 8 and sb(8, 0) == 0 and sb(-1, 160) == 0
    ws = FAKE * 64
    assert g(7, FAKE, 8, 160, FAKE * 2, 10, 0.01, FAKE * 4, ws, need, None) == PN_EINVAL      # type
    assert g(124, FAKE, 8, 161, FAKE * 2, 10, 0.01, FAKE * 4, ws, need, None) == PN_EINVAL    # K
    assert g(124, FAKE, 8, 160, FAKE * 2, 0, 0.01, FAKE * 4, ws, need, None) == PN_EINVAL     # n
    assert g(124, FAKE, 8, 160, FAKE * 2, 10, 0.0, FAKE * 4, ws, need, None) == PN_EINVAL     # damp
    assert g(124, FAKE, 8, 160, FAKE * 2, 10, 0.01, FAKE * 4, ws, need - 1, None) == PN_EINVAL  # scratch
    assert g(124, FAKE + 2, 8, 160, FAKE * 2, 10, 0.01, FAKE * 4, ws, need, None) == PN_EALIGN
    assert g(124, FAKE, 8, 160, FAKE * 2, 10, 0.01, FAKE * 4, ws + 16, need, None) == PN_EALIGN
    assert g(124, FAKE, 0, 160, FAKE * 2, 10, 0.01, FAKE * 4, ws, need, None) == 0            # nothing to do
    assert g(125, FAKE, 8, 65600, FAKE * 2, 10, 0.01, FAKE * 4, ws, 1 << 62, None) == PN_EINVAL  # K too wide


def test_prefill_checks(lib):
    # checks that come before any device query or launch
    u, g, p = lib.pn_unpack_f16, lib.pn_gemm_f16, lib.pn_prefill
    assert u(7, FAKE, 4, 80, FAKE * 2, None) == PN_EINVAL                  # unknown type
    assert u(124, FAKE, 4, 81, FAKE * 2, None) == PN_EINVAL                # K not whole blocks
    assert u(124, FAKE, 4, 80, FAKE * 2 + 2, None) == PN_EALIGN            # w16 not 4-byte aligned
    assert u(125, FAKE, 4, 64, FAKE + 16, None) == PN_EINVAL               # w16 overlaps W
    assert u(124, FAKE, 0, 80, FAKE * 2, None) == 0                        # nothing to do
    ws = FAKE * 8
    assert g(FAKE, 16, 100, FAKE * 2, 4, FAKE * 4, 16, ws, 1 << 20, None) == PN_EINVAL   # K % 8
    assert g(FAKE, 16, 128, FAKE * 2, 4, FAKE * 4, 15, ws, 1 << 20, None) == PN_EINVAL   # ldy < N
    assert g(FAKE, 16, 128, FAKE * 2, 0, FAKE * 4, 16, ws, 1 << 20, None) == PN_EINVAL   # M = 0
    assert g(FAKE, 16, 128, FAKE * 2 + 8, 4, FAKE * 4, 16, ws, 1 << 20, None) == PN_EALIGN   # x
    assert g(FAKE, 16, 128, FAKE * 2, 4, FAKE * 4 + 2, 16, ws, 1 << 20, None) == PN_EALIGN   # y
    assert g(FAKE, 16, 128, FAKE * 2, 4, FAKE * 4, 16, ws + 16, 1 << 20, None) == PN_EINVAL  # workspace
    assert g(FAKE, 0, 128, FAKE * 2, 4, FAKE * 4, 16, ws, 1 << 20, None) == 0
    assert p(124, FAKE, 16, 100, FAKE * 2, 4, FAKE * 4, FAKE * 16, 1 << 20, ws, 1 << 20, None) == PN_EINVAL
    assert p(125, FAKE, 16, 128, FAKE * 2, 0, FAKE * 4, FAKE * 16, 1 << 20, ws, 1 << 20, None) == PN_EINVAL


def test_read_ranges_checks(lib):
    r = lib.pn_read_ranges
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE * 2)
    sizes = (ctypes.c_size_t * 2)(1024, 1024)
    assert r(ptrs, sizes, 0, FAKE * 4, None) == PN_EINVAL           # no ranges
    assert r(ptrs, sizes, 9, FAKE * 4, None) == PN_EINVAL           # more than PN_MAX_LAYER
    assert r(None, sizes, 2, FAKE * 4, None) == PN_EINVAL
    assert r(ptrs, sizes, 2, None, None) == PN_EINVAL
    bad = (ctypes.c_void_p * 2)(FAKE, FAKE * 2 + 8)
    assert r(bad, sizes, 2, FAKE * 4, None) == PN_EALIGN            # range not 16-byte aligned
    assert r(ptrs, sizes, 2, FAKE * 4 + 2, None) == PN_EALIGN       # sink not 4-byte aligned
