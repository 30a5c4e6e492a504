"""Seeded synthetic inputs for the PN GEMV workloads.

This module only draws random numbers. It holds none of the PN arithmetic (no
packing, no decoding, no dot products), so that both the CPU oracle and the CUDA
path can take their inputs from it without sharing any of the method.

Generator (reproducible in any language):

* ``splitmix64``: draw ``i`` of stream ``seed`` is ``mix(seed + (i + 1) * G)``
  with ``G = 0x9E3779B97F4A7C15`` and the standard splitmix64 finaliser
  ``mix(z) = z3 ^ (z3 >> 31)``, ``z2 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9``,
  ``z3 = (z2 ^ (z2 >> 27)) * 0x94D049BB133111EB`` (all mod 2**64).
* uniform ``u = (draw >> 11) * 2**-53`` in [0, 1).
* normal ``i`` uses draws ``2i`` and ``2i+1``: Box-Muller in fp64,
  ``sqrt(-2 ln(1 - u0)) * cos(2 pi u1)``.

Workloads (the decode-GEMV widths of a 27B-class model: K = 5120 for pn3t,
K = 6144 and 17408 for pn4t):

* weights: fp32 ``0.02 * normal`` (then quantised by a PN packer);
* activations x: fp16 round-to-nearest-even of ``normal``;
* seeds: ``0x504E0000 + 16 * config + tensor`` for weights, ``+ 8`` for x.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

PN3T = 124
PN4T = 125

SEED_BASE = 0x504E0000


def splitmix64(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the splitmix64 stream ``seed`` (uint64)."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _G
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Uniform fp64 in [0, 1) from the top 53 bits of each draw."""
    return (splitmix64(seed, count, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_CHUNK = 1 << 22


def normal(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Standard normal fp64 samples ``start .. start+count-1`` (Box-Muller, cosine branch)."""
    out = np.empty(count, dtype=np.float64)
    for lo in range(0, count, _CHUNK):
        n = min(_CHUNK, count - lo)
        u = uniform(seed, 2 * n, 2 * (start + lo))
        out[lo:lo + n] = np.sqrt(-2.0 * np.log1p(-u[0::2])) * np.cos(2.0 * np.pi * u[1::2])
    return out


def _normal_f32(seed: int, count: int, scale: float) -> np.ndarray:
    """``scale * normal`` rounded to fp32; chunks run on a thread pool (numpy
    releases the GIL inside its loops), each chunk drawing its own counters."""
    out = np.empty(count, dtype=np.float32)

    def fill(lo):
        n = min(_CHUNK, count - lo)
        out[lo:lo + n] = scale * normal(seed, n, lo)

    starts = range(0, count, _CHUNK)
    if count <= _CHUNK:
        for lo in starts:
            fill(lo)
    else:
        with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as pool:
            list(pool.map(fill, starts))
    return out


def weight_seed(config: int, tensor: int) -> int:
    return SEED_BASE + 16 * config + tensor


def x_seed(config: int, tensor: int) -> int:
    return weight_seed(config, tensor) + 8


def weights(seed: int, n: int, k: int, std: float = 0.02) -> np.ndarray:
    """fp32 weights [n][k], ``std * normal``."""
    return _normal_f32(seed, n * k, std).reshape(n, k)


def activations(seed: int, m: int, k: int) -> np.ndarray:
    """fp16 activations [m][k] (RNE of a standard normal), returned as float16."""
    return normal(seed, m * k).astype(np.float16).reshape(m, k)


def weight_rows(seed: int, n: int, k: int, rows, std: float = 0.02) -> np.ndarray:
    """Rows ``rows`` of ``weights(seed, n, k, std)``, drawn without the other rows."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, k), dtype=np.float32)
    for i, r in enumerate(rows):
        if not 0 <= r < n:
            raise IndexError(r)
        out[i] = std * normal(seed, k, int(r) * k)
    return out


# The workloads: (type, K, N) per tensor.
LAYER_27B = (
    (PN3T, 5120, 6144),
    (PN3T, 5120, 17408),
    (PN3T, 5120, 17408),
    (PN4T, 5120, 1024),
    (PN4T, 5120, 1024),
    (PN4T, 6144, 5120),
    (PN4T, 17408, 5120),
)

CONFIGS = {
    0: dict(name="pn3t N=1024 K=5120 M=1", tensors=((PN3T, 5120, 1024),), M=1),
    1: dict(name="pn3t N=17408 K=5120 M=1", tensors=((PN3T, 5120, 17408),), M=1),
    2: dict(name="pn4t N=5120 K=17408 M=1", tensors=((PN4T, 17408, 5120),), M=1),
    3: dict(name="27B-class layer, 7 tensors, M=1", tensors=LAYER_27B, M=1),
    4: dict(name="27B-class layer, 7 tensors, M=8", tensors=LAYER_27B, M=8),
    # the M 9 .. 16 band: one token plus 15 drafts over the same layer
    5: dict(name="27B-class layer, 7 tensors, M=16", tensors=LAYER_27B, M=16),
    # prefill: a 4096-token prompt through one FFN gate/up tensor
    6: dict(name="prefill: pn3t 5120->17408, M=4096", tensors=((PN3T, 5120, 17408),), M=4096, prefill=True),
}
