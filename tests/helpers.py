"""Shared test helpers: golden fixtures, on-grid blocks and the GEMV tolerance.

Nothing here computes a PN encoding or decoding for the oracle to be compared
with; the helpers only build inputs (weights that already sit on a quantisation
grid, so that their decoded values are known without any decoder) and state the
tolerance of the GEMV check.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

PN3T, PN4T = 124, 125
# (weights per block, codes per word, bits per code, zero point), from the
# format page's block table and the mid-tread reading.
GEOMETRY = {PN3T: (80, 10, 3, 4), PN4T: (64, 8, 4, 8)}

# GEMV bound: |y - y_ref| <= REL * sum_k |w_k x_k| + ABS per element.
REL, ABS = 1e-5, 1e-6


def read_worked_blocks():
    """Parse tests/golden/pn_worked_blocks.txt into a list of dicts."""
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "pn_worked_blocks.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(" ")
            if key == "block":
                cur = {"name": val}
                blocks.append(cur)
            elif key == "type":
                cur["type"] = int(val)
            elif key == "scale":
                cur["scale"] = int(val, 16)
            elif key == "codes":
                cur["codes"] = [int(v) for v in val.split()]
            elif key == "bytes":
                cur["bytes"] = bytes(int(v, 16) for v in val.split())
    return blocks


def f16_bits_to_f64(bits) -> np.ndarray:
    """fp16 bit patterns -> fp64 values (numpy's own conversion)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def on_grid_weights(rng: np.random.Generator, pn_type: int, n_rows: int, n_blocks: int,
                    scale_range=(-12, -4)):
    """Weights that already sit on a PN grid, with the grid step known.

    Each block gets an fp16 scale d (random sign and exponent in ``scale_range``,
    random 10-bit mantissa) and integer steps q in [-z, z-1] with at least one
    q = -z; the weight is the exact fp32 product d*q.  Such a block quantises
    back to exactly d and q under the signed-scale rule, so its decoded weights
    are known in advance.  Returns (w fp32 [N][K], d fp64 [N][nb], q int [N][K]).
    """
    bpb, _, _, z = GEOMETRY[pn_type]
    K = n_blocks * bpb
    e = rng.integers(scale_range[0], scale_range[1], size=(n_rows, n_blocks))
    mant = rng.integers(0, 1024, size=(n_rows, n_blocks))
    sign = rng.choice([-1.0, 1.0], size=(n_rows, n_blocks))
    d = sign * (1.0 + mant / 1024.0) * np.exp2(e.astype(np.float64))
    d = d.astype(np.float16).astype(np.float64)          # exactly an fp16 value
    q = rng.integers(-z, z, size=(n_rows, K))
    pos = rng.integers(0, bpb, size=(n_rows, n_blocks))
    for b in range(n_blocks):
        q[np.arange(n_rows), b * bpb + pos[:, b]] = -z   # one full-range step per block
    w = (np.repeat(d, bpb, axis=1) * q).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), np.repeat(d, bpb, axis=1) * q)
    return w, d, q


def assert_gemv_close(y, y_ref, abs_sum, rel=REL, abs_=ABS):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    bound = rel * np.asarray(abs_sum, dtype=np.float64) + abs_
    err = np.abs(y - y_ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: got {y[tuple(i)]!r} want {y_ref[tuple(i)]!r} "
                           f"bound {bound[tuple(i)]:.3g}" for i in idx)
        raise AssertionError(f"{int(bad.sum())} of {bad.size} outputs out of tolerance: {detail}")
    return float(np.max(err / bound)) if err.size else 0.0


def read_hadamard_cases():
    """Parse tests/golden/hadamard_worked.txt: list of (name, block, x fp16, out bits)."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "hadamard_worked.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(" ")
            if key == "case":
                cur = {"name": val}
                cases.append(cur)
            elif key == "block":
                cur["block"] = int(val)
            elif key == "x":
                cur["x"] = np.array([float(v) for v in val.split()], dtype=np.float16)
            elif key == "out":
                cur["out"] = np.array([int(v, 16) for v in val.split()], dtype=np.uint16)
    return cases


def sylvester_hadamard(n: int) -> np.ndarray:
    """H_n in Sylvester order (H_1 = [1], H_2n = [[H, H], [H, -H]]), fp64."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def zero_code_case(rng: np.random.Generator, pn_type: int, n_rows: int, n_blocks: int, M: int,
                   scale_exp=(-14, 3), tiny=1e-4, big=1e3):
    """Weights dominated by the zero code, with activations that punish any
    computation which does not subtract the zero point code by code.

    Format page, "Zero is a code, and the scale has a sign": n = z decodes to
    an exact zero.  In every block a few positions S_b (the same for all rows)
    hold the only non-zero steps: the first is the full-range step q = -z (so
    the block's scale is exactly d), the others random in [-z, z-1].  Every
    other code is n = z (weight 0).  x is tiny (about ``tiny``) at S_b and
    large (up to ``big``, random sign) everywhere else, so the exact outputs
    are small while sum_k |x_k| over a block is large: a kernel that forms
    sum n*x - z*sum x loses the answer to rounding, one that multiplies
    exact (n - z) values does not.  Scales d have random sign, 10-bit
    mantissa and exponent in ``scale_exp`` (|d| from 2^-14 to about 8 with the
    default); a few rows get fp16-subnormal scales.  Returns (w fp32 [N][K],
    x fp16 [M][K]); the weights sit on their grid, so the packer reproduces d
    and q exactly.
    """
    bpb, _, _, z = GEOMETRY[pn_type]
    K = n_blocks * bpb
    x = np.empty((M, K), dtype=np.float64)
    sign = rng.choice([-1.0, 1.0], size=(M, K))
    x[:] = sign * rng.uniform(1.0, big, size=(M, K))
    q = np.zeros((n_rows, K), dtype=np.int64)
    for b in range(n_blocks):
        s = int(rng.integers(1, 4))
        pos = b * bpb + rng.choice(bpb, size=s, replace=False)
        x[:, pos] = rng.choice([-1.0, 1.0], size=(M, s)) * rng.uniform(0.5, 1.5, size=(M, s)) * tiny
        q[:, pos[0]] = -z
        if s > 1:
            q[:, pos[1:]] = rng.integers(-z, z, size=(n_rows, s - 1))
    e = rng.integers(scale_exp[0], scale_exp[1], size=(n_rows, n_blocks))
    mant = rng.integers(0, 1024, size=(n_rows, n_blocks))
    dsign = rng.choice([-1.0, 1.0], size=(n_rows, n_blocks))
    d = dsign * (1.0 + mant / 1024.0) * np.exp2(e.astype(np.float64))
    sub = rng.random(n_rows) < 0.05
    d[sub] = dsign[sub] * rng.integers(1, 1024, size=(int(sub.sum()), n_blocks)) * 2.0 ** -24
    d = d.astype(np.float16).astype(np.float64)
    w = (np.repeat(d, bpb, axis=1) * q).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), np.repeat(d, bpb, axis=1) * q)
    return w, x.astype(np.float16)
