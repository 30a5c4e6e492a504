"""Pins for the CPU oracle: what the format page and the mathematics fix.

Every check compares the oracle with something other than itself: numbers the
page prints (block size, bits per weight), IEEE arithmetic done by numpy or
Python (fp16 conversion, exact products, exact rational sums), weights that sit
on a grid so their decoded values are known, a hand-assembled worked block, and
structural properties the page states (no code straddles the word halves, even
and odd codes share offsets, one code is exactly zero, the largest weight gets
the full range).  The ``pin_*`` functions take an oracle instance so that the
mutation test at the end can run them against copies of the oracle with one
planted mistake each.
"""
from __future__ import annotations

import math
import os
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle as oracle_mod
from helpers import (GEOMETRY, PN3T, PN4T, f16_bits_to_f64, on_grid_weights,
                     read_hadamard_cases, read_worked_blocks, sylvester_hadamard)

TYPES = (PN3T, PN4T)


# ------------------------------------------------------------- pin functions --

def pin_block_geometry(o):
    # "Both PN types use the same block: a 2-byte scale and eight 32-bit words";
    # pn3t 80 weights / 3.40 bits, pn4t 64 weights / 4.25 bits; 5120 = 64 pn3t
    # blocks; 6144 and 17408 are not multiples of 80 but are of 64.
    assert o.row_bytes(PN3T, 80) == 34 and o.row_bytes(PN4T, 64) == 34
    assert o.row_bytes(PN3T, 5120) == 64 * 34 == 2176
    assert o.row_bytes(PN4T, 5120) == 2720
    assert o.row_bytes(PN4T, 6144) == 3264
    assert o.row_bytes(PN4T, 17408) == 9248
    assert o.row_bytes(PN3T, 6144) == 0 and o.row_bytes(PN3T, 17408) == 0
    assert o.row_bytes(PN4T, 80) == 0 and o.row_bytes(PN3T, 64) == 0
    assert 8 * o.row_bytes(PN3T, 5120) / 5120 == pytest.approx(3.40, abs=1e-12)
    assert 8 * o.row_bytes(PN4T, 17408) / 17408 == pytest.approx(4.25, abs=1e-12)


def pin_worked_blocks(o):
    for blk in read_worked_blocks():
        t = blk["type"]
        bpb, _, _, z = GEOMETRY[t]
        d = float(f16_bits_to_f64([blk["scale"]])[0])
        want = np.array([d * (n - z) for n in blk["codes"]], dtype=np.float64)
        assert np.array_equal(want.astype(np.float32).astype(np.float64), want)
        got = o.unpack(t, np.frombuffer(blk["bytes"], dtype=np.uint8)[None, :], bpb)
        assert np.array_equal(got[0].astype(np.float64), want), blk["name"]
        packed = o.pack(t, want.astype(np.float32)[None, :])
        assert packed.tobytes() == blk["bytes"], blk["name"]


def pin_fp16_conversion(o):
    # The oracle's own fp16 conversions against numpy's IEEE binary16 (RNE).
    bits = np.arange(65536, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    got = np.array([o.half_to_float(int(b)) for b in bits], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    rng = np.random.default_rng(7)
    f = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 18, 20000))).astype(np.float32),
        # ties and thresholds: halfway points around subnormals, normals, overflow
        np.array([65504, 65519.996, 65520, 65536, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -25 * 1.0000001, 1.5 * 2.0 ** -24, 2.5 * 2.0 ** -24, 2.0 ** -14,
                  (1 + 2.0 ** -11) * 2.0 ** -14, (1 + 3 * 2.0 ** -11), 1 + 2.0 ** -11,
                  0.0, -0.0, 1e-30, -1e-30, 3e38, -3e38], dtype=np.float32),
    ])
    f = np.concatenate([f, -f])
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    got = np.array([o.float_to_half(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def _block_bytes(scale_bits, words):
    out = bytearray(scale_bits.to_bytes(2, "little"))
    for w in words:
        out += int(w).to_bytes(4, "little")
    return bytes(out)


def _replicate(n, bits, per_half):
    v = 0
    for i in range(per_half):
        v |= n << (bits * i)
    return v | (v << 16)


def pin_decode_exact_all_scales(o):
    # w = d*(n - z) is exact in fp32 for every finite fp16 d and every code, and
    # the zero code gives a zero whose sign is the IEEE product's.
    all_bits = np.arange(65536, dtype=np.uint16)
    finite_bits = all_bits[np.isfinite(all_bits.view(np.float16))]
    assert finite_bits.size == 63488
    dvals = finite_bits.view(np.float16).astype(np.float64)
    for t in TYPES:
        bpb, cpw, bits, z = GEOMETRY[t]
        for n in range(1 << bits):
            word = _replicate(n, bits, cpw // 2).to_bytes(4, "little")
            blk = np.empty((finite_bits.size, 34), dtype=np.uint8)
            blk[:, 0:2] = finite_bits.view(np.uint8).reshape(-1, 2)
            blk[:, 2:] = np.frombuffer(word * 8, dtype=np.uint8)
            got = o.unpack(t, blk, bpb).astype(np.float64)
            want = dvals * float(n - z)                      # exact in fp64
            assert np.array_equal(want.astype(np.float32).astype(np.float64), want)
            assert np.array_equal(got, np.repeat(want[:, None], bpb, axis=1))
            assert np.array_equal(np.signbit(got), np.repeat(np.signbit(want)[:, None], bpb, axis=1))


def pin_half_structure(o):
    # Even codes fill the low 16 bits, odd codes the high 16 bits, at the same
    # offsets; no code crosses the middle; pn3t leaves bits 15 and 31 unused.
    rng = np.random.default_rng(11)
    for t in TYPES:
        bpb, cpw, bits, z = GEOMETRY[t]
        d = 2.0 ** -7
        for trial in range(40):
            q = rng.integers(-z, z, size=bpb)
            q[rng.integers(0, bpb)] = -z
            base = o.pack(t, (d * q).astype(np.float32)[None, :])[0]
            k = int(rng.integers(0, bpb))
            q2 = q.copy()
            choices = [v for v in range(-z, z) if v != q[k] and v != -z]
            q2[k] = rng.choice(choices) if q[k] != -z or (q == -z).sum() > 1 else q[k]
            other = o.pack(t, (d * q2).astype(np.float32)[None, :])[0]
            w0 = np.frombuffer(base[2:].tobytes(), dtype="<u4")
            w1 = np.frombuffer(other[2:].tobytes(), dtype="<u4")
            diff = w0 ^ w1
            j = k // cpw
            assert all(diff[i] == 0 for i in range(8) if i != j)
            if q2[k] != q[k]:
                other_half = 0x0000FFFF if (k % cpw) % 2 else 0xFFFF0000
                assert int(diff[j]) != 0 and (int(diff[j]) & other_half) == 0
        # equal code pairs (2i, 2i+1) give equal halves
        qp = rng.integers(-z, z, size=bpb // 2)
        qp[0] = -z
        q = np.repeat(qp, 2)
        words = np.frombuffer(o.pack(t, (d * q).astype(np.float32)[None, :])[0, 2:].tobytes(),
                              dtype="<u4")
        assert np.array_equal(words & 0xFFFF, words >> 16)
        if t == PN3T:
            q = np.full(bpb, z - 1)
            q[0] = -z
            words = np.frombuffer(o.pack(t, (d * q).astype(np.float32)[None, :])[0, 2:].tobytes(),
                                  dtype="<u4")
            assert np.all(words & 0x80008000 == 0)
            raw = o.pack(t, (d * q).astype(np.float32)[None, :])
            flipped = raw.copy()
            fw = np.frombuffer(flipped[0, 2:].tobytes(), dtype="<u4") | 0x80008000
            flipped[0, 2:] = np.frombuffer(fw.astype("<u4").tobytes(), dtype=np.uint8)
            assert np.array_equal(o.unpack(t, raw, bpb), o.unpack(t, flipped, bpb))


def pin_every_half_round_trips(o):
    # All 2^15 (pn3t, bits 15 cleared) / 2^16 (pn4t) values of one half: decode,
    # re-quantise, and the bytes come back (word 7 holds a code 0 so the scale is
    # recovered exactly).
    for t in TYPES:
        bpb, cpw, bits, z = GEOMETRY[t]
        span = 1 << (bits * (cpw // 2))
        h = np.arange(span, dtype=np.uint32)
        blk = np.zeros((span, 34), dtype=np.uint8)
        blk[:, 0:2] = np.frombuffer(np.float16(0.125).tobytes(), dtype=np.uint8)
        mid = _replicate(z, bits, cpw // 2)
        words = np.empty((span, 8), dtype="<u4")
        words[:, :] = mid
        words[:, 0] = h | (h << 16)
        words[:, 7] = mid & 0xFFFF0000          # low half all code 0 -> step -z
        blk[:, 2:] = words.view(np.uint8).reshape(span, 32)
        w = o.unpack(t, blk, bpb)
        assert np.array_equal(o.pack(t, w), blk)


def pin_full_range_and_bound(o):
    rng = np.random.default_rng(3)
    for t in TYPES:
        bpb, _, _, z = GEOMETRY[t]
        N, nb = 64, 24
        v = (0.02 * rng.standard_normal((N, nb * bpb))).astype(np.float32)
        v[:8] *= np.float32(1e-4)               # small scales, subnormal fp16 d
        v[8:16] *= np.float32(300.0)
        W = o.pack(t, v)
        w = o.unpack(t, W, nb * bpb)
        blocks = W.reshape(N, nb, 34)
        d = f16_bits_to_f64(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
        vb = v.reshape(N, nb, bpb).astype(np.float64)
        wb = w.reshape(N, nb, bpb).astype(np.float64)
        jmax = np.argmax(np.abs(vb), axis=2)    # numpy: first index on ties
        a = np.take_along_axis(vb, jmax[:, :, None], axis=2)[:, :, 0]
        nz = d != 0
        # largest weight decodes to step -z: d*(-z), and d's sign is opposite a's
        dec = np.take_along_axis(wb, jmax[:, :, None], axis=2)[:, :, 0]
        assert np.array_equal(dec[nz], -z * d[nz])
        assert np.all(np.sign(d[nz]) == -np.sign(a[nz]))
        # some weight uses the full range in every non-zero block
        steps = wb / np.where(nz, d, 1.0)[:, :, None]
        assert np.all(steps[nz].min(axis=1) == -z)
        assert np.all(steps == np.round(steps)) and steps.min() >= -z and steps.max() <= z - 1
        # rounding error: within half a step unless clamped at the top of the range
        ratio = vb / np.where(nz, d, 1.0)[:, :, None]
        err = np.abs(vb - wb)
        step = np.broadcast_to(np.abs(d)[:, :, None], vb.shape)
        nzb = np.broadcast_to(nz[:, :, None], vb.shape)
        clamped = ratio > (z - 1) + 0.5
        inner = ~clamped & nzb
        assert np.all(err[inner] <= step[inner] * 0.5 * (1 + 2.0 ** -20))
        assert np.all(err[clamped] <= step[clamped] * 1.5 * (1 + 2.0 ** -9))
        # round trip: re-quantising the decoded weights gives the same bytes
        assert np.array_equal(o.pack(t, w), W)


def pin_on_grid_lossless(o):
    rng = np.random.default_rng(5)
    for t in TYPES:
        bpb, _, _, z = GEOMETRY[t]
        w, d, q = on_grid_weights(rng, t, 32, 10)
        W = o.pack(t, w)
        assert np.array_equal(o.unpack(t, W, w.shape[1]), w)
        blocks = W.reshape(32, 10, 34)
        dd = f16_bits_to_f64(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
        assert np.array_equal(dd, d)


def pin_special_blocks(o):
    for t in TYPES:
        bpb, cpw, bits, z = GEOMETRY[t]
        zero_word = _replicate(z, bits, cpw // 2)
        zero_block = _block_bytes(0, [zero_word] * 8)
        # all-zero block and a block whose scale underflows fp16 -> the zero block
        for vals in (np.zeros(bpb), np.full(bpb, -0.0), np.full(bpb, 1e-9), np.linspace(-1e-9, 2e-9, bpb)):
            W = o.pack(t, vals.astype(np.float32)[None, :])
            assert W.tobytes() == zero_block
        # first index wins a tie of magnitudes: +a before -a -> d < 0
        v = np.zeros(bpb, dtype=np.float32)
        v[3], v[9] = 0.5, -0.5
        W = o.pack(t, v[None, :])
        assert f16_bits_to_f64([int(W[0, 0]) | (int(W[0, 1]) << 8)])[0] == -0.5 / z
        v[3], v[9] = -0.5, 0.5
        W = o.pack(t, v[None, :])
        assert f16_bits_to_f64([int(W[0, 0]) | (int(W[0, 1]) << 8)])[0] == 0.5 / z
        # the zero code decodes to a zero with the sign of d*0
        for dbits in (0xBC00, 0x3C00, 0x8000, 0x0000, 0x0001, 0x8001):
            blk = np.frombuffer(_block_bytes(dbits, [zero_word] * 8), dtype=np.uint8)[None, :]
            w = o.unpack(t, blk, bpb)
            assert np.all(w == 0)
            assert np.all(np.signbit(w) == bool(dbits & 0x8000))
        # a scale beyond fp16 saturates at 65504 with the block's sign
        v = np.zeros(bpb, dtype=np.float32)
        v[0] = -1e7
        W = o.pack(t, v[None, :])
        assert (int(W[0, 0]) | (int(W[0, 1]) << 8)) == 0x7BFF


def pin_gemv_exact_tiny(o):
    # Brute force: K of one or two blocks, exact rational sums of on-grid weights
    # times fp16 activations; the oracle rounds its fp64 sum to fp32 once.
    rng = np.random.default_rng(13)
    for t in TYPES:
        bpb, _, _, z = GEOMETRY[t]
        for nb in (1, 2):
            K = nb * bpb
            w, _, _ = on_grid_weights(rng, t, 4, nb)
            x = rng.standard_normal((8, K)).astype(np.float16)
            y, a = o.gemv(t, o.pack(t, w), K, x)
            for m in range(8):
                for r in range(4):
                    terms = [Fraction(float(w[r, k])) * Fraction(float(x[m, k])) for k in range(K)]
                    exact = sum(terms, Fraction(0))
                    absx = sum((abs(p) for p in terms), Fraction(0))
                    tol = Fraction(K, 2 ** 52) * absx + Fraction(abs(float(np.spacing(np.float32(float(exact))))))
                    assert abs(Fraction(float(y[m, r])) - exact) <= tol
                    assert abs(Fraction(float(a[m, r])) - absx) <= Fraction(K, 2 ** 52) * absx


def pin_gemv_independent(o):
    # On-grid weights are known without decoding; their product with x in fp64
    # (numpy) checks rows, tokens, blocks and signs of the oracle's GEMV.
    rng = np.random.default_rng(17)
    for t in TYPES:
        bpb, _, _, z = GEOMETRY[t]
        nb, N, M = 9, 37, 5
        w, _, _ = on_grid_weights(rng, t, N, nb, scale_range=(-9, -5))
        x = rng.standard_normal((M, nb * bpb)).astype(np.float16)
        y, a = o.gemv(t, o.pack(t, w), nb * bpb, x)
        ref = x.astype(np.float64) @ w.astype(np.float64).T
        absref = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T
        assert np.all(np.abs(y - ref) <= 1e-12 * absref + np.abs(ref) * 2.0 ** -24)
        assert np.allclose(a, absref, rtol=1e-12, atol=0)
        # one-hot x returns a column of the weights; all-ones x returns row sums
        k = int(rng.integers(0, nb * bpb))
        e = np.zeros((1, nb * bpb), dtype=np.float16)
        e[0, k] = 1.0
        assert np.array_equal(o.gemv(t, o.pack(t, w), nb * bpb, e, want_abs=False)[0], w[:, k])
        ones = np.ones((1, nb * bpb), dtype=np.float16)
        rows = o.gemv(t, o.pack(t, w), nb * bpb, ones, want_abs=False)[0].astype(np.float64)
        assert np.all(np.abs(rows - w.astype(np.float64).sum(axis=1)) <= np.abs(rows) * 2.0 ** -24)
        # linearity in x
        x1 = rng.standard_normal((1, nb * bpb)).astype(np.float16)
        x2 = rng.standard_normal((1, nb * bpb)).astype(np.float16)
        x12 = (x1.astype(np.float32) + x2.astype(np.float32)).astype(np.float16)
        Wp = o.pack(t, w)
        lhs, al = o.gemv(t, Wp, nb * bpb, x12)
        y1, a1 = o.gemv(t, Wp, nb * bpb, x1)
        y2, a2 = o.gemv(t, Wp, nb * bpb, x2)
        rounding = np.abs(w.astype(np.float64)) @ np.abs(x12.astype(np.float64) - x1.astype(np.float64) - x2.astype(np.float64)).T
        assert np.all(np.abs(lhs - (y1 + y2)).T <= rounding + 1e-6 * (a1 + a2 + al).T)


# ------------------------------------------------------ Hadamard rotation ----

def pin_hadamard_worked(o):
    # hand-derived rotations of small blocks (tests/golden/hadamard_worked.txt)
    for case in read_hadamard_cases():
        got = o.hadamard(case["x"][None, :], case["block"])[0]
        assert np.array_equal(got.view(np.uint16), case["out"]), case["name"]


def pin_hadamard_dense(o):
    # the fp32 values before rounding equal H_B x / sqrt(B) computed densely in
    # fp64 (Sylvester matrix by numpy) up to the fp32 rounding of log2(B)
    # butterfly stages and one scale; the fp16 output is their rounding (numpy's)
    rng = np.random.default_rng(23)
    for B, K, M in ((2, 6, 2), (4, 12, 3), (8, 40, 2), (64, 192, 2), (1024, 2048, 2), (2048, 6144, 1),
                    (4096, 8192, 1)):
        x = rng.standard_normal((M, K)).astype(np.float16)
        out, o32 = o.hadamard(x, B, want_f32=True)
        m = int(math.log2(B))
        xb = x.astype(np.float64).reshape(M, K // B, B)
        ref = (xb @ sylvester_hadamard(B).T / math.sqrt(B)).reshape(M, K)
        bound = (m + 2) * 2.0 ** -24 * (np.abs(xb).sum(axis=2, keepdims=True) / math.sqrt(B))
        bound = np.broadcast_to(bound, xb.shape).reshape(M, K)
        assert np.all(np.abs(o32.astype(np.float64) - ref) <= bound), B
        assert np.array_equal(out.view(np.uint16), o32.astype(np.float16).view(np.uint16)), B


def pin_hadamard_structure(o):
    # one-hot rows give +-1/sqrt(B) everywhere; constant rows give sqrt(B) times
    # the constant in slot 0 and zeros elsewhere; rotating twice gives x back
    # up to the two fp16 roundings; a row's blocks are rotated independently
    for B in (2, 4, 8, 16, 256, 2048):
        K = 2 * B
        e = np.zeros((1, K), dtype=np.float16)
        e[0, B + 3 % B] = 1.0
        _, o32 = o.hadamard(e, B, want_f32=True)
        assert np.all(o32[0, :B] == 0.0)
        assert np.allclose(np.abs(o32[0, B:]), 1.0 / math.sqrt(B), rtol=2.0 ** -22, atol=0)
        c = np.full((1, K), 0.5, dtype=np.float16)
        _, o32 = o.hadamard(c, B, want_f32=True)
        for blk in range(2):
            v = o32[0, blk * B:(blk + 1) * B].astype(np.float64)
            assert v[0] == pytest.approx(0.5 * math.sqrt(B), rel=2.0 ** -22) and np.all(v[1:] == 0.0)
        rng = np.random.default_rng(B)
        x = rng.standard_normal((2, K)).astype(np.float16)
        back = o.hadamard(o.hadamard(x, B), B).astype(np.float64)
        assert np.all(np.abs(back - x.astype(np.float64)) <= 2.0 ** -9 * np.abs(x).max() * 4)


def _uniform_block(pn_type, dbits, j):
    """One block whose every code is n = j + z, with scale bits dbits."""
    bpb, cpw, bits, z = GEOMETRY[pn_type]
    word = _replicate(j + z, bits, cpw // 2)
    return np.frombuffer(_block_bytes(dbits, [word] * 8), dtype=np.uint8)[None, :]


def pin_unpack_f16_worked(o):
    # Hand-derived fp16 roundings of the exact product d*(n - z) (reading R11):
    # (1 + 2^-10)*3 = 3 + 3*2^-10 is halfway between two fp16 values and goes up
    # to the even one, (1 + 3*2^-10)*3 is halfway and goes down to the even one,
    # (1 + 2^-10)*7 rounds up, products on the fp16 grid stay exact, 65504*2
    # overflows to inf, 2^-24*3 is the subnormal 3*2^-24, and -d*0 is -0.
    cases = [(PN3T, 0x3C01, 3, 0x4202), (PN3T, 0x3C03, 3, 0x4204), (PN3T, 0x3C01, -3, 0xC202),
             (PN3T, 0x3C01, 2, 0x4001), (PN3T, 0x3C01, -4, 0xC401), (PN4T, 0x3C01, 7, 0x4702),
             (PN4T, 0x7BFF, 1, 0x7BFF), (PN4T, 0x7BFF, 2, 0x7C00), (PN3T, 0x7BFF, -4, 0xFC00),
             (PN3T, 0x0001, 3, 0x0003), (PN3T, 0xBC01, 0, 0x8000), (PN4T, 0x3C00, -8, 0xC800)]
    for t, dbits, j, want in cases:
        bpb = GEOMETRY[t][0]
        got = o.unpack_f16(t, _uniform_block(t, dbits, j), bpb)
        assert np.all(got.view(np.uint16) == want), (t, hex(dbits), j)


def pin_unpack_f16_is_rounded_decode(o):
    # Each reconstructed weight is numpy's fp16 rounding (an independent IEEE
    # implementation) of the pinned exact decode, for scales across the whole
    # fp16 range, every code, and several blocks and rows.
    rng = np.random.default_rng(29)
    for t in TYPES:
        bpb, cpw, bits, z = GEOMETRY[t]
        nb, N = 3, 40
        W = np.zeros((N, nb * 34), dtype=np.uint8)
        for r in range(N):
            for b in range(nb):
                dbits = int(rng.integers(0, 0x7C00)) | (int(rng.integers(0, 2)) << 15)
                words = [int(v) for v in rng.integers(0, 2 ** 32, size=8, dtype=np.uint64)]
                W[r, b * 34:(b + 1) * 34] = np.frombuffer(_block_bytes(dbits, words), dtype=np.uint8)
        with np.errstate(over="ignore"):
            want = o.unpack(t, W, nb * bpb).astype(np.float16)
        got = o.unpack_f16(t, W, nb * bpb)
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), t


def pin_gemm_f16_exact_tiny(o):
    # Brute force with exact rationals: the oracle's GEMM is the fp32 rounding
    # of sum_k w[n][k] x[m][k]; rows, tokens and the abs sum checked one by one.
    rng = np.random.default_rng(31)
    N, K, M = 3, 24, 4
    w = (0.05 * rng.standard_normal((N, K))).astype(np.float16)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y, a = o.gemm_f16(w, x)
    assert y.shape == (M, N)
    for m in range(M):
        for n in range(N):
            terms = [Fraction(float(w[n, k])) * Fraction(float(x[m, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            absx = sum((abs(p) for p in terms), Fraction(0))
            tol = Fraction(K, 2 ** 52) * absx + Fraction(abs(float(np.spacing(np.float32(float(exact))))))
            assert abs(Fraction(float(y[m, n])) - exact) <= tol
            assert abs(Fraction(float(a[m, n])) - absx) <= Fraction(K, 2 ** 52) * absx


def pin_gemm_f16_matches_gemv_on_grid(o):
    # Scales with a 7-bit mantissa times steps of at most 3 bits need at most
    # 11 significant bits, so those weights are exact in fp16: the GEMM of the
    # reconstructed weights must then equal the (pinned) PN GEMV bit for bit,
    # and a one-hot x returns a column of the reconstructed weights.
    rng = np.random.default_rng(37)
    for t in TYPES:
        bpb, _, _, z = GEOMETRY[t]
        nb, N, M = 5, 21, 6
        d = (rng.choice([-1.0, 1.0], size=(N, nb)) * (1.0 + 8 * rng.integers(0, 128, size=(N, nb)) / 1024.0)
             * np.exp2(rng.integers(-9, -5, size=(N, nb)).astype(np.float64)))
        q = rng.integers(-z, z, size=(N, nb * bpb))
        q[:, ::bpb] = -z                                  # one full-range step per block
        w = (np.repeat(d, bpb, axis=1) * q).astype(np.float32)
        assert np.array_equal(w.astype(np.float16).astype(np.float32), w)
        W = o.pack(t, w)
        assert np.array_equal(o.unpack(t, W, nb * bpb), w)
        x = rng.standard_normal((M, nb * bpb)).astype(np.float16)
        w16 = o.unpack_f16(t, W, nb * bpb)
        assert np.array_equal(w16.astype(np.float32), w)
        assert np.array_equal(o.gemm_f16(w16, x, want_abs=False), o.gemv(t, W, nb * bpb, x, want_abs=False))
        k = int(rng.integers(0, nb * bpb))
        e = np.zeros((1, nb * bpb), dtype=np.float16)
        e[0, k] = 1.0
        assert np.array_equal(o.gemm_f16(w16, e, want_abs=False)[0], w[:, k])


# ---------------------------------------------------------------- GPTQ ----
# Reading R12: the published GPTQ procedure (Frantar et al., ICLR 2023,
# Algorithm 1) with PN blocks as its groups.  Its pins: a Hessian without
# off-diagonal terms leaves nothing to feed forward, so the result is the
# pinned round-to-nearest packer's; an independent fp64 restatement in the
# optimal-brain-quantiser form (explicit inverse, downdated after every
# column) gives the same codes and scales; and on correlated inputs the
# feedback lowers the output error below round-to-nearest's.

def _gptq_reference(pn_type, w, X, damp):
    """Decoded weights [N][K] of GPTQ in the explicit-inverse form (numpy fp64)."""
    bpb, _, _, z = GEOMETRY[pn_type]
    N, K = w.shape
    Xd = X.astype(np.float64)
    H = 2.0 * Xd.T @ Xd
    H += damp * np.mean(np.diag(H)) * np.eye(K)
    Hinv = np.linalg.inv(H)
    W = w.astype(np.float64).copy()
    out = np.zeros((N, K))
    d = np.zeros(N, dtype=np.float32)
    for k in range(K):
        if k % bpb == 0:
            blk = W[:, k:k + bpb].astype(np.float32)
            j = np.argmax(np.abs(blk), axis=1)                  # first index on ties
            a = blk[np.arange(N), j]
            d = (a / np.float32(-z)).astype(np.float16).astype(np.float32)
        v = W[:, k].astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = np.clip(np.rint(v / np.where(d == 0, np.float32(1), d)), -z, z - 1).astype(np.float32)
        q = np.where(d == 0, np.float32(0), q)
        wq = (d * q).astype(np.float32).astype(np.float64)
        out[:, k] = wq
        err = (W[:, k] - wq) / Hinv[k, k]
        W[:, k + 1:] -= np.outer(err, Hinv[k, k + 1:])
        Hinv = Hinv - np.outer(Hinv[:, k], Hinv[k, :]) / Hinv[k, k]
    return out


def pin_gptq_diagonal_is_rtn(o):
    rng = np.random.default_rng(41)
    for t in (PN3T, PN4T):
        bpb = GEOMETRY[t][0]
        K = 2 * bpb
        w = (0.02 * rng.standard_normal((5, K))).astype(np.float32)
        X = np.diag(rng.uniform(0.5, 2.0, K)).astype(np.float32)   # orthogonal columns: H is diagonal
        assert np.array_equal(o.gptq(t, w, X, 0.01), o.pack(t, w))


def pin_gptq_matches_obq(o):
    rng = np.random.default_rng(42)
    for t in (PN3T, PN4T):
        bpb = GEOMETRY[t][0]
        N, K, n = 6, 2 * bpb, 3 * bpb
        w = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
        A = rng.standard_normal((K, K)) * 0.3 + np.eye(K)
        X = (rng.standard_normal((n, K)) @ A).astype(np.float32)
        got = o.unpack(t, o.gptq(t, w, X, 0.01), K).astype(np.float64)
        want = _gptq_reference(t, w, X, 0.01)
        assert np.array_equal(got, want)


def pin_gptq_beats_rtn(o):
    rng = np.random.default_rng(43)
    for t in (PN3T, PN4T):
        bpb = GEOMETRY[t][0]
        N, K, n = 16, 3 * bpb, 4 * bpb
        w = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
        A = rng.standard_normal((K, K)) * 0.5 + np.eye(K)
        X = (rng.standard_normal((n, K)) @ A).astype(np.float32)
        e_gptq = np.linalg.norm((w - o.unpack(t, o.gptq(t, w, X, 0.01), K)).astype(np.float64) @ X.T.astype(np.float64))
        e_rtn = np.linalg.norm((w - o.unpack(t, o.pack(t, w), K)).astype(np.float64) @ X.T.astype(np.float64))
        assert e_gptq < 0.8 * e_rtn, (e_gptq, e_rtn)


ALL_PINS = [pin_block_geometry, pin_worked_blocks, pin_fp16_conversion, pin_decode_exact_all_scales,
            pin_half_structure, pin_every_half_round_trips, pin_full_range_and_bound,
            pin_on_grid_lossless, pin_special_blocks, pin_gemv_exact_tiny, pin_gemv_independent,
            pin_hadamard_worked, pin_hadamard_dense, pin_hadamard_structure,
            pin_unpack_f16_worked, pin_unpack_f16_is_rounded_decode, pin_gemm_f16_exact_tiny,
            pin_gemm_f16_matches_gemv_on_grid, pin_gptq_diagonal_is_rtn, pin_gptq_matches_obq,
            pin_gptq_beats_rtn]


# ------------------------------------------------------------------- tests ----

@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(oracle, pin):
    pin(oracle)


def test_oracle_rejects_bad_arguments(oracle):
    with pytest.raises(ValueError):
        oracle.pack(PN3T, np.zeros((2, 64), dtype=np.float32))
    with pytest.raises(ValueError):
        oracle.unpack(PN4T, np.zeros((2, 34), dtype=np.uint8), 80)
    assert oracle.lib.oracle_pack(99, None, 1, 80, None) != 0
    x = np.zeros((1, 24), dtype=np.float16)
    for block in (3, 1, 8192, 16):       # not a power of two, too small, too large, not dividing K
        with pytest.raises(ValueError):
            oracle.hadamard(x if block != 8192 else np.zeros((1, 8192), dtype=np.float16), block)


def test_gemv_threads_match_single(oracle):
    rng = np.random.default_rng(1)
    w = (0.02 * rng.standard_normal((33, 160))).astype(np.float32)
    x = rng.standard_normal((3, 160)).astype(np.float16)
    W = oracle.pack(PN3T, w)
    assert np.array_equal(oracle.gemv_threads(PN3T, W, 160, x, 4), oracle.gemv(PN3T, W, 160, x, want_abs=False))


# Each mutation edits one expression of a copy of the oracle source.  Every one
# is a plausible slip (a dropped term, a wrong sign or index, a transposed
# operand, a different rounding); some pin must fail for each.
MUTATIONS = {
    "codes_straddle": ("return 16 * (c & 1) + f->bits * (c >> 1);", "return f->bits * c;"),
    "halves_swapped": ("return 16 * (c & 1) + f->bits * (c >> 1);", "return 16 * (1 - (c & 1)) + f->bits * (c >> 1);"),
    "words_interleaved": ("static int code_word(const oracle_fmt* f, int k) { return k / f->per_word; }",
                          "static int code_word(const oracle_fmt* f, int k) { (void)f; return k % 8; }"),
    "zero_point_sign": ("out[k] = d * (float)(n - f->zero);", "out[k] = d * (float)(n + f->zero);"),
    "zero_point_value": ("f->per_block = 80; f->per_word = 10; f->bits = 3; f->zero = 4;",
                         "f->per_block = 80; f->per_word = 10; f->bits = 3; f->zero = 3;"),
    "tie_last_index": ("++j) {\n        if (fabsf(v[j]) > amax)", "++j) {\n        if (fabsf(v[j]) >= amax)"),
    "unsigned_step": ("float d32 = a / (float)(-z);", "float d32 = a / (float)(z);"),
    "truncating_codes": ("float q = rintf(v[k] / d);", "float q = truncf(v[k] / d);"),
    "fp16_ties_away": ("if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) r++;", "if (rem >= 0x1000u) r++;"),
    "scale_last": ("uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));",
                   "uint16_t dbits = (uint16_t)(blk[32] | (blk[33] << 8));"),
    "token_zero_only": ("double xv = (double)oracle_half_to_float(xm[b * f.per_block + k]);",
                        "double xv = (double)oracle_half_to_float(x[b * f.per_block + k]);"),
    "last_block_dropped": ("for (int64_t b = 0; b < nb; ++b) {\n                decode_block",
                           "for (int64_t b = 0; b + 1 < nb; ++b) {\n                decode_block"),
    "rows_reversed": ("y[(int64_t)m * N + r] = (float)acc;", "y[(int64_t)m * N + (N - 1 - r)] = (float)acc;"),
    "fp32_accumulate": ("double acc = 0.0, acc_abs = 0.0;", "float acc = 0.0f; double acc_abs = 0.0;"),
    "hadamard_difference_sign": ("v[i + h] = a - b;", "v[i + h] = b - a;"),
    "hadamard_odd_scale": ("if (m % 2) s = ldexpf(sqrt2, -(m + 1) / 2);", "if (m % 2) s = ldexpf(1.0f, -(m + 1) / 2);"),
    "hadamard_block_offset": ("const int64_t off = (int64_t)row * K + base;", "const int64_t off = (int64_t)row * K;"),
    "hadamard_partner": ("const float a = v[i], b = v[i + h];", "const float a = v[i], b = v[(i + h) % B];\n                    if (h > 1) continue;"),
    "f16_block_offset": ("w16[r * K + b * f.per_block + k] = oracle_float_to_half(wblk[k]);",
                         "w16[r * K + k] = oracle_float_to_half(wblk[k]);"),
    "f16_scale_rounded_first": ("w16[r * K + b * f.per_block + k] = oracle_float_to_half(wblk[k]);",
                                "w16[r * K + b * f.per_block + k] = oracle_float_to_half(wblk[k] + wblk[k] * 0x1p-12f);"),
    "gemm_transposed_weights": ("double p = (double)oracle_half_to_float(wrow[k]) * (double)oracle_half_to_float(xrow[k]);",
                                "double p = (double)oracle_half_to_float(w16[k * N + n]) * (double)oracle_half_to_float(xrow[k]);"),
    "gemm_fp32_accumulate": ("double sum = 0.0, sum_abs = 0.0;", "float sum = 0.0f; double sum_abs = 0.0;"),
    "gemm_token_zero": ("const uint16_t* xrow = x + (int64_t)m * K;", "const uint16_t* xrow = x;"),
    "gptq_no_feedback": ("for (int64_t j = k + 1; j < K; ++j) W[r * K + j] -= err * C[j * K + k];",
                         "for (int64_t j = k + 1; j < K; ++j) W[r * K + j] -= 0.0 * err * C[j * K + k];"),
    "gptq_factor_of_h": ("if (!cholesky_lower(Hi, C, K))", "if (!cholesky_lower(H, C, K))"),
    "gptq_transposed_factor": ("W[r * K + j] -= err * C[j * K + k];", "W[r * K + j] -= err * C[k * K + j] + err * C[j * K + k] * (j == k + 1);"),
    "gptq_scale_from_original": ("cur[j] = (float)W[r * K + b * f.per_block + j];", "cur[j] = w[r * K + b * f.per_block + j];"),
    "gptq_no_damping": ("H[i * K + i] += damp * mean_diag;", "H[i * K + i] += 1e-9 * damp * mean_diag;"),
    "gptq_error_not_scaled": ("const double err = (W[r * K + k] - (double)wq) / ukk;",
                              "const double err = (W[r * K + k] - (double)wq);"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name):
    find, repl = MUTATIONS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(find) == 1, f"mutation anchor not found: {name}"
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as fh:
            fh.write(src.replace(find, repl))
        lib = oracle_mod.compile_oracle(path, os.path.join(tmp, "libmutant.so"))
        mutant = oracle_mod.Oracle(oracle_mod.load(lib))
        failed = []
        for pin in ALL_PINS:
            try:
                pin(mutant)
            except Exception as exc:  # noqa: BLE001 - any failure counts as caught
                failed.append((pin.__name__, type(exc).__name__))
        assert failed, f"no pin caught mutation {name}"
