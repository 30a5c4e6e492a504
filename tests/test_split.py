"""The tensor-core GEMV's work split, checked on the host (no GPU).

pn_tc_split returns the unit ranges the kernel's thread blocks take.  The
kernel relies on them being contiguous, covering every unit once, and each
holding at least one whole tile (so that a tile cut by a range boundary has
exactly two owners, whose partial sums the kernel adds); and on the split
being a function of the call's shapes alone.
"""
from __future__ import annotations

import bisect
import random

import pytest

from bit_weight_only_pn_gb300 import pn

PN3T, PN4T = 124, 125
LAYER_27B = [(PN3T, 6144, 5120), (PN3T, 17408, 5120), (PN3T, 17408, 5120), (PN4T, 1024, 5120),
             (PN4T, 1024, 5120), (PN4T, 5120, 6144), (PN4T, 5120, 17408)]      # (type, N, K)


@pytest.fixture(scope="module", autouse=True)
def built():
    from bit_weight_only_pn_gb300 import build
    build.build()


def units_of(shapes):
    """(first unit, chunks, tiles) of each tensor, and the total."""
    out, u = [], 0
    for t, N, K in shapes:
        chunks = K // (80 if t == PN3T else 64) // 8
        tiles = (N + 15) // 16
        out.append((u, chunks, tiles))
        u += chunks * tiles
    return out, u


def check_split(shapes, M, sms):
    starts = pn.tc_split(shapes, M, sms)
    layout, total = units_of(shapes)
    max_chunks = max(c for _, c, _ in layout)
    grid = len(starts) - 1
    assert 1 <= grid <= min(sms, 256)
    assert starts[0] == 0 and starts[-1] == total
    for c in range(grid):
        assert starts[c + 1] - starts[c] >= max_chunks, (c, starts[c], starts[c + 1])
    # every tile has one or two owners: the ranges holding its first and last unit
    for base, chunks, tiles in layout:
        for tile in range(tiles):
            lo, hi = base + tile * chunks, base + (tile + 1) * chunks
            owners = bisect.bisect_right(starts, hi - 1) - bisect.bisect_right(starts, lo) + 1
            assert owners in (1, 2), (tile, owners)
    return starts


def test_layer_split_uses_every_sm():
    for M in (3, 8, 12, 16):
        starts = check_split(LAYER_27B, M, 152)
        assert len(starts) - 1 == 152


def test_random_shapes_keep_the_invariants():
    rng = random.Random(20261202)
    for _ in range(150):
        n = rng.randint(1, 8)
        shapes = []
        for _ in range(n):
            t = rng.choice((PN3T, PN4T))
            chunks = rng.randint(1, 40) if rng.random() < 0.7 else rng.randint(1, 4)
            N = rng.randint(1, 4000) if rng.random() < 0.7 else rng.randint(1, 64)
            shapes.append((t, N, chunks * 8 * (80 if t == PN3T else 64)))
        check_split(shapes, rng.randint(3, 16), rng.randint(1, 300))


def test_tiny_problems_fall_back_to_few_blocks():
    # one tile of one chunk: a single range, whatever the SM count
    assert pn.tc_split([(PN4T, 16, 512)], 8, 152) == [0, 1]
    # 3 tiles of 34 chunks: at most three blocks, each with a whole tile
    starts = check_split([(PN4T, 48, 17408)], 8, 152)
    assert len(starts) - 1 <= 3


def test_split_depends_only_on_the_shapes():
    first = {M: pn.tc_split(LAYER_27B, M, 152) for M in (3, 8, 16)}
    # fill and cycle the cache of splits with other shapes, then ask again
    for N in range(16, 16 * 40, 16):
        pn.tc_split([(PN3T, N, 5120), (PN4T, 2 * N, 4096)], 8, 152)
    for M in (3, 8, 16):
        assert pn.tc_split(LAYER_27B, M, 152) == first[M]


def test_argument_checks():
    lib = pn.lib()
    bad = [
        ([(7, 64, 5120)], 8, 152),             # unknown type
        ([(PN3T, 64, 5200)], 8, 152),          # K not a multiple of 8 blocks
        ([(PN4T, 64, 4608 + 64)], 8, 152),
        ([(PN3T, 0, 5120)], 8, 152),           # no rows
        ([(PN3T, 64, 5120)], 2, 152),          # M below the kernel's range
        ([(PN3T, 64, 5120)], 17, 152),         # M above it
        ([(PN3T, 64, 5120)], 8, 0),            # no SMs
        ([(PN3T, 64, 5120)] * 9, 8, 152),      # too many tensors
        ([], 8, 152),                          # none
    ]
    for shapes, M, sms in bad:
        with pytest.raises(pn.PnError) as err:
            pn.tc_split(shapes, M, sms)
        assert err.value.status == 1, (shapes, M, sms)
    # null pointers
    assert lib.pn_tc_split(None, None, None, 1, 8, 152, None, None) == 1
