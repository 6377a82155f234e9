"""The score/select kernel's work split, restated on the CPU.

The kernel gives CTA c (of nC = min(grid, T) participating CTAs) the tiles
[c*T/nC, (c+1)*T/nC) of the global tile sequence, finds the CTA of tile t as
((t+1)*nC - 1) // T, counts a work row's segments as c_last - c_first + 1 and
stores CTA c's part of work row w in slot c + w. These tests check that
arithmetic for many shapes: every participating CTA has a tile, the segment
count equals the number of CTAs that really touch the row (so exactly one
becomes the merger), and slots are unique and inside the workspace.
"""
import numpy as np


def split(T, grid):
    nC = min(grid, T)
    return nC, [(c * T // nC, (c + 1) * T // nC) for c in range(nC)]


def cta_of(t, T, nC):
    return ((t + 1) * nC - 1) // T


def check(tiles, grid):
    starts = np.concatenate([[0], np.cumsum(tiles)])
    T = int(starts[-1])
    if T == 0:
        return
    nC, ranges = split(T, grid)
    assert all(b > a for a, b in ranges)
    for t in range(T):
        c = cta_of(t, T, nC)
        assert ranges[c][0] <= t < ranges[c][1]
    slots = set()
    for w, n in enumerate(tiles):
        if n == 0:
            continue
        rs, re = int(starts[w]), int(starts[w + 1])
        touching = [c for c, (a, b) in enumerate(ranges) if a < re and b > rs]
        c_first, c_last = cta_of(rs, T, nC), cta_of(re - 1, T, nC)
        assert touching == list(range(c_first, c_last + 1))
        for c in touching:
            s = c + w
            assert s not in slots and s < grid + len(tiles)
            slots.add(s)


def test_schedule_small_and_ragged():
    rng = np.random.default_rng(0)
    for _ in range(300):
        R = int(rng.integers(1, 40))
        tiles = rng.integers(0, 30, R)
        tiles[rng.random(R) < 0.3] = 0
        for grid in (1, 2, 7, 152, 500):
            check(tiles.tolist(), grid)


def test_schedule_workload_shapes():
    check([24 * 0, 0, 24, 32], 152)                        # the tiny workload: T < grid
    check([1024] * 128, 152)                                # long context
    rng = np.random.default_rng(1)
    check(((rng.integers(2048, 32769, 32) + 127) // 128).tolist(), 152)
