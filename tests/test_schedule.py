"""The score/select kernel's work split, restated on the CPU.

Work row w owns tiles [wts[w], wts[w+1]) of the global tile sequence. The
split charges every work row that has tiles a penalty of P virtual tiles after
its last tile (the segment finalisation its CTA performs), cuts the virtual
sequence evenly over nC = min(grid, T) CTAs and maps the cuts back to tiles;
CTA c's start is clamped to [c, T - nC + c] and a prefix max of start - c
makes the starts strictly increasing, so every participating CTA has a tile.
A work row's segments are the CTAs from the one holding its first tile to the
one holding its last (found by search over the starts), and CTA c's part of
work row w is stored in slot c + w. These tests check, for many shapes, that
the split covers the tiles exactly once, that the segment count equals the
number of CTAs that really touch the row (so exactly one becomes the merger),
that slots are unique and inside the workspace, and that the penalty moves
tiles away from CTAs that finish a row inside their range.
"""
import numpy as np


def split(tiles, grid, penalty=0):
    wts = np.concatenate([[0], np.cumsum(tiles)]).astype(np.int64)
    T = int(wts[-1])
    nC = min(grid, T)
    nz = np.asarray(tiles) > 0
    vs = wts[:-1] + penalty * np.concatenate([[0], np.cumsum(nz)])[:-1]
    V = T + penalty * int(nz.sum())
    starts = []
    for c in range(nC + 1):
        if c == nC:
            t = T
        else:
            v = c * V // nC
            w = int(np.searchsorted(vs, v, side="right")) - 1
            t = int(wts[w] + min(v - vs[w], wts[w + 1] - wts[w]))
        starts.append(max(min(t, T - nC + c), c) - c)
    starts = np.maximum.accumulate(starts) + np.arange(nC + 1)
    return nC, [(int(starts[c]), int(starts[c + 1])) for c in range(nC)]


def cta_of(t, ranges):
    return max(c for c, (a, _) in enumerate(ranges) if a <= t)


def check(tiles, grid, penalty=0):
    starts = np.concatenate([[0], np.cumsum(tiles)])
    T = int(starts[-1])
    if T == 0:
        return None
    nC, ranges = split(tiles, grid, penalty)
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    assert all(b > a for a, b in ranges)
    assert all(ranges[c][1] == ranges[c + 1][0] for c in range(nC - 1))
    slots = set()
    for w, n in enumerate(tiles):
        if n == 0:
            continue
        rs, re = int(starts[w]), int(starts[w + 1])
        touching = [c for c, (a, b) in enumerate(ranges) if a < re and b > rs]
        c_first, c_last = cta_of(rs, ranges), cta_of(re - 1, ranges)
        assert touching == list(range(c_first, c_last + 1))
        for c in touching:
            s = c + w
            assert s not in slots and s < grid + len(tiles)
            slots.add(s)
    return ranges


def test_schedule_small_and_ragged():
    rng = np.random.default_rng(0)
    for _ in range(300):
        R = int(rng.integers(1, 40))
        tiles = rng.integers(0, 30, R)
        tiles[rng.random(R) < 0.3] = 0
        for grid in (1, 2, 7, 152, 500):
            for penalty in (0, 1, 2, 6, 12):
                check(tiles.tolist(), grid, penalty)


def test_schedule_workload_shapes():
    check([24 * 0, 0, 24, 32], 152)                        # the tiny workload: T < grid
    check([1024] * 128, 152)                                # long context
    rng = np.random.default_rng(1)
    check(((rng.integers(2048, 32769, 32) + 127) // 128).tolist(), 152)


def test_row_end_penalty_balances_finalising_ctas():
    """With the penalty, a CTA that finishes a work row inside its range gets
    fewer tiles than one that does not, by about the penalty."""
    rng = np.random.default_rng(2)
    tiles = ((rng.integers(2048, 32769, 32) + 127) // 128).tolist()
    ends = np.cumsum(tiles)
    for penalty in (0, 6):
        ranges = check(tiles, 304, penalty)
        inner = [b - a for a, b in ranges if any(a < e < b for e in ends)]
        plain = [b - a for a, b in ranges if not any(a < e < b for e in ends)]
        gap = np.mean(plain) - np.mean(inner)
        if penalty == 0:
            assert abs(gap) < 1.5
        else:
            assert penalty - 2 <= gap <= penalty + 2
