"""The decode kernel's work partition as arithmetic, checked on the host.

The kernel deals out the line of (sequence, KV head) runs by cost: tile x of
run r sits at cost position x + 3r, and CTA b takes the tiles whose cost
position lies in [b, b + 1) * ceil(cost_total / grid). Its range ends are
found by the thread that holds the sequence whose cost span contains each
end, while the prefix sum is written (no search); the walk's first piece
(the part of the range in the run holding its last tile) is recorded by the
same thread when that run is its sequence's; cursor look-ups elsewhere are
warp-parallel searches (32 chunks per round, then a ballot for the run).
This model restates those steps and checks them against a plain search of
the prefix sum: every CTA's range, every first piece, every cursor."""
import numpy as np
import pytest

PIECE_COST = 3


def div_small(a, b):
    """The kernel's quotient: a float estimate corrected to the exact one."""
    q = int(np.float32(a) / np.float32(b))
    while q > 0 and q * b > a:
        q -= 1
    while (q + 1) * b <= a:
        q += 1
    return q


def first_tile_at(scan, hkv, y, cost_total):
    """Plain definition: the first tile whose cost position is >= y."""
    total = hkv * scan[-1]
    if y >= cost_total:
        return total
    x = 0
    for r in range(hkv * len(scan)):
        s, g = divmod(r, hkv)
        nb = scan[s] - (scan[s - 1] if s else 0)
        for j in range(nb):
            if x + PIECE_COST * r >= y:
                return x
            x += 1
    return total


def owner_ends(tiles, hkv, grid, b):
    """The owner threads' computation of CTA b's range and first piece."""
    per_head = sum(tiles)
    cost_total = hkv * (per_head + PIECE_COST * len(tiles))
    cchunk = -(-cost_total // grid)
    y_lo, y_hi = b * cchunk, (b + 1) * cchunk
    ends, first, run = [None, None], None, 0
    for s, n in enumerate(tiles):
        before = run
        run += n
        c0 = hkv * (before + PIECE_COST * s)
        c1 = c0 + hkv * (n + PIECE_COST)

        def tile_at(y):
            g = div_small(y - c0, n + PIECE_COST)
            return hkv * before + g * n + min(y - c0 - g * (n + PIECE_COST), n)
        if c0 <= y_lo < c1:
            ends[0] = tile_at(y_lo)
        if c0 <= y_hi < c1:
            g = div_small(y_hi - c0, n + PIECE_COST)
            r = min(y_hi - c0 - g * (n + PIECE_COST), n)
            hi_t = hkv * before + g * n + r
            ends[1] = hi_t
            if n > 0 and (r > 0 or g > 0):
                gl = g if r > 0 else g - 1
                seg = hkv * before + gl * n
                split = max(seg, tile_at(y_lo)) if y_lo >= c0 else seg
                if hi_t > split:
                    first = (s, gl, split - seg, split)
    if y_lo >= cost_total:
        ends[0] = hkv * per_head
    if y_hi >= cost_total:
        ends[1] = hkv * per_head
    return ends, first, cost_total, cchunk


def warp_first_true(n, pred):
    lo, length = 0, n
    while length > 1:
        step = (length + 31) >> 5
        bits = [pred(min(lo + (lane + 1) * step, lo + length) - 1) for lane in range(32)]
        c = bits.index(True)
        lo += c * step
        length = min(step, length - c * step)
    return lo


def locate_warp(scan, hkv, x):
    s = warp_first_true(len(scan), lambda i: hkv * scan[i] > x)
    nb = scan[s] - (scan[s - 1] if s else 0)
    off = x - hkv * (scan[s] - nb)
    g = sum(1 for lane in range(1, hkv) if lane * nb <= off) if hkv <= 32 else off // nb
    return s, g, off - g * nb


def locate_plain(scan, hkv, x):
    per_head = x // hkv
    s = next(i for i, v in enumerate(scan) if v > per_head)
    nb = scan[s] - (scan[s - 1] if s else 0)
    off = x - hkv * (scan[s] - nb)
    return s, off // nb, off % nb


CASES = [
    ([3, 0, 7, 1, 0, 0, 12], 2, 5),
    ([1] * 40, 8, 37),
    ([0, 0, 5, 0, 9], 1, 4),
    ([86, 12, 375, 1, 44, 0, 63, 200], 8, 152),
    ([2] * 70, 33, 19),
]


@pytest.mark.parametrize("tiles,hkv,grid", CASES)
def test_range_ends_and_first_piece(tiles, hkv, grid):
    scan = list(np.cumsum(tiles))
    found = nonempty = 0
    for b in range(grid):
        (lo, hi), first, cost_total, cchunk = owner_ends(tiles, hkv, grid, b)
        assert lo == first_tile_at(scan, hkv, b * cchunk, cost_total)
        assert hi == first_tile_at(scan, hkv, (b + 1) * cchunk, cost_total)
        if lo >= hi:
            assert first is None  # nothing is copied for an empty range
            continue
        # the walk's first piece: from max(start of the run holding hi - 1, lo) to hi
        s, g, blk = locate_plain(scan, hkv, hi - 1)
        nb = tiles[s]
        seg = hi - 1 - blk
        split = max(seg, lo)
        want = (*locate_plain(scan, hkv, split), split)
        nonempty += 1
        if first is not None:
            found += 1
            assert first == want
            assert want[2] + (hi - split) <= nb  # the piece lies in one run
    assert found >= nonempty // 2  # the plan finds the first piece for most CTAs


@pytest.mark.parametrize("tiles,hkv,grid", CASES)
def test_warp_search_matches_plain_search(tiles, hkv, grid):
    scan = list(np.cumsum(tiles))
    for x in range(hkv * scan[-1]):
        assert locate_warp(scan, hkv, x) == locate_plain(scan, hkv, x)


def test_div_small_is_exact():
    rng = np.random.default_rng(0)
    for _ in range(5000):
        b = int(rng.integers(1, 5000))
        a = int(rng.integers(0, 64)) * b + int(rng.integers(0, b))
        assert div_small(a, b) == a // b
