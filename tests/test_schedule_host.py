"""Host model of the balanced schedule the MLA decode kernels derive on the GPU.

The kernels lay the sequences' tiles end to end (T tiles), charge every
sequence start kPC tiles (tile t of sequence b sits at cost t + kPC (b + 1)),
cut the cost line of length T + kPC B into parts = min(chunks, that) equal
parts, and find a tile's chunk in closed form, floor(cost * parts / total).
Chunk k starts at the first tile whose cost reaches ceil(k * total / parts),
searched as the first non-empty sequence whose last tile reaches it.  The
count of a split sequence expects one piece from every chunk between the
chunks of its first and last tile, and each chunk has two partial slots: 2c
for a piece whose sequence began earlier, 2c + 1 for one that begins in c.
This restates those rules in plain Python and checks the invariants the
count and the merge rely on, for 32- and 64-token tiles and the charges the
kernels use (2 and 3) and one more (4).
"""
import numpy as np
import pytest


def tiles_of(lens, tile):
    return [(max(0, L) + tile - 1) // tile for L in lens]


def cut_starts(n, kpc, nc):
    """First tile of every chunk (the kernels' search), plus T at the end."""
    T = sum(n)
    B = len(n)
    total = T + kpc * B
    parts = min(nc, total)
    pre = np.concatenate([[0], np.cumsum(n)]).astype(np.int64)
    starts = []
    for k in range(nc + 1):
        if k >= parts:
            starts.append(T)
            continue
        x = -(-k * total // parts)  # ceil
        g = T
        for b in range(B):
            if n[b] == 0:
                continue
            last = pre[b] + n[b] - 1 + kpc * (b + 1)
            if last >= x:
                t = x - kpc * (b + 1)
                g = max(int(t), int(pre[b]))
                break
        starts.append(g)
    return starts, total, parts, pre


def chunk_of(t, b, kpc, total, parts):
    return (t + kpc * (b + 1)) * parts // total


def check(lens, tile, kpc, nc):
    n = tiles_of(lens, tile)
    starts, total, parts, pre = cut_starts(n, kpc, nc)
    T = sum(n)
    assert starts[0] == 0 and starts[-1] == T
    assert all(starts[k] <= starts[k + 1] for k in range(nc))
    # every tile in exactly one chunk, and the closed form agrees
    owner = {}
    for k in range(nc):
        for t in range(starts[k], starts[k + 1]):
            assert t not in owner
            owner[t] = k
    assert len(owner) == T
    for b in range(len(n)):
        for t in range(pre[b], pre[b] + n[b]):
            assert chunk_of(t, b, kpc, total, parts) == owner[t], (b, t)
    # a split sequence has one piece in every chunk of its span, and the
    # count's target equals its number of pieces
    slots = {}
    for b in range(len(n)):
        if n[b] == 0:
            continue
        first, last = int(pre[b]), int(pre[b] + n[b] - 1)
        c_first = chunk_of(first, b, kpc, total, parts)
        c_last = chunk_of(last, b, kpc, total, parts)
        pieces = {owner[t] for t in range(first, last + 1)}
        assert pieces == set(range(c_first, c_last + 1)), (b, c_first, c_last, pieces)
        if c_last > c_first:
            # slots: 2 c_first + 1 for the first piece, 2c for the others
            for c in range(c_first, c_last + 1):
                s = 2 * c + 1 if c == c_first else 2 * c
                assert s not in slots, (b, c, s, slots.get(s))
                slots[s] = b
    assert all(s < 2 * nc for s in slots)


@pytest.mark.parametrize("tile,kpc", [(32, 2), (64, 3), (64, 2), (64, 4), (32, 4)])
def test_balanced_cut_invariants(tile, kpc):
    rng = np.random.default_rng(1000 * tile + kpc)
    for case in range(120):
        B = int(rng.integers(1, 140))
        nc = int(rng.choice([1, 2, 7, 76, 152, 304]))
        kind = case % 4
        if kind == 0:
            lens = rng.integers(512, 4097, size=B)       # the decode workload's mix
        elif kind == 1:
            lens = rng.integers(0, 301, size=B)          # short, some empty
        elif kind == 2:
            lens = rng.choice([0, 1, tile, tile + 1, 20000], size=B)
        else:
            lens = rng.integers(0, 2 * tile + 2, size=B)
        check([int(x) for x in lens], tile, kpc, nc)


def test_balanced_cut_workload_shapes():
    """The benchmark's cut: B = 64, contexts 512..4096, 76 clusters of 64-token
    tiles (128 heads, charge 4) and 152 CTAs of 64-token tiles (16 heads,
    charge 3): every chunk has work."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(512, 4097, size=64)]
    for nc, kpc in ((76, 4), (152, 3)):
        check(lens, 64, kpc, nc)
        starts, _, _, _ = cut_starts(tiles_of(lens, 64), kpc, nc)
        assert all(starts[k + 1] > starts[k] for k in range(nc))
