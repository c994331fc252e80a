"""The balanced schedule's cut rule, as mla_decode_plan documents it, against
the bounds the plan sizes the workspace with.

Rows of g key groups are laid end to end; the sequence is cut every
W = cdiv(total, pairs) groups; a cut closer than W / 8 to a row's ends is
dropped. The plan reserves rows + pairs items and 2 * pairs partial slots;
the device list must never need more, whatever the lengths. This checks the
rule itself on adversarial length sets (the GPU tests read the device's list
back and check it piece by piece).
"""
import numpy as np
import pytest


def cut_rule(groups, tiles, pairs):
    """The CTA pair's rule. W is a worker's share of all row tiles' groups;
    the units' g groups are laid end to end and cut at the multiples of W
    inside each unit, none within W / 8 of its ends; all T row tiles of a
    unit are cut there. Returns the rows (one per tile), each row's piece
    sizes, and W."""
    total = sum(g * t for g, t in zip(groups, tiles))
    W = -(-total // pairs) if total > 0 else 1
    d = W // 8
    rows, pieces, pos = [], [], 0
    for g, t in zip(groups, tiles):
        a = pos
        lo, hi = a + d + 1, a + g - d - 1
        bounds = []
        if g > 1 and hi >= lo and t > 0:
            c = -(-lo // W) * W
            while c <= hi:
                bounds.append(c - a)
                c += W
        edges = [0] + bounds + [g]
        sizes = [edges[i + 1] - edges[i] for i in range(len(edges) - 1)]
        for _ in range(t):
            rows.append(g)
            pieces.append(list(sizes))
        pos += g
    return rows, pieces, W


def ranked_list(groups, tiles, pairs):
    """The list a batch of at most 256 units gets: the cut rule's pieces,
    enumerated unit by unit (piece j of unit u), ordered by size, largest
    first, ties in enumeration order; a piece's T row tiles are consecutive
    items. A split unit (k > 1 pieces) owns k T partial slots from the prefix
    over the units before it, tile t's piece j at slot base + t k + j.
    Returns (unit, tile, first key, end key, slot or -1) per item."""
    _, pieces, _ = cut_rule(groups, tiles, pairs)
    enum, base, r = [], 0, 0
    for u, (g, t) in enumerate(zip(groups, tiles)):
        if t == 0:
            continue
        sizes = pieces[r]
        r += t
        k = len(sizes)
        edge = 0
        for j, size in enumerate(sizes):
            enum.append((size, u, t, edge, j, k, base))
            edge += size
        if k > 1:
            base += k * t
    order = sorted(range(len(enum)), key=lambda i: (-enum[i][0], i))
    items = []
    for i in order:
        size, u, t, edge, j, k, b = enum[i]
        for tt in range(t):
            items.append((u, tt, edge * 128, (edge + size) * 128, b + tt * k + j if k > 1 else -1))
    return items


@pytest.mark.parametrize("name", ["equal", "one_long", "zeros", "mixed_tiles"])
def test_ranked_list_covers_every_row_once(name):
    """The small-batch list is a permutation of the cut rule's pieces, its
    sizes never grow, and the split units' slots are distinct."""
    groups, tiles = CASES[name]
    items = ranked_list(groups, tiles, 76)
    _, pieces, _ = cut_rule(groups, tiles, 76)
    assert len(items) == sum(len(p) for p in pieces)
    sizes = [(ke - kb) // 128 for _, _, kb, ke, _ in items]
    assert all(a >= b for a, b in zip(sizes, sizes[1:]))
    slots = [s for *_, s in items if s >= 0]
    assert len(set(slots)) == len(slots)
    for u, (g, t) in enumerate(zip(groups, tiles)):
        for tt in range(t):
            mine = sorted((kb, ke) for uu, ti, kb, ke, _ in items if uu == u and ti == tt)
            assert mine[0][0] == 0 and mine[-1][1] == g * 128
            assert all(a[1] == b[0] for a, b in zip(mine, mine[1:]))


CASES = {
    "equal": ([128] * 52, [1] * 52),
    "one_long": ([8192], [1]),
    "many_short": ([1] * 5000, [1] * 5000),
    "zeros": ([0] * 10, [1] * 10),
    "mixed_tiles": ([300, 5, 0, 4000, 77], [4, 1, 2, 3, 1]),
}


@pytest.mark.parametrize("pairs", [1, 7, 76])
@pytest.mark.parametrize("name", sorted(CASES) + ["random"])
def test_cut_rule_stays_inside_the_workspace(name, pairs):
    if name == "random":
        rng = np.random.default_rng(pairs)
        groups = rng.integers(0, 600, size=300).tolist()
        tiles = rng.integers(1, 5, size=300).tolist()
    else:
        groups, tiles = CASES[name]
    rows, pieces, W = cut_rule(groups, tiles, pairs)
    tmax = max(tiles)
    n_items = sum(len(p) for p in pieces)
    slots = sum(len(p) for p in pieces if len(p) > 1)
    assert n_items <= len(rows) + tmax * pairs     # plan: max_items = rows + T_max * pairs
    assert slots <= 2 * tmax * pairs               # plan: split_items = 2 * T_max * pairs slots
    for g, p in zip(rows, pieces):
        assert sum(p) == g and all(x >= 0 for x in p)  # each row covered once
    # no sliver next to a row's ends, no piece above W; every tile of a unit
    # cut at the same keys
    r = 0
    for g, t in zip(groups, tiles):
        p = pieces[r]
        assert all(pieces[r + k] == p for k in range(t))
        if len(p) > 1:
            assert p[0] > W // 8 and p[-1] > W // 8
            assert all(x <= W for x in p[1:-1])
        r += t


def contiguous_rule(groups, tiles, workers):
    """The rows-as-N kernel's schedule: every multiple of W inside a row is a
    cut, items in sequence order, a piece owned by the worker its first group
    falls to (an empty row: the worker of its position, at most the last).
    Returns the items [(unit, tile, first group, end group, partial slot or
    -1)], worker_first and W."""
    total = sum(g * t for g, t in zip(groups, tiles))
    W = -(-total // workers) if total > 0 else 1
    items, owners, pos, slot = [], [], 0, 0
    for u, (g, t) in enumerate(zip(groups, tiles)):
        for tt in range(t):
            a, b = pos, pos + g
            cuts = list(range((a // W + 1) * W, b, W)) if g > 1 else []
            bounds = [a] + cuts + [b]
            k = len(bounds) - 1
            for j in range(k):
                items.append((u, tt, bounds[j] - a, bounds[j + 1] - a, slot + j if k > 1 else -1))
                owners.append(min(bounds[j] // W, workers - 1))
            if k > 1:
                slot += k
            pos = b
    first = [int(np.searchsorted(owners, w, side="left")) for w in range(workers)] + [len(items)]
    return items, first, W


@pytest.mark.parametrize("workers", [1, 7, 76, 152])
@pytest.mark.parametrize("name", sorted(CASES) + ["random"])
def test_contiguous_rule_balances_exactly(name, workers):
    if name == "random":
        rng = np.random.default_rng(workers + 1000)
        groups = rng.integers(0, 600, size=300).tolist()
        tiles = rng.integers(1, 3, size=300).tolist()
    else:
        groups, tiles = CASES[name]
    items, first, W = contiguous_rule(groups, tiles, workers)
    rows = sum(tiles)
    total = sum(g * t for g, t in zip(groups, tiles))
    assert len(items) <= rows + workers                          # plan: max_items
    assert len({it[4] for it in items if it[4] >= 0}) == sum(it[4] >= 0 for it in items)
    assert all(it[4] < 2 * workers for it in items)              # plan: split_items slots
    assert first[0] == 0 and first[-1] == len(items) and np.all(np.diff(first) >= 0)
    # worker w's pieces are exactly the groups [w W, (w + 1) W) of the sequence
    for w in range(workers):
        load = sum(it[3] - it[2] for it in items[first[w]:first[w + 1]])
        assert load == max(0, min(W, total - w * W)), (w, load)
    # each row covered once, in order
    for u, (g, t) in enumerate(zip(groups, tiles)):
        for tt in range(t):
            mine = [it for it in items if it[0] == u and it[1] == tt]
            assert mine[0][2] == 0 and mine[-1][3] == g
            assert all(x[3] == y[2] for x, y in zip(mine, mine[1:]))
