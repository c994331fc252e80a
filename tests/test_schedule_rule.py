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
    rows = [g for g, t in zip(groups, tiles) for _ in range(t)]
    total = sum(rows)
    W = -(-total // pairs) if total > 0 else 1
    d = W // 8
    pieces, pos = [], 0
    for g in rows:
        a, b = pos, pos + g
        lo, hi = a + d + 1, b - d - 1
        cuts = []
        if g > 0 and hi >= lo:
            c = -(-lo // W) * W
            while c <= hi:
                cuts.append(c)
                c += W
        bounds = [a] + cuts + [b]
        pieces.append([bounds[i + 1] - bounds[i] for i in range(len(bounds) - 1)])
        pos = b
    return rows, pieces, W


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
    n_items = sum(len(p) for p in pieces)
    slots = sum(len(p) for p in pieces if len(p) > 1)
    assert n_items <= len(rows) + pairs            # plan: max_items = rows + pairs
    assert slots <= 2 * pairs                      # plan: split_items = 2 * pairs slots
    for g, p in zip(rows, pieces):
        assert sum(p) == g and all(x >= 0 for x in p)  # each row covered once
        if len(p) > 1:                             # no sliver next to a row's ends
            assert p[0] > W // 8 and p[-1] > W // 8
            assert all(x <= W for x in p[1:-1])
