"""The pair tiling of the symmetric outputs, and why it discards what it does (CPU).

X X^T and b A + c A A compute only the tiles on or above the diagonal of their
m x m output.  A CTA pair's tcgen05 product covers 256 x 256: two 128-row
blocks of the output (one per CTA) times two 128-column blocks.  Restated
here, in blocks of 128 for T = m / 128 blocks: pair tile (I, J), J >= I,
covers rows {2I, 2I+1} x columns {2J, 2J+1}, enumerated row by row as the
kernel's tile decode does.  The checks: every block on or above the diagonal
is computed exactly once, and the blocks computed and discarded (below the
diagonal) are one per diagonal pair tile.

That discard is the least any tiling by such units can have.  A unit covers
exactly two blocks of each block row it spans.  Block row r needs the T - r
blocks from the diagonal to the right edge, so when T - r is odd one block of
that row is computed twice or lies below the diagonal; with T even that holds
for every odd r, T/2 rows, and each discarded block serves one row.  So no
arrangement of pair units (any rows, any columns, any order) computes fewer
than T/2 discarded blocks, which is what the diagonal tiles discard.
"""

import pytest


def pair_tiles(T):
    """[(rows, cols)] of the kernel's symmetric tile order (block units)."""
    P = T // 2
    out = []
    for t in range(P * (P + 1) // 2):
        # decode: row tile i holds column tiles i..P-1
        i, r = 0, t
        while r >= P - i:
            r -= P - i
            i += 1
        j = i + r
        out.append(((2 * i, 2 * i + 1), (2 * j, 2 * j + 1)))
    return out


@pytest.mark.parametrize("T", [2, 4, 6, 14, 48])
def test_pair_tiling_covers_the_triangle_once_and_discards_the_minimum(T):
    seen = {}
    discarded = 0
    for rows, cols in pair_tiles(T):
        for r in rows:
            for c in cols:
                if c >= r:
                    seen[(r, c)] = seen.get((r, c), 0) + 1
                else:
                    discarded += 1
    assert set(seen) == {(r, c) for r in range(T) for c in range(r, T)}
    assert all(v == 1 for v in seen.values())
    parity_bound = sum(1 for r in range(T) if (T - r) % 2 == 1)
    assert discarded == parity_bound == T // 2


def test_no_unit_arrangement_beats_the_parity_bound_on_small_triangles():
    # exhaustive for T = 4: every cover of the 10 upper blocks by units
    # {r0, r1} x {c0, c1} (r0 != r1, c0 != c1) needs at least 2 extra blocks
    import itertools
    T = 4
    need = {(r, c) for r in range(T) for c in range(r, T)}
    units = [(rs, cs) for rs in itertools.combinations(range(T), 2) for cs in itertools.combinations(range(T), 2)]
    best = None
    for k in range(1, 4):
        for combo in itertools.combinations(units, k):
            cells = [(r, c) for rs, cs in combo for r in rs for c in cs]
            if need <= set(cells):
                extra = len(cells) - len(need)
                best = extra if best is None else min(best, extra)
        if best is not None:
            break
    assert best == T // 2
