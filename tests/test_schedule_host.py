"""The work count behind the packed-sequence schedule, pinned to the visibility rule by
brute force (CPU).  A unit's work is the number of the other side's 128-row tiles
(tiles never cross a shard) that hold at least one visible (query, key) pair with a row
of the unit; the schedule kernel and its host restatement in tests/test_gpu_schedule.py
count it as the tiles intersecting one position interval.  Here every pair is checked
one by one on small packed layouts."""
import numpy as np
import pytest

from test_gpu_schedule import ROWS, _cu



def _interval_count(cu, L, P, causal, kind, u):
    """Tiles intersecting the unit's visible interval (the schedule's definition)."""
    Ls = L // P
    n_t = -(-Ls // ROWS)
    per = -(-n_t // 2) if kind == 0 else n_t
    rows = 2 * ROWS if kind == 0 else ROWS
    s, i = divmod(u, per)
    a = s * Ls + i * rows
    b = min(s * Ls + Ls - 1, a + rows - 1)
    cu = np.asarray(cu)
    span = lambda pos: (int(cu[np.searchsorted(cu[:-1], pos, side="right") - 1]),
                        int(cu[np.searchsorted(cu[:-1], pos, side="right")]) - 1)
    (fa, _), (_, lb) = span(a), span(b)
    lo, hi = ((a if causal else fa), lb) if kind == 1 else (fa, (b if causal else lb))
    n = 0
    for sh in range(P):
        base = sh * Ls
        x, y = max(lo, base), min(hi, base + Ls - 1)
        if x <= y:
            n += (y - base) // ROWS - (x - base) // ROWS + 1
    return n


def _brute_count(cu, L, P, causal, kind, u):
    """Tiles holding a key (kind 0, 2) or query (kind 1) visible with a row of the unit."""
    Ls = L // P
    n_t = -(-Ls // ROWS)
    per = -(-n_t // 2) if kind == 0 else n_t
    rows = 2 * ROWS if kind == 0 else ROWS
    s, i = divmod(u, per)
    unit_rows = range(s * Ls + i * rows, min(s * Ls + Ls, s * Ls + i * rows + rows))
    seq = np.searchsorted(np.asarray(cu), np.arange(L), side="right") - 1
    tiles = set()
    for x in unit_rows:
        for y in range(L):
            if seq[x] != seq[y]:
                continue
            q, k = (y, x) if kind == 1 else (x, y)
            if causal and k > q:
                continue
            tiles.add((y // Ls, (y % Ls) // ROWS))
    return len(tiles)


CASES = [
    ([300, 1, 1000, 0, 747], 4),
    ([5, 7, 100, 200], 4),            # shards shorter than a tile
    ([17, 900, 83, 302, 1, 1, 1, 93], 3),
    ([640], 5),
    ([129, 383, 256], 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "n%d_P%d" % (len(c[0]), c[1]))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_work_count_is_visible_tiles(case, causal, kind):
    lengths, P = case
    cu = _cu(lengths)
    L = cu[-1]
    assert L % P == 0
    Ls = L // P
    n_t = -(-Ls // ROWS)
    per = -(-n_t // 2) if kind == 0 else n_t
    for u in range(P * per):
        assert _interval_count(cu, L, P, causal, kind, u) == _brute_count(cu, L, P, causal, kind, u), \
            (lengths, P, causal, kind, u)
