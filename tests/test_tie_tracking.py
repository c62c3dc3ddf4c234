"""The streaming repeated-maximum flag of the forward kernel, checked on the CPU against
the whole-row definition.

The fix of Qiu & Yao (priors.kr post, the fix paragraph of paper §4; bud-325 note,
Method) changes the shift of rows whose maximum repeats: at least two scores within
eps of the row maximum. The kernel sees a row one 128-column tile at a time and keeps
that flag exactly with two facts, restated here in plain numpy so that a mistake in
either would show:

* two entries of a tile reach a threshold iff two of its eight 16-column block maxima
  do or two of its sixteen column-class (column mod 16) maxima do;
* with running maximum m1 and tile maximum t1, the flag becomes "the tile holds two
  entries >= t1 - eps" when t1 > m1 + eps, becomes true when m1 - eps <= t1 <= m1 + eps,
  and is unchanged otherwise; with a new maximum within eps above m1 the old maximum
  itself is the second entry.

These tests need no GPU and do not use the oracle: the reference is the definition.
"""
import numpy as np
import pytest

TILE, BLOCK = 128, 16


def two_by_partitions(x, thr):
    """Two entries >= thr, decided from block and class maxima only."""
    blocks = x.reshape(TILE // BLOCK, BLOCK)
    nb = int((blocks.max(axis=1) >= thr).sum())
    ne = int((blocks.max(axis=0) >= thr).sum())
    return nb >= 2 or ne >= 2


def streamed_flag(row, eps):
    """The flag after every tile, updated as the kernel does."""
    m1, rep, out = -np.inf, False, []
    for j in range(0, row.size, TILE):
        x = row[j:j + TILE]
        t1 = x.max()
        thr = t1 - eps
        if t1 > m1:
            rep = two_by_partitions(x, thr) if m1 < thr else True
        elif t1 >= m1 - eps and t1 > -np.inf:
            rep = True
        m1 = max(m1, t1)
        out.append(rep)
    return out


def whole_row_flag(prefix, eps):
    m = prefix.max()
    return int((prefix >= m - eps).sum()) >= 2


@pytest.mark.parametrize("seed", range(40))
def test_partition_count_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    for _ in range(50):
        x = rng.integers(-8, 9, TILE).astype(np.float64) / 8
        k = rng.integers(0, 4)
        top = x.max()
        for c in rng.choice(TILE, size=k, replace=False):
            x[c] = top                      # planted ties, in any block and class
        thr = x.max() - rng.choice([0.0, 1e-3, 0.125, 0.5])
        assert two_by_partitions(x, thr) == (int((x >= thr).sum()) >= 2)


def test_partition_pairs_in_same_block_and_same_class():
    x = np.full(TILE, -1.0)
    for a, b in [(3, 5), (3, 19), (3, 40), (0, 127), (16, 32)]:
        y = x.copy()
        y[a] = y[b] = 2.0
        assert two_by_partitions(y, 2.0)
        y[b] = 1.5
        assert not two_by_partitions(y, 2.0)


@pytest.mark.parametrize("seed", range(30))
@pytest.mark.parametrize("eps", [0.0, 1e-3, 0.125])
def test_streamed_flag_equals_whole_row_definition(seed, eps):
    rng = np.random.default_rng(1000 + seed)
    n = TILE * int(rng.integers(1, 6))
    row = rng.integers(-16, 17, n).astype(np.float64) / 8   # a 1/8 grid: exact ties
    # Plant near-maximum entries in later tiles, some within eps of each other.
    for _ in range(int(rng.integers(0, 4))):
        c = int(rng.integers(0, n))
        row[c] = row.max() + rng.choice([0.0, eps / 2 if eps else 0.0, 0.125, 0.25])
    flags = streamed_flag(row, eps)
    for t, f in enumerate(flags):
        assert f == whole_row_flag(row[:TILE * (t + 1)], eps), (t, f)


def test_masked_tail_is_ignored():
    row = np.full(2 * TILE, -np.inf)
    row[:TILE + 10] = np.linspace(-1.0, 0.0, TILE + 10)
    assert streamed_flag(row, 1e-3) == [False, False]
    row[5] = 0.0
    assert streamed_flag(row, 1e-3) == [False, True]


def test_tile_maximum_just_below_the_running_maximum():
    # A later tile whose maximum lies within eps below the running maximum makes
    # the row repeated; one just outside eps does not.
    for below, expect in [(1 / 16, True), (1 / 8, True), (3 / 16, False)]:
        row = np.full(2 * TILE, -4.0)
        row[7] = 2.0
        row[TILE + 30] = 2.0 - below
        assert streamed_flag(row, 0.125) == [False, expect]


@pytest.mark.parametrize("seed", range(30))
def test_streamed_flag_with_descending_tiles(seed):
    # Every tile has a unique maximum, each a random step below the one before, so
    # that a later tile's maximum often falls within eps below the running maximum
    # instead of tying it.
    rng = np.random.default_rng(5000 + seed)
    n_t = int(rng.integers(2, 6))
    tiles, top = [], 2.0
    for _ in range(n_t):
        x = rng.integers(-32, 0, TILE) / 16.0
        x[int(rng.integers(0, TILE))] = top
        tiles.append(x)
        top -= rng.choice([1 / 32, 1 / 16, 1 / 8, 3 / 16])
    row = np.concatenate(tiles)
    for eps in (1 / 32, 1 / 16, 1 / 8):
        flags = streamed_flag(row, eps)
        for t, f in enumerate(flags):
            assert f == whole_row_flag(row[:TILE * (t + 1)], eps), (eps, t, f)
