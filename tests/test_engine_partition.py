"""Host-side checks of the split-K engine's work partition (no GPU).

The engine cuts the sequence of all (tile, k-block) pairs of a launch into one
contiguous range per CTA: CTA c holds [c*W // G, (c+1)*W // G). A tile that
straddles several ranges is split into pieces, one per CTA that holds some of
its k-blocks, and its partial sums go to slot 2c (the piece is the CTA's first
segment) or 2c + 1 (its last). The CTA holding the tile's first piece finishes
the tile; it must be at the end of its range there, so that every MMA of the
CTA has completed and its shared-memory ring is idle when it stages the other
pieces. This file restates those index formulas and checks these properties
on the workload's shapes and on edge cases."""
import pytest

K_MAX_PIECES = 256  # the engine's bound on pieces per tile (grid <= this)


def range_start(c, W, G):
    return c * W // G


def cta_of(j, W, G):
    """The CTA whose range holds k-block index j."""
    return ((j + 1) * G - 1) // W


def segments(c, W, G, KB):
    """The (tile, kb0, kb1) segments of CTA c, in order."""
    j, j1 = range_start(c, W, G), range_start(c + 1, W, G)
    out = []
    while j < j1:
        tau, kb0 = divmod(j, KB)
        kb1 = min(KB, kb0 + (j1 - j))
        out.append((tau, kb0, kb1))
        j += kb1 - kb0
    return out


def pieces(tau, W, G, KB):
    """The non-empty CTAs holding pieces of tile tau, in k order, with their slots."""
    kfirst = tau * KB
    res = []
    for cc in range(cta_of(kfirst, W, G), cta_of(kfirst + KB - 1, W, G) + 1):
        st = range_start(cc, W, G)
        if range_start(cc + 1, W, G) <= st:
            continue
        res.append((cc, cc * 2 + (0 if st >= kfirst else 1)))
    return res


SHAPES = [
    # (tiles, KB, grid): dense projections of the workload at 3 / 4 sub-blocks per stage
    (96, 38, 152), (96, 28, 152), (56, 43, 152), (56, 32, 152),
    # grouped launches: U experts x 16 gate/up tiles x 112 k-blocks, x 56 down tiles x 8 k-blocks
    (31 * 16, 112, 152), (277 * 16, 112, 152), (31 * 56, 8, 152), (277 * 56, 8, 152),
    # small and ragged: fewer k-blocks than CTAs (the host caps the grid), single tiles, odd grids
    (1, 1, 1), (1, 32, 32), (5, 6, 30), (3, 7, 20), (2, 5, 7), (1, 200, 152), (7, 3, 4), (40, 17, 151),
]


@pytest.mark.parametrize("capped", [True, False])
@pytest.mark.parametrize("tiles,KB,G", SHAPES)
def test_partition_properties(tiles, KB, G, capped):
    """Dense launches cap the grid at the number of k-blocks; grouped launches
    do not (their size is read from the device), so CTAs may hold nothing."""
    W = tiles * KB
    if capped:
        G = min(G, W)
    # every k-block belongs to exactly one CTA, and cta_of agrees with the ranges
    owner = {}
    for c in range(G):
        for j in range(range_start(c, W, G), range_start(c + 1, W, G)):
            assert j not in owner
            owner[j] = c
            assert cta_of(j, W, G) == c
    assert sorted(owner) == list(range(W))
    # the CTAs' segments: the slot each CTA writes for a split tile
    writes = {}
    for c in range(G):
        segs = segments(c, W, G, KB)
        for s, (tau, kb0, kb1) in enumerate(segs):
            whole = kb0 == 0 and kb1 == KB
            if not whole:
                slot = c * 2 + (0 if s == 0 else 1)
                assert (tau, c) not in writes
                writes[(tau, c)] = (slot, s == len(segs) - 1, kb0, kb1)
    # per split tile: pieces in k order cover the tile once; slots match what the CTAs write
    for tau in range(tiles):
        p = pieces(tau, W, G, KB)
        assert 1 <= len(p) <= K_MAX_PIECES
        if len(p) == 1:
            assert (tau, p[0][0]) not in writes  # a whole tile: no partials
            continue
        covered = 0
        for i, (cc, slot) in enumerate(p):
            wslot, is_last_seg, kb0, kb1 = writes[(tau, cc)]
            assert wslot == slot
            assert kb0 == covered  # k order, contiguous
            covered = kb1
            if i == 0:
                # the finishing CTA: its piece is the end of its range
                assert is_last_seg
        assert covered == KB
        # two slots per CTA, so distinct pieces never share one
        assert len({slot for _, slot in p}) == len(p)


def test_middle_pieces_occur_at_the_workload_shapes():
    """At the workload's dense shapes some tiles have three or more pieces: a CTA
    whose whole range lies inside the tile (the case the finishing CTA's bounded
    wait serves, as its piece ends together with the first piece)."""
    W, G, KB = 56 * 43, 152, 43
    assert any(len(pieces(t, W, G, KB)) >= 3 for t in range(56))
