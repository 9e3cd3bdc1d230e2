"""Pins for the mask side of the oracle (CPU only).

Each check ties the oracle to something other than its own code: the paper's Region C worked
example (hand-evaluated fixture), closed-form visible-pair counts, the tile census of a causal
mask, the transpose relation between the forward and backward descriptors, and the unsigned
interval test the paper uses for visibility checks (CompileMask section 4.4).
"""
import json
import os

import numpy as np
import pytest

from masked_flashattention_gb300 import workloads as W
from oracle import masks as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small_cases():
    for wid in (1, 2, 3, 4, 5, 6):
        for S in (256, 512, 1024):
            for seed in range(3):
                seg, nseg = W.segments(wid, 2, S, seed=seed * 7 + wid)
                for b in range(2):
                    yield wid, S, seg[b], int(nseg[b])


# ------------------------------------------------------------------------------------------------
# the paper's worked example
# ------------------------------------------------------------------------------------------------
def test_region_c_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "region_c_example.json")))
    seg, nseg, S, tile = np.array(g["seg"]), g["nseg"], g["S"], g["tile"]
    fwd = M.interval_table_fwd(3, seg, nseg, S)          # [2, S, 2]
    assert fwd.transpose(1, 0, 2).tolist() == g["fwd_intervals"]
    bwd = M.interval_table_bwd(3, seg, nseg, S)
    assert bwd.transpose(1, 0, 2).tolist() == g["bwd_intervals"]
    states = M.tile_states(3, seg, nseg, S, tile=tile)
    assert states.tolist() == g["fwd_tile_states"]
    assert M.pack_tile_states(states)[:, 0].tolist() == g["fwd_bitmap_words"]
    bstates = M.tile_states(3, seg, nseg, S, tile=tile, backward=True)
    assert M.pack_tile_states(bstates)[:, 0].tolist() == g["bwd_bitmap_words"]
    assert int(M.dense_mask(3, seg, nseg, S).sum()) == g["visible_pairs"]


# ------------------------------------------------------------------------------------------------
# two formulations agree: closed-form slots vs the dense predicate (and its transpose)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", list(_small_cases()), ids=lambda c: f"w{c[0]}-S{c[1]}")
def test_interval_union_equals_dense_rows(case):
    wid, S, seg, nseg = case
    dense = M.dense_mask(wid, seg, nseg, S)
    fwd = M.interval_table_fwd(wid, seg, nseg, S)
    bwd = M.interval_table_bwd(wid, seg, nseg, S)
    assert fwd.shape[0] == M.num_intervals(wid)[0] and bwd.shape[0] == M.num_intervals(wid)[1]
    assert np.array_equal(M.intervals_to_mask(fwd, S), dense)
    assert np.array_equal(M.intervals_to_mask(bwd, S), dense.T)
    # canonical form: every stored interval is (0, 0) or non-empty and inside [0, S]
    for t in (fwd, bwd):
        lo, hi = t[..., 0], t[..., 1]
        assert ((hi > lo) | ((lo == 0) & (hi == 0))).all()
        assert (lo >= 0).all() and (hi <= S).all()


# ------------------------------------------------------------------------------------------------
# closed-form visible-pair counts (per head), written from the workload definitions
# ------------------------------------------------------------------------------------------------
def closed_form_visible(wid, seg, nseg, S):
    L = [int(seg[k + 1] - seg[k]) for k in range(nseg)]
    if wid == 1:
        return sum(l * (l + 1) // 2 for l in L)
    if wid == 2:
        return S * (S + 1) // 2
    if wid == 3:
        P = L[0]
        return P * (P + 1) // 2 + sum(l * P + l * (l + 1) // 2 for l in L[1:])
    if wid == 4:
        h = L[0]
        return h * (h + 1) // 2 + (S - h) * (h + 1)
    if wid == 5:
        b = L[0]
        tot = b * (b + 1) // 2
        for d in range(1, nseg):
            tot += L[d] * b + L[d] * (L[d] + 1) // 2
            if d >= 2:
                tot += L[d] * min(64, L[d - 1])
        return tot
    if wid == 6:  # per user: a causal history of h rows, then c candidates that see h + 1 keys
        tot = 0
        for u in range(0, nseg, 2):
            h, c = L[u], L[u + 1]
            tot += h * (h + 1) // 2 + c * (h + 1)
        return tot
    raise ValueError(wid)


@pytest.mark.parametrize("case", list(_small_cases()), ids=lambda c: f"w{c[0]}-S{c[1]}")
def test_visible_count_closed_form_small(case):
    wid, S, seg, nseg = case
    assert int(M.dense_mask(wid, seg, nseg, S).sum()) == closed_form_visible(wid, seg, nseg, S)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_visible_count_closed_form_full_size(wid):
    w = W.WORKLOADS[wid]
    seg, nseg = W.segments(wid, w.B, w.S)
    for b in range(w.B):
        t = M.interval_table_fwd(wid, seg[b], int(nseg[b]), w.S)
        lens = (t[..., 1] - t[..., 0]).astype(np.int64)
        # the slots of a row are disjoint, so their lengths add up to the row's visible count
        starts = np.where(lens > 0, t[..., 0], np.iinfo(np.int32).max)
        order = np.argsort(starts, axis=0)
        s_sorted = np.take_along_axis(t[..., 0], order, 0)
        e_sorted = np.take_along_axis(t[..., 1], order, 0)
        l_sorted = np.take_along_axis(lens, order, 0)
        for n in range(1, t.shape[0]):
            ok = (l_sorted[n] == 0) | (l_sorted[n - 1] == 0) | (e_sorted[n - 1] <= s_sorted[n])
            assert ok.all()
        assert int(lens.sum()) == closed_form_visible(wid, seg[b], int(nseg[b]), w.S)
    if wid == 2:
        assert closed_form_visible(2, seg[0], 1, 8192) == 33_558_528


# ------------------------------------------------------------------------------------------------
# Tile-State Bitmaps
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("S", [256, 1024, 8192])
def test_causal_tile_census(S):
    seg, nseg = W.segments(2, 1, S)
    st = M.tile_states(2, seg[0], int(nseg[0]), S, tile=128)
    n = S // 128
    assert int((st == M.FULL).sum()) == n * (n - 1) // 2
    assert int((st == M.EMPTY).sum()) == n * (n - 1) // 2
    assert int((st == M.PARTIAL).sum()) == n
    assert all(st[t, t] == M.PARTIAL for t in range(n))


@pytest.mark.parametrize("case", list(_small_cases())[::3], ids=lambda c: f"w{c[0]}-S{c[1]}")
def test_backward_bitmap_is_transpose(case):
    wid, S, seg, nseg = case
    f = M.tile_states(wid, seg, nseg, S, tile=128)
    b = M.tile_states(wid, seg, nseg, S, tile=128, backward=True)
    assert np.array_equal(f.T, b)
    # a tile is non-empty exactly when some visible pair falls in it
    dense = M.dense_mask(wid, seg, nseg, S)
    nonempty = dense.reshape(S // 128, 128, S // 128, 128).any(axis=(1, 3))
    assert np.array_equal(f != M.EMPTY, nonempty)


def test_tile_states_brute_force_tiny():
    rng = np.random.default_rng(5)
    for _ in range(50):
        m = rng.random((8, 12)) < rng.random()
        st = M.tile_states_of(m, 4, 3)
        for r in range(2):
            for c in range(4):
                blk = [m[i, j] for i in range(4 * r, 4 * r + 4) for j in range(3 * c, 3 * c + 3)]
                want = 2 if all(blk) else (1 if any(blk) else 0)
                assert st[r, c] == want


def test_pack_tile_states_bit_positions():
    codes = np.zeros((1, 20), dtype=np.uint8)
    codes[0, 0] = 1
    codes[0, 15] = 2
    codes[0, 16] = 1
    codes[0, 19] = 2
    words = M.pack_tile_states(codes)
    assert words.shape == (1, 2)
    assert int(words[0, 0]) == (1 << 0) | (2 << 30)
    assert int(words[0, 1]) == (1 << 0) | (2 << 6)


# ------------------------------------------------------------------------------------------------
# the unsigned visibility test (section 4.4): j in [s, e) <=> (u32)(j - s) < (u32)(e - s)
# ------------------------------------------------------------------------------------------------
def test_unsigned_interval_check_exhaustive():
    r = np.arange(0, 130)
    s, e, j = np.meshgrid(r, r, r, indexing="ij")
    s, e, j = s.ravel(), e.ravel(), j.ravel()
    two = (j >= s) & (j < e)
    one = ((j - s).astype(np.uint32)) < ((e - s).astype(np.uint32))
    canonical = e >= s
    assert np.array_equal(two[canonical], one[canonical])
    # why empty intervals are stored as (0, 0): an inverted pair would make the test accept
    assert one[~canonical].mean() > 0.4
    assert not one[(s == 0) & (e == 0)].any()


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_interval_count_matches_visible_runs(wid):
    """The forward interval count is tight: some row has exactly that many separate visible
    runs (workload 5 rows see three, which a two-interval encoding could not hold); no row or
    column has more runs than its descriptor has slots."""
    S = 4096
    seg, nseg = W.segments(wid, 1, S, seed=11)
    dense = M.dense_mask(wid, seg[0], int(nseg[0]), S)

    def runs(m):
        return (m[:, 0].astype(int) + (m[:, 1:] & ~m[:, :-1]).sum(axis=1))

    nif, nib = M.num_intervals(wid)
    assert int(runs(dense).max()) == nif
    assert int(runs(dense.T).max()) <= nib


def test_varlen_users_are_independent():
    """Workload 6 packs users back to back: no query row sees a key of another user, and a
    user's block of the mask equals the single-sample HSTU mask (workload 4) of that user's
    history and candidates, shifted to the user's offset."""
    S = 2048
    seg, nseg = W.segments(6, 1, S, seed=3)
    seg, n = seg[0], int(nseg[0])
    dense = M.dense_mask(6, seg, n, S)
    for u in range(0, n, 2):
        a, h_end, e = int(seg[u]), int(seg[u + 1]), int(seg[u + 2])
        block = dense[a:e, a:e]
        one = np.array([0, h_end - a, e - a, e - a], dtype=np.int64)
        np.testing.assert_array_equal(block, M.dense_mask(4, one, 2, e - a))
        assert not dense[a:e, :a].any() and not dense[a:e, e:].any()


# ------------------------------------------------------------------------------------------------
# the other reading of workload 5's prefix rows (behind an oracle flag)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(3))
def test_w5_bidirectional_prefix_reading(seed):
    """With prefix_bidirectional the prefix rows see all of [0, b): exactly the b(b-1)/2 pairs of
    the prefix block above its diagonal are added, nothing else changes, and the flagged Interval
    Tables and bitmaps describe the flagged mask."""
    S = 1024
    seg, nseg = W.segments(5, 2, S, seed=100 + seed)
    for b in range(2):
        sb, nb = seg[b], int(nseg[b])
        P = int(sb[1])
        base = M.dense_mask(5, sb, nb, S)
        alt = M.dense_mask(5, sb, nb, S, prefix_bidirectional=True)
        added = alt & ~base
        ii, jj = np.nonzero(added)
        assert (ii < P).all() and (jj < P).all() and (jj > ii).all()
        assert int(added.sum()) == P * (P - 1) // 2
        assert not (base & ~alt).any()
        assert int(alt.sum()) == closed_form_visible(5, sb, nb, S) + P * (P - 1) // 2
        fwd = M.interval_table_fwd(5, sb, nb, S, prefix_bidirectional=True)
        bwd = M.interval_table_bwd(5, sb, nb, S, prefix_bidirectional=True)
        assert np.array_equal(M.intervals_to_mask(fwd, S), alt)
        assert np.array_equal(M.intervals_to_mask(bwd, S), alt.T)
        states = M.tile_states(5, sb, nb, S, prefix_bidirectional=True)
        assert np.array_equal(states, M.tile_states_of(alt, 128, 128))
        bstates = M.tile_states(5, sb, nb, S, backward=True, prefix_bidirectional=True)
        assert np.array_equal(bstates, states.T)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_interval_union_equals_dense_many_seeds(wid):
    """The slot form against the dense predicate (and its transpose) on 200 seeded segmentations
    per workload at S = 256 and 384, so short and uneven segments are covered."""
    for seed in range(100):
        for S in (256, 384):
            seg, nseg = W.segments(wid, 1, S, seed=10_000 + 131 * seed + wid)
            sb, nb = seg[0], int(nseg[0])
            dense = M.dense_mask(wid, sb, nb, S)
            assert np.array_equal(M.intervals_to_mask(M.interval_table_fwd(wid, sb, nb, S), S), dense)
            assert np.array_equal(M.intervals_to_mask(M.interval_table_bwd(wid, sb, nb, S), S), dense.T)


# ------------------------------------------------------------------------------------------------
# masked form of the Interval Table (the representation of the paper's section 4.4 ablation)
# ------------------------------------------------------------------------------------------------
def test_masked_runs_region_c_worked_example():
    """Hand-derived masked runs of the Region C instance (fixture), forward and backward."""
    g = json.load(open(os.path.join(GOLDEN, "region_c_example.json")))
    seg, nseg, S = np.array(g["seg"]), g["nseg"], g["S"]
    dense = M.dense_mask(3, seg, nseg, S)
    assert M.masked_runs_table(dense, 3).transpose(1, 0, 2).tolist() == g["fwd_masked_runs"]
    assert M.masked_runs_table(dense.T, 2).transpose(1, 0, 2).tolist() == g["bwd_masked_runs"]


def test_masked_runs_are_maximal_and_cover_the_complement():
    """Brute force on tiny random masks: the runs are increasing, disjoint, each bounded by a
    visible cell or an edge on both sides, and together cover exactly the invisible cells."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        R, C = int(rng.integers(1, 6)), int(rng.integers(1, 40))
        mask = rng.random((R, C)) < rng.uniform(0.1, 0.9)
        t = M.masked_runs_table(mask, C)
        for r in range(R):
            runs = [tuple(x) for x in t[:, r].tolist() if x != [0, 0]]
            covered = np.zeros(C, dtype=bool)
            prev_end = -1
            for s, e in runs:
                assert s < e and s > prev_end          # increasing, disjoint, not adjacent
                assert s == 0 or mask[r, s - 1]        # maximal on the left
                assert e == C or mask[r, e]            # maximal on the right
                covered[s:e] = True
                prev_end = e
            np.testing.assert_array_equal(covered, ~mask[r])


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_masked_runs_fit_one_slot_more(wid):
    """NI visible intervals leave at most NI + 1 masked runs per row, for every workload rule
    (forward and backward), so the masked table has NI + 1 slots."""
    nif, nib = M.num_intervals(wid)
    for S in (256, 640):
        seg, nseg = W.segments(wid, 2, S, seed=17 + wid)
        for b in range(2):
            dense = M.dense_mask(wid, seg[b], int(nseg[b]), S)
            M.masked_runs_table(dense, nif + 1)      # asserts the run count fits
            M.masked_runs_table(dense.T, nib + 1)
