"""Oracle: dense visibility masks, canonical Interval Tables and Tile-State Bitmaps.

Test infrastructure only (see the package header).

What the paper fixes (CompileMask, sections 2.1, 3.3.1, 3.3.2):
  * visibility is a property of each (query row i, key column j) pair; the mask boundaries come
    from per-batch metadata (sequence lengths, segment boundaries), section 1 / 2.2;
  * the Execution Descriptor holds, per row, the visible key intervals, padded with zero-length
    intervals up to the count the compiler derived (section 3.3.1);
  * it also holds two bits per tile telling whether the tile is empty, full or partial
    (section 3.3.1), which is the classification tiled attention needs (section 2.1);
  * forward and backward traversals get their own descriptors (section 3.2.2 / 3.3): the backward
    one lists, per key column, the visible query intervals.

Readings taken where the pages are silent (each is listed in the design notes):
  * an interval is stored as (start, end), half open; an empty or padding interval is (0, 0);
  * tile codes 0 = empty, 1 = partial, 2 = full, packed 16 tiles per uint32, tile t of a row at
    bits 2*(t % 16) of word t // 16;
  * slot order within a row is the order in which the rule names the intervals;
  * workload 5: prefix rows are causal over the prefix; the "previous document" of the first
    document is empty, and the prefix is not a document.  The other reading of the prefix rows
    (each sees the whole prefix [0, b)) is available with prefix_bidirectional=True in
    dense_mask, the Interval Tables and tile_states; the library's specs follow the causal one.

Segment conventions: seg_row[k] is the first position of segment k, seg_row[nseg] = S.
  workload 3: segment 0 is the prompt (P = seg_row[1]), segments 1..4 the responses;
  workload 4: segment 0 is the history (h = seg_row[1]), segment 1 the candidates;
  workload 5: segment 0 is the system prefix (b = seg_row[1]), segments 1.. the documents;
  workload 6: variable-length packing of users, each as two consecutive segments: segment 2u
  is user u's history, segment 2u + 1 its candidates (the HSTU rule applied per user).
"""
from __future__ import annotations

import numpy as np

PREV_DOC_HEAD = 64  # workload 5: tokens of the previous document that stay visible


def num_intervals(wid: int) -> tuple[int, int]:
    """Forward / backward interval counts of each workload's rule (max over its regions)."""
    return {1: (1, 1), 2: (1, 1), 3: (2, 1), 4: (2, 1), 5: (3, 2), 6: (2, 1)}[wid]


def segment_index(seg_row: np.ndarray, nseg: int, pos: np.ndarray) -> np.ndarray:
    """Index k of the segment holding each position: seg_row[k] <= pos < seg_row[k+1]."""
    bounds = np.asarray(seg_row[: nseg + 1], dtype=np.int64)
    return np.searchsorted(bounds, pos, side="right") - 1


# ------------------------------------------------------------------------------------------------
# dense masks: the visibility rule of each workload, written directly as a predicate on (i, j)
# ------------------------------------------------------------------------------------------------
def dense_mask(wid: int, seg_row: np.ndarray, nseg: int, S: int,
               rows: np.ndarray | None = None, cols: np.ndarray | None = None,
               prefix_bidirectional: bool = False) -> np.ndarray:
    """bool [len(rows), len(cols)]: True where query row i may attend to key column j.

    prefix_bidirectional (workload 5 only): prefix rows see the whole prefix instead of being
    causal over it (the other reading of the pages' three-interval workload)."""
    i = (np.arange(S) if rows is None else np.asarray(rows)).astype(np.int64)[:, None]
    j = (np.arange(S) if cols is None else np.asarray(cols)).astype(np.int64)[None, :]
    seg = np.asarray(seg_row, dtype=np.int64)
    ki = segment_index(seg, nseg, i)          # segment of the query row
    start_i = seg[ki]                         # first position of that segment
    if wid == 1:   # packed documents: row i sees [doc_start(i), i + 1)
        return (j >= start_i) & (j <= i)
    if wid == 2:   # causal: row i sees [0, i + 1)
        return np.broadcast_to(j <= i, (i.shape[0], j.shape[1])).copy()
    if wid == 3:   # prompt rows causal; a response row sees [0, P) and [resp_start(i), i + 1)
        P = seg[1]
        prompt = (i < P) & (j <= i)
        response = (i >= P) & ((j < P) | ((j >= start_i) & (j <= i)))
        return prompt | response
    if wid == 4:   # history rows causal; candidate row i sees [0, h) and [i, i + 1)
        h = seg[1]
        history = (i < h) & (j <= i)
        candidate = (i >= h) & ((j < h) | (j == i))
        return history | candidate
    if wid == 5:   # prefix causal; document row sees [0, b), head of previous doc, own doc causal
        b = seg[1]
        prefix = (i < b) & ((j < b) if prefix_bidirectional else (j <= i))
        prev = np.maximum(ki - 1, 0)
        prev_start = seg[prev]
        prev_len = seg[np.minimum(prev + 1, nseg)] - prev_start
        head_end = prev_start + np.minimum(PREV_DOC_HEAD, prev_len)
        has_prev_doc = ki >= 2
        doc = (i >= b) & ((j < b)
                          | (has_prev_doc & (j >= prev_start) & (j < head_end))
                          | ((j >= start_i) & (j <= i)))
        return prefix | doc
    if wid == 6:   # per user: history rows causal within the history; a candidate row sees the
        #           user's history and itself
        in_hist = (ki % 2) == 0
        hist_start = np.where(in_hist, start_i, seg[np.maximum(ki - 1, 0)])
        history = in_hist & (j >= start_i) & (j <= i)
        candidate = (~in_hist) & (((j >= hist_start) & (j < start_i)) | (j == i))
        return history | candidate
    raise ValueError(wid)


# ------------------------------------------------------------------------------------------------
# canonical Interval Tables (closed form per region, in the rule's slot order)
# ------------------------------------------------------------------------------------------------
def _slot(lo: int, hi: int, S: int) -> tuple[int, int]:
    lo = min(max(lo, 0), S)
    hi = min(max(hi, 0), S)
    return (lo, hi) if hi > lo else (0, 0)


def interval_table_fwd(wid: int, seg_row: np.ndarray, nseg: int, S: int,
                       prefix_bidirectional: bool = False) -> np.ndarray:
    """int32 [NI_f, S, 2]: the visible key intervals of every query row (prefix_bidirectional:
    see dense_mask)."""
    ni, _ = num_intervals(wid)
    out = np.zeros((ni, S, 2), dtype=np.int32)
    seg = [int(x) for x in seg_row[: nseg + 1]]
    for i in range(S):
        k = int(segment_index(np.asarray(seg), nseg, np.array([i]))[0])
        if wid == 1:
            slots = [(seg[k], i + 1)]
        elif wid == 2:
            slots = [(0, i + 1)]
        elif wid == 3:
            slots = [(0, i + 1)] if k == 0 else [(0, seg[1]), (seg[k], i + 1)]
        elif wid == 4:
            slots = [(0, i + 1)] if k == 0 else [(0, seg[1]), (i, i + 1)]
        elif wid == 5:
            if k == 0:
                slots = [(0, seg[1])] if prefix_bidirectional else [(0, i + 1)]
            elif k == 1:
                slots = [(0, seg[1]), (0, 0), (seg[k], i + 1)]
            else:
                ps, pe = seg[k - 1], seg[k]
                slots = [(0, seg[1]), (ps, min(ps + PREV_DOC_HEAD, pe)), (seg[k], i + 1)]
        elif wid == 6:
            slots = [(seg[k], i + 1)] if k % 2 == 0 else [(seg[k - 1], seg[k]), (i, i + 1)]
        else:
            raise ValueError(wid)
        for n, (lo, hi) in enumerate(slots):
            out[n, i] = _slot(lo, hi, S)
    return out


def interval_table_bwd(wid: int, seg_row: np.ndarray, nseg: int, S: int,
                       prefix_bidirectional: bool = False) -> np.ndarray:
    """int32 [NI_b, S, 2]: for every key column j, the query rows that see it (prefix_bidirectional:
    see dense_mask)."""
    _, ni = num_intervals(wid)
    out = np.zeros((ni, S, 2), dtype=np.int32)
    seg = [int(x) for x in seg_row[: nseg + 1]]
    for j in range(S):
        k = int(segment_index(np.asarray(seg), nseg, np.array([j]))[0])
        end_k = seg[k + 1]
        if wid == 1:
            slots = [(j, end_k)]
        elif wid == 2:
            slots = [(j, S)]
        elif wid == 3:
            slots = [(j, S)] if k == 0 else [(j, end_k)]
        elif wid == 4:
            slots = [(j, S)] if k == 0 else [(j, j + 1)]
        elif wid == 5:
            if k == 0:  # a prefix key: the prefix rows from j on (or all of them), every document row
                slots = [(0, S)] if prefix_bidirectional else [(j, S)]
            else:
                nxt = (0, 0)
                if j < seg[k] + PREV_DOC_HEAD and k + 1 < nseg:
                    nxt = (seg[k + 1], seg[k + 2])
                slots = [(j, end_k), nxt]
        elif wid == 6:
            # a history key is seen by the later history rows and every candidate of its user
            # (the candidate segment follows the history); a candidate key only by itself
            slots = [(j, seg[k + 2])] if k % 2 == 0 else [(j, j + 1)]
        else:
            raise ValueError(wid)
        for n, (lo, hi) in enumerate(slots):
            out[n, j] = _slot(lo, hi, S)
    return out


def masked_runs_table(mask: np.ndarray, nslots: int) -> np.ndarray:
    """int32 [nslots, R, 2]: the masked form of an Interval Table, the representation the paper's
    section 4.4 compares its visible intervals with.  For every row of the dense bool mask
    [R, C], the maximal runs of invisible columns as half-open (start, end) in increasing order,
    then (0, 0) padding.  Reading (the pages give no layout): same slot-major layout as the
    visible table, with one slot more than the rule's interval count, since NI disjoint visible
    intervals leave at most NI + 1 gaps."""
    R, C = mask.shape
    out = np.zeros((nslots, R, 2), dtype=np.int32)
    for r in range(R):
        hidden = np.concatenate(([0], (~mask[r]).astype(np.int8), [0]))
        edges = np.diff(hidden)
        starts = np.flatnonzero(edges == 1)
        ends = np.flatnonzero(edges == -1)
        assert len(starts) <= nslots, (r, len(starts), nslots)
        out[: len(starts), r, 0] = starts
        out[: len(starts), r, 1] = ends
    return out


def intervals_to_mask(table: np.ndarray, S: int) -> np.ndarray:
    """Dense bool [S, S] of the union of each row's intervals (row r, column c)."""
    c = np.arange(S)[None, :]
    m = np.zeros((table.shape[1], S), dtype=bool)
    for n in range(table.shape[0]):
        m |= (c >= table[n, :, 0:1]) & (c < table[n, :, 1:2])
    return m


# ------------------------------------------------------------------------------------------------
# Tile-State Bitmaps
# ------------------------------------------------------------------------------------------------
EMPTY, PARTIAL, FULL = 0, 1, 2


def tile_states_of(mask: np.ndarray, tile_r: int, tile_c: int) -> np.ndarray:
    """uint8 [R/tile_r, C/tile_c]: 0 if no pair of the tile is visible, 2 if all are, else 1."""
    R, C = mask.shape
    assert R % tile_r == 0 and C % tile_c == 0
    t = mask.reshape(R // tile_r, tile_r, C // tile_c, tile_c)
    anyv = t.any(axis=(1, 3))
    allv = t.all(axis=(1, 3))
    return np.where(allv, FULL, np.where(anyv, PARTIAL, EMPTY)).astype(np.uint8)


def tile_states(wid: int, seg_row: np.ndarray, nseg: int, S: int, tile: int = 128,
                backward: bool = False, prefix_bidirectional: bool = False) -> np.ndarray:
    """Tile states of the forward mask, or of its transpose for the backward descriptor.

    Built one tile-row at a time from the dense predicate so that 32K masks fit in memory.
    prefix_bidirectional: see dense_mask.
    """
    nt = S // tile
    out = np.zeros((nt, nt), dtype=np.uint8)
    for t in range(nt):
        span = np.arange(t * tile, (t + 1) * tile)
        if backward:  # rows of the transposed mask = key columns of the forward mask
            block = dense_mask(wid, seg_row, nseg, S, rows=None, cols=span,
                               prefix_bidirectional=prefix_bidirectional).T
        else:
            block = dense_mask(wid, seg_row, nseg, S, rows=span, cols=None,
                               prefix_bidirectional=prefix_bidirectional)
        out[t] = tile_states_of(block, tile, tile)[0]
    return out


def pack_tile_states(codes: np.ndarray) -> np.ndarray:
    """uint32 [R, ceil(C/16)]: 2 bits per tile, tile c at bits 2*(c % 16) of word c // 16."""
    R, C = codes.shape
    W = (C + 15) // 16
    out = np.zeros((R, W), dtype=np.uint64)
    for c in range(C):
        out[:, c // 16] |= codes[:, c].astype(np.uint64) << np.uint64(2 * (c % 16))
    return out.astype(np.uint32)
