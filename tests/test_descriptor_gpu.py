"""GPU parity of the Execution Descriptor: the preprocess kernel vs the oracle, bit-exact.

Interval Tables (visible and masked forms) and Tile-State Bitmaps (forward and backward) must
equal the oracle's on the six workloads at full size and on many small seeded segmentations
(ragged tails included); the schedules must be longest-first permutations of the tile rows.
"""
import numpy as np
import pytest
import torch

from masked_flashattention_gb300 import workloads as W
from oracle import masks as M

pytestmark = pytest.mark.gpu


def _lib():
    from masked_flashattention_gb300 import binding as B
    B.lib()
    return B


MODES = ["generated", "generic"]


def _set_mode(B, mode):
    B.cm_set_preprocess_mode(B.CM_PREPROCESS_GENERIC if mode == "generic"
                             else B.CM_PREPROCESS_GENERATED)


def _build(B, wid, seg, nseg, S, mode="generated", form=0):
    from masked_flashattention_gb300 import specs
    _set_mode(B, mode)
    f = B.cm_compile_spec(specs.FWD[wid])
    b = B.cm_compile_spec(specs.BWD[wid])
    desc = B.Descriptor(f, b, seg.shape[0], S, form=form)
    try:
        B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
        torch.cuda.synchronize()
    finally:
        _set_mode(B, "generated")
    assert B.cm_get_status(desc) == 0
    return desc


def _masked_tables(wid, seg_row, n, S, block=1024):
    """The oracle's masked-form tables, forward and backward, built a block of rows at a time."""
    nif, nib = M.num_intervals(wid)
    tf = np.zeros((nif + 1, S, 2), dtype=np.int32)
    tb = np.zeros((nib + 1, S, 2), dtype=np.int32)
    for r0 in range(0, S, block):
        span = np.arange(r0, min(S, r0 + block))
        tf[:, span] = M.masked_runs_table(M.dense_mask(wid, seg_row, n, S, rows=span), nif + 1)
        tb[:, span] = M.masked_runs_table(M.dense_mask(wid, seg_row, n, S, cols=span).T, nib + 1)
    return tf, tb


def _check(desc, wid, seg, nseg, S):
    itf, itb = desc.interval_table_fwd(), desc.interval_table_bwd()
    bmf, bmb = desc.bitmap_fwd(), desc.bitmap_bwd()
    for b in range(seg.shape[0]):
        n = int(nseg[b])
        if desc.form == 1:
            tf, tb = _masked_tables(wid, seg[b], n, S)
            np.testing.assert_array_equal(itf[b], tf)
            np.testing.assert_array_equal(itb[b], tb)
        else:
            np.testing.assert_array_equal(itf[b], M.interval_table_fwd(wid, seg[b], n, S))
            np.testing.assert_array_equal(itb[b], M.interval_table_bwd(wid, seg[b], n, S))
        sf = M.tile_states(wid, seg[b], n, S, tile=128)
        sb = M.tile_states(wid, seg[b], n, S, tile=128, backward=True)
        np.testing.assert_array_equal(bmf[b], M.pack_tile_states(sf))
        np.testing.assert_array_equal(bmb[b], M.pack_tile_states(sb))
    # schedules: permutations of (b, tile), non-increasing non-empty tile counts
    NT = S // 128
    for sched, bm in ((desc.sched_f, bmf), (desc.sched_b, bmb)):
        s = sched.cpu().numpy()
        bb, tt = s >> 16, s & 0xFFFF
        assert sorted(zip(bb.tolist(), tt.tolist())) == [(x, y) for x in range(seg.shape[0])
                                                        for y in range(NT)]
        words = bm[bb, tt]  # [n, W]
        x = (words | (words >> 1)) & 0x55555555
        counts = np.array([sum(bin(int(v)).count("1") for v in row) for row in x])
        assert (np.diff(counts) <= 0).all()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_descriptor_full_size(wid, mode):
    B = _lib()
    w = W.WORKLOADS[wid]
    seg, nseg = W.segments(wid, w.B, w.S)
    desc = _build(B, wid, seg, nseg, w.S, mode)
    _check(desc, wid, seg, nseg, w.S)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("S", [128, 384, 1024, 2048])
def test_descriptor_small_seeded(wid, S, mode):
    B = _lib()
    for seed in range(4):
        if wid == 5 and S < 1024:
            continue  # the prefix/document rule needs room for documents
        seg, nseg = W.segments(wid, 3, S, seed=100 * seed + S + wid)
        desc = _build(B, wid, seg, nseg, S, mode)
        _check(desc, wid, seg, nseg, S)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("S", [384, 1024])
def test_masked_form_small_seeded(wid, S, mode):
    """The masked form of the descriptor (maximal runs of invisible indices per row, the
    representation of the paper's section 4.4 ablation) is bit-exact with the oracle; the
    bitmaps and schedules are those of the visible form."""
    B = _lib()
    for seed in range(2):
        if wid == 5 and S < 1024:
            continue
        seg, nseg = W.segments(wid, 3, S, seed=300 * seed + S + wid)
        desc = _build(B, wid, seg, nseg, S, mode, form=B.CM_FORM_MASKED)
        _check(desc, wid, seg, nseg, S)


@pytest.mark.parametrize("wid", [4, 5])
def test_masked_form_full_size(wid):
    B = _lib()
    w = W.WORKLOADS[wid]
    seg, nseg = W.segments(wid, w.B, w.S)
    desc = _build(B, wid, seg, nseg, w.S, form=B.CM_FORM_MASKED)
    _check(desc, wid, seg, nseg, w.S)


def test_bad_metadata_is_reported_not_faulted():
    B = _lib()
    from masked_flashattention_gb300 import specs
    f = B.cm_compile_spec(specs.FWD[1])
    b = B.cm_compile_spec(specs.BWD[1])
    S = 256
    seg = np.array([[0, 100, 90, S]], dtype=np.int32)  # not increasing
    nseg = np.array([3], dtype=np.int32)
    desc = B.Descriptor(f, b, 1, S)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    assert B.cm_get_status(desc) == B.CM_ERR_DEVICE_CHECK
    # a valid build afterwards clears the status
    seg = np.array([[0, 100, 200, S]], dtype=np.int32)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    assert B.cm_get_status(desc) == B.CM_OK


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_generated_kernels_load_and_agree_with_the_generic_kernel(wid):
    """The mask-specific kernels compile and load on this GPU (so the default mode really runs
    them), and build the same bytes as the generic kernel on a batch of several samples."""
    B = _lib()
    from masked_flashattention_gb300 import specs
    for text in (specs.FWD[wid], specs.BWD[wid]):
        rc, log = B.cm_spec_kernel_status(B.cm_compile_spec(text), load=True)
        assert rc == B.CM_OK, log
    rc, log = B.cm_descriptor_kernel_status(B.cm_compile_spec(specs.FWD[wid]),
                                            B.cm_compile_spec(specs.BWD[wid]), load=True)
    assert rc == B.CM_OK, log
    S = 4096
    seg, nseg = W.segments(wid, 5, S, seed=11 + wid)
    a = _build(B, wid, seg, nseg, S, "generated")
    g = _build(B, wid, seg, nseg, S, "generic")
    for x, y in ((a.itab_f, g.itab_f), (a.bm_f, g.bm_f), (a.itab_b, g.itab_b), (a.bm_b, g.bm_b)):
        assert torch.equal(x, y)
