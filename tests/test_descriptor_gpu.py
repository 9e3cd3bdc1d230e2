"""GPU parity of the Execution Descriptor: the preprocess kernels vs the oracle, bit-exact.

Interval Tables and Tile-State Bitmaps (forward and backward) must equal the oracle's on the five
workloads at full size and on many small seeded segmentations (ragged tails included); the
schedule must be a longest-first permutation of the tile rows.
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


def _build(B, wid, seg, nseg, S):
    from masked_flashattention_gb300 import specs
    f = B.cm_compile_spec(specs.FWD[wid])
    b = B.cm_compile_spec(specs.BWD[wid])
    desc = B.Descriptor(f, b, seg.shape[0], S)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == 0
    return desc


def _check(desc, wid, seg, nseg, S):
    itf, itb = desc.interval_table_fwd(), desc.interval_table_bwd()
    bmf, bmb = desc.bitmap_fwd(), desc.bitmap_bwd()
    for b in range(seg.shape[0]):
        n = int(nseg[b])
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


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_descriptor_full_size(wid):
    B = _lib()
    w = W.WORKLOADS[wid]
    seg, nseg = W.segments(wid, w.B, w.S)
    desc = _build(B, wid, seg, nseg, w.S)
    _check(desc, wid, seg, nseg, w.S)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("S", [128, 384, 1024, 2048])
def test_descriptor_small_seeded(wid, S):
    B = _lib()
    for seed in range(4):
        if wid == 5 and S < 1024:
            continue  # the prefix/document rule needs room for documents
        seg, nseg = W.segments(wid, 3, S, seed=100 * seed + S + wid)
        desc = _build(B, wid, seg, nseg, S)
        _check(desc, wid, seg, nseg, S)


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
