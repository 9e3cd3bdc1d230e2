"""GPU parity of descriptor-guided attention (forward and backward) against the fp64 oracle.

Tolerance (per tensor O, LSE, dQ, dK, dV; inputs are bf16 N(0, 1)): relative L2 error <= 1e-2
and max-abs error <= 3e-2.  Small cases compare every head; the full-size workloads run all heads
on the GPU in the same launch configuration the benchmark uses and compare heads 0 and H-1 of
every sample (each sample's mask is shared by its heads, so those two heads cover every row and
column of every mask).
"""
import math

import numpy as np
import pytest
import torch

from masked_flashattention_gb300 import workloads as W
from oracle import attention as A
from oracle import masks as M

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS = 1e-2, 3e-2


def _lib():
    from masked_flashattention_gb300 import binding as B
    B.lib()
    return B


def _errs(got, want):
    got = got.double().cpu()
    want = want.double().cpu()
    fin = torch.isfinite(want)
    assert torch.equal(fin, torch.isfinite(got)), "non-finite pattern differs"
    g, w = got[fin], want[fin]
    rel = ((g - w).norm() / max(w.norm().item(), 1e-30)).item()
    mx = (g - w).abs().max().item() if g.numel() else 0.0
    return rel, mx


def _assert_close(name, got, want):
    rel, mx = _errs(got, want)
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{name}: rel_l2={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


def run_gpu(B, fwd_text, bwd_text, seg, nseg, Q, K, V, dO, form=0):
    f = B.cm_compile_spec(fwd_text)
    b = B.cm_compile_spec(bwd_text)
    Bn, H, S, d = Q.shape
    desc = B.Descriptor(f, b, Bn, S, form=form)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse = B.attention_forward(desc, q, k, v)
    dq, dk, dv = B.attention_backward(desc, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == 0
    return o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def check_heads(wid, seg, nseg, Q, K, V, dO, out, heads, mask_fn=None):
    o, lse, dq, dk, dv = out
    Bn, H, S, d = Q.shape
    for b in range(Bn):
        if mask_fn is None:
            n = int(nseg[b])
            mask = lambda r0, r1, b=b, n=n: M.dense_mask(wid, seg[b], n, S, rows=np.arange(r0, r1))
        else:
            mask = mask_fn
        for h in heads:
            q, k, v, do = Q[b, h], K[b, h], V[b, h], dO[b, h]
            ro, rl = A.attention_forward(q, k, v, mask, block_rows=2048)
            rq, rk, rv = A.attention_backward(q, k, v, do, mask, block_rows=2048)
            _assert_close(f"O b{b}h{h}", o[b, h], ro)
            _assert_close(f"LSE b{b}h{h}", lse[b, h], rl)
            _assert_close(f"dQ b{b}h{h}", dq[b, h], rq)
            _assert_close(f"dK b{b}h{h}", dk[b, h], rk)
            _assert_close(f"dV b{b}h{h}", dv[b, h], rv)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("d", [64, 128])
def test_small_all_heads(wid, d):
    from masked_flashattention_gb300 import specs
    B = _lib()
    S = 1024
    w = W.scaled(W.WORKLOADS[wid], S, B=2, H=2, d=d)
    seg, nseg = W.segments(wid, w.B, S, seed=77 + wid)
    Q, K, V, dO = W.full_tensors(w, seed=9 + wid)
    out = run_gpu(B, specs.FWD[wid], specs.BWD[wid], seg, nseg, Q, K, V, dO)
    check_heads(wid, seg, nseg, Q, K, V, dO, out, range(w.H))


@pytest.mark.parametrize("S", [128, 384, 640])
def test_ragged_tile_counts(S):
    """Sizes with few or odd numbers of tiles (one tile; 3 and 5 tiles per row)."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    for wid in (1, 3, 4):
        w = W.scaled(W.WORKLOADS[wid], S, B=2, H=3, d=128)
        seg, nseg = W.segments(wid, w.B, S, seed=S + wid)
        Q, K, V, dO = W.full_tensors(w, seed=S + 3 * wid)
        out = run_gpu(B, specs.FWD[wid], specs.BWD[wid], seg, nseg, Q, K, V, dO)
        check_heads(wid, seg, nseg, Q, K, V, dO, out, range(w.H))


def test_rows_and_columns_that_see_nothing():
    """Rows with no visible key give O = 0 and LSE = -inf; keys nobody sees get zero dK/dV."""
    B = _lib()
    S, d = 512, 64
    fwd = "region i >= 200 : j <= i && j >= 130"
    bwd = "region i >= 130 : j >= max(i, 200)"
    seg = np.array([[0, S]], dtype=np.int32)
    nseg = np.array([1], dtype=np.int32)
    w = W.Workload(0, "partial-visibility", 1, 2, S, d)
    Q, K, V, dO = W.full_tensors(w, seed=5)
    out = run_gpu(B, fwd, bwd, seg, nseg, Q, K, V, dO)
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    dense = (i >= 200) & (j <= i) & (j >= 130)
    o, lse = out[0], out[1]
    assert torch.all(o[:, :, :200] == 0)
    assert torch.all(torch.isneginf(lse[:, :, :200]))
    assert torch.all(out[3][:, :, :130] == 0) and torch.all(out[4][:, :, :130] == 0)
    check_heads(0, seg, nseg, Q, K, V, dO, out, range(2), mask_fn=lambda r0, r1: dense[r0:r1])


def check_row_blocks_every_head(wid, seg, nseg, Q, K, V, dO, out, row0s):
    """Every (sample, head) on a few 128-row blocks of query rows, against the oracle run on
    those rows only: O, LSE and dQ of the rows, and for the last block (rows [S - 128, S)) the
    complete dK and dV of the last 128 keys, which no earlier row sees in these masks (every
    rule here is causal: key j is visible only to rows i >= j)."""
    o, lse, dq, dk, dv = out
    Bn, H, S, d = Q.shape
    for b in range(Bn):
        n = int(nseg[b])
        for r0 in row0s:
            R = slice(r0, r0 + 128)
            rows = np.arange(r0, r0 + 128)
            dense = M.dense_mask(wid, seg[b], n, S, rows=rows)
            assert not dense[:, rows[-1] + 1:].any()  # causal: nothing right of the block
            for h in range(H):
                ro, rl = A.attention_forward(Q[b, h, R], K[b, h], V[b, h], dense)
                rq, rk, rv = A.attention_backward(Q[b, h, R], K[b, h], V[b, h], dO[b, h, R], dense)
                _assert_close(f"O b{b}h{h} rows {r0}+", o[b, h, R], ro)
                _assert_close(f"LSE b{b}h{h} rows {r0}+", lse[b, h, R], rl)
                _assert_close(f"dQ b{b}h{h} rows {r0}+", dq[b, h, R], rq)
                if r0 == S - 128:
                    _assert_close(f"dK b{b}h{h} last keys", dk[b, h, R], rk[R])
                    _assert_close(f"dV b{b}h{h} last keys", dv[b, h, R], rv[R])


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_full_size_sampled_heads(wid):
    """Full size, in the benchmark's launch configuration.  Heads 0 and H-1 of every sample are
    compared in full; every other head on its first, middle and last 128 query rows (and the
    last 128 keys), so that each head's place in the kernels' grid is checked too."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    w = W.WORKLOADS[wid]
    seg, nseg = W.segments(wid, w.B, w.S)
    Q, K, V, dO = W.full_tensors(w)
    out = run_gpu(B, specs.FWD[wid], specs.BWD[wid], seg, nseg, Q, K, V, dO)
    heads = range(w.H) if wid == 1 else sorted({0, w.H - 1})
    check_heads(wid, seg, nseg, Q, K, V, dO, out, heads)
    if wid != 1:
        check_row_blocks_every_head(wid, seg, nseg, Q, K, V, dO, out,
                                    (0, (w.S // 256) * 128, w.S - 128))


def test_every_head_of_every_sample_with_full_schedule_chunks():
    """The kernels take the longest-first schedule in chunks of 128 work items and walk every
    head inside a chunk (a different branch of the grid mapping than when the schedule holds
    fewer than 128 items).  B * S/128 = 17 * 16 = 272 work items make two full chunks and a
    partial one; every (sample, head) is compared with the oracle, element by element."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    wid, S, Bn, H, d = 1, 2048, 17, 4, 128
    w = W.scaled(W.WORKLOADS[wid], S, B=Bn, H=H, d=d)
    seg, nseg = W.segments(wid, w.B, S, seed=2024)
    Q, K, V, dO = W.full_tensors(w, seed=99)
    out = run_gpu(B, specs.FWD[wid], specs.BWD[wid], seg, nseg, Q, K, V, dO)
    check_heads(wid, seg, nseg, Q, K, V, dO, out, range(H))


# (check form, descriptor form) pairs other than the default (range masks, visible intervals):
# the four arms of the paper's section 4.4 ablation and range masks over masked intervals
ARMS = {"unsigned_visible": (0, 0), "two_compare_visible": (1, 0), "unsigned_masked": (0, 1),
        "two_compare_masked": (1, 1), "range_masked": (3, 1)}


@pytest.mark.parametrize("arm", sorted(ARMS))
@pytest.mark.parametrize("wid", [1, 3, 4, 5, 6])
def test_interval_check_forms_small(wid, arm):
    """Every form of the partial-tile check, on visible and on masked Interval Tables, gives the
    oracle's attention on masks with 1 to 3 intervals per row."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    check, form = ARMS[arm]
    S = 1024
    w = W.scaled(W.WORKLOADS[wid], S, B=2, H=2, d=128)
    seg, nseg = W.segments(wid, w.B, S, seed=31 + wid)
    Q, K, V, dO = W.full_tensors(w, seed=13 + wid)
    B.cm_set_interval_check(check)
    try:
        out = run_gpu(B, specs.FWD[wid], specs.BWD[wid], seg, nseg, Q, K, V, dO, form=form)
    finally:
        B.cm_set_interval_check(B.CM_CHECK_RANGE_MASK)
    check_heads(wid, seg, nseg, Q, K, V, dO, out, range(w.H))


@pytest.mark.parametrize("arm", sorted(ARMS))
def test_interval_check_forms_full_size_hstu(arm):
    """The ablation arms at the HSTU workload's full size (heads 0 and H-1 against the oracle)."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    check, form = ARMS[arm]
    w = W.WORKLOADS[4]
    seg, nseg = W.segments(4, w.B, w.S)
    Q, K, V, dO = W.full_tensors(w)
    B.cm_set_interval_check(check)
    try:
        out = run_gpu(B, specs.FWD[4], specs.BWD[4], seg, nseg, Q, K, V, dO, form=form)
    finally:
        B.cm_set_interval_check(B.CM_CHECK_RANGE_MASK)
    check_heads(4, seg, nseg, Q, K, V, dO, out, sorted({0, w.H - 1}))


def test_maximum_sequence_length_causal():
    """The largest supported sequence (S = 131072, 1024 tiles per row) on a causal mask.  The
    oracle runs on the first and the last 128 query rows against all keys: that gives O, LSE
    and dQ of those rows, and the complete dK and dV of the last 128 keys, which no other row
    sees.  The descriptor is checked against the closed-form causal tables and tile census."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    S, H, d = 131072, 1, 128
    seg = np.array([[0, S]], dtype=np.int32)
    nseg = np.array([1], dtype=np.int32)
    w = W.Workload(2, "causal@S131072", 1, H, S, d)
    Q, K, V, dO = W.full_tensors(w, seed=17)
    f = B.cm_compile_spec(specs.FWD[2])
    b = B.cm_compile_spec(specs.BWD[2])
    desc = B.Descriptor(f, b, 1, S)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse = B.attention_forward(desc, q, k, v)
    dq, dk, dv = B.attention_backward(desc, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == 0
    # descriptor: row i sees [0, i + 1); tile census n(n-1)/2 full, n partial, the rest empty
    itf = desc.interval_table_fwd()[0, 0]
    np.testing.assert_array_equal(itf[:, 0], np.zeros(S, dtype=np.int32))
    np.testing.assert_array_equal(itf[:, 1], np.arange(1, S + 1, dtype=np.int32))
    words = desc.bitmap_fwd()[0]
    codes = np.stack([(words >> (2 * t)) & 3 for t in range(16)], axis=-1).reshape(words.shape[0], -1)
    n = S // 128
    assert int((codes == 2).sum()) == n * (n - 1) // 2 and int((codes == 1).sum()) == n
    for r0 in (0, S - 128):
        R = slice(r0, r0 + 128)
        mask = lambda a, c, r0=r0: (np.arange(S)[None, :] <= (r0 + np.arange(a, c))[:, None])
        ro, rl = A.attention_forward(Q[0, 0, R], K[0, 0], V[0, 0], mask)
        rq, rk, rv = A.attention_backward(Q[0, 0, R], K[0, 0], V[0, 0], dO[0, 0, R], mask)
        _assert_close(f"O rows {r0}+", o[0, 0, R].cpu(), ro)
        _assert_close(f"LSE rows {r0}+", lse[0, 0, R].cpu(), rl)
        _assert_close(f"dQ rows {r0}+", dq[0, 0, R].cpu(), rq)
        if r0 == S - 128:
            _assert_close("dK last keys", dk[0, 0, R].cpu(), rk[R])
            _assert_close("dV last keys", dv[0, 0, R].cpu(), rv[R])


@pytest.mark.parametrize("d", [64, 128])
def test_backward_stages_with_the_standalone_prologue(d):
    """The dK/dV stage after the standalone prologue (no dQ stage) gives the oracle's dK and dV,
    and the prologue's per-row constants (-D, -LSE*log2e) agree with the ones the dQ stage
    writes into its workspace (same values up to the order of the fp32 sums)."""
    from masked_flashattention_gb300 import specs
    B = _lib()
    wid, S = 3, 1024
    w = W.scaled(W.WORKLOADS[wid], S, B=2, H=2, d=d)
    seg, nseg = W.segments(wid, w.B, S, seed=41)
    Q, K, V, dO = W.full_tensors(w, seed=42)
    f, b = B.cm_compile_spec(specs.FWD[wid]), B.cm_compile_spec(specs.BWD[wid])
    desc = B.Descriptor(f, b, w.B, S)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse = B.attention_forward(desc, q, k, v)
    n = B.cm_attn_bwd_workspace_size(w.B, w.H, S, d)
    ws_pro = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ws_dq = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dk, dv, dq = torch.empty_like(k), torch.empty_like(v), torch.empty_like(q)
    B.cm_attn_bwd_prologue(o, lse, do, ws_pro)
    B.cm_attn_bwd_dkdv(desc, q, k, v, do, dk, dv, ws_pro)
    B.cm_attn_bwd_dq(desc, q, k, v, o, lse, do, dq, ws_dq)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == 0
    a, c = ws_pro.view(torch.float32).cpu(), ws_dq.view(torch.float32).cpu()
    assert torch.equal(torch.isfinite(a), torch.isfinite(c))
    fin = torch.isfinite(a)
    assert torch.allclose(a[fin], c[fin], rtol=1e-4, atol=1e-5)
    dk, dv = dk.cpu(), dv.cpu()
    for bb in range(w.B):
        nb = int(nseg[bb])
        mask = lambda r0, r1, bb=bb, nb=nb: M.dense_mask(wid, seg[bb], nb, S, rows=np.arange(r0, r1))
        for h in range(w.H):
            _, rk, rv = A.attention_backward(Q[bb, h], K[bb, h], V[bb, h], dO[bb, h], mask,
                                             block_rows=2048)
            _assert_close(f"dK b{bb}h{h}", dk[bb, h], rk)
            _assert_close(f"dV b{bb}h{h}", dv[bb, h], rv)
