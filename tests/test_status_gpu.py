"""Device-side failure reporting on the GPU, without faulting it.

The pages describe no failure handling; this is the library's own.  Every wait inside the
attention kernels is bounded.  A CTA whose wait expires records CM_ERR_TIMEOUT in the
descriptor's status word, lets the TMA copies and MMAs it already issued complete, frees its TMEM
and exits, so the context stays usable.  The dK/dV kernel also checks that the backward
Tile-State Bitmap is the transpose of the forward one (each traversal direction has its own
descriptor, CompileMask section 3.3, and both must describe the same mask).
"""
import numpy as np
import pytest
import torch

from masked_flashattention_gb300 import workloads as W
from oracle import attention as A
from oracle import masks as M

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS = 1e-2, 3e-2


def _close(name, got, want):
    got, want = got.double().cpu(), want.double().cpu()
    rel = ((got - want).norm() / want.norm()).item()
    mx = (got - want).abs().max().item()
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{name}: rel_l2={rel:.3e} max_abs={mx:.3e}"


def _setup(B, wid, S, Bn, H, d, fwd_text, bwd_text, seed):
    w = W.scaled(W.WORKLOADS[wid], S, B=Bn, H=H, d=d)
    seg, nseg = W.segments(wid, Bn, S, seed=seed)
    f, b = B.cm_compile_spec(fwd_text), B.cm_compile_spec(bwd_text)
    desc = B.Descriptor(f, b, Bn, S)
    meta = (torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda())
    B.cm_build_descriptor(f, b, meta[0], meta[1], desc)
    tensors = W.full_tensors(w, seed=seed)
    return w, seg, nseg, f, b, desc, meta, tensors


def test_expired_waits_are_reported_and_the_next_call_is_correct():
    """With a wait limit of 1 ns, ordinary waits (a TMA copy in flight, an MMA running) expire:
    forward and backward must return CM_ERR_TIMEOUT through the status word.  With the default
    limit restored, the same calls on the same context must succeed and match the oracle."""
    from masked_flashattention_gb300 import binding as B
    from masked_flashattention_gb300 import specs
    B.lib()
    wid = 3
    w, seg, nseg, f, b, desc, meta, (Q, K, V, dO) = _setup(
        B, wid, 1024, 2, 2, 128, specs.FWD[wid], specs.BWD[wid], seed=71)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    B.cm_set_wait_limit_ns(1)
    try:
        o, lse = B.attention_forward(desc, q, k, v)
        B.attention_backward(desc, q, k, v, o, lse, do)
        torch.cuda.synchronize()
        assert B.cm_get_status(desc) == B.CM_ERR_TIMEOUT
    finally:
        B.cm_set_wait_limit_ns(0)
    # the status word keeps the first error until the descriptor is rebuilt
    B.cm_build_descriptor(f, b, meta[0], meta[1], desc)
    o, lse = B.attention_forward(desc, q, k, v)
    dq, dk, dv = B.attention_backward(desc, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == B.CM_OK
    for bb in range(w.B):
        mask = M.dense_mask(wid, seg[bb], int(nseg[bb]), w.S)
        for h in range(w.H):
            ro, rl = A.attention_forward(Q[bb, h], K[bb, h], V[bb, h], mask)
            rq, rk, rv = A.attention_backward(Q[bb, h], K[bb, h], V[bb, h], dO[bb, h], mask)
            for name, got, want in (("O", o, ro), ("LSE", lse, rl), ("dQ", dq, rq),
                                    ("dK", dk, rk), ("dV", dv, rv)):
                _close(f"{name} b{bb}h{h}", got[bb, h], want)


def test_mismatched_forward_and_backward_specs_are_reported():
    """A backward MaskSpec that describes another mask (plain causal against the shared-prompt
    reward-model mask): the backward reports CM_ERR_DESC_MISMATCH, and the forward alone, which
    uses only the forward half of the descriptor, does not."""
    from masked_flashattention_gb300 import binding as B
    from masked_flashattention_gb300 import specs
    B.lib()
    w, seg, nseg, f, b, desc, meta, (Q, K, V, dO) = _setup(
        B, 3, 2048, 1, 2, 64, specs.FWD[3], specs.BWD[2], seed=5)
    # the two descriptors really differ (response rows do not see the other responses' keys)
    bmf, bmb = desc.bitmap_fwd()[0], desc.bitmap_bwd()[0]
    codes = lambda words: np.stack([(words >> (2 * t)) & 3 for t in range(16)], -1).reshape(
        words.shape[0], -1)[:, : w.S // 128]
    assert not np.array_equal(codes(bmb), codes(bmf).T)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse = B.attention_forward(desc, q, k, v)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == B.CM_OK
    B.attention_backward(desc, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == B.CM_ERR_DESC_MISMATCH
