"""Pins for the attention side of the oracle (CPU only, fp64).

The oracle's forward is checked against PyTorch's scaled_dot_product_attention (a library
routine that shares no code with it), its LSE against closed forms, and its backward against
torch.autograd through that library routine and against central finite differences.  Each
planted-mistake test breaks the oracle on purpose (on the CPU) and shows a pin catching it.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from masked_flashattention_gb300 import workloads as W
from oracle import attention as A
from oracle import masks as M


def _inputs(S, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(S, d, generator=g, dtype=torch.float64) for _ in range(4)]


def _sdpa(q, k, v, mask):
    return F.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None],
                                          attn_mask=torch.as_tensor(mask)[None, None])[0, 0]


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_forward_matches_library_sdpa(wid):
    S, d = 256, 64
    seg, nseg = W.segments(wid, 1, S, seed=3)
    mask = M.dense_mask(wid, seg[0], int(nseg[0]), S)
    q, k, v, _ = _inputs(S, d, wid)
    o, _ = A.attention_forward(q, k, v, mask)
    assert torch.allclose(o, _sdpa(q, k, v, mask), rtol=1e-12, atol=1e-12)


def test_forward_causal_matches_is_causal():
    S, d = 300, 32
    q, k, v, _ = _inputs(S, d, 1)
    mask = np.tril(np.ones((S, S), dtype=bool))
    o, _ = A.attention_forward(q, k, v, mask)
    ref = F.scaled_dot_product_attention(q[None, None], k[None, None], v[None, None],
                                         is_causal=True)[0, 0]
    assert torch.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_all_visible_is_textbook_softmax_attention():
    S, d = 64, 16
    q, k, v, _ = _inputs(S, d, 2)
    o, lse = A.attention_forward(q, k, v, np.ones((S, S), dtype=bool))
    s = (q @ k.T) / math.sqrt(d)
    assert torch.allclose(o, torch.softmax(s, dim=1) @ v, rtol=1e-12, atol=1e-12)
    assert torch.allclose(lse, torch.log(torch.exp(s).sum(1)), rtol=1e-12, atol=1e-12)


def test_lse_closed_forms():
    S, d = 8, 4
    q, k, v, _ = _inputs(S, d, 3)
    # a row that sees exactly one key: lse = its score
    mask = np.eye(S, dtype=bool)
    _, lse = A.attention_forward(q, k, v, mask)
    want = (q * k).sum(1) / math.sqrt(d)
    assert torch.allclose(lse, want, rtol=1e-13, atol=1e-13)
    # equal scores over n keys: lse = c + log n
    qz = torch.zeros(S, d, dtype=torch.float64)
    mask = np.tril(np.ones((S, S), dtype=bool))
    _, lse = A.attention_forward(qz, k, v, mask)
    assert torch.allclose(lse, torch.log(torch.arange(1, S + 1, dtype=torch.float64)))


def test_fully_masked_row():
    S, d = 16, 8
    q, k, v, do = _inputs(S, d, 4)
    mask = np.tril(np.ones((S, S), dtype=bool))
    mask[5] = False
    o, lse = A.attention_forward(q, k, v, mask)
    assert torch.all(o[5] == 0) and lse[5] == float("-inf")
    dq, dk, dv = A.attention_backward(q, k, v, do, mask)
    assert torch.all(dq[5] == 0)
    assert torch.isfinite(dk).all() and torch.isfinite(dv).all()


@pytest.mark.parametrize("wid", [1, 3, 5])
def test_backward_matches_autograd_of_library(wid):
    S, d = 128, 32
    seg, nseg = W.segments(wid, 1, S, seed=5)
    mask = M.dense_mask(wid, seg[0], int(nseg[0]), S)
    q, k, v, do = _inputs(S, d, 10 + wid)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = _sdpa(qq, kk, vv, mask)
    out.backward(do)
    dq, dk, dv = A.attention_backward(q, k, v, do, mask)
    for got, want in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
        assert torch.allclose(got, want, rtol=1e-10, atol=1e-12)


def test_backward_finite_differences():
    S, d = 24, 8
    seg, nseg = W.segments(5, 1, S * 64, seed=2)  # any mask shape; take the causal part
    mask = np.tril(np.ones((S, S), dtype=bool))
    mask[10:, :3] = False
    q, k, v, do = _inputs(S, d, 7)

    def loss(q_, k_, v_):
        o, _ = A.attention_forward(q_, k_, v_, mask)
        return float((o * do).sum())

    dq, dk, dv = A.attention_backward(q, k, v, do, mask)
    h = 1e-6
    rng = np.random.default_rng(0)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(12):
            r, c = int(rng.integers(S)), int(rng.integers(d))
            args_p = [q.clone(), k.clone(), v.clone()]
            args_m = [q.clone(), k.clone(), v.clone()]
            args_p[which][r, c] += h
            args_m[which][r, c] -= h
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - float(grad[r, c])) < 1e-6 * max(1.0, abs(fd))


def test_row_blocking_is_exact():
    S, d = 200, 16
    seg, nseg = W.segments(3, 1, 256, seed=1)
    mask = M.dense_mask(3, seg[0], int(nseg[0]), 256)[:S, :S]
    q, k, v, do = _inputs(S, d, 8)
    o1, l1 = A.attention_forward(q, k, v, mask)
    o2, l2 = A.attention_forward(q, k, v, lambda a, b: mask[a:b], block_rows=37)
    assert torch.allclose(o1, o2, rtol=1e-13, atol=1e-13) and torch.allclose(l1, l2)
    g1 = A.attention_backward(q, k, v, do, mask)
    g2 = A.attention_backward(q, k, v, do, mask, block_rows=37)
    for a, b in zip(g1, g2):
        assert torch.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_delta_identity():
    """D_i = sum_j p_ij dp_ij equals rowsum(dO * O), the form kernels use."""
    S, d = 96, 16
    q, k, v, do = _inputs(S, d, 9)
    mask = np.tril(np.ones((S, S), dtype=bool))
    o, lse = A.attention_forward(q, k, v, mask)
    s = (q @ k.T) / math.sqrt(d)
    p = torch.where(torch.as_tensor(mask), torch.exp(s - lse[:, None]), torch.zeros_like(s))
    D = (p * (do @ v.T)).sum(1)
    assert torch.allclose(D, (do * o).sum(1), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# ------------------------------------------------------------------------------------------------
def test_planted_transposed_dk_is_caught(monkeypatch):
    orig = A.attention_backward

    def broken(q, k, v, do, mask, scale=None, block_rows=None):
        dq, dk, dv = orig(q, k, v, do, mask, scale, block_rows)
        return dq, dk.flip(0), dv  # plausible indexing slip in dk's rows
    monkeypatch.setattr(A, "attention_backward", broken)
    with pytest.raises(AssertionError):
        test_backward_matches_autograd_of_library(3)


def test_planted_missing_scale_is_caught(monkeypatch):
    orig = A.attention_forward

    def broken(q, k, v, mask, scale=None, block_rows=None):
        return orig(q, k, v, mask, 1.0, block_rows)  # forgot 1/sqrt(d)
    monkeypatch.setattr(A, "attention_forward", broken)
    with pytest.raises(AssertionError):
        test_forward_matches_library_sdpa(2)


def test_planted_off_by_one_interval_is_caught(monkeypatch):
    orig = M.interval_table_fwd

    def broken(wid, seg_row, nseg, S):
        t = orig(wid, seg_row, nseg, S).copy()
        nz = t[..., 1] > 0
        t[..., 1][nz] -= 1  # [s, i) instead of [s, i + 1)
        return t
    monkeypatch.setattr(M, "interval_table_fwd", broken)
    from tests import test_oracle_masks as TM
    case = next(iter(TM._small_cases()))
    with pytest.raises(AssertionError):
        TM.test_interval_union_equals_dense_rows(case)
