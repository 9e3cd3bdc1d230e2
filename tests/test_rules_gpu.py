"""GPU checks of the compiler + preprocess + attention on MaskSpecs beyond the five workloads.

Each rule comes as a forward MaskSpec, the backward MaskSpec for the transposed traversal, and a
hand-written numpy predicate of the same rule (independent of the compiler).  The descriptor the
preprocess kernel builds must reproduce the predicate exactly (interval union per row, and the
2-bit tile states of the dense mask and of its transpose); attention on the descriptor must match
the fp64 oracle run on the predicate's dense mask.
"""
import numpy as np
import pytest
import torch

from masked_flashattention_gb300 import workloads as W
from oracle import attention as A
from oracle import masks as M

pytestmark = pytest.mark.gpu


def _seg_arrays(seg_row, nseg, S):
    pos = np.arange(S)
    k = np.searchsorted(seg_row[: nseg + 1], pos, side="right") - 1
    return k, seg_row[k], seg_row[np.minimum(k + 1, nseg)]


# (name, forward spec, backward spec, predicate(i, j, seg_row, nseg, S) -> bool [rows, cols])
def _window(i, j, sg, n, S):
    return (j > i - 200) & (j <= i)


def _doc_sink(i, j, sg, n, S):
    k, start, _ = _seg_arrays(sg, n, S)
    return (j <= i) & ((j >= start[i]) | (j < 16))


def _doc_bidir_global(i, j, sg, n, S):
    k, start, end = _seg_arrays(sg, n, S)
    return ((j >= start[i]) & (j < end[i])) | (i < 32) | (j < 32)


def _not_self_causal(i, j, sg, n, S):
    return (j <= i) & (j != i) | ((i == 0) & (j == 0))


RULES = [
    ("sliding_window_200",
     "region all : j > i - 200 && j <= i",
     "region all : j >= i && j < i + 200",
     _window),
    ("document_causal_with_16_sink_tokens",
     "region all : j <= i && (j >= seg_start(i) || j < 16)",
     "region i < 16 : j >= i\n"
     "region all : j >= i && j < seg_end(i)",
     _doc_sink),
    ("bidirectional_documents_plus_global_tokens",
     "region i < 32 : j >= 0\n"
     "region all : (j >= seg_start(i) && j < seg_end(i)) || j < 32",
     "region i < 32 : j >= 0\n"
     "region all : (j >= seg_start(i) && j < seg_end(i)) || j < 32",
     _doc_bidir_global),
    ("causal_without_the_diagonal",
     "region i == 0 : j == 0\n"
     "region all : j < i",
     "region all : j > i || (i == 0 && j == 0)",
     _not_self_causal),
]


def _dense(pred, seg_row, nseg, S):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    return np.asarray(pred(i, j, seg_row, nseg, S), dtype=bool)


def _build(B, fwd_text, bwd_text, seg, nseg, S):
    f, b = B.cm_compile_spec(fwd_text), B.cm_compile_spec(bwd_text)
    desc = B.Descriptor(f, b, seg.shape[0], S)
    B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
    torch.cuda.synchronize()
    assert B.cm_get_status(desc) == 0
    return desc


@pytest.mark.parametrize("rule", RULES, ids=[r[0] for r in RULES])
@pytest.mark.parametrize("S", [256, 640, 1024])
def test_descriptor_matches_hand_predicate(rule, S):
    from masked_flashattention_gb300 import binding as B
    B.lib()
    name, ftxt, btxt, pred = rule
    seg, nseg = W.random_segments(3, S, max_segs=6, seed=S + len(name))
    desc = _build(B, ftxt, btxt, seg, nseg, S)
    itf, itb = desc.interval_table_fwd(), desc.interval_table_bwd()
    bmf, bmb = desc.bitmap_fwd(), desc.bitmap_bwd()
    for b in range(seg.shape[0]):
        dense = _dense(pred, seg[b], int(nseg[b]), S)
        assert np.array_equal(M.intervals_to_mask(itf[b], S), dense)
        assert np.array_equal(M.intervals_to_mask(itb[b], S), dense.T)
        np.testing.assert_array_equal(bmf[b], M.pack_tile_states(M.tile_states_of(dense, 128, 128)))
        np.testing.assert_array_equal(bmb[b], M.pack_tile_states(M.tile_states_of(dense.T, 128, 128)))


@pytest.mark.parametrize("rule", RULES, ids=[r[0] for r in RULES])
def test_attention_on_custom_rule(rule):
    from masked_flashattention_gb300 import binding as B
    B.lib()
    name, ftxt, btxt, pred = rule
    S, H, d = 1024, 2, 128
    seg, nseg = W.random_segments(2, S, max_segs=5, seed=3)
    desc = _build(B, ftxt, btxt, seg, nseg, S)
    w = W.Workload(0, name, 2, H, S, d)
    Q, K, V, dO = W.full_tensors(w, seed=11)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse = B.attention_forward(desc, q, k, v)
    dq, dk, dv = B.attention_backward(desc, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    for b in range(2):
        dense = _dense(pred, seg[b], int(nseg[b]), S)
        for h in range(H):
            ro, rl = A.attention_forward(Q[b, h], K[b, h], V[b, h], dense)
            rq, rk, rv = A.attention_backward(Q[b, h], K[b, h], V[b, h], dO[b, h], dense)
            for nm, got, want in (("O", o, ro), ("LSE", lse, rl), ("dQ", dq, rq), ("dK", dk, rk),
                                  ("dV", dv, rv)):
                g = got[b, h].double().cpu()
                rel = ((g - want).norm() / want.norm()).item()
                mx = (g - want).abs().max().item()
                assert rel <= 1e-2 and mx <= 3e-2, f"{name} {nm} b{b}h{h}: {rel:.3e} {mx:.3e}"
