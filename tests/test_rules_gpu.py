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


def _four_intervals(i, j, sg, n, S):
    k, start, _ = _seg_arrays(sg, n, S)
    ki = k[i]

    def head(m):  # the first 8 positions of segment m (fewer if it is shorter)
        h0 = sg[np.clip(m, 0, n)]
        h1 = np.minimum(h0 + 8, sg[np.clip(m + 1, 0, n)])
        return (j >= h0) & (j < h1)

    far = (ki >= 2) & (head(ki - 2) | head(ki - 1))
    return (j < 16) | ((j >= start[i]) & (j <= i)) | far


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
    # four visible intervals per row (the compiler's slot limit; the CLEAR-style multi-interval
    # case): 16 sink tokens, the heads of the two previous segments, the own segment causally
    ("sink_two_previous_heads_and_own_segment",
     "region seg_idx(i) >= 2 : j < 16 "
     "|| (j >= seg_start_at(seg_idx(i) - 2) && j < min(seg_start_at(seg_idx(i) - 2) + 8, seg_end_at(seg_idx(i) - 2))) "
     "|| (j >= seg_start_at(seg_idx(i) - 1) && j < min(seg_start_at(seg_idx(i) - 1) + 8, seg_end_at(seg_idx(i) - 1))) "
     "|| (j >= seg_start(i) && j <= i)\n"
     "region all : j < 16 || (j >= seg_start(i) && j <= i)",
     "region i < 16 : j >= 0\n"
     "region seg_idx(i) == 0 && i < seg_start(i) + 8 : (j >= i && j < seg_end(i)) || (j >= seg_start_at(2) && j < seg_end_at(2))\n"
     "region i < seg_start(i) + 8 : (j >= i && j < seg_end(i)) || (j >= seg_start_at(seg_idx(i) + 1) && j < seg_end_at(seg_idx(i) + 2))\n"
     "region all : j >= i && j < seg_end(i)",
     _four_intervals),
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
    assert B.cm_get_status(desc) == B.CM_OK
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


def test_four_interval_rule_uses_four_slots():
    from masked_flashattention_gb300 import binding as B
    B.lib()
    rule = [r for r in RULES if r[0] == "sink_two_previous_heads_and_own_segment"][0]
    assert B.cm_spec_num_intervals(B.cm_compile_spec(rule[1])) == 4
    assert B.cm_spec_num_intervals(B.cm_compile_spec(rule[2])) == 2
