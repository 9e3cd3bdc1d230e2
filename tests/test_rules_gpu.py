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


def _heads_rule(p):
    """Sink tokens [0, 16), the first 8 tokens of each of the p previous segments, and the own
    segment causally: p + 2 visible intervals per row (CLEAR-style multi-interval rows)."""
    fwd_terms = ["j < 16", "(j >= seg_start(i) && j <= i)"]
    for m in range(1, p + 1):
        fwd_terms.append(f"(j >= seg_start_at(seg_idx(i) - {m}) && "
                         f"j < min(seg_start_at(seg_idx(i) - {m}) + 8, seg_end_at(seg_idx(i) - {m})))")
    fwd = "region all : " + " || ".join(fwd_terms)
    # key columns: sink keys are seen by every row; a key among the first 8 of its segment by the
    # rows of the p following segments; every key by the later rows of its own segment
    bwd = ("region i < 16 : j >= 0\n"
           "region i < seg_start(i) + 8 : (j >= i && j < seg_end(i)) || "
           f"(j >= seg_start_at(seg_idx(i) + 1) && j < seg_end_at(seg_idx(i) + {p}))\n"
           "region all : j >= i && j < seg_end(i)")

    def pred(i, j, sg, n, S):
        k, start, _ = _seg_arrays(sg, n, S)
        ki = k[i]
        vis = (j < 16) | ((j >= start[i]) & (j <= i))
        for m in range(1, p + 1):
            km = ki - m
            h0 = sg[np.clip(km, 0, n)]
            h1 = np.minimum(h0 + 8, sg[np.clip(km + 1, 0, n)])
            vis = vis | ((km >= 0) & (j >= h0) & (j < h1))
        return vis

    return (f"sink_{p}_previous_heads_and_own_segment", fwd, bwd, pred)


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
    # five, six and eight visible intervals per row (eight is the compiler's limit)
    _heads_rule(3),
    _heads_rule(4),
    _heads_rule(6),
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
    seg, nseg = W.random_segments(3, S, max_segs=12, seed=S + len(name))
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
    seg, nseg = W.random_segments(2, S, max_segs=10, seed=3)
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


@pytest.mark.parametrize("p", [3, 4, 6])
def test_multi_interval_rules_derive_their_interval_count(p):
    """The compiler derives the interval count from the rule (no preset count): p previous-segment
    heads, the sink and the own segment give p + 2 forward slots; the backward rule has 2."""
    from masked_flashattention_gb300 import binding as B
    B.lib()
    _, ftxt, btxt, _ = _heads_rule(p)
    assert B.cm_spec_num_intervals(B.cm_compile_spec(ftxt)) == p + 2
    assert B.cm_spec_num_intervals(B.cm_compile_spec(btxt)) == 2


@pytest.mark.parametrize("rule", [r for r in RULES if r[0].startswith("sink_")],
                         ids=lambda r: r[0])
def test_multi_interval_rules_masked_form_and_per_score_checks(rule):
    """Rules with 4 to 8 intervals per row (5 to 9 masked runs) with the per-score forms of the
    check, on visible and on masked Interval Tables: attention equals the oracle."""
    from masked_flashattention_gb300 import binding as B
    B.lib()
    name, ftxt, btxt, pred = rule
    S, H, d = 1024, 1, 64
    seg, nseg = W.random_segments(2, S, max_segs=12, seed=8)
    f, b = B.cm_compile_spec(ftxt), B.cm_compile_spec(btxt)
    w = W.Workload(0, name, 2, H, S, d)
    Q, K, V, dO = W.full_tensors(w, seed=21)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    for check, form in ((B.CM_CHECK_UNSIGNED, B.CM_FORM_VISIBLE), (B.CM_CHECK_TWO_COMPARE, B.CM_FORM_MASKED),
                        (B.CM_CHECK_RANGE_MASK, B.CM_FORM_MASKED)):
        desc = B.Descriptor(f, b, 2, S, form=form)
        B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(), desc)
        B.cm_set_interval_check(check)
        try:
            o, lse = B.attention_forward(desc, q, k, v)
            dq, dk, dv = B.attention_backward(desc, q, k, v, o, lse, do)
            torch.cuda.synchronize()
        finally:
            B.cm_set_interval_check(B.CM_CHECK_RANGE_MASK)
        assert B.cm_get_status(desc) == B.CM_OK
        for bb in range(2):
            dense = _dense(pred, seg[bb], int(nseg[bb]), S)
            if form == B.CM_FORM_MASKED:
                nif = B.cm_spec_num_intervals(f)
                np.testing.assert_array_equal(desc.interval_table_fwd()[bb],
                                              M.masked_runs_table(dense, nif + 1))
            ro, rl = A.attention_forward(Q[bb, 0], K[bb, 0], V[bb, 0], dense)
            rq, rk, rv = A.attention_backward(Q[bb, 0], K[bb, 0], V[bb, 0], dO[bb, 0], dense)
            for nm, got, want in (("O", o, ro), ("LSE", lse, rl), ("dQ", dq, rq), ("dK", dk, rk),
                                  ("dV", dv, rv)):
                g = got[bb, 0].double().cpu()
                fin = torch.isfinite(want)
                rel = ((g[fin] - want[fin]).norm() / want[fin].norm()).item()
                mx = (g[fin] - want[fin]).abs().max().item()
                assert rel <= 1e-2 and mx <= 3e-2, f"{name} {check}/{form} {nm} b{bb}: {rel:.3e} {mx:.3e}"
