"""CPU checks of the C ABI: the library loads and exports every declared symbol, the offline
compiler lowers MaskSpecs as the paper describes (section 3.2.2), and host-side validation
rejects bad arguments before anything reaches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from masked_flashattention_gb300 import build as bld
    bld.build()
    from masked_flashattention_gb300 import binding
    binding.lib()
    return binding


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "cm.h")).read()
    return re.findall(r"CM_API\s+[\w\s\*]+?\b(cm_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(B):
    names = declared_symbols()
    assert len(names) >= 11
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_region_c_lowering(B):
    """The paper's Region C: the response rule keeps [0, b) and [s(i), i + 1) as two slots."""
    from masked_flashattention_gb300 import specs
    s = B.cm_compile_spec(specs.FWD[3])
    text = B.cm_spec_describe(s)
    assert B.cm_spec_num_intervals(s) == 2
    region1 = text.split("region 1")[1]
    assert "slot 0: [0, seg_end_at(0))" in region1
    assert "slot 1: [seg_start(i), i + 1)" in region1


@pytest.mark.parametrize("wid,nif,nib", [(1, 1, 1), (2, 1, 1), (3, 2, 1), (4, 2, 1), (5, 3, 2), (6, 2, 1)])
def test_interval_counts(B, wid, nif, nib):
    from masked_flashattention_gb300 import specs
    from oracle import masks as M
    assert (nif, nib) == M.num_intervals(wid)
    assert B.cm_spec_num_intervals(B.cm_compile_spec(specs.FWD[wid])) == nif
    assert B.cm_spec_num_intervals(B.cm_compile_spec(specs.BWD[wid])) == nib


@pytest.mark.parametrize("rule,slots", [
    ("j <= i", ["[0, i + 1)"]),
    ("!(j > i)", ["[0, i + 1)"]),
    ("j != i", ["[0, i)", "[i + 1, S)"]),
    ("i >= j && j >= i - 3", ["[i - 3, i + 1)"]),
    ("j == i || j == i", ["[i, i + 1)"]),
    ("j < 0", []),
    ("j >= i + 1 && j <= i", []),
    ("(j < 10 || j >= 20) && j < 30", ["[0, 10)", "[20, 30)"]),
    ("2 * i - j >= 0 - i", ["[0, 3*i + 1)"]),
    ("j - seg_start(i) < 64 && j >= seg_start(i)", ["[seg_start(i), seg_start(i) + 64)"]),
])
def test_dnf_and_interval_extraction(B, rule, slots):
    s = B.cm_compile_spec(f"region all : {rule}")
    got = [line.split(": ", 1)[1].split(" if ")[0]
           for line in B.cm_spec_describe(s).splitlines() if line.strip().startswith("slot")]
    assert got == slots


def test_conditions_without_j_become_slot_conditions(B):
    s = B.cm_compile_spec("region all : j <= i || (i < 100 && j == 200)")
    text = B.cm_spec_describe(s)
    assert "slot 1: [200, 201) if i - 100 < 0" in text


def test_modulo_by_a_constant():
    """'%' by a positive constant: a guard on the parity of the segment index lowers to a
    remainder term; constant remainders fold; other divisors are rejected."""
    from masked_flashattention_gb300 import binding as B
    d = B.cm_spec_describe(B.cm_compile_spec("region seg_idx(i) % 2 == 1 : j <= i"))
    assert "mod(seg_idx(i), 2) == 1" in d
    d = B.cm_spec_describe(B.cm_compile_spec("region all : j < 7 % 4 + i"))
    assert "[0, i + 3)" in d
    for bad in ("region all : j < i % 0", "region all : j < i % i", "region all : j % 2 < i"):
        with pytest.raises(B.CMError):
            B.cm_compile_spec(bad)


@pytest.mark.parametrize("bad", [
    "region all j <= i",            # missing ':'
    "region j < 3 : j <= i",        # j in a guard
    "region all : 2 * j <= i",      # coefficient 2
    "region all : min(j, i) <= 3",  # j inside min
    "region all : j <= i * i",      # non-constant product
    "region all : j <= foo(i)",     # unknown name
    "region all : j < i < 3",       # chained comparison
    "",                             # no region
])
def test_parse_errors(B, bad):
    with pytest.raises(B.CMError) as e:
        B.cm_compile_spec(bad)
    assert e.value.code == B.CM_ERR_PARSE


def test_descriptor_sizes(B):
    from masked_flashattention_gb300 import specs
    f, b = B.cm_compile_spec(specs.FWD[5]), B.cm_compile_spec(specs.BWD[5])
    sizes = B.cm_descriptor_sizes(f, b, 2, 32768)
    NT = 256
    # status: the status word, the preprocess kernel's grid barrier and its two histograms of
    # per-row tile counts (0..NT)
    assert sizes == [2 * 3 * 32768 * 8, 2 * NT * 16 * 4, 2 * 2 * 32768 * 8, 2 * NT * 16 * 4,
                     2 * NT * 4, 2 * NT * 4, 4 * (2 + 2 * (NT + 1) + 6)]
    # masked form: one more slot per row (the runs around ni visible intervals)
    msizes = B.cm_descriptor_sizes(f, b, 2, 32768, form=B.CM_FORM_MASKED)
    assert msizes[0] == 2 * 4 * 32768 * 8 and msizes[2] == 2 * 3 * 32768 * 8
    assert msizes[1:2] == sizes[1:2] and msizes[3:] == sizes[3:]
    with pytest.raises(B.CMError):
        B.cm_descriptor_sizes(f, b, 2, 32768, form=2)
    with pytest.raises(B.CMError):
        B.cm_descriptor_sizes(f, b, 2, 1000)   # S not a multiple of 128
    with pytest.raises(B.CMError):
        B.cm_descriptor_sizes(f, b, 2, 32768, tile=64)


def _fake_desc(B, Bn, S, ni_f=1, ni_b=1, form=0):
    p = 1 << 20  # never dereferenced: validation fails first
    return B.cm_descriptor(Bn, S, 128, ni_f, ni_b, form, p, p, p, p, p, p, p)


def test_attention_argument_validation_happens_on_the_host(B):
    L = B.lib()
    p = ctypes.c_void_p(1 << 20)
    d = _fake_desc(B, 1, 256)
    # unsupported head dim
    assert L.cm_attn_fwd(ctypes.byref(d), p, p, p, p, p, 1, 2, 256, 96, 0.1, None) == B.CM_ERR_UNSUPPORTED
    # S not a multiple of the tile
    d2 = _fake_desc(B, 1, 200)
    assert L.cm_attn_fwd(ctypes.byref(d2), p, p, p, p, p, 1, 2, 200, 64, 0.1, None) == B.CM_ERR_UNSUPPORTED
    # descriptor built for another shape
    assert L.cm_attn_fwd(ctypes.byref(d), p, p, p, p, p, 2, 2, 256, 64, 0.1, None) == B.CM_ERR_INVALID_ARG
    # null tensor
    assert L.cm_attn_fwd(ctypes.byref(d), None, p, p, p, p, 1, 2, 256, 64, 0.1, None) == B.CM_ERR_INVALID_ARG
    # misaligned tensor
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert L.cm_attn_fwd(ctypes.byref(d), odd, p, p, p, p, 1, 2, 256, 64, 0.1, None) == B.CM_ERR_INVALID_ARG
    # non-finite scale
    assert L.cm_attn_fwd(ctypes.byref(d), p, p, p, p, p, 1, 2, 256, 64, float("nan"), None) == B.CM_ERR_INVALID_ARG
    # head count: at least 1, at most 2^24 (the kernels' grid mapping)
    assert L.cm_attn_fwd(ctypes.byref(d), p, p, p, p, p, 1, 0, 256, 64, 0.1, None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_fwd(ctypes.byref(d), p, p, p, p, p, 1, (1 << 24) + 1, 256, 64, 0.1,
                         None) == B.CM_ERR_UNSUPPORTED
    assert L.cm_attn_bwd(ctypes.byref(d), p, p, p, p, p, p, p, p, p, p, 1 << 40, 1, (1 << 24) + 1,
                         256, 64, 0.1, None) == B.CM_ERR_UNSUPPORTED
    # backward: workspace too small
    need = B.cm_attn_bwd_workspace_size(1, 2, 256, 64)
    assert need == 2 * (1 * 2 * 256 * 4)  # D and LSE * log2(e), fp32 per row
    assert L.cm_attn_bwd(ctypes.byref(d), p, p, p, p, p, p, p, p, p, p, need - 1, 1, 2, 256, 64,
                         0.1, None) == B.CM_ERR_INVALID_ARG
    # metadata pointer missing
    from masked_flashattention_gb300 import specs
    f, b = B.cm_compile_spec(specs.FWD[1]), B.cm_compile_spec(specs.BWD[1])
    meta = B.cm_meta(None, None, 3)
    assert L.cm_build_descriptor(f.handle, b.handle, ctypes.byref(meta), 1, 256, ctypes.byref(d),
                                 None) == B.CM_ERR_INVALID_ARG


def test_backward_stage_validation_happens_on_the_host(B):
    """The three stages of the backward check their arguments like cm_attn_bwd does."""
    L = B.lib()
    p = ctypes.c_void_p(1 << 20)
    d = _fake_desc(B, 1, 256)
    need = B.cm_attn_bwd_workspace_size(1, 2, 256, 64)
    # prologue: unsupported head dim, null tensor, short workspace, S not a multiple of the tile
    assert L.cm_attn_bwd_prologue(p, p, p, p, need, 1, 2, 256, 96, None) == B.CM_ERR_UNSUPPORTED
    assert L.cm_attn_bwd_prologue(None, p, p, p, need, 1, 2, 256, 64, None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_bwd_prologue(p, p, p, p, need - 1, 1, 2, 256, 64, None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_bwd_prologue(p, p, p, p, need, 1, 2, 200, 64, None) == B.CM_ERR_INVALID_ARG
    # dK/dV and dQ stages: descriptor for another shape, misaligned output, short workspace
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert L.cm_attn_bwd_dkdv(ctypes.byref(d), p, p, p, p, p, p, p, need, 2, 2, 256, 64, 0.1,
                              None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_bwd_dkdv(ctypes.byref(d), p, p, p, p, odd, p, p, need, 1, 2, 256, 64, 0.1,
                              None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_bwd_dq(ctypes.byref(d), p, p, p, p, p, p, p, p, need - 1, 1, 2, 256, 64, 0.1,
                            None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_bwd_dq(ctypes.byref(d), p, p, p, p, p, p, p, p, need, 1, 2, 256, 64,
                            float("inf"), None) == B.CM_ERR_INVALID_ARG
    assert L.cm_attn_bwd_dq(ctypes.byref(d), p, p, p, None, p, p, p, p, need, 1, 2, 256, 64, 0.1,
                            None) == B.CM_ERR_INVALID_ARG  # o is read for D
    # cm_attn_bwd checks everything before its first stage: a bad dq pointer is caught even
    # though the prologue's own arguments are fine
    assert L.cm_attn_bwd(ctypes.byref(d), p, p, p, p, p, p, None, p, p, p, need, 1, 2, 256, 64,
                         0.1, None) == B.CM_ERR_INVALID_ARG


def test_wait_limit_validation(B):
    L = B.lib()
    assert L.cm_set_wait_limit_ns(61 * 10**9) == B.CM_ERR_INVALID_ARG
    B.cm_set_wait_limit_ns(1)
    B.cm_set_wait_limit_ns(0)  # back to the default


def test_error_strings(B):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert B.cm_error_string(code)
    assert "transpose" in B.cm_error_string(B.CM_ERR_DESC_MISMATCH)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_generated_preprocess_kernels_compile(B, wid):
    """Each workload spec's mask-specific preprocess kernel (section 3.1) compiles with NVRTC for
    sm_103a (host only; loading needs a GPU and is checked by the GPU tests)."""
    from masked_flashattention_gb300 import specs
    for text in (specs.FWD[wid], specs.BWD[wid]):
        spec = B.cm_compile_spec(text)
        src = B.cm_spec_kernel_source(spec)
        assert 'extern "C" __global__' in src and "cm_generated_descriptor" in src
        ni = B.cm_spec_num_intervals(spec)
        assert f"descriptor_kernel<{ni}, {ni}>" in src
        rc, log = B.cm_spec_kernel_status(spec, load=False)
        if rc == B.CM_ERR_UNSUPPORTED:
            pytest.skip("NVRTC is not available here: " + log)
        assert rc == B.CM_OK, log


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5, 6])
def test_generated_pair_kernels_compile(B, wid):
    """The kernel cm_build_descriptor runs for a workload is generated from its forward and
    backward specs together (one launch builds both halves); it compiles with NVRTC."""
    from masked_flashattention_gb300 import specs
    f, b = B.cm_compile_spec(specs.FWD[wid]), B.cm_compile_spec(specs.BWD[wid])
    src = B.cm_descriptor_kernel_source(f, b)
    nf, nb = B.cm_spec_num_intervals(f), B.cm_spec_num_intervals(b)
    assert f"descriptor_kernel<{nf}, {nb}>" in src
    assert "struct EvalFwd" in src and "struct EvalBwd" in src
    rc, log = B.cm_descriptor_kernel_status(f, b, load=False)
    if rc == B.CM_ERR_UNSUPPORTED:
        pytest.skip("NVRTC is not available here: " + log)
    assert rc == B.CM_OK, log


def test_generated_source_follows_the_lowered_slots(B):
    """The generated evaluator holds the Region C slots of the lowered form: [0, b) and
    [s(i), i + 1) for response rows (seg_idx(i) >= 1), one causal slot for prompt rows."""
    from masked_flashattention_gb300 import specs
    src = B.cm_spec_kernel_source(B.cm_compile_spec(specs.FWD[3]))
    assert "if ((ki == (0))) {" in src
    assert "lo[0] = (0);\n      hi[0] = cmcore::wadd(i, (1));" in src
    assert "hi[0] = cmcore::seg_end_at(seg, nseg, (0));" in src
    assert "lo[1] = cmcore::seg_start_at(seg, nseg, ki);" in src


def test_preprocess_mode_validation(B):
    L = B.lib()
    assert L.cm_set_preprocess_mode(7) == B.CM_ERR_INVALID_ARG
    assert L.cm_set_preprocess_mode(-1) == B.CM_ERR_INVALID_ARG
    B.cm_set_preprocess_mode(B.CM_PREPROCESS_GENERIC)
    B.cm_set_preprocess_mode(B.CM_PREPROCESS_GENERATED)
    assert L.cm_spec_kernel_status(None, 0, None, 0) == B.CM_ERR_INVALID_ARG


def test_interval_check_mode_validation(B):
    L = B.lib()
    assert L.cm_set_interval_check(4) == B.CM_ERR_INVALID_ARG
    assert L.cm_set_interval_check(-1) == B.CM_ERR_INVALID_ARG
    assert L.cm_set_interval_check(2) == B.CM_ERR_INVALID_ARG
    for mode in (B.CM_CHECK_TWO_COMPARE, B.CM_CHECK_UNSIGNED, B.CM_CHECK_RANGE_MASK):
        B.cm_set_interval_check(mode)


def test_interval_count_limit_is_eight(B):
    """Rules may need up to 8 intervals per row; a ninth is refused with a parse error naming
    the limit (the kernels keep the row's intervals in registers)."""
    terms = ["j < 4"] + [f"(j >= {10 * m} && j < {10 * m + 3})" for m in range(1, 8)]
    assert B.cm_spec_num_intervals(B.cm_compile_spec("region all : " + " || ".join(terms))) == 8
    terms.append("(j >= 100 && j <= i)")
    with pytest.raises(B.CMError) as e:
        B.cm_compile_spec("region all : " + " || ".join(terms))
    assert e.value.code == B.CM_ERR_PARSE and "limit 8" in str(e.value)
