"""The backward entry point that allocates nothing (cm_attn_bwd_noalloc).

It serves callers that cannot allocate device memory (a host framework that owns all device
memory, or a thread that must not call cudaMalloc): the library's fixed scratch array replaces
the caller's workspace.  Here it is called through the C ABI twice in a row, on different inputs,
and each result is compared with the workspace entry point (cm_attn_bwd) on the same inputs and
with the fp64 oracle, with the tolerance of the other attention tests.  The second call is a
smaller problem, so it also shows that what the first call left in the shared array does not leak
into the next result.  This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

REL_L2, MAX_ABS = 1e-2, 3e-2


def _close(name, got, want):
    got, want = got.double().cpu(), want.double().cpu()
    rel = ((got - want).norm() / want.norm()).item()
    mx = (got - want).abs().max().item()
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{name}: rel_l2={rel:.3e} max_abs={mx:.3e}"


def test_noalloc_backward_matches_workspace_backward_twice():
    from masked_flashattention_gb300 import binding as B
    from masked_flashattention_gb300 import specs
    from masked_flashattention_gb300 import workloads as W
    from oracle import attention as A
    from oracle import masks as M

    B.lib()
    wid, d = 3, 128
    f, b = B.cm_compile_spec(specs.FWD[wid]), B.cm_compile_spec(specs.BWD[wid])
    # two calls in a row on different inputs; the second problem is smaller than the first, so
    # it reads only part of what the first call left in the shared array
    for call, (S, Bn, H, seed) in enumerate(((2048, 2, 4, 7), (1024, 1, 2, 8))):
        w = W.scaled(W.WORKLOADS[wid], S, B=Bn, H=H, d=d)
        seg, nseg = W.segments(wid, w.B, S, seed=41 + call)
        desc = B.Descriptor(f, b, w.B, S)
        B.cm_build_descriptor(f, b, torch.from_numpy(seg).cuda(), torch.from_numpy(nseg).cuda(),
                              desc)
        Q, K, V, dO = W.full_tensors(w, seed=seed)
        q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
        o, lse = B.attention_forward(desc, q, k, v)
        ref = B.attention_backward(desc, q, k, v, o, lse, do)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        B.cm_attn_bwd_noalloc(desc, q, k, v, o, lse, do, dq, dk, dv)
        torch.cuda.synchronize()
        assert B.cm_get_status(desc) == B.CM_OK
        for name, got, want in (("dQ", dq, ref[0]), ("dK", dk, ref[1]), ("dV", dv, ref[2])):
            _close(f"call {call} {name}", got, want)
        # and against the fp64 oracle, head by head
        for bb in range(w.B):
            mask = M.dense_mask(wid, seg[bb], int(nseg[bb]), S)
            for h in range(w.H):
                rq, rk, rv = A.attention_backward(Q[bb, h], K[bb, h], V[bb, h], dO[bb, h], mask)
                for name, got, want in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
                    _close(f"call {call} {name} b{bb}h{h} vs oracle", got[bb, h], want)


def test_noalloc_rejects_problems_beyond_the_scratch_array():
    from masked_flashattention_gb300 import binding as B
    from masked_flashattention_gb300 import specs

    B.lib()
    S, H, d = 32768, 160, 64  # 5.2M rows: needs > 32 MiB of scratch
    need = B.cm_attn_bwd_workspace_size(1, H, S, d)
    assert need > B.NOALLOC_SCRATCH_BYTES
    f, b = B.cm_compile_spec(specs.FWD[2]), B.cm_compile_spec(specs.BWD[2])
    desc = B.Descriptor(f, b, 1, S)
    t = torch.empty(1, H, S, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, H, S, dtype=torch.float32, device="cuda")
    with pytest.raises(B.CMError) as e:
        B.cm_attn_bwd_noalloc(desc, t, t, t, t, lse, t, t, t, t)
    assert e.value.code == B.CM_ERR_UNSUPPORTED
