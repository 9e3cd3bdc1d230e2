"""Thin ctypes binding of libcm.so, with the same names as the C ABI (include/cm.h).

Argument marshalling only: every step of the hot path runs in the library's CUDA kernels.
PyTorch supplies device memory (tensor data pointers) and streams; nothing here computes a
descriptor or an attention value, and there is no fallback when the library is missing.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcm.so")

CM_OK = 0
CM_ERR_PARSE = -1
CM_ERR_INVALID_ARG = -2
CM_ERR_UNSUPPORTED = -3
CM_ERR_CUDA = -4
CM_ERR_TIMEOUT = -5
CM_ERR_DEVICE_CHECK = -6
CM_ERR_DESC_MISMATCH = -7

TILE = 128


class CMError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        self.code = code
        msg = f"{what}: {cm_error_string(code)} ({code})"
        super().__init__(msg + (f": {detail}" if detail else ""))


class cm_meta(ctypes.Structure):
    _fields_ = [("seg", ctypes.c_void_p), ("nseg", ctypes.c_void_p), ("nseg_max", ctypes.c_int32)]


class cm_descriptor(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("ni_f", ctypes.c_int32), ("ni_b", ctypes.c_int32), ("form", ctypes.c_int32),
                ("itab_f", ctypes.c_void_p), ("bm_f", ctypes.c_void_p),
                ("itab_b", ctypes.c_void_p), ("bm_b", ctypes.c_void_p),
                ("sched_f", ctypes.c_void_p), ("sched_b", ctypes.c_void_p),
                ("status", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no other code path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "masked_flashattention_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.cm_compile_spec.argtypes = [ctypes.c_char_p, ctypes.POINTER(vp), ctypes.c_char_p, sz]
        L.cm_spec_free.argtypes = [vp]
        L.cm_spec_free.restype = None
        L.cm_spec_num_intervals.argtypes = [vp, ctypes.POINTER(i32)]
        L.cm_spec_describe.argtypes = [vp, ctypes.c_char_p, sz, ctypes.POINTER(sz)]
        L.cm_spec_kernel_source.argtypes = [vp, ctypes.c_char_p, sz, ctypes.POINTER(sz)]
        L.cm_spec_kernel_status.argtypes = [vp, i32, ctypes.c_char_p, sz]
        L.cm_descriptor_kernel_source.argtypes = [vp, vp, ctypes.c_char_p, sz, ctypes.POINTER(sz)]
        L.cm_descriptor_kernel_status.argtypes = [vp, vp, i32, ctypes.c_char_p, sz]
        L.cm_set_preprocess_mode.argtypes = [i32]
        L.cm_set_interval_check.argtypes = [i32]
        L.cm_descriptor_sizes.argtypes = [vp, vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
        L.cm_build_descriptor.argtypes = [vp, vp, ctypes.POINTER(cm_meta), i32, i32,
                                          ctypes.POINTER(cm_descriptor), vp]
        L.cm_attn_fwd.argtypes = [ctypes.POINTER(cm_descriptor), vp, vp, vp, vp, vp,
                                  i32, i32, i32, i32, ctypes.c_float, vp]
        L.cm_attn_bwd_workspace_size.argtypes = [i32, i32, i32, i32, ctypes.POINTER(sz)]
        L.cm_attn_bwd.argtypes = [ctypes.POINTER(cm_descriptor), vp, vp, vp, vp, vp, vp, vp, vp,
                                  vp, vp, sz, i32, i32, i32, i32, ctypes.c_float, vp]
        L.cm_attn_bwd_prologue.argtypes = [vp, vp, vp, vp, sz, i32, i32, i32, i32, vp]
        L.cm_attn_bwd_dkdv.argtypes = [ctypes.POINTER(cm_descriptor), vp, vp, vp, vp, vp, vp, vp,
                                       sz, i32, i32, i32, i32, ctypes.c_float, vp]
        L.cm_attn_bwd_dq.argtypes = [ctypes.POINTER(cm_descriptor), vp, vp, vp, vp, vp, vp, vp,
                                     vp, sz, i32, i32, i32, i32, ctypes.c_float, vp]
        L.cm_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        L.cm_attn_bwd_noalloc.argtypes = [ctypes.POINTER(cm_descriptor), vp, vp, vp, vp, vp, vp,
                                          vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp]
        L.cm_get_status.argtypes = [ctypes.POINTER(cm_descriptor), vp]
        L.cm_error_string.argtypes = [i32]
        L.cm_error_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def cm_error_string(code: int) -> str:
    try:
        return lib().cm_error_string(code).decode()
    except RuntimeError:
        return f"error {code}"


def _check(rc: int, what: str, detail: str = "") -> None:
    if rc != CM_OK:
        raise CMError(rc, what, detail)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------------------------------------------
# compiler
# ------------------------------------------------------------------------------------------------
class Spec:
    """Owns a compiled MaskSpec (host memory inside the library)."""

    def __init__(self, handle: int, text: str):
        self.handle = ctypes.c_void_p(handle)
        self.text = text

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None and self.handle.value:
            _lib.cm_spec_free(self.handle)
            self.handle = ctypes.c_void_p(0)


def cm_compile_spec(text: str) -> Spec:
    out = ctypes.c_void_p()
    err = ctypes.create_string_buffer(512)
    rc = lib().cm_compile_spec(text.encode(), ctypes.byref(out), err, 512)
    _check(rc, "cm_compile_spec", err.value.decode())
    return Spec(out.value, text)


def cm_spec_num_intervals(spec: Spec) -> int:
    n = ctypes.c_int()
    _check(lib().cm_spec_num_intervals(spec.handle, ctypes.byref(n)), "cm_spec_num_intervals")
    return n.value


def cm_spec_describe(spec: Spec) -> str:
    need = ctypes.c_size_t()
    _check(lib().cm_spec_describe(spec.handle, None, 0, ctypes.byref(need)), "cm_spec_describe")
    buf = ctypes.create_string_buffer(need.value)
    _check(lib().cm_spec_describe(spec.handle, buf, need.value, None), "cm_spec_describe")
    return buf.value.decode()


def cm_spec_kernel_source(spec: Spec) -> str:
    """CUDA C++ source of the spec's mask-specific preprocess kernel."""
    need = ctypes.c_size_t()
    _check(lib().cm_spec_kernel_source(spec.handle, None, 0, ctypes.byref(need)),
           "cm_spec_kernel_source")
    buf = ctypes.create_string_buffer(need.value)
    _check(lib().cm_spec_kernel_source(spec.handle, buf, need.value, None), "cm_spec_kernel_source")
    return buf.value.decode()


def cm_descriptor_kernel_source(fwd: Spec, bwd: Spec) -> str:
    """CUDA C++ source of the mask-specific preprocess kernel of a (forward, backward) pair."""
    need = ctypes.c_size_t()
    _check(lib().cm_descriptor_kernel_source(fwd.handle, bwd.handle, None, 0, ctypes.byref(need)),
           "cm_descriptor_kernel_source")
    buf = ctypes.create_string_buffer(need.value)
    _check(lib().cm_descriptor_kernel_source(fwd.handle, bwd.handle, buf, need.value, None),
           "cm_descriptor_kernel_source")
    return buf.value.decode()


def cm_descriptor_kernel_status(fwd: Spec, bwd: Spec, load: bool = True) -> tuple[int, str]:
    """(code, log) of the pair's generated kernel: compiled (load=False, host only) or compiled
    and loaded on the current GPU (load=True), as cm_build_descriptor does on first use."""
    buf = ctypes.create_string_buffer(1 << 16)
    rc = lib().cm_descriptor_kernel_status(fwd.handle, bwd.handle, 1 if load else 0, buf, len(buf))
    return rc, buf.value.decode(errors="replace")


def cm_spec_kernel_status(spec: Spec, load: bool = True) -> tuple[int, str]:
    """(code, log): CM_OK when the spec's generated preprocess kernel compiles (load=False, host
    only) or compiles and loads on the current GPU (load=True); otherwise the code and the reason."""
    buf = ctypes.create_string_buffer(1 << 16)
    rc = lib().cm_spec_kernel_status(spec.handle, 1 if load else 0, buf, len(buf))
    return rc, buf.value.decode(errors="replace")


CM_PREPROCESS_GENERATED = 0
CM_PREPROCESS_GENERIC = 1


def cm_set_preprocess_mode(mode: int) -> None:
    """Process-wide choice of descriptor kernels: generated per spec (default) or generic."""
    _check(lib().cm_set_preprocess_mode(mode), "cm_set_preprocess_mode")


CM_CHECK_UNSIGNED = 0
CM_CHECK_TWO_COMPARE = 1
CM_CHECK_RANGE_MASK = 3

CM_FORM_VISIBLE = 0
CM_FORM_MASKED = 1


def cm_set_interval_check(mode: int) -> None:
    """Process-wide form of the attention kernels' partial-tile check: per-row range masks
    (default), or per score the unsigned test or two comparisons (the paper's section 4.4
    forms)."""
    _check(lib().cm_set_interval_check(mode), "cm_set_interval_check")


def cm_descriptor_sizes(fwd: Spec, bwd: Spec, B: int, S: int, tile: int = TILE,
                        form: int = CM_FORM_VISIBLE) -> list[int]:
    sizes = (ctypes.c_size_t * 7)()
    _check(lib().cm_descriptor_sizes(fwd.handle, bwd.handle, B, S, tile, form, sizes),
           "cm_descriptor_sizes")
    return list(sizes)


# ------------------------------------------------------------------------------------------------
# descriptor
# ------------------------------------------------------------------------------------------------
class Descriptor:
    """Device buffers of an Execution Descriptor, allocated with torch on ``device``.  ``form``:
    CM_FORM_VISIBLE (visible intervals per row) or CM_FORM_MASKED (the masked runs)."""

    def __init__(self, fwd: Spec, bwd: Spec, B: int, S: int, device="cuda",
                 form: int = CM_FORM_VISIBLE):
        sizes = cm_descriptor_sizes(fwd, bwd, B, S, form=form)
        self.fwd, self.bwd, self.B, self.S, self.form = fwd, bwd, B, S, form
        self.ni_f = cm_spec_num_intervals(fwd) + form
        self.ni_b = cm_spec_num_intervals(bwd) + form
        self.NT = S // TILE
        self.W = (self.NT + 15) // 16
        self.itab_f = torch.empty(sizes[0] // 4, dtype=torch.int32, device=device)
        self.bm_f = torch.empty(sizes[1] // 4, dtype=torch.int32, device=device)
        self.itab_b = torch.empty(sizes[2] // 4, dtype=torch.int32, device=device)
        self.bm_b = torch.empty(sizes[3] // 4, dtype=torch.int32, device=device)
        self.sched_f = torch.empty(sizes[4] // 4, dtype=torch.int32, device=device)
        self.sched_b = torch.empty(sizes[5] // 4, dtype=torch.int32, device=device)
        self.status = torch.zeros((sizes[6] + 3) // 4, dtype=torch.int32, device=device)
        self.c = cm_descriptor(B, S, TILE, self.ni_f, self.ni_b, form,
                               self.itab_f.data_ptr(), self.bm_f.data_ptr(),
                               self.itab_b.data_ptr(), self.bm_b.data_ptr(),
                               self.sched_f.data_ptr(), self.sched_b.data_ptr(),
                               self.status.data_ptr())

    def nbytes(self) -> int:
        return sum(t.numel() * 4 for t in (self.itab_f, self.bm_f, self.itab_b, self.bm_b,
                                           self.sched_f, self.sched_b, self.status))

    # host views for checking
    def interval_table_fwd(self):
        return self.itab_f.view(self.B, self.ni_f, self.S, 2).cpu().numpy()

    def interval_table_bwd(self):
        return self.itab_b.view(self.B, self.ni_b, self.S, 2).cpu().numpy()

    def bitmap_fwd(self):
        return self.bm_f.view(self.B, self.NT, self.W).cpu().numpy().view("uint32")

    def bitmap_bwd(self):
        return self.bm_b.view(self.B, self.NT, self.W).cpu().numpy().view("uint32")


def cm_build_descriptor(fwd: Spec, bwd: Spec, seg: torch.Tensor, nseg: torch.Tensor,
                        desc: Descriptor, stream=None) -> None:
    """seg: device int32 [B, nseg_max + 1]; nseg: device int32 [B]."""
    for t in (seg, nseg):
        if not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
            raise ValueError("metadata must be contiguous int32 CUDA tensors")
    meta = cm_meta(seg.data_ptr(), nseg.data_ptr(), seg.shape[1] - 1)
    _check(lib().cm_build_descriptor(fwd.handle, bwd.handle, ctypes.byref(meta), desc.B, desc.S,
                                     ctypes.byref(desc.c), _stream(stream)),
           "cm_build_descriptor")


def cm_get_status(desc: Descriptor, stream=None) -> int:
    return lib().cm_get_status(ctypes.byref(desc.c), _stream(stream))


# ------------------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------------------
def _bhsd(t: torch.Tensor, name: str):
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 4 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, H, S, d]")
    return t.shape


def cm_attn_fwd(desc: Descriptor, q, k, v, o, lse, scale: float | None = None,
                stream=None) -> None:
    B, H, S, d = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o")):
        if _bhsd(t, n) != (B, H, S, d):
            raise ValueError(f"{n} shape mismatch")
    if not (lse.is_cuda and lse.dtype == torch.float32 and lse.shape == (B, H, S)):
        raise ValueError("lse must be fp32 CUDA [B, H, S]")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(lib().cm_attn_fwd(ctypes.byref(desc.c), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                             o.data_ptr(), lse.data_ptr(), B, H, S, d, scale, _stream(stream)),
           "cm_attn_fwd")


def cm_attn_bwd_workspace_size(B: int, H: int, S: int, d: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().cm_attn_bwd_workspace_size(B, H, S, d, ctypes.byref(n)),
           "cm_attn_bwd_workspace_size")
    return n.value


def cm_attn_bwd(desc: Descriptor, q, k, v, o, lse, d_o, dq, dk, dv, workspace: torch.Tensor,
                scale: float | None = None, stream=None) -> None:
    B, H, S, d = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (d_o, "dO"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        if _bhsd(t, n) != (B, H, S, d):
            raise ValueError(f"{n} shape mismatch")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().cm_attn_bwd(ctypes.byref(desc.c), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                             o.data_ptr(), lse.data_ptr(), d_o.data_ptr(), dq.data_ptr(),
                             dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), nbytes,
                             B, H, S, d, scale, _stream(stream)),
           "cm_attn_bwd")


def _bwd_shapes(q, others):
    B, H, S, d = _bhsd(q, "q")
    for t, n in others:
        if _bhsd(t, n) != (B, H, S, d):
            raise ValueError(f"{n} shape mismatch")
    return B, H, S, d


def cm_attn_bwd_prologue(o, lse, d_o, workspace: torch.Tensor, stream=None) -> None:
    """Per-row -D and -LSE * log2(e) of every row into the workspace, for callers that run
    cm_attn_bwd_dkdv without cm_attn_bwd_dq (cm_attn_bwd itself does not use it)."""
    B, H, S, d = _bwd_shapes(o, ((d_o, "dO"),))
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().cm_attn_bwd_prologue(o.data_ptr(), lse.data_ptr(), d_o.data_ptr(),
                                      workspace.data_ptr(), nbytes, B, H, S, d, _stream(stream)),
           "cm_attn_bwd_prologue")


def cm_attn_bwd_dkdv(desc: Descriptor, q, k, v, d_o, dk, dv, workspace: torch.Tensor,
                     scale: float | None = None, stream=None) -> None:
    """Second stage of cm_attn_bwd: dK and dV along key tiles (backward descriptor); reads the
    per-row constants that cm_attn_bwd_dq (or cm_attn_bwd_prologue) wrote into the workspace."""
    B, H, S, d = _bwd_shapes(q, ((k, "k"), (v, "v"), (d_o, "dO"), (dk, "dk"), (dv, "dv")))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().cm_attn_bwd_dkdv(ctypes.byref(desc.c), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                  d_o.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                  workspace.data_ptr(), nbytes, B, H, S, d, scale, _stream(stream)),
           "cm_attn_bwd_dkdv")


def cm_attn_bwd_dq(desc: Descriptor, q, k, v, o, lse, d_o, dq, workspace: torch.Tensor,
                   scale: float | None = None, stream=None) -> None:
    """First stage of cm_attn_bwd: dQ along query tiles (forward descriptor); also writes the
    workspace's per-row constants (-D and -LSE*log2e) that cm_attn_bwd_dkdv reads."""
    B, H, S, d = _bwd_shapes(q, ((k, "k"), (v, "v"), (o, "O"), (d_o, "dO"), (dq, "dq")))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().cm_attn_bwd_dq(ctypes.byref(desc.c), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                o.data_ptr(), lse.data_ptr(), d_o.data_ptr(), dq.data_ptr(),
                                workspace.data_ptr(), nbytes, B, H, S, d, scale, _stream(stream)),
           "cm_attn_bwd_dq")


def cm_set_wait_limit_ns(ns: int) -> None:
    """Process-wide limit of the attention kernels' bounded waits (0 = the 2 s default).  A
    diagnostic hook: a tiny limit makes ordinary waits expire and exercises the time-out path."""
    _check(lib().cm_set_wait_limit_ns(int(ns)), "cm_set_wait_limit_ns")


def cm_attn_bwd_noalloc(desc: Descriptor, q, k, v, o, lse, d_o, dq, dk, dv,
                        scale: float | None = None, stream=None) -> None:
    """cm_attn_bwd without a workspace, for callers that cannot allocate device memory.

    The library's fixed scratch array (CM_NOALLOC_SCRATCH_BYTES per GPU) stands in for the
    workspace; see include/cm.h for its limit and for the rule that overlapping calls race."""
    B, H, S, d = _bhsd(q, "q")
    for t, n in ((k, "k"), (v, "v"), (o, "o"), (d_o, "dO"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        if _bhsd(t, n) != (B, H, S, d):
            raise ValueError(f"{n} shape mismatch")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(lib().cm_attn_bwd_noalloc(ctypes.byref(desc.c), q.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), o.data_ptr(), lse.data_ptr(), d_o.data_ptr(),
                                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, d,
                                     scale, _stream(stream)),
           "cm_attn_bwd_noalloc")


NOALLOC_SCRATCH_BYTES = 32 << 20


# ------------------------------------------------------------------------------------------------
# convenience: one call for each pass, allocating outputs with torch
# ------------------------------------------------------------------------------------------------
def attention_forward(desc: Descriptor, q, k, v, scale=None, stream=None):
    B, H, S, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device)
    cm_attn_fwd(desc, q, k, v, o, lse, scale, stream)
    return o, lse


def attention_backward(desc: Descriptor, q, k, v, o, lse, d_o, scale=None, stream=None,
                       workspace=None):
    B, H, S, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(cm_attn_bwd_workspace_size(B, H, S, d), dtype=torch.uint8,
                                device=q.device)
    cm_attn_bwd(desc, q, k, v, o, lse, d_o, dq, dk, dv, workspace, scale, stream)
    return dq, dk, dv
