"""Python binding of the C ABI in include/ta.h (ctypes; argument marshalling only).

Every step of the computation runs in the CUDA kernels of libta.so; this
module only allocates outputs and workspaces with torch, passes raw device
pointers and the current CUDA stream, and turns a non-OK status into an
exception.  There is no fallback: if libta.so is missing the import of
``lib()`` fails loudly.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libta.so")

TA_OK, TA_ERR_INVALID_ARG, TA_ERR_UNSUPPORTED, TA_ERR_WORKSPACE, TA_ERR_CUDA = range(5)
TA_F32, TA_BF16 = 0, 1
TA_DEVERR_SEQLEN, TA_DEVERR_TIMEOUT, TA_DEVERR_RANGE, TA_DEVERR_PAGE = 1, 2, 4, 8
STATUS_NAMES = {0: "TA_OK", 1: "TA_ERR_INVALID_ARG", 2: "TA_ERR_UNSUPPORTED", 3: "TA_ERR_WORKSPACE",
                4: "TA_ERR_CUDA"}


class TAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class DecodePlan(ctypes.Structure):
    _fields_ = [("n_split", ctypes.c_int32), ("chunk", ctypes.c_int32), ("levels", ctypes.c_int32),
                ("fanin", ctypes.c_int32), ("grid", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


class DecodeParams(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("S", ctypes.c_int32), ("D", ctypes.c_int32), ("scale", ctypes.c_float),
                ("seqlens", ctypes.c_void_p), ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("chunk", ctypes.c_int32), ("n_split", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("stream", ctypes.c_void_p), ("wait_limit_ns", ctypes.c_uint64)]


class PagedDecodeParams(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seqlens", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("scale", ctypes.c_float), ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("chunk", ctypes.c_int32), ("n_split", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("stream", ctypes.c_void_p), ("wait_limit_ns", ctypes.c_uint64)]


class PrefillParams(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("S", ctypes.c_int32), ("D", ctypes.c_int32), ("scale", ctypes.c_float),
                ("cu_seqlens", ctypes.c_void_p), ("total_tokens", ctypes.c_int32), ("out_dtype", ctypes.c_int),
                ("wait_limit_ns", ctypes.c_uint64), ("stream", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libta.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with long_context_decode_04_b300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, st, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        L.ta_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
        L.ta_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
        L.ta_decode_ex.argtypes = [ctypes.POINTER(DecodeParams)]
        L.ta_decode_paged.argtypes = [ctypes.POINTER(PagedDecodeParams)]
        L.ta_decode_pi.argtypes = [ctypes.POINTER(DecodeParams), i, i]
        L.ta_decode_fp8.argtypes = [ctypes.POINTER(DecodeParams), vp, vp]
        L.ta_decode_nvfp4.argtypes = [ctypes.POINTER(DecodeParams), vp, vp, vp, vp]
        L.ta_decode_pi_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i, i, i]
        L.ta_decode_pi_workspace_bytes.restype = st
        L.ta_decode_partials.argtypes = [ctypes.POINTER(DecodeParams), vp, vp, vp]
        L.ta_decode_plan_for.argtypes = [i, i, i, i, i, i, i, i, i, ctypes.POINTER(DecodePlan)]
        L.ta_decode_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        L.ta_decode_workspace_bytes.restype = st
        L.ta_decode_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
        L.ta_combine.argtypes = [vp, vp, vp, i, i, i, vp, i, vp, vp, st, vp]
        L.ta_combine_workspace_bytes.argtypes = [i, i, i]
        L.ta_combine_workspace_bytes.restype = st
        L.ta_prefill_causal.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        L.ta_prefill_causal_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
        L.ta_prefill_causal_ex.argtypes = [ctypes.POINTER(PrefillParams)]
        L.ta_decode_noalloc_setup.argtypes = []
        L.ta_decode_noalloc_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.ta_test_fail_next_launches.argtypes = [i]
        L.ta_test_fail_next_launches.restype = ctypes.c_int
        L.ta_test_stall_next_launches.argtypes = [i]
        L.ta_test_stall_next_launches.restype = ctypes.c_int
        L.ta_last_error.argtypes = []
        L.ta_last_error.restype = ctypes.c_char_p
        for fn in ("ta_decode", "ta_decode_noalloc", "ta_decode_ex", "ta_decode_paged", "ta_decode_pi", "ta_decode_fp8",
                   "ta_prefill_causal_varlen", "ta_decode_partials", "ta_decode_plan_for", "ta_decode_status", "ta_combine",
                   "ta_prefill_causal", "ta_prefill_causal_ex", "ta_decode_noalloc_setup", "ta_decode_noalloc_status",
                   "ta_decode_nvfp4"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != TA_OK:
        raise TAError(status, lib().ta_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return TA_BF16
    if dt == torch.float32:
        return TA_F32
    raise TypeError(f"unsupported dtype {dt}")


def plan_decode(B, Hq, Hkv, S, D, *, chunk=0, n_split=0, varlen=False, sm_count=0) -> DecodePlan:
    """The split-KV plan the library would use (host computation only)."""
    p = DecodePlan()
    _check(lib().ta_decode_plan_for(B, Hq, Hkv, S, D, chunk, n_split, int(bool(varlen)), sm_count,
                                    ctypes.byref(p)))
    return p


def chunk_bounds(plan: DecodePlan, S: int):
    """[(start, end)] of the plan's chunks over S keys (include/ta.h)."""
    return [(min(c * plan.chunk, S), min((c + 1) * plan.chunk, S)) for c in range(plan.n_split)]


def decode_workspace(B, Hq, Hkv, S, D, *, chunk=0, n_split=0, varlen=False, device="cuda") -> torch.Tensor:
    """A zeroed device workspace big enough for ``decode(..., workspace=...)``."""
    plan = plan_decode(B, Hq, Hkv, S, D, chunk=chunk, n_split=n_split, varlen=varlen)
    return torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device=device)


def decode(q, k, v, *, seqlens=None, scale=None, out_dtype=None, chunk=0, n_split=0, workspace=None,
           out=None, lse=None, wait_limit_ns=0):
    """Split-KV decode.  q [B,Hq,D], k/v [B,Hkv,S,D] (bf16 or fp32, CUDA), seqlens [B] int32.

    Returns (out [B,Hq,D], lse [B,Hq] fp32).  ``workspace`` (uint8 CUDA tensor
    from ``decode_workspace``) makes the call allocation-free; without it the
    library uses its own per-device workspace.
    """
    B, Hq, D = q.shape
    _, Hkv, S, _ = k.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    p = DecodeParams()
    p.q, p.k, p.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    p.out, p.lse = out.data_ptr(), lse.data_ptr()
    p.B, p.Hq, p.Hkv, p.S, p.D = B, Hq, Hkv, S, D
    p.scale = scale
    p.seqlens = seqlens.data_ptr() if seqlens is not None else None
    p.in_dtype = _dtype_code(q.dtype)
    p.out_dtype = _dtype_code(out.dtype)
    p.chunk, p.n_split = chunk, n_split
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    p.stream = torch.cuda.current_stream(q.device).cuda_stream
    p.wait_limit_ns = int(wait_limit_ns)
    _check(lib().ta_decode_ex(ctypes.byref(p)))
    return out, lse


def decode_pi(q, k, v, window, period, *, seqlens=None, scale=None, out_dtype=None, chunk=0, n_split=0,
              workspace=None, out=None, lse=None, wait_limit_ns=0):
    """Decode over the pi-Attention key set: the window of the last ``window``
    keys plus every ``period``-th key before it, counted back from the
    newest.  Shapes as ``decode``; returns (out, lse)."""
    B, Hq, D = q.shape
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    p = _params(q, k, v, seqlens, scale, chunk, n_split, workspace, out=out, lse=lse, out_dtype=out.dtype,
                wait_limit_ns=wait_limit_ns)
    _check(lib().ta_decode_pi(ctypes.byref(p), int(window), int(period)))
    return out, lse


def decode_fp8(q, k8, v8, *, k_scale=None, v_scale=None, seqlens=None, scale=None, out_dtype=None, chunk=0,
               n_split=0, workspace=None, out=None, lse=None, wait_limit_ns=0):
    """Decode over an E4M3 KV cache.  q [B,Hq,D] bf16; k8/v8 [B,Hkv,S,D] uint8
    (E4M3 bit patterns); k_scale/v_scale [B*Hkv] fp32 or None.  Returns
    (out, lse).  The queries are used as fp16 values: an element of magnitude
    2^16 or more sets TA_DEVERR_RANGE (read with decode_status)."""
    B, Hq, D = q.shape
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    p = _params(q, k8, v8, seqlens, scale, chunk, n_split, workspace, out=out, lse=lse, out_dtype=out.dtype,
                wait_limit_ns=wait_limit_ns)
    _check(lib().ta_decode_fp8(ctypes.byref(p), _ptr(k_scale), _ptr(v_scale)))
    return out, lse


def decode_nvfp4(q, k4, v4, k_bs, v_bs, *, k_factor=None, v_factor=None, seqlens=None, scale=None, out_dtype=None,
                 chunk=0, n_split=0, workspace=None, out=None, lse=None, wait_limit_ns=0):
    """Decode over an NVFP4 KV cache.  q [B,Hq,D] bf16; k4/v4 [B,Hkv,S,D/2] uint8
    (E2M1 codes, even element in the low nibble); k_bs/v_bs [B,Hkv,S,D/16] uint8
    (E4M3 block scales); k_factor/v_factor [B*Hkv] fp32 or None.  Returns (out,
    lse).  As for decode_fp8, a query element of magnitude 2^16 or more sets
    TA_DEVERR_RANGE."""
    B, Hq, D = q.shape
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    p = _params(q, k4, v4, seqlens, scale, chunk, n_split, workspace, out=out, lse=lse, out_dtype=out.dtype,
                wait_limit_ns=wait_limit_ns)
    p.D = D  # the code tensors' last dimension is D/2
    _check(lib().ta_decode_nvfp4(ctypes.byref(p), _ptr(k_bs), _ptr(v_bs), _ptr(k_factor), _ptr(v_factor)))
    return out, lse


def decode_pi_workspace(B, Hq, Hkv, S, D, window, period, *, chunk=0, n_split=0, varlen=False, device="cuda"):
    n = int(lib().ta_decode_pi_workspace_bytes(B, Hq, Hkv, S, D, chunk, n_split, int(bool(varlen)), window,
                                               period))
    if n == 0:
        raise TAError(TA_ERR_INVALID_ARG, "bad pi-Attention workspace arguments")
    return torch.zeros(max(256, n), dtype=torch.uint8, device=device)


def decode_paged(q, k_pages, v_pages, block_table, seqlens, *, scale=None, out_dtype=None, chunk=0, n_split=0,
                 workspace=None, out=None, lse=None, wait_limit_ns=0):
    """Split-KV decode over a paged KV cache.

    q [B,Hq,D]; k_pages/v_pages [num_pages,Hkv,page_size,D]; block_table
    [B,pages_per_seq] int32; seqlens [B] int32 (all CUDA).  Returns
    (out [B,Hq,D], lse [B,Hq] fp32).
    """
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    pages_per_seq = block_table.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    p = PagedDecodeParams()
    p.q, p.k_pages, p.v_pages = q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr()
    p.block_table, p.seqlens = block_table.data_ptr(), seqlens.data_ptr()
    p.out, p.lse = out.data_ptr(), lse.data_ptr()
    p.B, p.Hq, p.Hkv, p.D = B, Hq, Hkv, D
    p.page_size, p.pages_per_seq, p.num_pages = page_size, pages_per_seq, num_pages
    p.scale = scale
    p.in_dtype = _dtype_code(q.dtype)
    p.out_dtype = _dtype_code(out.dtype)
    p.chunk, p.n_split = chunk, n_split
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    p.stream = torch.cuda.current_stream(q.device).cuda_stream
    p.wait_limit_ns = int(wait_limit_ns)
    _check(lib().ta_decode_paged(ctypes.byref(p)))
    return out, lse


def _params(q, k, v, seqlens, scale, chunk, n_split, workspace, out=None, lse=None, out_dtype=None,
            wait_limit_ns=0):
    B, Hq, D = q.shape
    _, Hkv, S, _ = k.shape
    p = DecodeParams()
    p.q, p.k, p.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    p.out = out.data_ptr() if out is not None else None
    p.lse = lse.data_ptr() if lse is not None else None
    p.B, p.Hq, p.Hkv, p.S, p.D = B, Hq, Hkv, S, D
    p.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    p.seqlens = seqlens.data_ptr() if seqlens is not None else None
    p.in_dtype = _dtype_code(q.dtype)
    p.out_dtype = _dtype_code(out_dtype if out_dtype is not None else q.dtype)
    p.chunk, p.n_split = chunk, n_split
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    p.stream = torch.cuda.current_stream(q.device).cuda_stream
    p.wait_limit_ns = int(wait_limit_ns)
    return p


def decode_partials(q, k, v, *, seqlens=None, scale=None, chunk=0, n_split=0, workspace=None,
                    m=None, l=None, o=None):
    """The split phase alone: (m, l [B*Hq, n_split], o [B*Hq, n_split, D]) fp32 partials."""
    B, Hq, D = q.shape
    _, Hkv, S, _ = k.shape
    plan = plan_decode(B, Hq, Hkv, S, D, chunk=chunk, n_split=n_split, varlen=seqlens is not None)
    N = plan.n_split
    if m is None:
        m = torch.empty((B * Hq, N), dtype=torch.float32, device=q.device)
        l = torch.empty((B * Hq, N), dtype=torch.float32, device=q.device)
        o = torch.empty((B * Hq, N, D), dtype=torch.float32, device=q.device)
    p = _params(q, k, v, seqlens, scale, chunk, n_split, workspace)
    _check(lib().ta_decode_partials(ctypes.byref(p), _ptr(m), _ptr(l), _ptr(o)))
    return m, l, o


def decode_bf16(q, k, v, out, lse, scale, seqlens=None):
    """The plain ``ta_decode`` entry point (bf16 in and out, library workspace)."""
    B, Hq, D = q.shape
    _, Hkv, S, _ = k.shape
    _check(lib().ta_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, float(scale),
                           _ptr(seqlens), _stream(q.device)))
    return out, lse


def decode_noalloc(q, k, v, out, lse, scale, seqlens=None):
    """``ta_decode_noalloc``: bf16 decode whose scratch is the library's fixed device array."""
    B, Hq, D = q.shape
    _, Hkv, S, _ = k.shape
    _check(lib().ta_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D,
                                   float(scale), _ptr(seqlens), _stream(q.device)))
    return out, lse


def decode_noalloc_setup() -> None:
    """``ta_decode_noalloc_setup``: load the device code and find the fixed scratch on the current device."""
    _check(lib().ta_decode_noalloc_setup())


def decode_noalloc_status(device="cuda") -> int:
    """Read and clear the status word of ``ta_decode_noalloc``'s fixed scratch (TA_DEVERR_* bits)."""
    flags = ctypes.c_int32(0)
    _check(lib().ta_decode_noalloc_status(_stream(torch.device(device)), ctypes.byref(flags)))
    return flags.value


def test_fail_next_launches(count: int) -> int:
    """``ta_test_fail_next_launches``: refuse the next ``count`` kernel launches; returns the number pending."""
    return int(lib().ta_test_fail_next_launches(int(count)))


def test_stall_next_launches(count: int) -> int:
    """``ta_test_stall_next_launches``: the next ``count`` decode / prefill launches
    run out their wait time limit; returns the number pending."""
    return int(lib().ta_test_stall_next_launches(int(count)))


def decode_status(workspace=None, device="cuda") -> int:
    """Read and clear the device status word (TA_DEVERR_* bits)."""
    flags = ctypes.c_int32(0)
    _check(lib().ta_decode_status(_ptr(workspace), _stream(torch.device(device)), ctypes.byref(flags)))
    return flags.value


def combine(m, l, o, *, out_dtype=torch.float32, workspace=None, out=None, lse=None):
    """Log-sum-exp merge of partials m, l [R,N], o [R,N,D] (fp32, CUDA) -> (out [R,D], lse [R])."""
    R, N = m.shape
    D = o.shape[2]
    if out is None:
        out = torch.empty((R, D), dtype=out_dtype, device=m.device)
    if lse is None:
        lse = torch.empty((R,), dtype=torch.float32, device=m.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ta_combine(_ptr(m), _ptr(l), _ptr(o), R, N, D, _ptr(out), _dtype_code(out.dtype), _ptr(lse),
                            _ptr(workspace), ws_bytes, _stream(m.device)))
    return out, lse


def combine_workspace_bytes(R, N, D) -> int:
    return int(lib().ta_combine_workspace_bytes(R, N, D))


def _prefill_ex(q, k, v, out, lse, B, H, Hkv, S, D, scale, cu_seqlens, total_tokens, wait_limit_ns):
    p = PrefillParams()
    p.q, p.k, p.v, p.out, p.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr()
    p.B, p.H, p.Hkv, p.S, p.D = B, H, Hkv, S, D
    p.scale = scale
    p.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    p.total_tokens = total_tokens
    p.out_dtype = _dtype_code(out.dtype)
    p.wait_limit_ns = int(wait_limit_ns)
    p.stream = torch.cuda.current_stream(q.device).cuda_stream
    _check(lib().ta_prefill_causal_ex(ctypes.byref(p)))


def prefill_causal(q, k, v, *, scale=None, out=None, lse=None, out_dtype=None, wait_limit_ns=0):
    """Causal prefill. q [B,H,S,D], k/v [B,Hkv,S,D] bf16 CUDA -> (out [B,H,S,D], lse [B,H,S] fp32).

    ``out_dtype`` torch.bfloat16 (default) or torch.float32; the plain
    ``ta_prefill_causal`` entry point serves the defaults, ``ta_prefill_causal_ex``
    the rest."""
    B, H, S, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if out.dtype == torch.bfloat16 and not wait_limit_ns:
        _check(lib().ta_prefill_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, S, D, scale,
                                       _stream(q.device)))
    else:
        _prefill_ex(q, k, v, out, lse, B, H, Hkv, S, D, scale, None, 0, wait_limit_ns)
    return out, lse


def prefill_causal_varlen(q, k, v, cu_seqlens, max_seqlen, *, scale=None, out=None, lse=None, out_dtype=None,
                          wait_limit_ns=0):
    """Causal prefill of packed variable-length sequences.  q [T,H,D], k/v
    [T,Hkv,D] bf16, cu_seqlens [num_seqs+1] int32 (CUDA) -> (out [T,H,D], lse
    [H,T] fp32); ``out_dtype`` as ``prefill_causal``."""
    T, H, D = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    if out.dtype == torch.bfloat16 and not wait_limit_ns:
        _check(lib().ta_prefill_causal_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
                                              cu_seqlens.numel() - 1, int(max_seqlen), T, H, Hkv, D, scale,
                                              _stream(q.device)))
    else:
        _prefill_ex(q, k, v, out, lse, cu_seqlens.numel() - 1, H, Hkv, int(max_seqlen), D, scale, cu_seqlens, T,
                    wait_limit_ns)
    return out, lse
