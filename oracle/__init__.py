"""Python access to the float64 CPU oracle (oracle/oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package.  It shares no code with
the CUDA library; both take their inputs from the seeded generator module.

Every function takes the exact tensors the GPU sees (torch CPU tensors or
numpy arrays, bf16 or fp32) and returns float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16, F64 = 0, 1, 2

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32p, i64p, dp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        cl, ci, cd = ctypes.c_long, ctypes.c_int, ctypes.c_double
        L.oracle_decode.argtypes = [vp, ci, vp, vp, ci, cl, cl, cl, cl, cl, cd, i32p, i64p, cl, dp, dp, ci]
        L.oracle_prefill_causal.argtypes = [vp, vp, vp, ci, cl, cl, cl, cl, cl, cd, i64p, cl, dp, dp, ci]
        L.oracle_decode_partials.argtypes = [vp, ci, vp, vp, ci, cl, cl, cl, cl, cl, cd, i32p, cl, cl,
                                             i64p, cl, dp, dp, dp]
        L.oracle_combine.argtypes = [dp, dp, dp, cl, cl, cl, dp, dp]
        for f in (L.oracle_decode, L.oracle_prefill_causal, L.oracle_decode_partials, L.oracle_combine):
            f.restype = ci
        _lib = L
    return _lib


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def _raw(t):
    """(contiguous numpy array holding the exact element bits, dtype code)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().contiguous().cpu()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), BF16
            if t.dtype == torch.float32:
                return t.numpy(), F32
            raise TypeError(f"oracle takes bf16 or fp32 tensors, got {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.uint16:  # raw bf16 bits
        return a, BF16
    raise TypeError(f"oracle takes float32 or raw-bf16 uint16 arrays, got {a.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def decode(q, k, v, scale, seqlens=None, rows=None, threads=None):
    """Decode attention. q [B,Hq,D], k/v [B,Hkv,S,D].  Returns (out [n,D], lse [n])
    for the rows b*Hq+h listed in ``rows`` (all rows in order when None)."""
    qa, qt = _raw(q)
    ka, kt = _raw(k)
    va, vt = _raw(v)
    assert kt == vt
    B, Hq, D = qa.shape
    _, Hkv, S, Dk = ka.shape
    assert Dk == D and va.shape == ka.shape and ka.shape[0] == B
    sl = None if seqlens is None else np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    rw = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = B * Hq if rw is None else len(rw)
    out = np.zeros((n, D))
    lse = np.zeros(n)
    rc = lib().oracle_decode(_ptr(qa), qt, _ptr(ka), _ptr(va), kt, B, Hq, Hkv, S, D, float(scale),
                             _ptr(sl), _ptr(rw), n, _ptr(out), _ptr(lse), threads or default_threads())
    _check(rc, "decode")
    return out, lse


def prefill_causal(q, k, v, scale, rows=None, threads=None):
    """Causal prefill. q [B,H,S,D], k/v [B,Hkv,S,D].  Returns (out [n,D], lse [n]) for
    the rows (b*H+h)*S+i listed in ``rows`` (all rows in order when None)."""
    qa, qt = _raw(q)
    ka, kt = _raw(k)
    va, vt = _raw(v)
    assert qt == kt == vt
    B, H, S, D = qa.shape
    _, Hkv, Sk, Dk = ka.shape
    assert Sk == S and Dk == D and va.shape == ka.shape
    rw = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = B * H * S if rw is None else len(rw)
    out = np.zeros((n, D))
    lse = np.zeros(n)
    rc = lib().oracle_prefill_causal(_ptr(qa), _ptr(ka), _ptr(va), qt, B, H, Hkv, S, D, float(scale),
                                     _ptr(rw), n, _ptr(out), _ptr(lse), threads or default_threads())
    _check(rc, "prefill_causal")
    return out, lse


def decode_partials(q, k, v, scale, b, h, bounds, seqlens=None):
    """Split-KV partials (m, l, o) of decode row (b, h); chunk c = [bounds[c], bounds[c+1])."""
    qa, qt = _raw(q)
    ka, kt = _raw(k)
    va, vt = _raw(v)
    B, Hq, D = qa.shape
    _, Hkv, S, _ = ka.shape
    bd = np.ascontiguousarray(np.asarray(bounds, dtype=np.int64))
    N = len(bd) - 1
    sl = None if seqlens is None else np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    m = np.zeros(N)
    l = np.zeros(N)
    o = np.zeros((N, D))
    rc = lib().oracle_decode_partials(_ptr(qa), qt, _ptr(ka), _ptr(va), kt, B, Hq, Hkv, S, D,
                                      float(scale), _ptr(sl), b, h, _ptr(bd), N, _ptr(m), _ptr(l), _ptr(o))
    _check(rc, "decode_partials")
    return m, l, o


def combine(m, l, o):
    """Log-sum-exp merge. m, l [R,N]; o [R,N,D] -> (out [R,D], lse [R])."""
    m = np.ascontiguousarray(np.asarray(m, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(l, dtype=np.float64))
    o = np.ascontiguousarray(np.asarray(o, dtype=np.float64))
    R, N = m.shape
    D = o.shape[2]
    out = np.zeros((R, D))
    lse = np.zeros(R)
    rc = lib().oracle_combine(_ptr(m), _ptr(l), _ptr(o), R, N, D, _ptr(out), _ptr(lse))
    _check(rc, "combine")
    return out, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, scale, rows=None, threads=None):
    """Decode over a paged KV cache: sequence b's key j is row j % page_size of
    page block_table[b, j // page_size] of the [num_pages, Hkv, page_size, D]
    pools.  The definition is unchanged (attention over keys [0, L_b) of each
    sequence); the pages are gathered into the contiguous cache first with
    numpy indexing (a library gather) and ``decode`` does the rest."""
    kp, kt = _raw(k_pages)
    vp, vt = _raw(v_pages)
    table = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(seqlens, dtype=np.int64)
    B, P = table.shape
    _, Hkv, page, D = kp.shape
    S = P * page
    kc = np.zeros((B, Hkv, S, D), dtype=kp.dtype)
    vc = np.zeros((B, Hkv, S, D), dtype=vp.dtype)
    for b in range(B):
        npg = (int(lens[b]) + page - 1) // page
        for pg in range(npg):
            kc[b, :, pg * page:(pg + 1) * page] = kp[table[b, pg]]
            vc[b, :, pg * page:(pg + 1) * page] = vp[table[b, pg]]
    return decode(q, kc, vc, scale, seqlens=lens.astype(np.int32), rows=rows, threads=threads)


def pi_key_set(L, window, period):
    """The keys the newest query (position i = L - 1) attends under pi-Attention
    (pi-Attention explainer, technical summary section 2A): the ring-local
    window [i - window, i] and the periodic skips i - m * period (m >= 1)
    before it; past keys only.  Ascending list."""
    if L <= 0:
        return []
    i = L - 1
    keys = set(range(max(0, i - window), i + 1))
    j = i - period
    while j >= 0:
        keys.add(j)
        j -= period
    return sorted(keys)


def decode_pi(q, k, v, scale, window, period, seqlens=None, rows=None, threads=None):
    """Decode attention restricted to each sequence's pi-Attention key set: the
    definition of ``decode`` over the gathered keys (a numpy gather); the fusion
    gate of that page is not applied."""
    ka, kt = _raw(k)
    va, vt = _raw(v)
    B, Hkv, S, D = ka.shape
    lens = [S] * B if seqlens is None else [int(x) for x in seqlens]
    sets = [pi_key_set(L, window, period) for L in lens]
    n = max(1, max(len(x) for x in sets))
    kg = np.zeros((B, Hkv, n, D), dtype=ka.dtype)
    vg = np.zeros((B, Hkv, n, D), dtype=va.dtype)
    for b, idx in enumerate(sets):
        if idx:
            kg[b, :, :len(idx)] = ka[b][:, idx]
            vg[b, :, :len(idx)] = va[b][:, idx]
    glens = np.array([len(x) for x in sets], dtype=np.int32)
    return decode(q, kg, vg, scale, seqlens=glens, rows=rows, threads=threads)


def prefill_causal_varlen(q, k, v, cu_seqlens, scale, threads=None):
    """Causal prefill of packed variable-length sequences: q [T,H,D], k/v
    [T,Hkv,D]; sequence s is tokens [cu[s], cu[s+1]), and its row i attends
    keys 0..i of the same sequence.  Each sequence is sliced out (numpy) and
    given to ``prefill_causal``.  Returns (out [T,H,D], lse [H,T])."""
    qa, qt = _raw(q)
    ka, kt = _raw(k)
    va, vt = _raw(v)
    T, H, D = qa.shape
    Hkv = ka.shape[1]
    cu = [int(x) for x in cu_seqlens]
    out = np.zeros((T, H, D))
    lse = np.zeros((H, T))
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        if e <= a:
            continue
        qs = np.ascontiguousarray(qa[a:e].transpose(1, 0, 2))[None]
        ks = np.ascontiguousarray(ka[a:e].transpose(1, 0, 2))[None]
        vs = np.ascontiguousarray(va[a:e].transpose(1, 0, 2))[None]
        o, l = prefill_causal(qs, ks, vs, scale, threads=threads)
        out[a:e] = o.reshape(H, e - a, D).transpose(1, 0, 2)
        lse[:, a:e] = l.reshape(H, e - a)
    return out, lse


def e4m3_to_float(bits):
    """Values of FP8 E4M3 bit patterns (uint8): sign, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111
    is NaN and there is no infinity.  Written from the format definition."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def decode_fp8(q, k8, v8, k_scale, v_scale, scale, seqlens=None, rows=None, threads=None):
    """Decode over an E4M3 KV cache: the cache is dequantised first (value =
    e4m3 * scale of its (sequence, KV head), in float64, exact) and ``decode``
    does the rest.  k8/v8 [B,Hkv,S,D] uint8 bit patterns; k_scale/v_scale
    [B*Hkv] or None (1)."""
    kb = np.asarray(k8.cpu().numpy() if hasattr(k8, "cpu") else k8, dtype=np.uint8)
    vb = np.asarray(v8.cpu().numpy() if hasattr(v8, "cpu") else v8, dtype=np.uint8)
    B, Hkv = kb.shape[:2]
    ks = np.ones(B * Hkv) if k_scale is None else np.asarray(k_scale, dtype=np.float64).reshape(-1)
    vs = np.ones(B * Hkv) if v_scale is None else np.asarray(v_scale, dtype=np.float64).reshape(-1)
    kd = e4m3_to_float(kb) * ks.reshape(B, Hkv, 1, 1)
    vd = e4m3_to_float(vb) * vs.reshape(B, Hkv, 1, 1)
    return decode(q, np.ascontiguousarray(kd), np.ascontiguousarray(vd), scale, seqlens=seqlens, rows=rows,
                  threads=threads)


def e2m1_to_float(codes):
    """Values of FP4 E2M1 codes (the low 4 bits of each entry): sign, 2
    exponent bits with bias 1, 1 mantissa bit; exponent 0 is subnormal
    (m/2); no infinity or NaN (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).
    Written from the format definition."""
    c = np.asarray(codes).astype(np.int64) & 15
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m / 2.0, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag)


def nvfp4_dequantize(codes, block_scales, factor):
    """NVFP4 values in float64: codes [..., D/2] uint8 holding element 2i in
    the low nibble and element 2i + 1 in the high nibble (E2M1), block_scales
    [..., D/16] uint8 E4M3, one per 16 consecutive elements, and `factor` an
    fp32 array broadcastable to the leading dimensions.  value = e2m1 *
    e4m3(block scale) * factor (exact in float64)."""
    c = np.asarray(codes.cpu().numpy() if hasattr(codes, "cpu") else codes, dtype=np.uint8)
    bs = np.asarray(block_scales.cpu().numpy() if hasattr(block_scales, "cpu") else block_scales, dtype=np.uint8)
    lo = e2m1_to_float(c & 15)
    hi = e2m1_to_float(c >> 4)
    vals = np.stack([lo, hi], axis=-1).reshape(*c.shape[:-1], 2 * c.shape[-1])
    vals = vals * np.repeat(e4m3_to_float(bs), 16, axis=-1)
    return vals * np.asarray(factor, dtype=np.float64)


def decode_nvfp4(q, k4, k_bs, v4, v_bs, k_factor, v_factor, scale, seqlens=None, rows=None, threads=None):
    """Decode over an NVFP4 KV cache: K and V are dequantised first
    (``nvfp4_dequantize`` with the (sequence, KV head) factors; None = 1) and
    ``decode`` does the rest.  k4/v4 [B,Hkv,S,D/2] uint8, k_bs/v_bs
    [B,Hkv,S,D/16] uint8, k_factor/v_factor [B*Hkv]."""
    kb = np.asarray(k4.cpu().numpy() if hasattr(k4, "cpu") else k4, dtype=np.uint8)
    B, Hkv = kb.shape[:2]
    kf = np.ones(B * Hkv) if k_factor is None else np.asarray(k_factor, dtype=np.float64).reshape(-1)
    vf = np.ones(B * Hkv) if v_factor is None else np.asarray(v_factor, dtype=np.float64).reshape(-1)
    kd = nvfp4_dequantize(kb, k_bs, kf.reshape(B, Hkv, 1, 1))
    vd = nvfp4_dequantize(v4, v_bs, vf.reshape(B, Hkv, 1, 1))
    return decode(q, np.ascontiguousarray(kd), np.ascontiguousarray(vd), scale, seqlens=seqlens, rows=rows,
                  threads=threads)
