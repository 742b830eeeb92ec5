"""The C ABI on the host: exported symbols, the KV-chunk scheduler, and argument
validation (which rejects bad calls before any CUDA call, so it runs without a GPU)."""
import ctypes
import os
import re

import pytest
import torch

from long_context_decode_04_b300 import ta

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "ta.h")
SMS = 148


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ta_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert {"ta_decode", "ta_decode_ex", "ta_combine", "ta_prefill_causal", "ta_last_error"} <= set(names)
    L = ctypes.CDLL(ta.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, f"declared in include/ta.h but not exported: {missing}"


def _chunks(plan, S):
    return ta.chunk_bounds(plan, S)


@pytest.mark.parametrize("B,Hq,Hkv,S,D", [
    (1, 32, 8, 131072, 128), (16, 32, 8, 32768, 128), (1, 32, 8, 1 << 20, 128), (1, 1, 1, 4096, 64),
    (1, 1, 1, 1, 64), (3, 4, 2, 255, 128), (2, 8, 8, 257, 64), (1, 32, 8, 1000, 128), (64, 32, 8, 8192, 128)])
@pytest.mark.parametrize("varlen", [False, True])
def test_plan_covers_every_key_once(B, Hq, Hkv, S, D, varlen):
    plan = ta.plan_decode(B, Hq, Hkv, S, D, varlen=varlen, sm_count=SMS)
    ch = _chunks(plan, S)
    assert ch[0][0] == 0 and ch[-1][1] == S
    for (a0, a1), (b0, b1) in zip(ch, ch[1:]):
        assert a1 == b0 and a0 < a1  # contiguous, non-empty, no overlap
    assert ch[-1][0] < ch[-1][1]
    items = B * Hkv * plan.n_split
    assert plan.grid == min(items, SMS)
    if plan.n_split == 1 or (plan.n_split <= 128 and B * Hkv <= 4032):
        assert plan.levels == 0  # one chunk, or the decode kernel merges its chunks itself
    else:
        n, lv = plan.n_split, 1
        while n > plan.fanin:
            n, lv = -(-n // plan.fanin), lv + 1
        assert plan.levels == lv
    if S >= 256 * SMS and not varlen:
        assert items >= SMS  # every SM gets work


def test_plan_of_the_128k_workload_fills_the_sms_evenly():
    """Two items per SM: 8 KV heads x 37 chunks of 28 whole 128-key tiles."""
    plan = ta.plan_decode(1, 32, 8, 131072, 128, sm_count=SMS)
    items = 8 * plan.n_split
    assert items % SMS == 0 and plan.grid == SMS
    assert plan.chunk % 128 == 0 and plan.chunk >= 256  # whole 128-key tiles of the tensor-core kernel
    assert plan.levels == 0  # merged inside the decode kernel


@pytest.mark.parametrize("Hq,Hkv,D,tile", [(32, 8, 128, 128), (16, 8, 128, 128), (8, 8, 128, 120),
                                           (4, 4, 64, 120), (32, 8, 64, 120), (64, 8, 64, 120)])
def test_plan_chunks_are_whole_tiles_of_the_kernel_for_the_shape(Hq, Hkv, D, tile):
    """Chunks are whole 128-key tiles for the tensor-core shapes (D = 128, G = 2 or
    4) and whole 120-key tiles for the CUDA-core kernel's shapes, at least two."""
    for S in (300, 5000, 131072, 1 << 20):
        for varlen in (False, True):
            plan = ta.plan_decode(2, Hq, Hkv, S, D, varlen=varlen, sm_count=SMS)
            if plan.n_split > 1:
                assert plan.chunk % tile == 0 and plan.chunk >= 2 * tile, (S, varlen, plan.chunk)


def test_plan_overrides():
    p = ta.plan_decode(1, 32, 8, 1 << 20, 128, chunk=256, sm_count=SMS)
    assert p.chunk == 256 and p.n_split == 4096 and p.levels == 2
    p = ta.plan_decode(1, 32, 8, 1000, 128, n_split=7, sm_count=SMS)
    assert p.n_split == 7 and p.chunk == 143
    p = ta.plan_decode(1, 32, 8, 5, 128, n_split=9, sm_count=SMS)  # more splits than keys
    assert p.n_split == 5 and p.chunk == 1


def test_workspace_size_formula():
    def a256(x):
        return (x + 255) // 256 * 256
    B, Hq, Hkv, S, D = 1, 32, 8, 1 << 20, 128
    p = ta.plan_decode(B, Hq, Hkv, S, D, chunk=256, sm_count=SMS)
    R, N = B * Hq, p.n_split
    n1 = -(-N // 64)
    comb = 2 * (2 * a256(4 * R * n1) + a256(4 * R * n1 * D))
    control = 16384  # status word, work-queue counter and per-unit chunk counters
    assert p.workspace_bytes == control + 2 * a256(4 * R * N) + a256(4 * R * N * D) + comb
    p1 = ta.plan_decode(1, 1, 1, 100, 64, sm_count=SMS)
    assert p1.n_split == 1 and p1.workspace_bytes == 256


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), ta.TA_ERR_INVALID_ARG),
    (dict(S=0), ta.TA_ERR_INVALID_ARG),
    (dict(B=0), ta.TA_ERR_INVALID_ARG),
    (dict(D=96), ta.TA_ERR_UNSUPPORTED),
    (dict(Hq=16, Hkv=2, D=128), ta.TA_ERR_UNSUPPORTED),
    (dict(q=0x1008), ta.TA_ERR_INVALID_ARG),
    (dict(k=None), ta.TA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), ta.TA_ERR_INVALID_ARG),
    (dict(chunk=-1), ta.TA_ERR_INVALID_ARG),
    (dict(in_dtype=7), ta.TA_ERR_INVALID_ARG),
    (dict(in_dtype=ta.TA_F32, out_dtype=ta.TA_BF16), ta.TA_ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_arguments_before_launch(kw, status):
    base = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, B=1, Hq=8, Hkv=2, S=64, D=128,
                scale=0.1, seqlens=None, in_dtype=ta.TA_BF16, out_dtype=ta.TA_BF16, chunk=0, n_split=0,
                workspace=None, workspace_bytes=0, stream=None)
    base.update(kw)
    p = ta.DecodeParams(**base)
    rc = ta.lib().ta_decode_ex(ctypes.byref(p))
    assert rc == status
    assert len(ta.lib().ta_last_error()) > 0


def test_combine_and_prefill_reject_bad_arguments():
    L = ta.lib()
    vp = ctypes.c_void_p
    assert L.ta_combine(vp(0x1000), vp(0x2000), vp(0x3000), 4, 0, 128, vp(0x4000), ta.TA_F32, None, None, 0,
                        None) == ta.TA_ERR_INVALID_ARG
    assert L.ta_combine(vp(0x1000), vp(0x2000), vp(0x3000), 4, 2, 96, vp(0x4000), ta.TA_F32, None, None, 0,
                        None) == ta.TA_ERR_UNSUPPORTED
    assert L.ta_combine(None, vp(0x2000), vp(0x3000), 4, 2, 128, vp(0x4000), ta.TA_F32, None, None, 0,
                        None) == ta.TA_ERR_INVALID_ARG
    assert L.ta_prefill_causal(vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000), None, 1, 6, 4, 128, 128,
                               ctypes.c_float(0.1), None) == ta.TA_ERR_INVALID_ARG
    assert L.ta_prefill_causal(vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000), None, 1, 8, 2, 128, 64,
                               ctypes.c_float(0.1), None) == ta.TA_ERR_UNSUPPORTED
    assert L.ta_prefill_causal(vp(0x1004), vp(0x2000), vp(0x3000), vp(0x4000), None, 1, 8, 2, 128, 128,
                               ctypes.c_float(0.1), None) == ta.TA_ERR_INVALID_ARG
    assert L.ta_prefill_causal(vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000), None, 1, 8, 2, 128, 128,
                               ctypes.c_float(0.0), None) == ta.TA_ERR_UNSUPPORTED


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_cuda_error():
    p = ta.DecodeParams(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, B=1, Hq=8, Hkv=2, S=64, D=128,
                        scale=0.1, in_dtype=ta.TA_BF16, out_dtype=ta.TA_BF16)
    assert ta.lib().ta_decode_ex(ctypes.byref(p)) == ta.TA_ERR_CUDA
    assert b"cuda" in ta.lib().ta_last_error().lower()


@pytest.mark.parametrize("kw,status", [
    (dict(block_table=None), ta.TA_ERR_INVALID_ARG),
    (dict(seqlens=None), ta.TA_ERR_INVALID_ARG),
    (dict(page_size=0), ta.TA_ERR_INVALID_ARG),
    (dict(pages_per_seq=0), ta.TA_ERR_INVALID_ARG),
    (dict(num_pages=0), ta.TA_ERR_INVALID_ARG),
    (dict(block_table=0x6002), ta.TA_ERR_INVALID_ARG),
    (dict(k_pages=0x2008), ta.TA_ERR_INVALID_ARG),
    (dict(D=96), ta.TA_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), ta.TA_ERR_INVALID_ARG),
])
def test_paged_decode_rejects_bad_arguments_before_launch(kw, status):
    base = dict(q=0x1000, k_pages=0x2000, v_pages=0x3000, block_table=0x6000, seqlens=0x7000, out=0x4000,
                lse=0x5000, B=2, Hq=8, Hkv=2, D=128, page_size=16, pages_per_seq=4, num_pages=8, scale=0.1,
                in_dtype=ta.TA_BF16, out_dtype=ta.TA_BF16, chunk=0, n_split=0, workspace=None,
                workspace_bytes=0, stream=None)
    base.update(kw)
    p = ta.PagedDecodeParams(**base)
    assert ta.lib().ta_decode_paged(ctypes.byref(p)) == status
    assert len(ta.lib().ta_last_error()) > 0


def test_pi_decode_rejects_bad_window_and_period():
    p = ta.DecodeParams(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, B=1, Hq=8, Hkv=2, S=64, D=128,
                        scale=0.1, in_dtype=ta.TA_BF16, out_dtype=ta.TA_BF16)
    assert ta.lib().ta_decode_pi(ctypes.byref(p), -1, 4) == ta.TA_ERR_INVALID_ARG
    assert ta.lib().ta_decode_pi(ctypes.byref(p), 4, 0) == ta.TA_ERR_INVALID_ARG
    assert ta.lib().ta_decode_pi_workspace_bytes(1, 8, 2, 64, 128, 0, 0, 0, 4, 0) == 0


@pytest.mark.parametrize("S,window,period", [(1, 0, 1), (100, 0, 1), (100, 5, 7), (131072, 4096, 64),
                                             (1000, 2000, 3), (50, 3, 100)])
def test_pi_key_bound_covers_every_length(S, window, period):
    """The plan cuts the list of attended keys; its length bound must hold for
    every sequence length up to S (checked against the oracle's key set)."""
    import oracle
    bound = min(S, min(window + 1, S) + -(-max(0, S - 1 - window) // period))
    for L in sorted(x for x in {1, 2, S // 3, S // 2, S - 1, S} if 1 <= x <= S):
        assert len(oracle.pi_key_set(L, window, period)) <= bound


def test_varlen_prefill_rejects_bad_arguments():
    L = ta.lib()
    vp = ctypes.c_void_p
    f = ctypes.c_float(0.1)
    ok = dict(q=vp(0x1000), k=vp(0x2000), v=vp(0x3000), out=vp(0x4000), lse=None, cu=vp(0x5000))
    def call(**kw):
        a = dict(ok, **{k2: v2 for k2, v2 in kw.items() if k2 in ok})
        n = dict(num_seqs=2, max_seqlen=128, total=256, H=8, Hkv=2, D=128)
        n.update({k2: v2 for k2, v2 in kw.items() if k2 in n})
        return L.ta_prefill_causal_varlen(a["q"], a["k"], a["v"], a["out"], a["lse"], a["cu"], n["num_seqs"],
                                          n["max_seqlen"], n["total"], n["H"], n["Hkv"], n["D"], f, None)
    assert call(cu=None) == ta.TA_ERR_INVALID_ARG
    assert call(num_seqs=0) == ta.TA_ERR_INVALID_ARG
    assert call(H=6, Hkv=4) == ta.TA_ERR_INVALID_ARG
    assert call(D=64) == ta.TA_ERR_UNSUPPORTED
    assert call(q=vp(0x1008)) == ta.TA_ERR_INVALID_ARG
    assert call(cu=vp(0x5002)) == ta.TA_ERR_INVALID_ARG


def test_fp8_decode_rejects_unsupported_shapes():
    base = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, B=1, Hq=8, Hkv=2, S=64, D=128,
                scale=0.1, in_dtype=ta.TA_BF16, out_dtype=ta.TA_BF16)
    L = ta.lib()
    p = ta.DecodeParams(**dict(base, D=64))
    assert L.ta_decode_fp8(ctypes.byref(p), None, None) == ta.TA_ERR_UNSUPPORTED
    p = ta.DecodeParams(**dict(base, in_dtype=ta.TA_F32, out_dtype=ta.TA_F32))
    assert L.ta_decode_fp8(ctypes.byref(p), None, None) == ta.TA_ERR_INVALID_ARG
    p = ta.DecodeParams(**base)
    assert L.ta_decode_fp8(ctypes.byref(p), ctypes.c_void_p(0x6002), None) == ta.TA_ERR_INVALID_ARG


def test_prefill_ex_rejects_bad_arguments():
    L = ta.lib()

    def call(**kw):
        base = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, B=1, H=8, Hkv=2, S=128, D=128,
                    scale=0.1, cu_seqlens=None, total_tokens=0, out_dtype=ta.TA_F32, wait_limit_ns=0, stream=None)
        base.update(kw)
        p = ta.PrefillParams(**base)
        return L.ta_prefill_causal_ex(ctypes.byref(p))

    assert L.ta_prefill_causal_ex(None) == ta.TA_ERR_INVALID_ARG
    assert call(out_dtype=7) == ta.TA_ERR_INVALID_ARG
    assert call(H=6, Hkv=4) == ta.TA_ERR_INVALID_ARG
    assert call(out=0x4004) == ta.TA_ERR_INVALID_ARG
    assert call(D=64) == ta.TA_ERR_UNSUPPORTED
    assert call(scale=-1.0) == ta.TA_ERR_UNSUPPORTED
    assert call(cu_seqlens=0x6000, total_tokens=0) == ta.TA_ERR_INVALID_ARG  # packed needs tokens
    assert call(cu_seqlens=0x6002, total_tokens=256) == ta.TA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the hook ahead of the no-GPU error path")
def test_launch_failure_hook_refuses_launches_after_validation():
    """ta_test_fail_next_launches: a valid merge call whose launch is refused returns
    TA_ERR_CUDA naming the hook (the merge of <= 64 partials makes no CUDA call
    before its launch, so this runs without a GPU); a rejected call does not use
    up an injected failure; once the count is spent the real outcome returns."""
    L = ta.lib()
    vp = ctypes.c_void_p
    args = (vp(0x1000), vp(0x2000), vp(0x3000), 4, 2, 128, vp(0x4000), ta.TA_F32, None, None, 0, None)
    assert L.ta_test_fail_next_launches(2) == 0
    # bad arguments are rejected before the launch: no injected failure is used
    assert L.ta_combine(vp(0x1000), vp(0x2000), vp(0x3000), 4, 0, 128, vp(0x4000), ta.TA_F32, None, None, 0,
                        None) == ta.TA_ERR_INVALID_ARG
    for _ in range(2):
        assert L.ta_combine(*args) == ta.TA_ERR_CUDA
        assert b"ta_test_fail_next_launches" in L.ta_last_error()
    assert L.ta_test_fail_next_launches(0) == 0
    assert L.ta_combine(*args) == ta.TA_ERR_CUDA  # no GPU here: the real launch error
    assert b"ta_test_fail_next_launches" not in L.ta_last_error()
    assert L.ta_test_fail_next_launches(5) == 0
    assert L.ta_test_fail_next_launches(0) == 5  # cancelled with 5 pending


def test_nvfp4_decode_rejects_bad_arguments():
    base = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, B=1, Hq=8, Hkv=2, S=64, D=128,
                scale=0.1, in_dtype=ta.TA_BF16, out_dtype=ta.TA_BF16)
    L = ta.lib()
    vp = ctypes.c_void_p
    p = ta.DecodeParams(**base)
    assert L.ta_decode_nvfp4(ctypes.byref(p), None, vp(0x6000), None, None) == ta.TA_ERR_INVALID_ARG
    assert L.ta_decode_nvfp4(ctypes.byref(p), vp(0x6008), vp(0x6000), None, None) == ta.TA_ERR_INVALID_ARG
    assert L.ta_decode_nvfp4(ctypes.byref(p), vp(0x6000), vp(0x7000), vp(0x8002), None) == ta.TA_ERR_INVALID_ARG
    p = ta.DecodeParams(**dict(base, Hq=2))  # one query head per KV head
    assert L.ta_decode_nvfp4(ctypes.byref(p), vp(0x6000), vp(0x7000), None, None) == ta.TA_ERR_UNSUPPORTED
    p = ta.DecodeParams(**dict(base, S=70))  # S not a multiple of 16
    assert L.ta_decode_nvfp4(ctypes.byref(p), vp(0x6000), vp(0x7000), None, None) == ta.TA_ERR_UNSUPPORTED
    p = ta.DecodeParams(**dict(base, in_dtype=ta.TA_F32, out_dtype=ta.TA_F32))
    assert L.ta_decode_nvfp4(ctypes.byref(p), vp(0x6000), vp(0x7000), None, None) == ta.TA_ERR_INVALID_ARG
