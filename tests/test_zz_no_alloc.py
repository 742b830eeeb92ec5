"""ta_decode_noalloc, the decode entry point for callers that cannot allocate
device memory (their GPU memory is held by a pool allocator, or allocation
after start-up is forbidden): it must give what ta_decode gives, call after
call, using only its fixed scratch array, and its results must match the
float64 oracle within the usual tolerances.

Called through the C ABI.  Kept in a file that pytest collects last, so that
a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 8 << 20  # the fixed scratch size stated in include/ta.h


def _inputs(name, **kw):
    x = synth.make_inputs(synth.WORKLOADS[name], **kw)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    sl = None if x["seqlens"] is None else x["seqlens"].to(DEV)
    return x, (q, k, v, sl, x["scale"])


def _both(q, k, v, sl, scale):
    B, Hq, D = q.shape
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    ref_out = torch.empty_like(out)
    ref_lse = torch.empty_like(lse)
    ta.decode_noalloc(q, k, v, out, lse, scale, seqlens=sl)
    ta.decode_bf16(q, k, v, ref_out, ref_lse, scale, seqlens=sl)
    torch.cuda.synchronize()
    return out, lse, ref_out, ref_lse


def _compare(x, out, lse, ref_out, ref_lse):
    # against ta_decode (the same arithmetic: the tolerance is generous) ...
    check_out(out.float().cpu().numpy(), ref_out.double().cpu().numpy(), bf16=True)
    check_lse(lse.cpu().numpy(), ref_lse.double().cpu().numpy())
    # ... and against the float64 oracle
    sl = None if x["seqlens"] is None else x["seqlens"].numpy()
    ro, rl = oracle.decode(x["q"], x["k"], x["v"], x["scale"], seqlens=sl)
    check_out(out.float().cpu().numpy().reshape(ro.shape), ro, bf16=True)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


@pytest.mark.parametrize("name,kw", [
    ("gqa_32x8_d128_s131072", {}),                      # the 128K-token GQA workload, full size
    ("varlen_b16_32x8_d128_s1k_32k", {"S": 8192}),    # variable lengths, masked padding
])
def test_noalloc_matches_ta_decode_on_two_calls_in_a_row(name, kw):
    B, Hq, Hkv = (synth.WORKLOADS[name].B, synth.WORKLOADS[name].Hq, synth.WORKLOADS[name].Hkv)
    S = kw.get("S", synth.WORKLOADS[name].S)
    need = ta.plan_decode(B, Hq, Hkv, S, 128, varlen=name.startswith("varlen")).workspace_bytes
    assert need <= SCRATCH_BYTES
    x1, first = _inputs(name, **kw)
    x2, second = _inputs(name, seed=77, **kw)  # different values, same shape
    a = _both(*first)
    b = _both(*second)
    _compare(x1, *a)
    _compare(x2, *b)
    # the two calls really computed different things from the shared scratch
    assert not torch.equal(a[0], b[0])


def test_noalloc_separate_merge_path_over_128_chunks():
    """A plan with more than 128 chunks (so separate merge launches read the
    partials from, and write their intermediates into, the fixed scratch): one
    sequence with one KV head and 131072 keys passed with its length (the
    length-agnostic plan over-decomposes to about four items per SM), twice in
    a row."""
    w = synth.Workload("one_kv_head", 2, "decode", 1, 4, 1, 131072, 128, "bf16")
    plan = ta.plan_decode(1, 4, 1, w.S, 128, varlen=True)
    assert plan.n_split > 128 and plan.levels == 2 and plan.workspace_bytes <= SCRATCH_BYTES
    for seed in (None, 78):
        x = synth.make_inputs(w, seed=seed)
        x["seqlens"] = torch.tensor([w.S], dtype=torch.int32)
        q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
        res = _both(q, k, v, x["seqlens"].to(DEV), x["scale"])
        _compare(x, *res)


def test_noalloc_allocates_nothing_after_its_set_up():
    ta.decode_noalloc_setup()
    _, args = _inputs("gqa_32x8_d128_s131072", S=20000)
    q = args[0]
    out = torch.empty(1, 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 32, dtype=torch.float32, device=DEV)
    ta.decode_noalloc(q, args[1], args[2], out, lse, args[4])  # first call: module and scratch in place
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        ta.decode_noalloc(q, args[1], args[2], out, lse, args[4])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    assert ta.decode_noalloc_status() == 0


def test_noalloc_reports_device_flags_through_its_own_status_word():
    _, (q, k, v, sl, scale) = _inputs("varlen_b16_32x8_d128_s1k_32k", S=4096, B=3)
    out = torch.empty(3, 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(3, 32, dtype=torch.float32, device=DEV)
    bad = torch.tensor([4097, 100, -2], dtype=torch.int32, device=DEV)  # outside [0, S]: clamped
    ta.decode_noalloc(q, k, v, out, lse, scale, seqlens=bad)
    assert ta.decode_noalloc_status() & ta.TA_DEVERR_SEQLEN
    assert ta.decode_noalloc_status() == 0  # read and cleared
    ok = torch.tensor([4096, 100, 0], dtype=torch.int32, device=DEV)
    o2 = torch.empty_like(out)
    l2 = torch.empty_like(lse)
    ta.decode_noalloc(q, k, v, o2, l2, scale, seqlens=ok)
    torch.cuda.synchronize()
    assert ta.decode_noalloc_status() == 0
    # the clamped lengths are the lengths 4096 and 0
    assert torch.equal(out, o2) and torch.equal(torch.nan_to_num(lse), torch.nan_to_num(l2))


def test_noalloc_rejects_a_shape_beyond_its_scratch():
    # 192 sequences x 8 KV heads x 65536 keys: the default plan splits each
    # (sequence, KV head) in five and needs about 15 MiB of partials.  K/V
    # are real buffers of the full size (24 GiB, shared by K and V, never
    # written), so even a call that slipped through would stay in bounds.
    B, Hq, Hkv, S, D = 192, 32, 8, 65536, 128
    need = ta.plan_decode(B, Hq, Hkv, S, D).workspace_bytes
    assert need > SCRATCH_BYTES
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device=DEV)
    kv = torch.empty(B, Hkv, S, D, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    rc = ta.lib().ta_decode_noalloc(ta._ptr(q), ta._ptr(kv), ta._ptr(kv), ta._ptr(out), ta._ptr(lse), B, Hq, Hkv,
                                    S, D, ta.ctypes.c_float(0.1), None, ta._stream(q.device))
    assert rc == ta.TA_ERR_WORKSPACE
    assert b"scratch" in ta.lib().ta_last_error()
    del kv
    torch.cuda.synchronize()
