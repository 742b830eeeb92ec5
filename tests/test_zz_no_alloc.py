"""ta_decode_noalloc, the decode entry point for callers that cannot allocate
device memory (their GPU memory is held by a pool allocator, or allocation
after start-up is forbidden): it must give what ta_decode gives, call after
call, using only its fixed scratch array.

Called through the C ABI.  Kept in a file that pytest collects last, so that
a run stopping at the first failure has already run every other test.
"""
import pytest
import torch

from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 8 << 20  # the fixed scratch size stated in include/ta.h


def _inputs(name, **kw):
    x = synth.make_inputs(synth.WORKLOADS[name], **kw)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    sl = None if x["seqlens"] is None else x["seqlens"].to(DEV)
    return q, k, v, sl, x["scale"]


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


def _compare(out, lse, ref_out, ref_lse):
    check_out(out.float().cpu().numpy(), ref_out.double().cpu().numpy(), bf16=True)
    check_lse(lse.cpu().numpy(), ref_lse.double().cpu().numpy())


@pytest.mark.parametrize("name,kw", [
    ("gqa_32x8_d128_s131072", {}),                      # the 128K-token GQA workload, full size
    ("varlen_b16_32x8_d128_s1k_32k", {"S": 8192}),    # variable lengths, masked padding
])
def test_noalloc_matches_ta_decode_on_two_calls_in_a_row(name, kw):
    B, Hq, Hkv = (synth.WORKLOADS[name].B, synth.WORKLOADS[name].Hq, synth.WORKLOADS[name].Hkv)
    S = kw.get("S", synth.WORKLOADS[name].S)
    need = ta.plan_decode(B, Hq, Hkv, S, 128, varlen=name.startswith("varlen")).workspace_bytes
    assert need <= SCRATCH_BYTES
    first = _inputs(name, **kw)
    second = _inputs(name, seed=77, **kw)  # different values, same shape
    a = _both(*first)
    b = _both(*second)
    _compare(*a)
    _compare(*b)
    # the two calls really computed different things from the shared scratch
    assert not torch.equal(a[0], b[0])


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
