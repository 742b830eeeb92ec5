"""Failure detection on the GPU, in the forms that leave the GPU usable: device-side
conditions recorded in the status word and read on the host, a pipeline wait that
runs out its (per-launch) time limit because a test hook makes it wait on a
barrier nothing completes, and a launch refused on the host by a test hook.
None of these faults, traps or hangs the GPU: every wait in the kernels has a
time limit, and a launch that gives up lets its copies and tensor-core
operations finish and frees its tensor memory before it returns."""
import time

import numpy as np
import pytest
import torch

from long_context_decode_04_b300 import synth, ta

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT_NS = 2_000_000  # 2 ms: the per-launch limit the stalled launches run out


@pytest.fixture(autouse=True)
def _clean_hooks():
    ta.test_stall_next_launches(0)
    ta.test_fail_next_launches(0)
    ta.decode_status()
    yield
    ta.test_stall_next_launches(0)
    ta.test_fail_next_launches(0)
    torch.cuda.synchronize()


def _decode_inputs(Hq, Hkv, S, dtype="bf16", seed=50):
    w = synth.Workload("t", 9, "decode", 2, Hq, Hkv, S, 128, dtype)
    x = synth.make_inputs(w, seed=seed)
    return tuple(x[n].to(DEV) for n in ("q", "k", "v")) + (x["scale"],)


def test_prefill_flags_values_outside_fp16_range():
    w = synth.Workload("t", 5, "prefill", 1, 4, 2, 300, 128, "bf16")
    x = synth.make_inputs(w, seed=51)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    ta.prefill_causal(q, k, v)
    assert ta.decode_status() == 0
    v_big = v.clone()
    v_big[0, 1, 77, 5] = 70000.0  # bf16 70144 > 65280, the largest value that converts exactly
    ta.prefill_causal(q, k, v_big)
    assert ta.decode_status() & ta.TA_DEVERR_RANGE
    v_big[0, 1, 77, 5] = -65280.0  # the limit itself converts exactly
    ta.prefill_causal(q, k, v_big)
    assert ta.decode_status() == 0


@pytest.mark.parametrize("kind", ["tensor_core", "cuda_core", "fp8", "paged", "pi"])
def test_decode_wait_runs_out_its_limit_and_the_next_call_is_exact(kind):
    """A stalled launch gives up after its 2 ms limit (not the default 2 s), records
    TA_DEVERR_TIMEOUT, returns, and leaves the library workspace reusable once
    ta_decode_status has read the flag: the next decode is bit for bit the one
    before the stall."""
    if kind == "cuda_core":
        q, k, v, scale = _decode_inputs(2, 2, 20000)  # one query head per KV head
    else:
        q, k, v, scale = _decode_inputs(8, 2, 20000)
    if kind == "fp8":
        k8, ks = synth.to_e4m3(k.cpu())
        v8, vs = synth.to_e4m3(v.cpu())
        k8, ks, v8, vs = k8.to(DEV), ks.to(DEV), v8.to(DEV), vs.to(DEV)
        run = lambda **kw: ta.decode_fp8(q, k8, v8, k_scale=ks, v_scale=vs, scale=scale, **kw)
    elif kind == "paged":
        lens = [20000, 7777]
        kp, vp, bt = synth.to_pages(k.cpu(), v.cpu(), lens, 64, seed=3)
        kp, vp, bt = kp.to(DEV), vp.to(DEV), bt.to(DEV)
        sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
        run = lambda **kw: ta.decode_paged(q, kp, vp, bt, sl, scale=scale, **kw)
    elif kind == "pi":
        run = lambda **kw: ta.decode_pi(q, k, v, 1000, 9, scale=scale, **kw)
    else:
        run = lambda **kw: ta.decode(q, k, v, scale=scale, **kw)
    ref_out, ref_lse = run()
    torch.cuda.synchronize()
    assert ta.decode_status() == 0
    assert ta.test_stall_next_launches(1) == 0
    t0 = time.perf_counter()
    out, lse = run(wait_limit_ns=LIMIT_NS)  # returns TA_OK: the failure is on the device
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert ta.decode_status() & ta.TA_DEVERR_TIMEOUT
    assert took < 1.0, f"the stalled launch took {took:.3f} s: the 2 ms limit was not applied"
    assert ta.test_stall_next_launches(0) == 0  # the stall was used up
    out2, lse2 = run()
    torch.cuda.synchronize()
    assert ta.decode_status() == 0
    assert torch.equal(out2, ref_out) and torch.equal(lse2, ref_lse)


def test_prefill_wait_runs_out_its_limit_and_the_next_call_is_exact():
    w = synth.Workload("t", 5, "prefill", 1, 8, 2, 1000, 128, "bf16")
    x = synth.make_inputs(w, seed=52)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    ref = ta.prefill_causal(q, k, v)
    torch.cuda.synchronize()
    assert ta.decode_status() == 0
    ta.test_stall_next_launches(1)
    t0 = time.perf_counter()
    ta.prefill_causal(q, k, v, wait_limit_ns=LIMIT_NS)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0
    assert ta.decode_status() & ta.TA_DEVERR_TIMEOUT
    again = ta.prefill_causal(q, k, v)
    torch.cuda.synchronize()
    assert ta.decode_status() == 0
    assert torch.equal(again[0], ref[0]) and torch.equal(again[1], ref[1])


def test_caller_workspace_after_a_timeout_is_reusable_once_its_control_region_is_zeroed():
    q, k, v, scale = _decode_inputs(8, 2, 20000)
    ws = ta.decode_workspace(2, 8, 2, 20000, 128)
    ref = ta.decode(q, k, v, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    ta.test_stall_next_launches(1)
    ta.decode(q, k, v, scale=scale, workspace=ws, wait_limit_ns=LIMIT_NS)
    assert ta.decode_status(ws) & ta.TA_DEVERR_TIMEOUT
    ws[:16384].zero_()  # as include/ta.h asks after TA_DEVERR_TIMEOUT
    again = ta.decode(q, k, v, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    assert ta.decode_status(ws) == 0
    assert torch.equal(again[0], ref[0]) and torch.equal(again[1], ref[1])


def test_refused_launch_writes_nothing_and_the_next_call_works():
    q, k, v, scale = _decode_inputs(8, 2, 5000)
    out = torch.full((2, 8, 128), 9.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((2, 8), 9.0, dtype=torch.float32, device=DEV)
    ta.test_fail_next_launches(1)
    with pytest.raises(ta.TAError) as e:
        ta.decode(q, k, v, scale=scale, out=out, lse=lse)
    assert e.value.status == ta.TA_ERR_CUDA and "ta_test_fail_next_launches" in str(e.value)
    torch.cuda.synchronize()
    assert torch.all(out == 9.0) and torch.all(lse == 9.0)
    ta.decode(q, k, v, scale=scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.isfinite(lse).all() and not torch.all(out == 9.0)
    w = synth.Workload("t", 5, "prefill", 1, 4, 2, 300, 128, "bf16")
    x = synth.make_inputs(w, seed=53)
    pq, pk, pv = (x[n].to(DEV) for n in ("q", "k", "v"))
    pout = torch.full_like(pq, 5.0)
    ta.test_fail_next_launches(1)
    with pytest.raises(ta.TAError):
        ta.prefill_causal(pq, pk, pv, out=pout)
    torch.cuda.synchronize()
    assert torch.all(pout == 5.0)
    assert ta.decode_status() == 0
