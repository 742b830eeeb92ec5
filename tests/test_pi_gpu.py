"""Split-KV decode over the pi-Attention key set (ring-local window plus
periodic skips, causal) on the GPU through the C ABI, against the float64
oracle restricted to the same keys; with period 1 it is the dense decode, bit
for bit.  Keys past each sequence's length are NaN, so a wrong key shows."""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(S, B=2, name="gqa_32x8_d128_s131072", seed=None, pad=True):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, S=S, B=B, seed=seed)
    return x


def _run(x, window, period, seqlens=None, **kw):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = ta.decode_pi(q, k, v, window, period, seqlens=sl, scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("window,period", [(0, 2), (16, 64), (127, 7), (500, 120), (4000, 3), (10, 5000)])
def test_pi_matches_oracle(window, period):
    x = _inputs(5003, seed=900 + period)
    out, lse = _run(x, window, period, out_dtype=torch.float32)
    ro, rl = oracle.decode_pi(x["q"], x["k"], x["v"], x["scale"], window, period)
    check_out(out.cpu().numpy().reshape(-1, 128), ro, bf16=False)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_pi_varlen_nan_padding_and_forced_splits():
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w, S=4096, B=5, pad_value=float("nan"))
    lens = [int(v) for v in x["seqlens"]]
    for split in (0, 3, 40):
        out, lse = _run(x, 300, 17, seqlens=lens, n_split=split)
        ro, rl = oracle.decode_pi(x["q"], x["k"], x["v"], x["scale"], 300, 17, seqlens=lens)
        check_out(out.float().cpu().numpy().reshape(-1, 128), ro, bf16=True)
        check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_pi_period_one_is_the_dense_decode():
    x = _inputs(3000, seed=905)
    a = _run(x, 0, 1, out_dtype=torch.float32)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    b = ta.decode(q, k, v, scale=x["scale"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_pi_small_head_shapes():
    for name in ("single_head_d64_s4096_f32",):
        x = synth.make_inputs(synth.WORKLOADS[name], S=2000)
        out, lse = _run(x, 100, 9, out_dtype=torch.float32)
        ro, rl = oracle.decode_pi(x["q"], x["k"], x["v"], x["scale"], 100, 9)
        check_out(out.cpu().numpy().reshape(-1, 64), ro, bf16=False)
        check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_pi_full_128k_window_4096_period_64():
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    x = synth.make_inputs(w)
    ws = ta.decode_pi_workspace(1, 32, 8, w.S, 128, 4096, 64)
    out, lse = _run(x, 4096, 64, workspace=ws)
    ro, rl = oracle.decode_pi(x["q"], x["k"], x["v"], x["scale"], 4096, 64)
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro, bf16=True)
    check_lse(lse.cpu().numpy().reshape(-1), rl)
    assert ta.decode_status(ws) == 0
