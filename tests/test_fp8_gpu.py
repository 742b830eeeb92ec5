"""Split-KV decode over an FP8 (E4M3) KV cache on the GPU through the C ABI,
against the float64 oracle that dequantises the same bytes first.  Rows past
each sequence's length hold the E4M3 NaN pattern, so a wrong key shows."""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _quantised(name, **kw):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, **kw)
    k8, ks = synth.to_e4m3(x["k"])
    v8, vs = synth.to_e4m3(x["v"])
    return x, k8, v8, ks, vs


def _run(x, k8, v8, ks, vs, seqlens=None, **kw):
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = ta.decode_fp8(x["q"].to(DEV), k8.to(DEV), v8.to(DEV), k_scale=None if ks is None else ks.to(DEV),
                             v_scale=None if vs is None else vs.to(DEV), seqlens=sl, scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return out, lse


def _check(x, k8, v8, ks, vs, out, lse, bf16, seqlens=None):
    ro, rl = oracle.decode_fp8(x["q"], k8, v8, None if ks is None else ks.numpy(),
                               None if vs is None else vs.numpy(), x["scale"], seqlens=seqlens)
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro, bf16=bf16)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_fp8_full_128k():
    x, k8, v8, ks, vs = _quantised("gqa_32x8_d128_s131072")
    out, lse = _run(x, k8, v8, ks, vs)
    _check(x, k8, v8, ks, vs, out, lse, bf16=True)
    out, lse = _run(x, k8, v8, ks, vs, out_dtype=torch.float32)
    _check(x, k8, v8, ks, vs, out, lse, bf16=False)


@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("split", [0, 1, 9])
def test_fp8_head_groups_and_splits(G, split):
    w = synth.Workload("fp8", 2, "decode", 2, 2 * G, 2, 3001, 128, "bf16")
    x = synth.make_inputs(w, seed=1500 + G)
    k8, ks = synth.to_e4m3(x["k"])
    v8, vs = synth.to_e4m3(x["v"])
    out, lse = _run(x, k8, v8, ks, vs, out_dtype=torch.float32, n_split=split)
    _check(x, k8, v8, ks, vs, out, lse, bf16=False)


def test_fp8_varlen_nan_padding_and_unit_scales():
    x, k8, v8, ks, vs = _quantised("varlen_b16_32x8_d128_s1k_32k", S=4096, B=5)
    lens = [int(v) for v in x["seqlens"]]
    for b, L in enumerate(lens):
        k8[b, :, L:] = 0x7F  # E4M3 NaN
        v8[b, :, L:] = 0x7F
    out, lse = _run(x, k8, v8, ks, vs, seqlens=lens, out_dtype=torch.float32)
    _check(x, k8, v8, ks, vs, out, lse, bf16=False, seqlens=lens)
    # no scales: the bytes are the values
    out, lse = _run(x, k8, v8, None, None, seqlens=lens, out_dtype=torch.float32)
    _check(x, k8, v8, None, None, out, lse, bf16=False, seqlens=lens)
