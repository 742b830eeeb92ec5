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


# every E4M3 byte but the two NaN patterns: signed zeros, the subnormals
# (k * 2^-9, k = 1..7) and +-448 included
_FINITE_E4M3 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


@pytest.mark.parametrize("G,out_dtype", [(1, torch.float32), (2, torch.bfloat16), (4, torch.float32)])
def test_fp8_uniform_random_codes(G, out_dtype):
    """K and V bytes drawn uniformly over the 254 finite E4M3 patterns, with
    +-448 and the smallest subnormal also planted at fixed strides so that
    every tile holds them; factors 2^-6 (K) and 2^-8 (V) keep the scores of
    order one."""
    w = synth.Workload("fp8", 2, "decode", 2, 2 * G, 2, 3001, 128, "bf16")
    x = synth.make_inputs(w, seed=1600 + G)
    rng = np.random.Generator(np.random.PCG64(93 + G))
    shape = (2, 2, 3001, 128)
    k8 = _FINITE_E4M3[rng.integers(0, _FINITE_E4M3.size, size=shape)]
    v8 = _FINITE_E4M3[rng.integers(0, _FINITE_E4M3.size, size=shape)]
    k8[:, :, ::97, 5] = 0x7E   # +448
    k8[:, :, 1::89, 6] = 0xFE  # -448
    v8[:, :, ::83, 7] = 0xFE
    v8[:, :, 2::79, 8] = 0x7E
    k8[:, :, 3::101, 9] = 0x01  # 2^-9
    v8[:, :, 4::103, 10] = 0x81  # -2^-9
    k8, v8 = torch.from_numpy(k8), torch.from_numpy(v8)
    ks = torch.full((4,), 2.0 ** -6, dtype=torch.float32)
    vs = torch.full((4,), 2.0 ** -8, dtype=torch.float32)
    out, lse = _run(x, k8, v8, ks, vs, out_dtype=out_dtype)
    _check(x, k8, v8, ks, vs, out, lse, bf16=out_dtype == torch.bfloat16)


@pytest.mark.parametrize("G", [1, 4])
def test_fp8_flags_a_query_outside_fp16(G):
    """Queries are used as fp16 values: 65280, the largest bf16 value below
    2^16, fits; 2^16 and beyond do not, and record TA_DEVERR_RANGE."""
    w = synth.Workload("fp8", 2, "decode", 2, 2 * G, 2, 1024, 128, "bf16")
    x = synth.make_inputs(w, seed=1700 + G)
    k8, ks = synth.to_e4m3(x["k"])
    v8, vs = synth.to_e4m3(x["v"])
    ta.decode_status()
    for value, flagged in ((65280.0, False), (-65280.0, False), (65536.0, True), (-3.0e38, True)):
        q = x["q"].clone()
        q[1, 2 * G - 1, 77] = value
        ta.decode_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), k_scale=ks.to(DEV), v_scale=vs.to(DEV), scale=x["scale"])
        torch.cuda.synchronize()
        st = ta.decode_status()
        assert bool(st & ta.TA_DEVERR_RANGE) == flagged, (value, st)
        assert st & ~ta.TA_DEVERR_RANGE == 0, st
