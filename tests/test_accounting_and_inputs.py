"""Host-side facts: the byte-count function against the page's printed sizes,
and the seeded input generator's determinism and shapes."""
import os

import numpy as np
import pytest
import torch

from long_context_decode_04_b300 import accounting, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_sizing.txt")


def _rows():
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        s, d, e, h, layers, expected, unit, sig = line.split()
        yield int(s), int(d), int(e), int(h), int(layers), float(expected), unit, int(sig)


def _round_sig(x, sig):
    from math import floor, log10
    return round(x, sig - 1 - int(floor(log10(abs(x)))))


@pytest.mark.parametrize("row", list(_rows()))
def test_kv_cache_bytes_match_page(row):
    s, d, e, h, layers, expected, unit, sig = row
    got = accounting.kv_cache_bytes(s, d, heads=h, layers=layers, bytes_per_elem=e)
    div = {"MB": 1e6, "GB": 1e9}[unit]
    assert _round_sig(got / div, sig) == expected


def test_decode_bytes_of_the_128k_workload():
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    assert accounting.decode_kv_bytes(w.B, w.Hkv, w.D, w.S, 2) == 536_870_912
    # 4096 bytes of K and V per context token across the 8 KV heads
    assert accounting.decode_kv_bytes(1, 8, 128, 1, 2) == 4096


def test_prefill_flops_of_the_16k_workload():
    assert accounting.prefill_causal_flops(1, 32, 16384, 128) == 4 * 32 * 128 * (16384 * 16385 // 2)
    # brute count of causal pairs on a tiny case
    S = 7
    pairs = sum(1 for i in range(S) for j in range(S) if j <= i)
    assert accounting.prefill_causal_flops(1, 1, S, 1) == 4 * pairs


def test_inputs_are_seeded_and_thread_independent():
    a = synth._normal_f32(1234, 2, (1 << 24) + 77, threads=1)
    b = synth._normal_f32(1234, 2, (1 << 24) + 77, threads=8)
    assert np.array_equal(a, b)
    assert abs(float(a.mean())) < 1e-3 and abs(float(a.std()) - 1) < 1e-3


def test_workload_shapes():
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w, S=2048, B=4, pad_value=float("nan"))
    assert x["q"].shape == (4, 32, 128) and x["k"].shape == (4, 8, 2048, 128)
    assert x["q"].dtype == torch.bfloat16
    sl = x["seqlens"]
    assert sl.dtype == torch.int32 and int(sl.min()) >= 1 and int(sl.max()) <= 2048
    for b in range(4):
        assert torch.isnan(x["k"][b, :, int(sl[b]):].float()).all()
        assert not torch.isnan(x["k"][b, :, :int(sl[b])].float()).any()
    full = synth.seqlens_for(w)
    assert int(full.min()) >= 1024 and int(full.max()) <= 32768 and full.shape == (16,)
    p = synth.WORKLOADS["causal_prefill_32x8_d128_s16384"]
    y = synth.make_inputs(p, S=256)
    assert y["q"].shape == (1, 32, 256, 128) and y["k"].shape == (1, 8, 256, 128)
    c1 = synth.WORKLOADS["single_head_d64_s4096_f32"]
    z = synth.make_inputs(c1)
    assert z["q"].dtype == torch.float32 and z["k"].shape == (1, 1, 4096, 64)
