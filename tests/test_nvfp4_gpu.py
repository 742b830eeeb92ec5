"""Split-KV decode over an NVFP4 KV cache (E2M1 codes, one E4M3 scale per 16
elements, one fp32 factor per (sequence, KV head)) on the GPU through the C
ABI, against the float64 oracle that dequantises the same bytes first.  Rows
past each sequence's length have NaN block scales (E4M3 0x7f), so a wrong key
shows."""
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
    k4, kbs, kf = synth.to_nvfp4(x["k"])
    v4, vbs, vf = synth.to_nvfp4(x["v"])
    return x, (k4, kbs, kf, v4, vbs, vf)


def _run(x, c, seqlens=None, factors=True, **kw):
    k4, kbs, kf, v4, vbs, vf = c
    sl = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device=DEV)
    out, lse = ta.decode_nvfp4(x["q"].to(DEV), k4.to(DEV), v4.to(DEV), kbs.to(DEV), vbs.to(DEV),
                               k_factor=kf.to(DEV) if factors else None, v_factor=vf.to(DEV) if factors else None,
                               seqlens=sl, scale=x["scale"], **kw)
    torch.cuda.synchronize()
    return out, lse


def _check(x, c, out, lse, bf16, seqlens=None, factors=True):
    k4, kbs, kf, v4, vbs, vf = c
    ro, rl = oracle.decode_nvfp4(x["q"], k4, kbs, v4, vbs, kf.numpy() if factors else None,
                                 vf.numpy() if factors else None, x["scale"], seqlens=seqlens)
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro, bf16=bf16)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_nvfp4_full_128k():
    """The 128K-token GQA workload quantised to NVFP4, as the benchmark runs it."""
    x, c = _quantised("gqa_32x8_d128_s131072")
    out, lse = _run(x, c)
    _check(x, c, out, lse, bf16=True)
    out, lse = _run(x, c, out_dtype=torch.float32)
    _check(x, c, out, lse, bf16=False)


@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("chunk", [0, 128, 256, 1280])
def test_nvfp4_head_groups_and_chunks(G, chunk):
    w = synth.Workload("t", 9, "decode", 2, 2 * G, 2, 3008, 128, "bf16")
    x, c = _quantised_from(w)
    out, lse = _run(x, c, out_dtype=torch.float32, chunk=chunk)
    _check(x, c, out, lse, bf16=False)


def _quantised_from(w, **kw):
    x = synth.make_inputs(w, **kw)
    k4, kbs, kf = synth.to_nvfp4(x["k"])
    v4, vbs, vf = synth.to_nvfp4(x["v"])
    return x, (k4, kbs, kf, v4, vbs, vf)


def test_nvfp4_unit_factors_and_every_code():
    """No factors (1): codes drawn uniformly over all 256 bytes (every E2M1 code in
    both nibbles, signed zeros included), block scales uniform over 2^-3 .. 2^0
    (E4M3 0x20 .. 0x38, subnormal scales not included: they would make scores
    of order 2^-9 too small to test anything)."""
    w = synth.Workload("t", 9, "decode", 1, 8, 2, 2048, 128, "bf16")
    x = synth.make_inputs(w)
    rng = np.random.Generator(np.random.PCG64(91))
    k4 = torch.from_numpy(rng.integers(0, 256, size=(1, 2, 2048, 64)).astype(np.uint8))
    v4 = torch.from_numpy(rng.integers(0, 256, size=(1, 2, 2048, 64)).astype(np.uint8))
    kbs = torch.from_numpy(rng.integers(0x20, 0x39, size=(1, 2, 2048, 8)).astype(np.uint8))
    vbs = torch.from_numpy(rng.integers(0x20, 0x39, size=(1, 2, 2048, 8)).astype(np.uint8))
    c = (k4, kbs, None, v4, vbs, None)
    out, lse = _run(x, c, factors=False, out_dtype=torch.float32)
    _check(x, c, out, lse, bf16=False, factors=False)


def test_nvfp4_varlen_nan_padding():
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w, S=4096, B=5)
    lens = [int(v) for v in x["seqlens"]]
    k4, kbs, kf = synth.to_nvfp4(x["k"])
    v4, vbs, vf = synth.to_nvfp4(x["v"])
    for b, L in enumerate(lens):
        kbs[b, :, L:] = 0x7f  # E4M3 NaN: a key read past the length turns the row into NaN
        vbs[b, :, L:] = 0x7f
    c = (k4, kbs, kf, v4, vbs, vf)
    for split in (0, 8):
        out, lse = _run(x, c, seqlens=lens, n_split=split, out_dtype=torch.float32)
        _check(x, c, out, lse, bf16=False, seqlens=lens)


def test_nvfp4_attends_exactly_the_keys_up_to_each_length():
    """Zero codes make every score 0 and every weight 1: lse = ln(count) and, with V
    = 1.0 (code 2, scale 1.0) in dimension 0 everywhere and in dimension 1 on probe
    keys, out[1] = #probes / count."""
    B, Hq, Hkv, S, D = 3, 8, 2, 20000 // 16 * 16, 128
    lens = [1, 4097, S]
    k4 = torch.zeros(B, Hkv, S, D // 2, dtype=torch.uint8)
    kbs = torch.full((B, Hkv, S, D // 16), 0x38, dtype=torch.uint8)
    v4 = torch.zeros(B, Hkv, S, D // 2, dtype=torch.uint8)
    v4[..., 0] = 0x02  # element 0 = 1.0, element 1 = 0
    vbs = torch.full((B, Hkv, S, D // 16), 0x38, dtype=torch.uint8)
    fracs = []
    for b, L in enumerate(lens):
        j = np.arange(L)
        probe = (j % 128 == 0) | (j % 128 == 127) | (j == L - 1) | (j % 997 == 5)
        v4[b, :, j[probe], 0] = 0x22  # elements 0 and 1 = 1.0
        kbs[b, :, L:] = 0x7f
        vbs[b, :, L:] = 0x7f
        fracs.append(probe.sum() / L)
    q = torch.randn(B, Hq, D).to(torch.bfloat16)
    out, lse = ta.decode_nvfp4(q.to(DEV), k4.to(DEV), v4.to(DEV), kbs.to(DEV), vbs.to(DEV),
                               seqlens=torch.tensor(lens, dtype=torch.int32, device=DEV), scale=0.1,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    out = out.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for b, L in enumerate(lens):
        assert np.all(np.abs(lse[b] - np.log(L)) < 1e-5), (b, lse[b])
        assert np.all(np.abs(out[b, :, 0] - 1.0) < 1e-6)
        assert np.all(np.abs(out[b, :, 1] - fracs[b]) < 0.25 / L)
        assert np.all(out[b, :, 2:] == 0.0)


def test_nvfp4_flags_a_query_outside_fp16():
    """As for the E4M3 cache: a query element of magnitude 2^16 or more (not an
    fp16 value) records TA_DEVERR_RANGE; 65280 does not."""
    w = synth.Workload("t", 9, "decode", 2, 8, 2, 2048, 128, "bf16")
    x, c = _quantised_from(w)
    ta.decode_status()
    for value, flagged in ((65280.0, False), (65536.0, True)):
        q = x["q"].clone()
        q[0, 5, 100] = value
        _run(dict(x, q=q), c)
        st = ta.decode_status()
        assert bool(st & ta.TA_DEVERR_RANGE) == flagged, (value, st)
        assert st & ~ta.TA_DEVERR_RANGE == 0, st


def test_nvfp4_rejects_unsupported_shapes():
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device=DEV)
    k4 = torch.zeros(1, 8, 1000, 64, dtype=torch.uint8, device=DEV)  # S not a multiple of 16
    bs = torch.zeros(1, 8, 1000, 8, dtype=torch.uint8, device=DEV)
    with pytest.raises(ta.TAError) as e:
        ta.decode_nvfp4(q, k4, k4, bs, bs)
    assert e.value.status == ta.TA_ERR_UNSUPPORTED
    k4 = torch.zeros(1, 8, 1024, 64, dtype=torch.uint8, device=DEV)
    bs = torch.zeros(1, 8, 1024, 8, dtype=torch.uint8, device=DEV)
    with pytest.raises(ta.TAError) as e:  # one query head per KV head
        ta.decode_nvfp4(q, k4, k4, bs, bs)
    assert e.value.status == ta.TA_ERR_UNSUPPORTED
    q4 = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ta.TAError) as e:  # chunks that are not whole 128-key tiles
        ta.decode_nvfp4(q4, k4, k4, bs, bs, chunk=200)
    assert e.value.status == ta.TA_ERR_UNSUPPORTED
