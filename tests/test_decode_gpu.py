"""Split-KV decode on the GPU against the float64 oracle (through the C ABI).

Small shapes span several tiles, chunks and a ragged tail; the full-size
workloads run in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(x, out_dtype=None, **kw):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    sl = None if x["seqlens"] is None else x["seqlens"].to(DEV)
    out, lse = ta.decode(q, k, v, seqlens=sl, scale=x["scale"], out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle(x, rows=None):
    sl = None if x["seqlens"] is None else x["seqlens"].numpy()
    return oracle.decode(x["q"], x["k"], x["v"], x["scale"], seqlens=sl, rows=rows)


def _compare(x, out, lse, bf16, rows=None):
    ro, rl = _oracle(x, rows)
    D = x["q"].shape[-1]
    o = out.reshape(-1, D)
    l = lse.reshape(-1)
    if rows is not None:
        o, l = o[rows], l[rows]
    return check_out(o, ro, bf16), check_lse(l, rl)


# ------------------------------------------------------------ small shapes

@pytest.mark.parametrize("name", ["single_head_d64_s4096_f32", "gqa_32x8_d128_s131072",
                                  "varlen_b16_32x8_d128_s1k_32k"])
@pytest.mark.parametrize("S", [1, 7, 255, 256, 257, 1000, 3001])
def test_small_shapes_f32_out(name, S):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, S=S, B=min(w.B, 3), pad_value=float("nan"))
    out, lse = _run(x, out_dtype=torch.float32)
    _compare(x, out, lse, bf16=False)


@pytest.mark.parametrize("n_split", [1, 2, 3, 7, 64, 65, 128, 129, 200])
def test_forced_splits_and_levels(n_split):
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    x = synth.make_inputs(w, S=4099)
    out, lse = _run(x, out_dtype=torch.float32, n_split=n_split)
    _compare(x, out, lse, bf16=False)
    out_b, lse_b = _run(x, n_split=n_split)
    _compare(x, out_b, lse_b, bf16=True)


@pytest.mark.parametrize("chunk", [1, 16, 100, 127, 128, 129, 255, 256, 257])
def test_chunk_boundaries(chunk):
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    x = synth.make_inputs(w, S=777)
    out, lse = _run(x, out_dtype=torch.float32, chunk=chunk)
    _compare(x, out, lse, bf16=False)


@pytest.mark.parametrize("D,G,dtype", [(64, 1, "bf16"), (64, 2, "bf16"), (64, 4, "bf16"), (64, 8, "bf16"),
                                       (128, 1, "bf16"), (128, 2, "bf16"), (128, 4, "bf16"),
                                       (64, 1, "f32"), (64, 8, "f32"), (128, 4, "f32"), (128, 1, "f32")])
def test_every_supported_head_shape(D, G, dtype):
    w = synth.Workload("t", 9, "decode", 2, 2 * G, 2, 1500, D, dtype)
    x = synth.make_inputs(w)
    out, lse = _run(x, out_dtype=torch.float32, n_split=3)
    _compare(x, out, lse, bf16=False)
    if dtype == "bf16":
        out, lse = _run(x)
        _compare(x, out, lse, bf16=True)


def test_plain_entry_point_matches_ex():
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    x = synth.make_inputs(w, S=5000)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out = torch.empty(1, 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 32, dtype=torch.float32, device=DEV)
    ta.decode_bf16(q, k, v, out, lse, x["scale"])
    o2, l2 = ta.decode(q, k, v, scale=x["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_results_are_deterministic():
    """The dynamic work queue changes which CTA runs an item, never the arithmetic."""
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w, S=8192, B=6)
    a = _run(x)
    b = _run(x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ------------------------------------------------------------ exact attended set

@pytest.mark.parametrize("chunk", [0, 256])
def test_zero_keys_count_attended_keys_exactly(chunk):
    """K = 0 makes every score 0, so lse = ln(count): off-by-one in masking or chunk
    bounds moves lse by >= 1/count, far above the 1e-5 check (count <= 16384)."""
    B, Hq, Hkv, S, D = 5, 8, 2, 16384, 128
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16)
    lens = torch.tensor([1, 255, 256, 257, 16384], dtype=torch.int32)
    for b in range(B):
        k[b, :, lens[b]:] = float("nan")
        v[b, :, lens[b]:] = float("nan")
    out, lse = ta.decode(q.to(DEV), k.to(DEV), v.to(DEV), seqlens=lens.to(DEV), scale=0.1,
                         out_dtype=torch.float32, chunk=chunk)
    lse = lse.cpu().numpy()
    for b in range(B):
        assert np.all(np.abs(lse[b] - np.log(int(lens[b]))) < 1e-5), (b, lse[b])
        assert torch.isfinite(out[b]).all()


def test_probe_columns_at_large_counts():
    """Large counts.  With K = 0 every weight is exactly 1 in the kernel's exp2, so the
    sums are exact integers in fp32 and lse = ln(L) to a few ulp: a count off by one
    moves lse by 1/L = 7.6e-6 at L = 131072, above the 3e-6 check.  Probes pin which
    keys are attended: V[:,1] = 1 only on key 0, key L-1 and the first and last key
    of every chunk, so out[1] = #probes / L, and a missed probe moves it by 1/L."""
    B, Hq, Hkv, S, D = 2, 4, 1, 131072, 128
    lens = [131072, 100003]
    plan = ta.plan_decode(B, Hq, Hkv, S, D, varlen=True)
    k = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16)
    v[:, :, :, 0] = 1.0
    expect = []
    for b, L in enumerate(lens):
        probes = {0, L - 1}
        for c0, c1 in ta.chunk_bounds(plan, S):
            for j in (c0, c1 - 1):
                if 0 <= j < L:
                    probes.add(j)
        for j in probes:
            v[b, :, j, 1] = 1.0
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("nan")
        expect.append(len(probes) / L)
    q = torch.randn(B, Hq, D).to(torch.bfloat16)
    out, lse = ta.decode(q.to(DEV), k.to(DEV), v.to(DEV), seqlens=torch.tensor(lens, dtype=torch.int32).to(DEV),
                         scale=0.1, out_dtype=torch.float32)
    out = out.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for b, L in enumerate(lens):
        assert np.all(np.abs(lse[b] - np.log(L)) < 3e-6), (lse[b], np.log(L))
        assert np.all(np.abs(out[b, :, 0] - 1.0) < 1e-5)
        assert np.all(np.abs(out[b, :, 1] - expect[b]) < 0.25 / L), (out[b, :, 1], expect[b])


def test_empty_sequences_and_status_word():
    B, Hq, Hkv, S, D = 3, 4, 2, 600, 64
    g = torch.Generator().manual_seed(9)
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16).to(DEV)
    k = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn(B, Hkv, S, D, generator=g).to(torch.bfloat16).to(DEV)
    ws = ta.decode_workspace(B, Hq, Hkv, S, D, varlen=True)
    out, lse = ta.decode(q, k, v, seqlens=torch.tensor([0, 600, 5], dtype=torch.int32, device=DEV),
                         out_dtype=torch.float32, workspace=ws)
    assert ta.decode_status(ws) == 0
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.isfinite(lse[1:]).all()
    # a length past S is clamped and flagged, never read past the cache
    out, lse = ta.decode(q, k, v, seqlens=torch.tensor([601, -3, 600], dtype=torch.int32, device=DEV),
                         out_dtype=torch.float32, workspace=ws)
    assert ta.decode_status(ws) & ta.TA_DEVERR_SEQLEN
    o2, l2 = ta.decode(q, k, v, seqlens=torch.tensor([600, 0, 600], dtype=torch.int32, device=DEV),
                       out_dtype=torch.float32, workspace=ws)
    assert torch.equal(out, o2) and torch.equal(torch.nan_to_num(lse), torch.nan_to_num(l2))
    assert ta.decode_status(ws) == 0


def test_workspace_too_small_is_rejected():
    B, Hq, Hkv, S, D = 1, 8, 2, 50000, 128
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(B, Hkv, S, D, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(ta.TAError) as e:
        ta.decode(q, k, k, workspace=ws)
    assert e.value.status == ta.TA_ERR_WORKSPACE


def test_outputs_do_not_write_past_their_end():
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    x = synth.make_inputs(w, S=2000)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out_buf = torch.full((32 * 128 + 256,), 7.0, dtype=torch.float32, device=DEV)
    lse_buf = torch.full((32 + 64,), 7.0, dtype=torch.float32, device=DEV)
    out = out_buf[:32 * 128].view(1, 32, 128)
    lse = lse_buf[:32].view(1, 32)
    ta.decode(q, k, v, scale=x["scale"], out=out, lse=lse, n_split=9)
    torch.cuda.synchronize()
    assert torch.all(out_buf[32 * 128:] == 7.0) and torch.all(lse_buf[32:] == 7.0)


# ------------------------------------------------------------ full-size workloads

def test_full_single_head_d64_s4096_f32():
    w = synth.WORKLOADS["single_head_d64_s4096_f32"]
    x = synth.make_inputs(w)
    out, lse = _run(x)
    _compare(x, out, lse, bf16=False)


def test_full_gqa_s131072_all_rows():
    w = synth.WORKLOADS["gqa_32x8_d128_s131072"]
    x = synth.make_inputs(w)
    out, lse = _run(x)
    _compare(x, out, lse, bf16=True)
    out, lse = _run(x, out_dtype=torch.float32)
    _compare(x, out, lse, bf16=False)


def test_full_varlen_b16_nan_padding():
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w, pad_value=float("nan"))
    out, lse = _run(x)
    _compare(x, out, lse, bf16=True)


@pytest.mark.slow
def test_full_extreme_s1048576_chunk256():
    w = synth.WORKLOADS["gqa_32x8_d128_s1048576_c256"]
    x = synth.make_inputs(w)
    plan = ta.plan_decode(1, 32, 8, w.S, 128, chunk=w.chunk)
    assert plan.n_split == 4096 and plan.levels == 2
    out, lse = _run(x, chunk=w.chunk)
    _compare(x, out, lse, bf16=True)
