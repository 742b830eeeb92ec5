"""Split-KV decode over a paged KV cache (block table) on the GPU, through the
C ABI: against the float64 oracle, and against the contiguous decode of the
same cache (which runs on the tensor-core kernel for the bf16 G = 4 shape, so
the two agree to rounding).  Unreferenced pool rows are NaN, so a wrong page
or row shows."""
import numpy as np
import pytest
import torch

import oracle
from long_context_decode_04_b300 import synth, ta
from tests.parity import check_lse, check_out

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, Hq, Hkv, D, dtype, page, n_pages_per_seq, seed, lens=None):
    S = page * n_pages_per_seq
    w = synth.Workload("paged", 3, "decode", B, Hq, Hkv, S, D, dtype)
    x = synth.make_inputs(w, seed=seed)
    if lens is None:
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = [int(v) for v in rng.integers(1, S, size=B, endpoint=True)]
    kp, vp, bt = synth.to_pages(x["k"], x["v"], lens, page, seed=seed, pad_value=float("nan"))
    return x, lens, kp, vp, bt


def _paged(x, lens, kp, vp, bt, **kw):
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return ta.decode_paged(x["q"].to(DEV), kp.to(DEV), vp.to(DEV), bt.to(DEV), sl, scale=x["scale"], **kw)


@pytest.mark.parametrize("page", [1, 16, 64, 120, 128, 256, 1000])
def test_paged_matches_oracle_and_contiguous(page):
    n_pages = max(2, 3000 // page)
    x, lens, kp, vp, bt = _case(4, 32, 8, 128, "bf16", page, n_pages, seed=500 + page)
    out, lse = _paged(x, lens, kp, vp, bt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rl = oracle.decode_paged(x["q"], kp, vp, bt.numpy(), lens, x["scale"])
    check_out(out.cpu().numpy().reshape(-1, 128), ro, bf16=False)
    check_lse(lse.cpu().numpy().reshape(-1), rl)
    # the contiguous decode of the same cache (padded to the same S) agrees:
    # for this shape it runs on the tensor cores and the paged one on the CUDA
    # cores, so the two agree to rounding, within the oracle tolerances
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    o2, l2 = ta.decode(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), seqlens=sl, scale=x["scale"],
                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_out(out.cpu().numpy().reshape(-1, 128), o2.cpu().numpy().reshape(-1, 128).astype(np.float64), bf16=False)
    check_lse(lse.cpu().numpy().reshape(-1), l2.cpu().numpy().reshape(-1).astype(np.float64))
    assert ta.decode_status() == 0


@pytest.mark.parametrize("split", [0, 1, 7, 100])
def test_paged_forced_splits_bf16_out(split):
    x, lens, kp, vp, bt = _case(3, 8, 2, 128, "bf16", 64, 40, seed=600 + split)
    out, lse = _paged(x, lens, kp, vp, bt, n_split=split)
    torch.cuda.synchronize()
    ro, rl = oracle.decode_paged(x["q"], kp, vp, bt.numpy(), lens, x["scale"])
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro, bf16=True)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


@pytest.mark.parametrize("D,G,dtype", [(64, 1, "f32"), (64, 8, "bf16"), (128, 2, "f32")])
def test_paged_other_head_shapes(D, G, dtype):
    x, lens, kp, vp, bt = _case(2, 2 * G, 2, D, dtype, 32, 30, seed=700 + D + G)
    out, lse = _paged(x, lens, kp, vp, bt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rl = oracle.decode_paged(x["q"], kp, vp, bt.numpy(), lens, x["scale"])
    check_out(out.cpu().numpy().reshape(-1, D), ro, bf16=False)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_paged_empty_and_full_sequences():
    x, lens, kp, vp, bt = _case(3, 8, 2, 128, "bf16", 64, 10, seed=801, lens=[0, 640, 1])
    out, lse = _paged(x, lens, kp, vp, bt, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ro, rl = oracle.decode_paged(x["q"], kp, vp, bt.numpy(), lens, x["scale"])
    check_out(out.cpu().numpy().reshape(-1, 128)[8:], ro[8:], bf16=False)
    check_lse(lse.cpu().numpy().reshape(-1), rl)


def test_bad_page_ids_are_flagged_not_followed():
    x, lens, kp, vp, bt = _case(2, 8, 2, 128, "bf16", 64, 8, seed=802, lens=[300, 500])
    bt = bt.clone()
    bt[1, 2] = kp.shape[0] + 1000  # past the pool
    bt[0, 0] = -5
    ws = ta.decode_workspace(2, 8, 2, 64 * 8, 128, varlen=True)
    _paged(x, lens, kp, vp, bt, workspace=ws)
    assert ta.decode_status(ws) & ta.TA_DEVERR_PAGE
    _paged(x, lens, kp, vp, bt * 0 + torch.arange(8, dtype=torch.int32), workspace=ws)  # valid ids again
    assert ta.decode_status(ws) == 0


def test_full_varlen_b16_paged_64():
    """The 16-sequence variable-length workload (lengths 1K-32K, peaked keys),
    held in 64-key pages."""
    w = synth.WORKLOADS["varlen_b16_32x8_d128_s1k_32k"]
    x = synth.make_inputs(w)
    lens = [int(v) for v in x["seqlens"]]
    kp, vp, bt = synth.to_pages(x["k"], x["v"], lens, 64, seed=11, pad_value=float("nan"))
    out, lse = _paged(x, lens, kp, vp, bt)
    torch.cuda.synchronize()
    ro, rl = oracle.decode_paged(x["q"], kp, vp, bt.numpy(), lens, x["scale"])
    check_out(out.float().cpu().numpy().reshape(-1, 128), ro, bf16=True)
    check_lse(lse.cpu().numpy().reshape(-1), rl)
